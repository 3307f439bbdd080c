// choice.cu -- option log-probabilities at the readout rows.
//
// Flide, section 3.1, Eq. 1: p_i(o) = exp(w_o^T h_i) / sum_o' exp(w_o'^T h_i)
// with h_i the hidden state at the last token of question i; section 3.3.3:
// only the readout rows, listed in a fixed-size index buffer, are read.
//
// One thread block per readout row.  Every dot product is summed in the same
// order whatever the round holds: thread i accumulates elements i, i+256, ...
// in fp32, then a fixed shuffle tree and a fixed cross-warp order.
#include <cuda_bf16.h>

#include "device.cuh"

using namespace hsm;
using hsd::Meta;

namespace {

constexpr int kThreads = 256;
constexpr int kMaxOpt = 32;

template <typename T>
__global__ void __launch_bounds__(kThreads)
choice_kernel(const int32_t* __restrict__ meta, const T* __restrict__ hidden, long long stride, int dim,
              const float* __restrict__ W, int n_opt, float* __restrict__ logprobs, int32_t* status) {
  __shared__ float part[kThreads / 32][kMaxOpt];
  __shared__ float z[kMaxOpt];
  Meta M{meta};
  const int i = blockIdx.x;
  if (i >= M.h(H_N_READOUT)) return;
  const int row = M.readout()[i];
  if (row < 0 || row >= M.h(H_N_TOK)) {
    hsd::set_status(status, HS_DEV_BAD_META);
    return;
  }
  const T* hr = hidden + (size_t)row * stride;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int o = 0; o < n_opt; ++o) {
    float acc = 0.f;
    for (int e = threadIdx.x; e < dim; e += kThreads) acc = fmaf(hsd::to_f(hr[e]), W[(size_t)o * dim + e], acc);
    acc = hsd::warp_sum(acc);
    if (lane == 0) part[warp][o] = acc;
  }
  __syncthreads();
  if (threadIdx.x < n_opt) {
    float s = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) s += part[w][threadIdx.x];
    z[threadIdx.x] = s;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = -INFINITY;
    for (int o = 0; o < n_opt; ++o) m = fmaxf(m, z[o]);
    float l = 0.f;
    for (int o = 0; o < n_opt; ++o) l += expf(z[o] - m);
    const float lse = m + logf(l);
    for (int o = 0; o < n_opt; ++o) logprobs[(size_t)i * n_opt + o] = z[o] - lse;
  }
}

}  // namespace

extern "C" hs_status hs_choice_logprobs(const hs_round_caps* caps, const void* dev_meta, hs_dtype dt,
                                        const void* hidden, int64_t hidden_stride, int32_t hidden_dim,
                                        const float* option_rows, int32_t n_opt, float* logprobs,
                                        int32_t* dev_status, void* stream) {
  HS_CHECK_ARG(caps && dev_meta && hidden && option_rows && logprobs, "null argument");
  HS_CHECK_ARG(hidden_dim > 0 && hidden_stride >= hidden_dim, "bad hidden shape");
  HS_CHECK_ARG(n_opt >= 1 && n_opt <= kMaxOpt, "n_opt must be in [1, %d]", kMaxOpt);
  if (dt != HS_F32 && dt != HS_BF16) return hs::fail(HS_EUNSUPPORTED, "dtype %d", (int)dt);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return hs::fail(HS_ECUDA, "no CUDA device");
  if (caps->max_readouts <= 0) return HS_OK;
  cudaStream_t st = (cudaStream_t)stream;
  if (dt == HS_BF16)
    choice_kernel<__nv_bfloat16><<<caps->max_readouts, kThreads, 0, st>>>(
        (const int32_t*)dev_meta, (const __nv_bfloat16*)hidden, hidden_stride, hidden_dim, option_rows, n_opt,
        logprobs, dev_status);
  else
    choice_kernel<float><<<caps->max_readouts, kThreads, 0, st>>>((const int32_t*)dev_meta, (const float*)hidden,
                                                                  hidden_stride, hidden_dim, option_rows, n_opt,
                                                                  logprobs, dev_status);
  HS_LAUNCH_CHECK("choice_logprobs");
  return HS_OK;
}
