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

// eight consecutive elements as floats (16-byte aligned source)
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&h)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[2 * i] = __uint_as_float(w[i] << 16);
    h[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void load8(const float* p, float (&h)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  h[0] = a.x; h[1] = a.y; h[2] = a.z; h[3] = a.w; h[4] = b.x; h[5] = b.y; h[6] = b.z; h[7] = b.w;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
choice_kernel(const int32_t* __restrict__ meta, const T* __restrict__ hidden, long long stride, int dim,
              const float* __restrict__ W, int n_opt, float* __restrict__ logprobs, int32_t* status) {
  hsd::pdl_wait();  // (launched with launch_pdl: nothing global before this)
  hsd::pdl_trigger();
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
  // eight elements at a time in 16-byte loads when the row and the option rows allow it, four options per
  // pass over the row (the loads of a pass are independent, so they are in flight together)
  const bool vec = dim % 8 == 0 && ((uintptr_t)hr & 15) == 0 && ((uintptr_t)W & 15) == 0;
  for (int o0 = 0; o0 < n_opt; o0 += 4) {
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (vec) {
      for (int e8 = threadIdx.x; e8 < dim / 8; e8 += kThreads) {
        float h[8];
        load8(hr + (size_t)e8 * 8, h);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          if (o0 + k < n_opt) {
            const float4* w4 = reinterpret_cast<const float4*>(W + (size_t)(o0 + k) * dim + (size_t)e8 * 8);
            const float4 a = w4[0], b = w4[1];
            float s = acc[k];
            s = fmaf(h[0], a.x, s); s = fmaf(h[1], a.y, s); s = fmaf(h[2], a.z, s); s = fmaf(h[3], a.w, s);
            s = fmaf(h[4], b.x, s); s = fmaf(h[5], b.y, s); s = fmaf(h[6], b.z, s); s = fmaf(h[7], b.w, s);
            acc[k] = s;
          }
        }
      }
    } else {
      for (int e = threadIdx.x; e < dim; e += kThreads) {
        const float he = hsd::to_f(hr[e]);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (o0 + k < n_opt) acc[k] = fmaf(he, W[(size_t)(o0 + k) * dim + e], acc[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float v = hsd::warp_sum(acc[k]);
      if (lane == 0 && o0 + k < n_opt) part[warp][o0 + k] = v;
    }
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
    hsd::launch_pdl(choice_kernel<__nv_bfloat16>, dim3(caps->max_readouts), dim3(kThreads), 0, st,
                    (const int32_t*)dev_meta, (const __nv_bfloat16*)hidden, (long long)hidden_stride, (int)hidden_dim,
                    option_rows, (int)n_opt, logprobs, dev_status);
  else
    hsd::launch_pdl(choice_kernel<float>, dim3(caps->max_readouts), dim3(kThreads), 0, st, (const int32_t*)dev_meta,
                    (const float*)hidden, (long long)hidden_stride, (int)hidden_dim, option_rows, (int)n_opt, logprobs,
                    dev_status);
  HS_LAUNCH_CHECK("choice_logprobs");
  return HS_OK;
}
