// stack.cu -- per-token parts of a hybrid attention / Gated DeltaNet stack.
//
// Flide, "Accelerating Decision Inference with Exact State Forking",
// section 3.2: pointwise operations (projections, norms, the MLP) act on
// every token alone and ignore the tree; the rotary embedding of a branch
// token uses the position it has in its standalone sequence (positions
// continue from the parent); section 3.2.2: a short causal convolution in
// front of the delta rule reads a token's predecessors through an index, so
// a question's first tokens see the last tokens of its state (and a resumed
// state's first tokens see the saved convolution window, section 3.4).
//
// Every kernel here handles each row independently and reduces in a fixed
// order, so a row's bits do not depend on the rest of the round.
#include <cuda_bf16.h>

#include <cmath>
#include <vector>

#include "device.cuh"

using namespace hsm;
using hsd::Meta;

namespace {

__device__ __forceinline__ float silu(float x) { return x / (1.f + expf(-x)); }
__device__ __forceinline__ float softplus(float x) { return x > 20.f ? x : log1pf(expf(x)); }

// eight consecutive elements as floats, and back (16-byte aligned; bf16 stores round to nearest even)
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&f)[8]) {
  hsd::cvt16(*reinterpret_cast<const float4*>(p), f, __nv_bfloat16());
}
__device__ __forceinline__ void load8(const float* p, float (&f)[8]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0], b = reinterpret_cast<const float4*>(p)[1];
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&f)[8]) {
  __nv_bfloat162 o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) o[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  *reinterpret_cast<float4*>(p) = *reinterpret_cast<float4*>(o);
}
__device__ __forceinline__ void store8(float* p, const float (&f)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(f[0], f[1], f[2], f[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(f[4], f[5], f[6], f[7]);
}

// ---------------------------------------------------------------- embedding
template <typename O>
__global__ void embed_kernel(const int32_t* __restrict__ ids, int T, const __nv_bfloat16* __restrict__ table,
                             int vocab, int dim, O* __restrict__ out, int32_t* status) {
  const int t = blockIdx.x;
  if (t >= T) return;
  const int id = ids[t];
  const bool ok = id >= 0 && id < vocab;
  if (!ok && threadIdx.x == 0) hsd::set_status(status, HS_DEV_BAD_META);
  for (int c = threadIdx.x * 8; c < dim; c += blockDim.x * 8) {
    float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (ok) load8(table + (size_t)id * dim + c, f);
    store8(out + (size_t)t * dim + c, f);
  }
}

// ------------------------------------------------------------------ RMSNorm
// one warp per row: lane-strided fp32 sums of squares, then a fixed butterfly
template <typename X, typename O>
__global__ void rmsnorm_kernel(const X* __restrict__ x, long long ldx, int T, int dim,
                               const __nv_bfloat16* __restrict__ w, float eps, O* __restrict__ out, long long ldo) {
  const int row = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= T) return;
  const X* xr = x + (size_t)row * ldx;
  float ss = 0.f;
  for (int c = lane * 8; c < dim; c += 256) {
    float f[8];
    load8(xr + c, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
  }
  ss = hsd::warp_sum(ss);
  const float inv = 1.f / sqrtf(ss / (float)dim + eps);
  O* orow = out + (size_t)row * ldo;
  for (int c = lane * 8; c < dim; c += 256) {
    float f[8], g[8];
    load8(xr + c, f);
    if (w) {
      load8(w + c, g);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) g[i] = 1.f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = f[i] * inv * g[i];
    store8(orow + c, f);
  }
}

// --------------------------------------------------------------------- RoPE
// rotate-half on n_heads heads of width d starting at column col0, at the
// token's standalone position (node pos0 + index in node)
__global__ void rope_kernel(const int32_t* __restrict__ meta, __nv_bfloat16* __restrict__ x, long long ldx,
                            int col0, int n_heads, int d, const float2* __restrict__ table, int max_pos,
                            int32_t* status) {
  Meta M{meta};
  const int t = blockIdx.x;
  if (t >= M.h(H_N_TOK)) return;
  const int32_t* tk = M.tok(t);
  const int pos = M.seg(tk[T_SEG])[S_POS0] + tk[T_IDX];
  if (pos < 0 || pos >= max_pos) {
    if (threadIdx.x == 0) hsd::set_status(status, HS_DEV_BAD_META);
    return;
  }
  const int half = d / 2;
  __nv_bfloat16* xr = x + (size_t)t * ldx + col0;
  for (int e = threadIdx.x; e < n_heads * half; e += blockDim.x) {
    const int h = e / half, i = e % half;
    const float2 cs = table[(size_t)pos * half + i];
    __nv_bfloat16* p = xr + h * d;
    const float a = __bfloat162float(p[i]), b = __bfloat162float(p[i + half]);
    p[i] = __float2bfloat16_rn(a * cs.x - b * cs.y);
    p[i + half] = __float2bfloat16_rn(a * cs.y + b * cs.x);
  }
}

// ------------------------------------------------------------ GDN front end
// One block per token: causal conv (kConvTaps taps, predecessors by index),
// SiLU, L2 norm of each q and k head, and the gates
//   alpha = exp(-0.1 softplus(a)),  beta = sigmoid(b).
constexpr int kPrepThreads = 256;
__global__ void __launch_bounds__(kPrepThreads)
gdn_prep_kernel(const int32_t* __restrict__ meta, const __nv_bfloat16* __restrict__ proj, long long ldp,
                const __nv_bfloat16* __restrict__ win, long long ldw, int n_win,
                const __nv_bfloat16* __restrict__ cw, int H, int d, __nv_bfloat16* __restrict__ qo,
                __nv_bfloat16* __restrict__ ko, __nv_bfloat16* __restrict__ vo, float* __restrict__ alpha,
                float* __restrict__ beta, int32_t* status) {
  extern __shared__ float ys[];  // [3 * H * d]
  Meta M{meta};
  const int t = blockIdx.x;
  if (t >= M.h(H_N_TOK)) return;
  const int C = 3 * H * d;
  const int32_t* pred = M.m + M.h(H_OFF_PRED) + t * kPredWords;
  const __nv_bfloat16* src[kConvTaps];
  src[0] = proj + (size_t)t * ldp;
  bool bad = false;
  for (int k = 1; k < kConvTaps; ++k) {
    const int pr = pred[k - 1];
    if (pr >= 0) {
      src[k] = proj + (size_t)pr * ldp;
    } else if (pr == -1) {
      src[k] = nullptr;
    } else {
      const int wr = -2 - pr;
      if (win && wr < n_win) {
        src[k] = win + (size_t)wr * ldw;
      } else {
        src[k] = nullptr;
        bad = true;
      }
    }
  }
  if (bad && threadIdx.x == 0) hsd::set_status(status, HS_DEV_BAD_META);
  for (int ch = threadIdx.x; ch < C; ch += blockDim.x) {
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < kConvTaps; ++k)
      if (src[k]) acc = fmaf(__bfloat162float(cw[(size_t)ch * kConvTaps + k]), __bfloat162float(src[k][ch]), acc);
    ys[ch] = silu(acc);
  }
  __syncthreads();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // 2H normalised vectors (q heads then k heads), then H plain v heads
  for (int vec = warp; vec < 3 * H; vec += kPrepThreads / 32) {
    const float* y = ys + vec * d;
    float inv = 1.f;
    if (vec < 2 * H) {
      float ss = 0.f;
      for (int i = lane; i < d; i += 32) ss = fmaf(y[i], y[i], ss);
      ss = hsd::warp_sum(ss);
      inv = 1.f / sqrtf(ss + 1e-6f);
    }
    __nv_bfloat16* dst = vec < H ? qo + ((size_t)t * H + vec) * d
                                 : vec < 2 * H ? ko + ((size_t)t * H + vec - H) * d : vo + ((size_t)t * H + vec - 2 * H) * d;
    for (int i = lane; i < d; i += 32) dst[i] = __float2bfloat16_rn(y[i] * inv);
  }
  if (threadIdx.x < H) {
    const float a = __bfloat162float(proj[(size_t)t * ldp + C + threadIdx.x]);
    const float b = __bfloat162float(proj[(size_t)t * ldp + C + H + threadIdx.x]);
    alpha[(size_t)t * H + threadIdx.x] = expf(-0.1f * softplus(a));
    beta[(size_t)t * H + threadIdx.x] = 1.f / (1.f + expf(-b));
  }
}

// -------------------------------------------------------------------- SwiGLU
__global__ void swiglu_kernel(const __nv_bfloat16* __restrict__ gu, long long ldg, int T, int F,
                              __nv_bfloat16* __restrict__ out, long long ldo) {
  const int t = blockIdx.x;
  if (t >= T) return;
  for (int i = threadIdx.x * 8; i < F; i += blockDim.x * 8) {
    float g[8], u[8];
    hsd::cvt16(*reinterpret_cast<const float4*>(gu + (size_t)t * ldg + i), g, __nv_bfloat16());
    hsd::cvt16(*reinterpret_cast<const float4*>(gu + (size_t)t * ldg + F + i), u, __nv_bfloat16());
    __nv_bfloat162 o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) o[j] = __floats2bfloat162_rn(silu(g[2 * j]) * u[2 * j], silu(g[2 * j + 1]) * u[2 * j + 1]);
    *reinterpret_cast<float4*>(out + (size_t)t * ldo + i) = *reinterpret_cast<float4*>(o);
  }
}

// ----------------------------------------------------------------- row copy
__global__ void copy_rows_kernel(const uint8_t* __restrict__ src, long long lds, const int32_t* src_rows,
                                 uint8_t* __restrict__ dst, long long ldd, const int32_t* dst_rows, int width16) {
  const int r = blockIdx.x;
  const float4* s = reinterpret_cast<const float4*>(src + (size_t)src_rows[r] * lds);
  float4* d = reinterpret_cast<float4*>(dst + (size_t)dst_rows[r] * ldd);
  for (int i = threadIdx.x; i < width16; i += blockDim.x) d[i] = s[i];
}

bool al16(const void* p) { return ((uintptr_t)p & 15) == 0; }

hs_status need_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return hs::fail(HS_ECUDA, "no CUDA device");
  return HS_OK;
}

}  // namespace

extern "C" hs_status hs_embed(const int32_t* ids, int32_t T, const void* table, int32_t vocab, int32_t dim,
                              void* out, hs_dtype out_dtype, int32_t* dev_status, void* stream) {
  HS_CHECK_ARG(ids && table && out, "null argument");
  HS_CHECK_ARG(T >= 0 && vocab > 0 && dim > 0 && dim % 8 == 0, "bad shape");
  HS_CHECK_ARG(al16(table) && al16(out), "16-byte alignment required");
  if (out_dtype != HS_BF16 && out_dtype != HS_F32) return hs::fail(HS_EUNSUPPORTED, "embed: output dtype %d", out_dtype);
  if (hs_status s = need_device()) return s;
  if (T == 0) return HS_OK;
  const cudaStream_t st = (cudaStream_t)stream;
  if (out_dtype == HS_F32)
    embed_kernel<<<T, 128, 0, st>>>(ids, T, (const __nv_bfloat16*)table, vocab, dim, (float*)out, dev_status);
  else
    embed_kernel<<<T, 128, 0, st>>>(ids, T, (const __nv_bfloat16*)table, vocab, dim, (__nv_bfloat16*)out, dev_status);
  HS_LAUNCH_CHECK("embed");
  return HS_OK;
}

extern "C" hs_status hs_rmsnorm(const void* x, int64_t ldx, hs_dtype x_dtype, int32_t T, int32_t dim, const void* w,
                                float eps, void* out, int64_t ldo, hs_dtype out_dtype, void* stream) {
  HS_CHECK_ARG(x && out, "null argument");
  HS_CHECK_ARG(T >= 0 && dim > 0 && dim % 8 == 0 && ldx >= dim && ldo >= dim && ldx % 8 == 0 && ldo % 8 == 0,
               "bad shape");
  HS_CHECK_ARG(al16(x) && al16(out) && al16(w), "16-byte alignment required");
  if ((x_dtype != HS_BF16 && x_dtype != HS_F32) || (out_dtype != HS_BF16 && out_dtype != HS_F32))
    return hs::fail(HS_EUNSUPPORTED, "rmsnorm: dtypes %d -> %d", x_dtype, out_dtype);
  if (hs_status s = need_device()) return s;
  if (T == 0) return HS_OK;
  const dim3 grid((T + 7) / 8), block(256);
  const cudaStream_t st = (cudaStream_t)stream;
  const __nv_bfloat16* wb = (const __nv_bfloat16*)w;
  if (x_dtype == HS_F32 && out_dtype == HS_F32)
    rmsnorm_kernel<<<grid, block, 0, st>>>((const float*)x, ldx, T, dim, wb, eps, (float*)out, ldo);
  else if (x_dtype == HS_F32)
    rmsnorm_kernel<<<grid, block, 0, st>>>((const float*)x, ldx, T, dim, wb, eps, (__nv_bfloat16*)out, ldo);
  else if (out_dtype == HS_F32)
    rmsnorm_kernel<<<grid, block, 0, st>>>((const __nv_bfloat16*)x, ldx, T, dim, wb, eps, (float*)out, ldo);
  else
    rmsnorm_kernel<<<grid, block, 0, st>>>((const __nv_bfloat16*)x, ldx, T, dim, wb, eps, (__nv_bfloat16*)out, ldo);
  HS_LAUNCH_CHECK("rmsnorm");
  return HS_OK;
}

extern "C" hs_status hs_rope_table(float* host_table, int32_t max_pos, int32_t d, double theta) {
  HS_CHECK_ARG(host_table && max_pos > 0 && d > 0 && d % 2 == 0 && theta > 1.0, "bad argument");
  const int half = d / 2;
  for (int p = 0; p < max_pos; ++p)
    for (int i = 0; i < half; ++i) {
      const double ang = (double)p * std::pow(theta, -2.0 * i / d);
      host_table[((size_t)p * half + i) * 2] = (float)std::cos(ang);
      host_table[((size_t)p * half + i) * 2 + 1] = (float)std::sin(ang);
    }
  return HS_OK;
}

extern "C" hs_status hs_rope_apply(const hs_round_caps* caps, const void* dev_meta, void* x, int64_t ldx,
                                   int32_t col0, int32_t n_heads, int32_t d, const float* table, int32_t max_pos,
                                   int32_t* dev_status, void* stream) {
  HS_CHECK_ARG(caps && dev_meta && x && table, "null argument");
  HS_CHECK_ARG(n_heads > 0 && d > 0 && d % 2 == 0 && col0 >= 0 && ldx >= col0 + (int64_t)n_heads * d, "bad shape");
  HS_CHECK_ARG(max_pos > 0 && ((uintptr_t)table & 7) == 0, "the cos/sin table must be 8-byte aligned");
  if (hs_status s = need_device()) return s;
  if (caps->max_tokens <= 0) return HS_OK;
  rope_kernel<<<caps->max_tokens, 128, 0, (cudaStream_t)stream>>>((const int32_t*)dev_meta, (__nv_bfloat16*)x, ldx,
                                                                  col0, n_heads, d, (const float2*)table, max_pos,
                                                                  dev_status);
  HS_LAUNCH_CHECK("rope");
  return HS_OK;
}

extern "C" hs_status hs_gdn_prep(const hs_round_caps* caps, const void* dev_meta, const void* proj, int64_t ldp,
                                 const void* window, int64_t ldw, int32_t n_window_rows, const void* conv_w, int32_t h,
                                 int32_t d, void* q, void* k, void* v, float* alpha, float* beta, int32_t* dev_status,
                                 void* stream) {
  HS_CHECK_ARG(caps && dev_meta && proj && conv_w && q && k && v && alpha && beta, "null argument");
  HS_CHECK_ARG(h > 0 && d > 0 && ldp >= 3 * (int64_t)h * d + 2 * h, "bad shape");
  HS_CHECK_ARG(!window || ldw >= 3 * (int64_t)h * d, "bad window stride");
  if (hs_status s = need_device()) return s;
  if (caps->max_tokens <= 0) return HS_OK;
  const size_t smem = sizeof(float) * 3 * (size_t)h * d;
  static std::atomic<bool> configured[hsd::kMaxDevices];  // zero-initialised: per device
  const int slot = hsd::device_slot();
  if (slot < 0) return hs::fail(HS_ECUDA, "gdn_prep: no usable CUDA device");
  if (!configured[slot].load()) {
    if (cudaFuncSetAttribute(gdn_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) != cudaSuccess)
      return hs::fail(HS_ECUDA, "gdn_prep: cannot raise the shared-memory limit");
    configured[slot].store(true);
  }
  HS_CHECK_ARG(smem <= 200 * 1024, "3*h*d too large");
  gdn_prep_kernel<<<caps->max_tokens, kPrepThreads, smem, (cudaStream_t)stream>>>(
      (const int32_t*)dev_meta, (const __nv_bfloat16*)proj, ldp, (const __nv_bfloat16*)window, ldw, n_window_rows,
      (const __nv_bfloat16*)conv_w, h, d, (__nv_bfloat16*)q, (__nv_bfloat16*)k, (__nv_bfloat16*)v, alpha, beta,
      dev_status);
  HS_LAUNCH_CHECK("gdn_prep");
  return HS_OK;
}

extern "C" hs_status hs_swiglu(const void* gu, int64_t ldg, int32_t T, int32_t F, void* out, int64_t ldo,
                               void* stream) {
  HS_CHECK_ARG(gu && out, "null argument");
  HS_CHECK_ARG(T >= 0 && F > 0 && F % 8 == 0 && ldg >= 2 * (int64_t)F && ldo >= F && ldg % 8 == 0 && ldo % 8 == 0,
               "bad shape");
  HS_CHECK_ARG(al16(gu) && al16(out), "16-byte alignment required");
  if (hs_status s = need_device()) return s;
  if (T == 0) return HS_OK;
  swiglu_kernel<<<T, 256, 0, (cudaStream_t)stream>>>((const __nv_bfloat16*)gu, ldg, T, F, (__nv_bfloat16*)out, ldo);
  HS_LAUNCH_CHECK("swiglu");
  return HS_OK;
}

extern "C" hs_status hs_copy_rows(const void* src, int64_t lds, const int32_t* src_rows, void* dst, int64_t ldd,
                                  const int32_t* dst_rows, int32_t n, int32_t width_bytes, void* stream) {
  HS_CHECK_ARG(src && dst && (n == 0 || (src_rows && dst_rows)), "null argument");
  HS_CHECK_ARG(n >= 0 && width_bytes > 0 && width_bytes % 16 == 0 && lds % 16 == 0 && ldd % 16 == 0, "bad shape");
  HS_CHECK_ARG(al16(src) && al16(dst), "16-byte alignment required");
  if (hs_status s = need_device()) return s;
  if (n == 0) return HS_OK;
  copy_rows_kernel<<<n, 128, 0, (cudaStream_t)stream>>>((const uint8_t*)src, lds, src_rows, (uint8_t*)dst, ldd,
                                                        dst_rows, width_bytes / 16);
  HS_LAUNCH_CHECK("copy_rows");
  return HS_OK;
}
