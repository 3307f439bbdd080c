// gdn.cu -- Gated DeltaNet fork prefill in chunks, and state checkpoints.
//
// Flide, "Accelerating Decision Inference with Exact State Forking":
//   section 3.2.2, Eq. 4 -- S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T)
//     + beta_t v_t k_t^T, o_t = S_t q_t; state segments run first, then each
//     question continues from its request's end-of-state S_P through an
//     index, without copying;
//   section 3.3.1 -- a fixed-length chunk list built per round;
//   section 3.4 -- the state at a checkpoint is the end state of the first
//     of two levels, saved during the same pass; a resumed state starts from
//     the saved slot;
//   section 3.5 -- every question's chunks start at the fork.
//
// Chunked form (gated delta rule regrouped by chunk of C <= 64 tokens, from
// the state S0 at the chunk start; g = cumulative sum of log alpha inside the
// chunk):
//   A_ts = beta_t e^{g_t-g_s} k_t.k_s (s<t),   P_ts = e^{g_t-g_s} q_t.k_s (s<=t)
//   (I + A) [W | Ut] = [diag(beta e^g) K | diag(beta) V]
//   U = Ut - W S0^T;  O = diag(e^g) Q S0^T + P U;  S = e^{g_C} S0 + U^T diag(e^{g_C-g}) K
// Phase A (all chunks of all levels in parallel) builds W, Ut, P, g; phase B
// walks each node's chunks in order, one launch per tree level, split over
// d_v slices (rows of S evolve independently, so the split is exact).
#include <cuda_bf16.h>

#include <mutex>

#include "device.cuh"
#include "gdn_ws.h"

using namespace hsm;
using hsd::Meta;

namespace {

constexpr int kThreads = 256;
constexpr int kDvSlice = 16;

template <int DK, int DV>
struct WsLayout {
  static constexpr size_t W = 0;
  static constexpr size_t UT = W + (size_t)kChunk * DK;
  static constexpr size_t P = UT + (size_t)kChunk * DV;
  static constexpr size_t G = P + (size_t)kChunk * kChunk;
  static constexpr size_t FLOATS = G + kChunk;  // per (chunk, head)
};

__host__ __device__ inline size_t ws_floats_per(int dk, int dv) {
  return (size_t)kChunk * dk + (size_t)kChunk * dv + (size_t)kChunk * kChunk + kChunk;
}

// Load `len` rows of a [T, H, D] tensor (head h) into smem rows of stride
// `ld` as fp32; rows >= len are zero.
template <typename T, int D>
__device__ __forceinline__ void load_rows(float* dst, int ld, const T* __restrict__ src, int row0, int len, int H,
                                          int h) {
  constexpr int VEC = 16 / sizeof(T);
  for (int e = threadIdx.x; e < kChunk * (D / VEC); e += blockDim.x) {
    const int r = e / (D / VEC), c = (e % (D / VEC)) * VEC;
    float f[8];
    if (r < len) {
      const float4 raw = *reinterpret_cast<const float4*>(src + ((size_t)(row0 + r) * H + h) * D + c);
      hsd::cvt16(raw, f, T());
    } else {
#pragma unroll
      for (int i = 0; i < VEC; ++i) f[i] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < VEC; ++i) dst[r * ld + c + i] = f[i];
  }
}

// ---------------------------------------------------------------------------
// Phase A: chunk-local quantities, one thread block per (chunk, head).
// ---------------------------------------------------------------------------
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThreads)
gdn_chunk_local_kernel(const int32_t* __restrict__ meta, int H, const T* __restrict__ q, const T* __restrict__ k,
                       const T* __restrict__ v, const float* __restrict__ alpha, const float* __restrict__ beta,
                       float* __restrict__ ws) {
  extern __shared__ float sm[];
  constexpr int LK = DK + 1;
  float* Ks = sm;                      // [64][LK]
  float* Qs = Ks + kChunk * LK;        // [64][LK]
  float* Vs = Qs + kChunk * LK;        // [64][DV]
  float* As = Vs + kChunk * DV;        // [64][65]
  float* gs = As + kChunk * (kChunk + 1);
  float* bs = gs + kChunk;

  Meta M{meta};
  const int c = blockIdx.x, h = blockIdx.y;
  if (c >= M.h(H_N_CHUNK)) return;
  const int32_t* ch = M.chunk(c);
  const int row0 = ch[C_ROW0], len = ch[C_LEN];
  load_rows<T, DK>(Ks, LK, k, row0, len, H, h);
  load_rows<T, DK>(Qs, LK, q, row0, len, H, h);
  load_rows<T, DV>(Vs, DV, v, row0, len, H, h);
  if (threadIdx.x < kChunk) {
    const int t = threadIdx.x;
    gs[t] = t < len ? logf(alpha[(size_t)(row0 + t) * H + h]) : 0.f;
    bs[t] = t < len ? beta[(size_t)(row0 + t) * H + h] : 0.f;
  }
  __syncthreads();
  if (threadIdx.x == 0) {  // inclusive cumulative sum, fixed order
    float acc = 0.f;
    for (int t = 0; t < kChunk; ++t) {
      acc += gs[t];
      gs[t] = acc;
    }
  }
  __syncthreads();

  float* wsp = ws + ((size_t)c * H + h) * WsLayout<DK, DV>::FLOATS;
  // A (strictly lower) into smem, P (lower incl.) straight to the workspace
  {
    const int t = threadIdx.x / 4, s0 = (threadIdx.x % 4) * 16;
    float a[16], p[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) a[j] = p[j] = 0.f;
    for (int cc = 0; cc < DK; ++cc) {
      const float kt = Ks[t * LK + cc], qt = Qs[t * LK + cc];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float ks = Ks[(s0 + j) * LK + cc];
        a[j] = fmaf(kt, ks, a[j]);
        p[j] = fmaf(qt, ks, p[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int s = s0 + j;
      const float dec = expf(gs[t] - gs[s]);
      As[t * (kChunk + 1) + s] = (s < t && t < len) ? bs[t] * dec * a[j] : 0.f;
      wsp[WsLayout<DK, DV>::P + t * kChunk + s] = (s <= t && t < len) ? dec * p[j] : 0.f;
    }
  }
  if (threadIdx.x < kChunk) wsp[WsLayout<DK, DV>::G + threadIdx.x] = gs[threadIdx.x];
  __syncthreads();
  // forward substitution (I + A) X = B, one column per thread, in registers
  const int col = threadIdx.x;
  if (col < DK + DV) {
    float x[kChunk];
#pragma unroll
    for (int t = 0; t < kChunk; ++t) {
      float acc = col < DK ? bs[t] * expf(gs[t]) * Ks[t * LK + col] : bs[t] * Vs[t * DV + (col - DK)];
      if (t >= len) acc = 0.f;
#pragma unroll
      for (int s = 0; s < t; ++s) acc = fmaf(-As[t * (kChunk + 1) + s], x[s], acc);
      x[t] = acc;
    }
    if (col < DK) {
#pragma unroll
      for (int t = 0; t < kChunk; ++t) wsp[WsLayout<DK, DV>::W + t * DK + col] = x[t];
    } else {
#pragma unroll
      for (int t = 0; t < kChunk; ++t) wsp[WsLayout<DK, DV>::UT + t * DV + (col - DK)] = x[t];
    }
  }
}

// ---------------------------------------------------------------------------
// Phase B: the chunk chain of every node of one tree level, per (node, head,
// d_v slice).  The state slice lives in shared memory across the chain.
// ---------------------------------------------------------------------------
template <typename T, int DK, int DV>
__global__ void __launch_bounds__(kThreads)
gdn_state_pass_kernel(const int32_t* __restrict__ meta, int level, int H, const T* __restrict__ q,
                      const T* __restrict__ k, const float* __restrict__ ws, float* __restrict__ state,
                      int n_slots, T* __restrict__ out, int32_t* status) {
  extern __shared__ float sm[];
  constexpr int LK = DK + 1;
  constexpr int J = kDvSlice;
  float* Ss = sm;                  // [J][LK]
  float* Ws = Ss + J * LK;         // [64][LK]
  float* Qs = Ws + kChunk * LK;    // [64][LK]
  float* Ks = Qs + kChunk * LK;    // [64][LK]
  float* Ps = Ks + kChunk * LK;    // [64][65]
  float* Uts = Ps + kChunk * (kChunk + 1);  // [64][J]
  float* Us = Uts + kChunk * J;             // [64][J]
  float* gs = Us + kChunk * J;              // [64]
  float* dk_s = gs + kChunk;                // [64] e^{g_C - g_t}

  Meta M{meta};
  if (level >= M.h(H_N_LEVEL)) return;
  const int lo = M.level_off()[level], hi = M.level_off()[level + 1];
  if ((int)blockIdx.x >= hi - lo) return;
  const int seg = M.level_seg()[lo + blockIdx.x];
  const int32_t* sg = M.seg(seg);
  const int h = blockIdx.y, j0 = blockIdx.z * J;
  const int init = sg[S_INIT_SLOT], endslot = sg[S_END_SLOT];
  if (init >= n_slots || endslot >= n_slots) {
    hsd::set_status(status, HS_DEV_BAD_SLOT);
    return;
  }
  for (int e = threadIdx.x; e < J * DK; e += blockDim.x) {
    const int j = e / DK, cc = e % DK;
    Ss[j * LK + cc] = init >= 0 ? state[(((size_t)init * H + h) * DV + j0 + j) * DK + cc] : 0.f;
  }
  const int c_off = sg[S_CHUNK_OFF], n_c = sg[S_N_CHUNK];
  for (int ci = 0; ci < n_c; ++ci) {
    const int32_t* ch = M.chunk(c_off + ci);
    const int row0 = ch[C_ROW0], len = ch[C_LEN];
    const float* wsp = ws + ((size_t)(c_off + ci) * H + h) * WsLayout<DK, DV>::FLOATS;
    __syncthreads();  // previous chunk done with every buffer
    for (int e = threadIdx.x; e < kChunk * DK; e += blockDim.x) {
      const int t = e / DK, cc = e % DK;
      Ws[t * LK + cc] = wsp[WsLayout<DK, DV>::W + e];
    }
    for (int e = threadIdx.x; e < kChunk * kChunk; e += blockDim.x) {
      const int t = e / kChunk, s = e % kChunk;
      Ps[t * (kChunk + 1) + s] = wsp[WsLayout<DK, DV>::P + e];
    }
    for (int e = threadIdx.x; e < kChunk * J; e += blockDim.x) {
      const int t = e / J, j = e % J;
      Uts[e] = wsp[WsLayout<DK, DV>::UT + t * DV + j0 + j];
    }
    if (threadIdx.x < kChunk) gs[threadIdx.x] = wsp[WsLayout<DK, DV>::G + threadIdx.x];
    load_rows<T, DK>(Qs, LK, q, row0, len, H, h);
    load_rows<T, DK>(Ks, LK, k, row0, len, H, h);
    __syncthreads();
    if (threadIdx.x < kChunk) dk_s[threadIdx.x] = threadIdx.x < len ? expf(gs[len - 1] - gs[threadIdx.x]) : 0.f;
    // U = Ut - W S^T  (4 outputs per thread: row t, columns jj..jj+3)
    const int t = threadIdx.x / 4, jj = (threadIdx.x % 4) * 4;
    {
      float u[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) u[i] = 0.f;
      for (int cc = 0; cc < DK; ++cc) {
        const float w = Ws[t * LK + cc];
#pragma unroll
        for (int i = 0; i < 4; ++i) u[i] = fmaf(w, Ss[(jj + i) * LK + cc], u[i]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) Us[t * J + jj + i] = t < len ? Uts[t * J + jj + i] - u[i] : 0.f;
    }
    __syncthreads();
    // O = e^g (Q S^T) + P U
    {
      float o1[4], o2[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) o1[i] = o2[i] = 0.f;
      for (int cc = 0; cc < DK; ++cc) {
        const float qv = Qs[t * LK + cc];
#pragma unroll
        for (int i = 0; i < 4; ++i) o1[i] = fmaf(qv, Ss[(jj + i) * LK + cc], o1[i]);
      }
      for (int s = 0; s <= t; ++s) {
        const float p = Ps[t * (kChunk + 1) + s];
#pragma unroll
        for (int i = 0; i < 4; ++i) o2[i] = fmaf(p, Us[s * J + jj + i], o2[i]);
      }
      if (t < len) {
        const float eg = expf(gs[t]);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          out[((size_t)(row0 + t) * H + h) * DV + j0 + jj + i] = hsd::from_f<T>(fmaf(eg, o1[i], o2[i]));
      }
    }
    __syncthreads();
    // S = e^{g_C} S + U^T diag(e^{g_C - g}) K
    {
      const float egc = expf(gs[len - 1]);
      const int j = threadIdx.x / 16, cl = threadIdx.x % 16;
      float acc[DK / 16];
#pragma unroll
      for (int i = 0; i < DK / 16; ++i) acc[i] = 0.f;
      for (int s = 0; s < len; ++s) {
        const float us = Us[s * J + j] * dk_s[s];
#pragma unroll
        for (int i = 0; i < DK / 16; ++i) acc[i] = fmaf(us, Ks[s * LK + cl + 16 * i], acc[i]);
      }
#pragma unroll
      for (int i = 0; i < DK / 16; ++i) {
        float* sp = &Ss[j * LK + cl + 16 * i];
        *sp = fmaf(egc, *sp, acc[i]);
      }
    }
  }
  __syncthreads();
  if (endslot >= 0) {
    for (int e = threadIdx.x; e < J * DK; e += blockDim.x) {
      const int j = e / DK, cc = e % DK;
      state[(((size_t)endslot * H + h) * DV + j0 + j) * DK + cc] = Ss[j * LK + cc];
    }
  }
}

// ---------------------------------------------------------------------------
// cp.async helpers (16-byte global -> shared copies; size 0 = zero fill)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ float dot4(const float4& a, const float4& b) {
  return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}

// ---------------------------------------------------------------------------
// Phase A, register-blocked: one thread block per (chunk, head).  Rows of
// K, Q, V are staged in fp32 with a 4-float pad so that float4 reads of 8
// different rows hit 32 different banks.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
gdn_chunk_local_v2(const int32_t* __restrict__ meta, int H, const T* __restrict__ q, const T* __restrict__ k,
                   const T* __restrict__ v, const float* __restrict__ alpha, const float* __restrict__ beta,
                   float* __restrict__ ws) {
  constexpr int L = D + 4;
  constexpr int LA = kChunk + 4;
  extern __shared__ __align__(16) float smA[];
  float* Ks = smA;
  float* Qs = Ks + kChunk * L;
  float* Vs = Qs + kChunk * L;
  float* As = Vs + kChunk * L;   // [64][LA] strictly lower
  float* Ps = As + kChunk * LA;  // [64][LA] lower incl.
  float* gs = Ps + kChunk * LA;
  float* bs = gs + kChunk;
  float* bg = bs + kChunk;        // beta_t e^{g_t}

  Meta M{meta};
  const int c = blockIdx.x, h = blockIdx.y;
  if (c >= M.h(H_N_CHUNK)) return;
  const int32_t* ch = M.chunk(c);
  const int row0 = ch[C_ROW0], len = ch[C_LEN];
  const int tid = threadIdx.x;
  load_rows<T, D>(Ks, L, k, row0, len, H, h);
  load_rows<T, D>(Qs, L, q, row0, len, H, h);
  load_rows<T, D>(Vs, L, v, row0, len, H, h);
  if (tid < kChunk) {
    gs[tid] = tid < len ? logf(alpha[(size_t)(row0 + tid) * H + h]) : 0.f;
    bs[tid] = tid < len ? beta[(size_t)(row0 + tid) * H + h] : 0.f;
  }
  __syncthreads();
  if (tid == 0) {  // inclusive cumulative sum, fixed order
    float acc = 0.f;
    for (int t = 0; t < kChunk; ++t) {
      acc += gs[t];
      gs[t] = acc;
    }
  }
  __syncthreads();
  if (tid < kChunk) bg[tid] = bs[tid] * expf(gs[tid]);
  {
    const int t = tid >> 2, sq = tid & 3;  // rows s = sq + 4 j
    float a[16], pp[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) a[j] = pp[j] = 0.f;
#pragma unroll 2
    for (int cc = 0; cc < D; cc += 4) {
      const float4 kt = *reinterpret_cast<const float4*>(&Ks[t * L + cc]);
      const float4 qt = *reinterpret_cast<const float4*>(&Qs[t * L + cc]);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float4 ks = *reinterpret_cast<const float4*>(&Ks[(sq + 4 * j) * L + cc]);
        a[j] += dot4(kt, ks);
        pp[j] += dot4(qt, ks);
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int s = sq + 4 * j;
      const bool low = s <= t && t < len;
      const float dec = low ? expf(gs[t] - gs[s]) : 0.f;
      As[t * LA + s] = (low && s < t) ? bs[t] * dec * a[j] : 0.f;
      Ps[t * LA + s] = low ? dec * pp[j] : 0.f;
    }
  }
  __syncthreads();
  float* wsp = ws + ((size_t)c * H + h) * WsLayout<D, D>::FLOATS;
  {
    for (int e = tid; e < kChunk * (kChunk / 4); e += blockDim.x) {
      const int t = e / (kChunk / 4), s4 = (e % (kChunk / 4)) * 4;
      *reinterpret_cast<float4*>(wsp + WsLayout<D, D>::P + t * kChunk + s4) =
          *reinterpret_cast<const float4*>(&Ps[t * LA + s4]);
    }
    if (tid < kChunk) wsp[WsLayout<D, D>::G + tid] = gs[tid];
  }
  // forward substitution (I + A) [W | Ut] = [diag(beta e^g) K | diag(beta) V], one column per thread
  if (tid < 2 * D) {
    const bool isW = tid < D;
    const int cc = isW ? tid : tid - D;
    const float* src = isW ? Ks : Vs;
    const float* scl = isW ? bg : bs;
    float x[kChunk];
#pragma unroll
    for (int t = 0; t < kChunk; ++t) x[t] = 0.f;
#pragma unroll
    for (int t = 0; t < kChunk; ++t) {
      float acc = scl[t] * src[t * L + cc];
#pragma unroll
      for (int s = 0; s < t; s += 4) {
        const float4 a4 = *reinterpret_cast<const float4*>(&As[t * LA + s]);
        acc = fmaf(-a4.x, x[s], acc);
        if (s + 1 < t) acc = fmaf(-a4.y, x[s + 1], acc);
        if (s + 2 < t) acc = fmaf(-a4.z, x[s + 2], acc);
        if (s + 3 < t) acc = fmaf(-a4.w, x[s + 3], acc);
      }
      x[t] = acc;
    }
    float* dst = wsp + (isW ? WsLayout<D, D>::W : WsLayout<D, D>::UT) + cc;
#pragma unroll
    for (int t = 0; t < kChunk; ++t) dst[t * D] = x[t];
  }
}

// ---------------------------------------------------------------------------
// Phase B, pipelined (bf16 inputs): one thread block per (node, head, 16-row
// slice of d_v).  The next chunk's W, P, Ut slice, g, Q and K are fetched
// with cp.async into the other half of a double buffer while the current
// chunk runs.  The state slice is kept transposed, S_T[c][j], so that four
// consecutive j are one float4.
// ---------------------------------------------------------------------------
template <typename T, int D>
struct StageB {
  static constexpr int LW = D + 4;                 // fp32 row of W
  static constexpr int LP = kChunk + 4;            // fp32 row of P
  static constexpr int LQ = D + 16 / sizeof(T);    // row of Q, K in elements (16-byte pad)
  static constexpr int W = 0;
  static constexpr int P = W + kChunk * LW * 4;
  static constexpr int UT = P + kChunk * LP * 4;
  static constexpr int Q = UT + kChunk * kDvSlice * 4;
  static constexpr int K = Q + kChunk * LQ * (int)sizeof(T);
  static constexpr int G = K + kChunk * LQ * (int)sizeof(T);
  static constexpr int BYTES = G + kChunk * 4;
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
gdn_state_pass_v2(const int32_t* __restrict__ meta, int level, int H, const T* __restrict__ q,
                  const T* __restrict__ k, const float* __restrict__ ws, float* __restrict__ state, int n_slots,
                  T* __restrict__ out, int32_t* status) {
  using SB = StageB<T, D>;
  constexpr int J = kDvSlice;
  constexpr int VEC = 16 / sizeof(T);
  extern __shared__ __align__(16) unsigned char smB[];
  float* ST = reinterpret_cast<float*>(smB + 2 * SB::BYTES);  // [D][J]
  float* Us = ST + D * J;                                       // [64][J]
  float* dks = Us + kChunk * J;                                 // [64]

  Meta M{meta};
  if (level >= M.h(H_N_LEVEL)) return;
  const int lo = M.level_off()[level], hi = M.level_off()[level + 1];
  if ((int)blockIdx.x >= hi - lo) return;
  const int seg = M.level_seg()[lo + blockIdx.x];
  const int32_t* sg = M.seg(seg);
  const int h = blockIdx.y, jb = blockIdx.z * J;
  const int init = sg[S_INIT_SLOT], endslot = sg[S_END_SLOT];
  if (init >= n_slots || endslot >= n_slots) {
    hsd::set_status(status, HS_DEV_BAD_SLOT);
    return;
  }
  const int tid = threadIdx.x;
  for (int e = tid; e < D * J; e += blockDim.x) {
    const int j = e / D, cc = e % D;  // coalesced along c in the pool
    ST[cc * J + j] = init >= 0 ? state[(((size_t)init * H + h) * D + jb + j) * D + cc] : 0.f;
  }
  const int c_off = sg[S_CHUNK_OFF], n_c = sg[S_N_CHUNK];

  auto prefetch = [&](int ci, unsigned char* sp) {
    const int32_t* chp = M.chunk(c_off + ci);
    const int row0 = chp[C_ROW0], len = chp[C_LEN];
    const float* wsp = ws + ((size_t)(c_off + ci) * H + h) * WsLayout<D, D>::FLOATS;
    for (int e = tid; e < kChunk * (D / 4); e += blockDim.x) {
      const int t = e / (D / 4), c4 = (e % (D / 4)) * 4;
      cp_async16(sp + SB::W + (t * SB::LW + c4) * 4, wsp + WsLayout<D, D>::W + t * D + c4, true);
    }
    for (int e = tid; e < kChunk * (kChunk / 4); e += blockDim.x) {
      const int t = e / (kChunk / 4), s4 = (e % (kChunk / 4)) * 4;
      cp_async16(sp + SB::P + (t * SB::LP + s4) * 4, wsp + WsLayout<D, D>::P + t * kChunk + s4, true);
    }
    for (int e = tid; e < kChunk * (J / 4); e += blockDim.x) {
      const int t = e / (J / 4), j4 = (e % (J / 4)) * 4;
      cp_async16(sp + SB::UT + (t * J + j4) * 4, wsp + WsLayout<D, D>::UT + t * D + jb + j4, true);
    }
    for (int e = tid; e < 2 * kChunk * (D / VEC); e += blockDim.x) {
      const int which = e >= kChunk * (D / VEC);
      const int ee = which ? e - kChunk * (D / VEC) : e;
      const int t = ee / (D / VEC), c8 = (ee % (D / VEC)) * VEC;
      const T* src = (which ? k : q) + ((size_t)(row0 + (t < len ? t : 0)) * H + h) * D + c8;
      cp_async16(sp + (which ? SB::K : SB::Q) + (t * SB::LQ + c8) * (int)sizeof(T), src, t < len);
    }
    if (tid < kChunk / 4) cp_async16(sp + SB::G + tid * 16, wsp + WsLayout<D, D>::G + tid * 4, true);
    cp_async_commit();
  };

  if (n_c > 0) prefetch(0, smB);
  const int t = tid >> 2, jl = (tid & 3) * 4;           // U / O: row t, columns jl..jl+3 of the slice
  const int jd = tid & 15, cd = (tid >> 4) * (D / 16);  // S update: column jd, rows cd..cd+D/16-1
  for (int ci = 0; ci < n_c; ++ci) {
    unsigned char* sp = smB + (ci & 1) * SB::BYTES;
    if (ci + 1 < n_c) {
      prefetch(ci + 1, smB + ((ci + 1) & 1) * SB::BYTES);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const int32_t* chp = M.chunk(c_off + ci);
    const int row0 = chp[C_ROW0], len = chp[C_LEN];
    const float* Wsm = reinterpret_cast<const float*>(sp + SB::W);
    const float* Psm = reinterpret_cast<const float*>(sp + SB::P);
    const float* Utm = reinterpret_cast<const float*>(sp + SB::UT);
    const T* Qsm = reinterpret_cast<const T*>(sp + SB::Q);
    const T* Ksm = reinterpret_cast<const T*>(sp + SB::K);
    const float* gsm = reinterpret_cast<const float*>(sp + SB::G);
    const float gC = gsm[len - 1];
    if (tid < kChunk) dks[tid] = tid < len ? expf(gC - gsm[tid]) : 0.f;
    // U = Ut - W S^T
    {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int cc = 0; cc < D; cc += 4) {
        const float4 w = *reinterpret_cast<const float4*>(&Wsm[t * SB::LW + cc]);
        const float4 s0 = *reinterpret_cast<const float4*>(&ST[(cc + 0) * J + jl]);
        const float4 s1 = *reinterpret_cast<const float4*>(&ST[(cc + 1) * J + jl]);
        const float4 s2 = *reinterpret_cast<const float4*>(&ST[(cc + 2) * J + jl]);
        const float4 s3 = *reinterpret_cast<const float4*>(&ST[(cc + 3) * J + jl]);
        acc.x = fmaf(w.x, s0.x, fmaf(w.y, s1.x, fmaf(w.z, s2.x, fmaf(w.w, s3.x, acc.x))));
        acc.y = fmaf(w.x, s0.y, fmaf(w.y, s1.y, fmaf(w.z, s2.y, fmaf(w.w, s3.y, acc.y))));
        acc.z = fmaf(w.x, s0.z, fmaf(w.y, s1.z, fmaf(w.z, s2.z, fmaf(w.w, s3.z, acc.z))));
        acc.w = fmaf(w.x, s0.w, fmaf(w.y, s1.w, fmaf(w.z, s2.w, fmaf(w.w, s3.w, acc.w))));
      }
      const float4 ut = *reinterpret_cast<const float4*>(&Utm[t * J + jl]);
      *reinterpret_cast<float4*>(&Us[t * J + jl]) =
          make_float4(ut.x - acc.x, ut.y - acc.y, ut.z - acc.z, ut.w - acc.w);
    }
    __syncthreads();
    // O = e^g (Q S^T) + P U, and the S-update products U^T diag(e^{gC-g}) K into registers
    {
      float4 o1 = make_float4(0.f, 0.f, 0.f, 0.f), o2 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 2
      for (int cc = 0; cc < D; cc += VEC) {
        float qf[8];
        hsd::cvt16(*reinterpret_cast<const float4*>(&Qsm[t * SB::LQ + cc]), qf, T());
#pragma unroll
        for (int i = 0; i < VEC; ++i) {
          const float4 s = *reinterpret_cast<const float4*>(&ST[(cc + i) * J + jl]);
          o1.x = fmaf(qf[i], s.x, o1.x);
          o1.y = fmaf(qf[i], s.y, o1.y);
          o1.z = fmaf(qf[i], s.z, o1.z);
          o1.w = fmaf(qf[i], s.w, o1.w);
        }
      }
#pragma unroll 4
      for (int s4 = 0; s4 < kChunk; s4 += 4) {
        const float4 pv = *reinterpret_cast<const float4*>(&Psm[t * SB::LP + s4]);
        const float pw[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 u = *reinterpret_cast<const float4*>(&Us[(s4 + i) * J + jl]);
          o2.x = fmaf(pw[i], u.x, o2.x);
          o2.y = fmaf(pw[i], u.y, o2.y);
          o2.z = fmaf(pw[i], u.z, o2.z);
          o2.w = fmaf(pw[i], u.w, o2.w);
        }
      }
      if (t < len) {
        const float eg = expf(gsm[t]);
        T* dst = out + ((size_t)(row0 + t) * H + h) * D + jb + jl;
        dst[0] = hsd::from_f<T>(fmaf(eg, o1.x, o2.x));
        dst[1] = hsd::from_f<T>(fmaf(eg, o1.y, o2.y));
        dst[2] = hsd::from_f<T>(fmaf(eg, o1.z, o2.z));
        dst[3] = hsd::from_f<T>(fmaf(eg, o1.w, o2.w));
      }
    }
    float su[D / 16];
#pragma unroll
    for (int i = 0; i < D / 16; ++i) su[i] = 0.f;
    for (int s = 0; s < len; ++s) {
      const float u = Us[s * J + jd] * dks[s];
      float kf[8];
      if constexpr (D / 16 == 8) {
        hsd::cvt16(*reinterpret_cast<const float4*>(&Ksm[s * SB::LQ + cd]), kf, T());
      } else {
#pragma unroll
        for (int i = 0; i < D / 16; ++i) kf[i] = hsd::to_f(Ksm[s * SB::LQ + cd + i]);
      }
#pragma unroll
      for (int i = 0; i < D / 16; ++i) su[i] = fmaf(u, kf[i], su[i]);
    }
    __syncthreads();  // every read of S_T and of this stage is done
    const float egc = expf(gC);
#pragma unroll
    for (int i = 0; i < D / 16; ++i) {
      float* sp2 = &ST[(cd + i) * J + jd];
      *sp2 = fmaf(egc, *sp2, su[i]);
    }
  }
  __syncthreads();
  if (endslot >= 0) {
    for (int e = tid; e < D * J; e += blockDim.x) {
      const int j = e / D, cc = e % D;
      state[(((size_t)endslot * H + h) * D + jb + j) * D + cc] = ST[cc * J + j];
    }
  }
}

__global__ void copy_state_kernel(const float4* __restrict__ src, float4* __restrict__ dst, size_t n4) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

template <int DK, int DV>
constexpr size_t smemA() {
  return sizeof(float) * ((size_t)kChunk * (DK + 1) * 2 + kChunk * DV + kChunk * (kChunk + 1) + 2 * kChunk);
}
template <int DK, int DV>
constexpr size_t smemB() {
  return sizeof(float) * ((size_t)kDvSlice * (DK + 1) + 3 * (size_t)kChunk * (DK + 1) + kChunk * (kChunk + 1) +
                          2 * kChunk * kDvSlice + 2 * kChunk);
}

}  // namespace

hs_status hs_gdn_chain_tc_launch(const hs_round_caps* caps, const int32_t* meta, int H, const void* q,
                                 const uint8_t* ws, uint8_t* scan, float* state, int n_slots, void* out,
                                 int32_t* status, cudaStream_t st);
static size_t scan_region_offset(const hs_round_caps* caps, int32_t h, int32_t dk, int32_t dv);
hs_status hs_gdn_prep_tc_launch(const hs_round_caps* caps, const int32_t* meta, int H, const void* q, const void* k,
                                const void* v, const float* alpha, const float* beta, uint8_t* ws, int32_t* status,
                                cudaStream_t st);

namespace {

template <int D>
constexpr size_t smemA2() {
  return sizeof(float) * ((size_t)3 * kChunk * (D + 4) + 2 * (size_t)kChunk * (kChunk + 4) + 3 * kChunk);
}
template <typename T, int D>
constexpr size_t smemB2() {
  return 2 * (size_t)StageB<T, D>::BYTES + sizeof(float) * ((size_t)D * kDvSlice + kChunk * kDvSlice + kChunk);
}

template <typename T, int D>
hs_status run_gdn(const hs_round_caps* caps, const int32_t* meta, int H, const void* q, const void* k,
                  const void* v, const float* alpha, const float* beta, float* state, int n_slots, void* out,
                  float* ws, int32_t* status, cudaStream_t st) {
  if constexpr (sizeof(T) == 2 && D == 128) {
    // tensor cores for both passes, through the compact bf16 workspace
    const hs_status s = hs_gdn_prep_tc_launch(caps, meta, H, q, k, v, alpha, beta, (uint8_t*)ws, status, st);
    if (s != HS_OK) return s;
    uint8_t* scan = (uint8_t*)ws + scan_region_offset(caps, H, D, D);
    return hs_gdn_chain_tc_launch(caps, meta, H, q, (const uint8_t*)ws, scan, state, n_slots, out, status, st);
  }
  // bf16 inputs take the pipelined state pass; fp32 rows do not fit its double buffer at d=128
  constexpr bool kPipelined = sizeof(T) == 2;
  static std::atomic<bool> configured[hsd::kMaxDevices];  // zero-initialised: per device
  const int slot = hsd::device_slot();
  if (slot < 0) return hs::fail(HS_ECUDA, "gdn: no usable CUDA device");
  auto ka = gdn_chunk_local_v2<T, D>;
  auto kb1 = gdn_state_pass_kernel<T, D, D>;
  auto kb2 = gdn_state_pass_v2<T, D>;
  if (!configured[slot].load()) {
    bool ok = cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smemA2<D>()) == cudaSuccess;
    if (kPipelined)
      ok = ok && cudaFuncSetAttribute(kb2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smemB2<T, D>()) ==
                     cudaSuccess;
    else
      ok = ok && cudaFuncSetAttribute(kb1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smemB<D, D>()) ==
                     cudaSuccess;
    if (!ok) return hs::fail(HS_ECUDA, "gdn: cannot raise the shared-memory limit");
    configured[slot].store(true);
  }
  if (caps->max_chunks > 0) {
    ka<<<dim3(caps->max_chunks, H), kThreads, smemA2<D>(), st>>>(meta, H, (const T*)q, (const T*)k, (const T*)v,
                                                                 alpha, beta, ws);
    HS_LAUNCH_CHECK("gdn_chunk_local");
  }
  for (int lev = 0; lev < caps->max_levels && caps->max_segments > 0; ++lev) {
    const dim3 grid(caps->max_segments, H, D / kDvSlice);
    if (kPipelined)
      kb2<<<grid, kThreads, smemB2<T, D>(), st>>>(meta, lev, H, (const T*)q, (const T*)k, ws, state, n_slots,
                                                   (T*)out, status);
    else
      kb1<<<grid, kThreads, smemB<D, D>(), st>>>(meta, lev, H, (const T*)q, (const T*)k, ws, state, n_slots,
                                                  (T*)out, status);
    HS_LAUNCH_CHECK("gdn_state_pass");
  }
  return HS_OK;
}

}  // namespace

// Per-chunk blocks, then (d = 128) the buffers of the two-level state scan.
static size_t scan_region_offset(const hs_round_caps* caps, int32_t h, int32_t dk, int32_t dv) {
  return ((size_t)caps->max_chunks * h * ws_floats_per(dk, dv) * sizeof(float) + 255) & ~(size_t)255;
}

extern "C" size_t hs_gdn_workspace_bytes(const hs_round_caps* caps, int32_t h, int32_t dk, int32_t dv) {
  if (!caps || h <= 0 || dk <= 0 || dv <= 0) return 0;
  size_t n = scan_region_offset(caps, h, dk, dv);
  if (dk == 128 && dv == 128) n += (size_t)scan_cap(caps->max_chunks) * h * gdnws::kScanBytes;
  return n;
}

namespace {
// The shapes and dtypes the GDN kernels are built for; both fork-prefill entry points check them first, so
// they report the same error for the same bad arguments.
hs_status gdn_shape_check(int32_t h, int32_t dk, int32_t dv, int32_t chunk, hs_dtype dt) {
  HS_CHECK_ARG(h > 0, "h must be > 0");
  if (chunk != kChunk) return hs::fail(HS_EUNSUPPORTED, "chunk %d (built: %d)", chunk, kChunk);
  if (dk != dv || (dk != 64 && dk != 128)) return hs::fail(HS_EUNSUPPORTED, "dk=%d dv=%d (built: 64, 128)", dk, dv);
  if (dt != HS_F32 && dt != HS_BF16) return hs::fail(HS_EUNSUPPORTED, "dtype %d", (int)dt);
  return HS_OK;
}
}  // namespace

extern "C" hs_status hs_gdn_fork_prefill(const hs_round_caps* caps, const void* dev_meta, hs_dtype dt, int32_t h,
                                         int32_t dk, int32_t dv, int32_t chunk, const void* q, const void* k,
                                         const void* v, const float* alpha, const float* beta, float* state_pool,
                                         int32_t n_slots, void* out, void* ws, size_t ws_bytes, int32_t* dev_status,
                                         void* stream) {
  HS_CHECK_ARG(caps && dev_meta && q && k && v && alpha && beta && out && ws, "null argument");
  HS_CHECK_ARG(n_slots >= 0 && (n_slots == 0 || state_pool), "bad state pool");
  if (hs_status s = gdn_shape_check(h, dk, dv, chunk, dt)) return s;
  const size_t need = hs_gdn_workspace_bytes(caps, h, dk, dv);
  HS_CHECK_ARG(ws_bytes >= need, "workspace of %zu bytes < %zu", ws_bytes, need);
  HS_CHECK_ARG(((uintptr_t)ws & 255) == 0, "workspace must be 256-byte aligned");
  HS_CHECK_ARG((((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)out) & 15) == 0,
               "q, k, v, out must be 16-byte aligned");
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return hs::fail(HS_ECUDA, "no CUDA device");
  cudaStream_t st = (cudaStream_t)stream;
  const int32_t* meta = (const int32_t*)dev_meta;
  if (dt == HS_BF16) {
    if (dk == 128)
      return run_gdn<__nv_bfloat16, 128>(caps, meta, h, q, k, v, alpha, beta, state_pool, n_slots, out, (float*)ws,
                                         dev_status, st);
    return run_gdn<__nv_bfloat16, 64>(caps, meta, h, q, k, v, alpha, beta, state_pool, n_slots, out, (float*)ws,
                                      dev_status, st);
  }
  if (dk == 128)
    return run_gdn<float, 128>(caps, meta, h, q, k, v, alpha, beta, state_pool, n_slots, out, (float*)ws, dev_status,
                               st);
  return run_gdn<float, 64>(caps, meta, h, q, k, v, alpha, beta, state_pool, n_slots, out, (float*)ws, dev_status, st);
}

extern "C" hs_status hs_gdn_state_checkpoint(float* state_pool, int32_t n_slots, int32_t src, int32_t dst, int32_t h,
                                             int32_t dk, int32_t dv, void* stream) {
  HS_CHECK_ARG(state_pool, "null state pool");
  HS_CHECK_ARG(src >= 0 && src < n_slots && dst >= 0 && dst < n_slots, "slot out of range (src %d, dst %d, n %d)",
               src, dst, n_slots);
  HS_CHECK_ARG(h > 0 && dk > 0 && dv > 0 && ((size_t)h * dk * dv) % 4 == 0, "bad state shape");
  HS_CHECK_ARG(((uintptr_t)state_pool & 15) == 0, "state pool must be 16-byte aligned");
  if (src == dst) return HS_OK;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return hs::fail(HS_ECUDA, "no CUDA device");
  const size_t per = (size_t)h * dk * dv;
  const size_t n4 = per / 4;
  int grid = (int)((n4 + 255) / 256);
  if (grid > 1024) grid = 1024;
  copy_state_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>((const float4*)(state_pool + (size_t)src * per),
                                                             (float4*)(state_pool + (size_t)dst * per), n4);
  HS_LAUNCH_CHECK("gdn_state_checkpoint");
  return HS_OK;
}

// ---------------------------------------------------------------------------
// Workspace-free variant for callers that cannot allocate device memory:
// the scratch lives in a file-scope device array (HS_GDN_NOALLOC_SCRATCH_BYTES
// per GPU that loads the library, held until exit).  Host code cannot use the
// array's name as a device address, so each device's address is looked up
// once with cudaGetSymbolAddress while that device is current.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_gdn_noalloc_scratch[HS_GDN_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};
}  // namespace

extern "C" hs_status hs_gdn_fork_prefill_noalloc(const hs_round_caps* caps, const void* dev_meta, hs_dtype dt,
                                                 int32_t h, int32_t dk, int32_t dv, int32_t chunk, const void* q,
                                                 const void* k, const void* v, const float* alpha, const float* beta,
                                                 float* state_pool, int32_t n_slots, void* out, int32_t* dev_status,
                                                 void* stream) {
  HS_CHECK_ARG(caps, "null caps");
  if (hs_status s = gdn_shape_check(h, dk, dv, chunk, dt)) return s;
  const size_t need = hs_gdn_workspace_bytes(caps, h, dk, dv);
  if (need > HS_GDN_NOALLOC_SCRATCH_BYTES)
    return hs::fail(HS_ECAPACITY, "round needs %zu bytes of GDN scratch; the built-in scratch holds %zu", need,
                    (size_t)HS_GDN_NOALLOC_SCRATCH_BYTES);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return hs::fail(HS_ECUDA, "no CUDA device");
  if (dev < 0 || dev >= kMaxDevices) return hs::fail(HS_EUNSUPPORTED, "device ordinal %d", dev);
  void* ptr = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
      cudaError_t e = cudaGetSymbolAddress(&g_scratch_ptr[dev], g_gdn_noalloc_scratch);
      if (e != cudaSuccess) {
        g_scratch_ptr[dev] = nullptr;
        return hs::fail(HS_ECUDA, "scratch address on device %d: %s", dev, cudaGetErrorString(e));
      }
    }
    ptr = g_scratch_ptr[dev];
  }
  return hs_gdn_fork_prefill(caps, dev_meta, dt, h, dk, dv, chunk, q, k, v, alpha, beta, state_pool, n_slots, out,
                             ptr, HS_GDN_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
