// gdn_prep_tc.cu -- chunk-local pass of the Gated DeltaNet prefill on tcgen05
// (bf16 inputs, d_k = d_v = 128, chunks of 64 tokens).
//
// Flide, "Accelerating Decision Inference with Exact State Forking", section
// 3.2.2 (Eq. 4, the gated delta rule) regrouped by chunk, every node's chunks
// starting at its first token (section 3.5).  For one chunk of one head, with
// g = cumulative sum of log alpha inside the chunk:
//
//   A_ts = beta_t e^{g_t - g_s} k_t.k_s  (s < t)      T = (I + A)^{-1}
//   P_ts = e^{g_t - g_s} q_t.k_s          (s <= t)
//   W  = T diag(beta e^g) K,   Ut = T diag(beta) V
//
// K' = diag(e^{g_C - g}) K, and the decay factors e^{g_t}, e^{g_C - g_t}, e^{g_C}
// (C = last token).  The
// results go to the compact workspace that the tensor-core state pass reads
// (layout in gdn_ws.h).
//
// One CTA = one chunk x two heads, so that the two heads' 64 tokens stack
// into the 128 rows of an MMA; two CTAs share an SM (96 KB of shared memory,
// 256 tensor-memory columns each), so one's copies and waits overlap the
// other's arithmetic:
//   warp 4      TMA of Q, K, V (both heads), tensor-memory allocation, and the
//               MMAs from one thread: K K^T and Q K^T (128 x 128, the two
//               64 x 64 diagonal blocks are used), then per head
//               W^T = K^T (T diag(beta e^g))^T and, once those are done,
//               Ut^T = V^T (T diag(beta))^T, with K and V read as MN-major A
//               operands straight from their TMA tiles and T split into a
//               bf16 high and low part.
//   warps 0..3  thread r = (head r / 64, token r % 64): the decay factors, the
//               masked rows of A and P, then column r % 64 of T by forward
//               substitution in fp32, then its row of K' = diag(e^{g_C-g}) K,
//               then (as thread = row k of W^T, Ut^T) the swizzled bf16 images
//               of W^T and Ut^T; the three images are copied out in bulk.
// Shared memory: Q | K | V, 32 KB each.  The Q buffer is reused for A (fp32)
// once Q K^T is done, then for the T operands, then for the W^T images.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "device.cuh"
#include "gdn_ws.h"
#include "tc_ptx.cuh"

using namespace hsm;
using hsd::Meta;

namespace {

constexpr int kD = 128;
constexpr int kThreads = 160;
constexpr long long kWaitCycles = 4000000000LL;
// shared memory (from a 1024-aligned base).  Q, K, V: two [128][64] slabs each
// (slab = 64 columns of d; rows 0..63 head a, 64..127 head b).
constexpr int kOffQ = 0, kOffK = 32768, kOffV = 65536;
constexpr int kSmem = 98304;
constexpr int kOffA = kOffQ;  // A^T, fp32 [2][64][64], 16-byte chunks swizzled by row (after Q K^T)
constexpr int kOffT = kOffQ;  // per head: T hi, T lo, each [64 s][64 t] bf16 MN-major (after the solve)
constexpr uint32_t kInTx = 3 * 32768;
// tensor-memory columns (256): K K^T and Q K^T, then W^T and Ut^T over them
constexpr uint32_t kTKK = 0, kTQK = 128;  // [128][128] fp32 each
constexpr uint32_t kTW = 0, kTU = 128;    // [128 (d)][64 (t)] per head, heads side by side

constexpr uint32_t kIdescSq = tc::idesc_bf16(128, 128, 0, 0);  // A, B K-major
constexpr uint32_t kIdescWU = tc::idesc_bf16(128, 64, 1, 1);   // A, B MN-major

struct Prm {
  const int32_t* meta;
  int H;
  const float* alpha;
  const float* beta;
  uint8_t* ws;
  int32_t* status;
};

// byte offset of A[u][s] in one head's block, stored transposed (row s holds column s of A: the
// entries A[u][s], u = 0..63), its 16-byte chunks swizzled by s
__device__ __forceinline__ int at_off(int s, int u) {
  return s * 256 + ((((u >> 2) ^ (s & 15))) << 4) + (u & 3) * 4;
}

// Row j of T diag(scale) as the MN-major B operand of one head: high part at
// `bt`, low part at `bt + 8192`.
__device__ __forceinline__ void write_t_operand(uint8_t* bt, int j, const float (&x)[64], float scale) {
  const int rowb = (j >> 3) * 1024 + (j & 7) * 128;
#pragma unroll
  for (int c8 = 0; c8 < 8; ++c8) {
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = x[c8 * 8 + 2 * e] * scale, b = x[c8 * 8 + 2 * e + 1] * scale;
      hi[e] = tc::pack_bf16x2(a, b);
      lo[e] = tc::pack_bf16x2(a - __uint_as_float(hi[e] << 16), b - __uint_as_float(hi[e] & 0xFFFF0000u));
    }
    const int off = rowb + ((c8 ^ (j & 7)) << 4);
    *reinterpret_cast<uint4*>(bt + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(bt + 8192 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
}

// No minimum-blocks hint: with one, ptxas kept fewer registers and spilled in
// the solve; without it the kernel takes 155 registers (25,600 per CTA) and two
// CTAs still fit on an SM.
__global__ void __launch_bounds__(kThreads)
gdn_chunk_prep_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const Prm p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_in, bar_d, bar_b1, bar_w1, bar_b2, bar_w2;
  __shared__ uint32_t tmem_slot;
  __shared__ float gsh[2][64], bsh[2][64];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);

  Meta M{p.meta};
  const int c = blockIdx.x, hp = blockIdx.y;
  if (c >= M.h(H_N_CHUNK)) return;
  const int32_t* ch = M.chunk(c);
  const int row0 = ch[C_ROW0], len = ch[C_LEN];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    tc::mbar_init(&bar_in, 1);
    tc::mbar_init(&bar_d, 1);
    tc::mbar_init(&bar_b1, 128);
    tc::mbar_init(&bar_w1, 1);
    tc::mbar_init(&bar_b2, 128);
    tc::mbar_init(&bar_w2, 1);
    tc::fence_mbar_init();
  }
  if (warp == 4) {
    tc::tmem_alloc(&tmem_slot, 256);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  // (launched with launch_pdl) Everything above reads only the round's metadata, which host copies write;
  // pages, inputs, workspace and state written by the earlier kernels in the stream are touched only after
  // the wait.  The next kernel may start launching only now, once every block of this one holds its tensor
  // memory: a block of the next kernel that took the columns first, then waited here for this kernel, would
  // block this kernel's allocation for good.
  hsd::pdl_trigger();
  hsd::pdl_wait();

  if (warp == 4) {
    // ------------------------------------------------------- copies and MMAs
    // (copies from lane 0; the MMAs from the converged warp: voted waits, one elected lane issues, descriptors
    // built once with a K step added to the start-address field)
    if (lane == 0) {
      tc::mbar_expect_tx(&bar_in, kInTx);
      for (int i = 0; i < 2; ++i) {
        const int hh = 2 * hp + i;  // head H (odd H) is out of range: zero fill
        for (int half = 0; half < 2; ++half) {
          const int o = half * 16384 + i * 8192;
          tc::tma_load_3d(smem + kOffQ + o, &tm_q, half * 64, hh, row0, &bar_in);
          tc::tma_load_3d(smem + kOffK + o, &tm_k, half * 64, hh, row0, &bar_in);
          tc::tma_load_3d(smem + kOffV + o, &tm_v, half * 64, hh, row0, &bar_in);
        }
      }
    }
    __syncwarp();
    bool ok = __all_sync(~0u, tc::mbar_wait(&bar_in, 0, kWaitCycles));
    if (ok) {
      tc::fence_after_sync();
      const uint64_t dq = tc::sdesc_sw128(tc::smem_u32(smem + kOffQ), 16, 1024);
      const uint64_t dk = tc::sdesc_sw128(tc::smem_u32(smem + kOffK), 16, 1024);
#pragma unroll
      for (int k = 0; k < 8; ++k) {  // K K^T, Q K^T over d (16 per step)
        const uint64_t off = (uint64_t)(((k >> 2) * 16384 + (k & 3) * 32) >> 4);
        tc::mma_bf16_ss_w(tmem + kTKK, dk + off, dk + off, kIdescSq, k > 0 ? 1u : 0u);
        tc::mma_bf16_ss_w(tmem + kTQK, dq + off, dk + off, kIdescSq, k > 0 ? 1u : 0u);
      }
      tc::mma_commit_w(&bar_d);
    }
    // W^T, then Ut^T, each from its T operand in the Q buffer
    for (int pass = 0; pass < 2 && ok; ++pass) {
      ok = __all_sync(~0u, tc::mbar_wait(pass == 0 ? &bar_b1 : &bar_b2, 0, kWaitCycles));
      if (!ok) break;
      tc::fence_after_sync();
      const int src = pass == 0 ? kOffK : kOffV;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint64_t da = tc::sdesc_sw128(tc::smem_u32(smem + src + i * 8192), 16384, 1024);
        const uint64_t db = tc::sdesc_sw128(tc::smem_u32(smem + kOffT + i * 16384), 8192, 1024);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // over the chunk's tokens s, 16 per step
            tc::mma_bf16_ss_w(tmem + (pass == 0 ? kTW : kTU) + 64 * i, da + (uint64_t)((k * 2048) >> 4),
                              db + (uint64_t)((part * 8192 + k * 2048) >> 4), kIdescWU, (part > 0 || k > 0) ? 1u : 0u);
          }
        }
      }
      tc::mma_commit_w(pass == 0 ? &bar_w1 : &bar_w2);
    }
    if (!ok && lane == 0) hsd::set_status(p.status, HS_DEV_TIMEOUT);
    __syncwarp();
  } else {
    // -------------------------------------------------------------- rows
    const int r = threadIdx.x;  // TMEM lane
    const int i = r >> 6, t = r & 63;
    const int hh = 2 * hp + i;
    const bool valid = hh < p.H;
    const uint32_t lb = (uint32_t)(warp * 32) << 16;
    uint8_t* wsi = p.ws + ((size_t)c * p.H + (valid ? hh : 0)) * gdnws::kBytes;
    {
      const size_t a = (size_t)(row0 + t) * p.H + hh;
      gsh[i][t] = (valid && t < len) ? logf(p.alpha[a]) : 0.f;
      bsh[i][t] = (valid && t < len) ? p.beta[a] : 0.f;
    }
    tc::named_sync(1, 128);
    if (t == 0) {  // inclusive cumulative sum, fixed order
      float acc = 0.f;
      for (int s = 0; s < 64; ++s) {
        acc += gsh[i][s];
        gsh[i][s] = acc;
      }
    }
    tc::named_sync(1, 128);
    const float gt = gsh[i][t], bt = bsh[i][t];
    const float gC = gsh[i][len - 1];
    if (valid) {
      float* gd = reinterpret_cast<float*>(wsi + gdnws::kG);
      gd[t] = t < len ? expf(gt) : 0.f;
      gd[64 + t] = t < len ? expf(gC - gt) : 0.f;
      if (t == 0) gd[128] = expf(gC);
    }
    bool ok = __all_sync(~0u, tc::mbar_wait(&bar_d, 0, kWaitCycles));
    if (ok) {
      tc::fence_after_sync();
      // row t of A (fp32, in the Q buffer: Q K^T is done) and of P (bf16, straight to the workspace)
      uint8_t* Ai = smem + kOffA + i * 16384;
      uint8_t* Pi = wsi + gdnws::kP;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t kk[32], qk[32];
        tc::tmem_ld32(tmem + lb + kTKK + 64 * i + 32 * half, kk);
        tc::tmem_ld32(tmem + lb + kTQK + 64 * i + 32 * half, qk);
        tc::tmem_wait_ld();
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          float av[4], pv[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s = half * 32 + c4 * 4 + e;
            const bool low = s <= t && t < len;
            // e^{g_t - g_s} = 2^{(g_t - g_s) log2 e}, g_t <= g_s (hardware 2^x: relative error ~2^-22)
            const float dec = low ? tc::ex2_approx((gt - gsh[i][s]) * 1.4426950408889634f) : 0.f;
            av[e] = (low && s < t) ? bt * dec * __uint_as_float(kk[c4 * 4 + e]) : 0.f;
            pv[e] = low ? dec * __uint_as_float(qk[c4 * 4 + e]) : 0.f;
            *reinterpret_cast<float*>(Ai + at_off(s, t)) = av[e];  // A[t][s] into row s of A^T
          }
          if (valid)  // four consecutive s: one half of a 16-byte chunk of P's swizzled row
            *reinterpret_cast<uint2*>(Pi + gdnws::sw128_off(t, half * 32 + c4 * 4, 64)) =
                make_uint2(tc::pack_bf16x2(pv[0], pv[1]), tc::pack_bf16x2(pv[2], pv[3]));
        }
      }
    }
    tc::named_sync(1, 128);
    // column j = t of T = (I + A)^{-1} by forward substitution, x_u = [u == j] - sum_{s<u} A_us x_s, in the
    // right-looking order: when x_s is final it is added into every later row at once (pairs of rows in
    // fp32x2), so the updates of a step are independent and only x_{s+1} waits on x_s.  The sums run over s
    // in increasing order, as in the plain recurrence.  A warp whose columns all lie at or past 32 starts
    // at s = 32 (its x_s is zero before: T is lower triangular).
    float x[64];
    {
      const uint8_t* Ai = smem + kOffA + i * 16384;
      uint64_t xp[32];  // x as pairs (x_{2k}, x_{2k+1}): partial sums until final
#pragma unroll
      for (int k = 0; k < 32; ++k) xp[k] = 0ull;
      const int s_lo = (t & 32) ? 32 : 0;  // warp-uniform: columns 32..63 are one warp of the head
#pragma unroll
      for (int s = 0; s < 64; ++s) {
        if (s < s_lo) continue;
        float lo, hi;
        tc::f2_unpack(xp[s >> 1], lo, hi);
        float xs;
        if ((s & 1) == 0) {
          lo = (s == t ? 1.f : 0.f) - lo;
          xs = lo;
          hi = fmaf(*reinterpret_cast<const float*>(Ai + at_off(s, s + 1)), xs, hi);  // row s + 1
        } else {
          hi = (s == t ? 1.f : 0.f) - hi;
          xs = hi;
        }
        xp[s >> 1] = tc::f2_pack(lo, hi);
        const uint64_t xs2 = tc::f2_pack(xs, xs);
        // rows 2k, 2k+1 for k >= k0, read four at a time from row s of A^T
        const int k0 = (s + 2) >> 1;
#pragma unroll
        for (int m = k0 >> 1; m < 16; ++m) {
          const float4 a4 = *reinterpret_cast<const float4*>(Ai + at_off(s, 4 * m));
          if (2 * m >= k0) xp[2 * m] = tc::f2_fma(tc::f2_pack(a4.x, a4.y), xs2, xp[2 * m]);
          xp[2 * m + 1] = tc::f2_fma(tc::f2_pack(a4.z, a4.w), xs2, xp[2 * m + 1]);
        }
      }
#pragma unroll
      for (int k = 0; k < 32; ++k) tc::f2_unpack(xp[k], x[2 * k], x[2 * k + 1]);
    }
    tc::named_sync(1, 128);  // A is read by every thread before the T operands overwrite it
    // row j of T diag(beta e^g) for W, then (once the W products are done) of T diag(beta) for Ut
    uint8_t* bt_i = smem + kOffT + i * 16384;
    write_t_operand(bt_i, t, x, t < len ? bt * expf(gt) : 0.f);
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    tc::mbar_arrive(&bar_b1);
    ok = ok && __all_sync(~0u, tc::mbar_wait(&bar_w1, 0, kWaitCycles));
    if (ok) {
      tc::fence_after_sync();
      write_t_operand(bt_i, t, x, bt);
    }
    tc::fence_proxy_async_smem();
    tc::fence_before_sync();
    tc::mbar_arrive(&bar_b2);
    ok = ok && __all_sync(~0u, tc::mbar_wait(&bar_w2, 0, kWaitCycles)) &&
         __all_sync(~0u, tc::mbar_wait(&bar_in, 0, kWaitCycles));  // (makes the TMA-written K tile visible here)
    if (ok) {
      tc::fence_after_sync();
      // K' = diag(e^{gC-g}) K: thread r = (head i, token t) scales its row of the K tile into the V buffer
      {
        const float dk = t < len ? expf(gC - gt) : 0.f;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int rowoff = hf * 16384 + i * 8192 + t * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int off = ((c ^ (t & 7)) << 4);
            const uint4 kv = *reinterpret_cast<const uint4*>(smem + kOffK + rowoff + off);
            const uint32_t w4[4] = {kv.x, kv.y, kv.z, kv.w};
            uint32_t o4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              o4[e] = tc::pack_bf16x2(dk * __uint_as_float(w4[e] << 16), dk * __uint_as_float(w4[e] & 0xFFFF0000u));
            *reinterpret_cast<uint4*>(smem + kOffV + i * 16384 + hf * 8192 + t * 128 + off) =
                make_uint4(o4[0], o4[1], o4[2], o4[3]);
          }
        }
      }
      tc::named_sync(1, 128);  // every row of the K tile is read before the Ut images overwrite it
      // thread r = row r of W^T and Ut^T: its 64 tokens as one swizzled 128-byte row of each image
      // (W images in the Q buffer, Ut images in the K buffer; every MMA is done with both)
      const int kd = r;
#pragma unroll
      for (int i2 = 0; i2 < 2; ++i2) {
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          uint8_t* stg = smem + (which == 0 ? kOffQ : kOffK) + i2 * 16384;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t v[32];
            tc::tmem_ld32(tmem + lb + (which == 0 ? kTW : kTU) + 64 * i2 + 32 * half, v);
            tc::tmem_wait_ld();
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              uint4 u;
              u.x = tc::pack_bf16x2(__uint_as_float(v[c4 * 8 + 0]), __uint_as_float(v[c4 * 8 + 1]));
              u.y = tc::pack_bf16x2(__uint_as_float(v[c4 * 8 + 2]), __uint_as_float(v[c4 * 8 + 3]));
              u.z = tc::pack_bf16x2(__uint_as_float(v[c4 * 8 + 4]), __uint_as_float(v[c4 * 8 + 5]));
              u.w = tc::pack_bf16x2(__uint_as_float(v[c4 * 8 + 6]), __uint_as_float(v[c4 * 8 + 7]));
              *reinterpret_cast<uint4*>(stg + gdnws::sw128_off(kd, half * 32 + c4 * 8, 128)) = u;
            }
          }
        }
      }
      tc::fence_proxy_async_smem();
      tc::named_sync(1, 128);
      if (r == 0) {
        for (int i2 = 0; i2 < 2; ++i2) {
          if (2 * hp + i2 >= p.H) continue;
          uint8_t* dst = p.ws + ((size_t)c * p.H + 2 * hp + i2) * gdnws::kBytes;
          tc::bulk_store(dst + gdnws::kW, smem + kOffQ + i2 * 16384, 16384);
          tc::bulk_store(dst + gdnws::kU, smem + kOffK + i2 * 16384, 16384);
          tc::bulk_store(dst + gdnws::kK, smem + kOffV + i2 * 16384, 16384);
        }
        tc::bulk_commit();
        tc::bulk_wait_read_all();  // the images may be overwritten once read; the writes finish on their own
      }
    } else {
      hsd::set_status(p.status, HS_DEV_TIMEOUT);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 4) tc::tmem_dealloc(tmem, 256);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)ptr;
  }
  return fn;
}

bool map_rows(CUtensorMap* m, const void* base, int H, long long T) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
  cuuint32_t box[3] = {64, 1, 64};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Chunk-local pass of every chunk and head into the compact workspace.
hs_status hs_gdn_prep_tc_launch(const hs_round_caps* caps, const int32_t* meta, int H, const void* q, const void* k,
                                const void* v, const float* alpha, const float* beta, uint8_t* ws, int32_t* status,
                                cudaStream_t st) {
  if (caps->max_chunks <= 0) return HS_OK;
  CUtensorMap mq, mk, mv;
  if (!map_rows(&mq, q, H, caps->max_tokens) || !map_rows(&mk, k, H, caps->max_tokens) ||
      !map_rows(&mv, v, H, caps->max_tokens))
    return hs::fail(HS_ECUDA, "gdn: tensor map encoding failed");
  static std::atomic<bool> configured[hsd::kMaxDevices];  // zero-initialised: per device
  const int slot = hsd::device_slot();
  if (slot < 0) return hs::fail(HS_ECUDA, "gdn_chunk_prep_tc: no usable CUDA device");
  if (!configured[slot].load()) {
    if (cudaFuncSetAttribute(gdn_chunk_prep_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem + 1024) !=
            cudaSuccess ||
        // two CTAs per SM: every SM configured for all of its shared memory
        cudaFuncSetAttribute(gdn_chunk_prep_tc_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
      return hs::fail(HS_ECUDA, "gdn_chunk_prep_tc: cannot raise the shared-memory limit");
    configured[slot].store(true);
  }
  Prm prm{meta, H, alpha, beta, ws, status};
  hsd::launch_pdl(gdn_chunk_prep_tc_kernel, dim3(caps->max_chunks, (H + 1) / 2), dim3(kThreads), kSmem + 1024, st, mq,
                  mk, mv, prm);
  HS_LAUNCH_CHECK("gdn_chunk_prep_tc");
  return HS_OK;
}
