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
// (C = last token).  The results go to the compact workspace that the
// tensor-core state pass reads (layout in gdn_ws.h).
//
// Persistent: two CTAs share an SM (96 KB of shared memory and 256
// tensor-memory columns each), and each walks the (chunk, head) items
// blockIdx.x, + gridDim.x, ... -- the barriers' phases follow the items it
// has taken and the tensor memory is allocated once.  The next item's K, Q
// and V are loaded as soon as the last MMA that reads this item's tiles has
// completed (its K' stores have read the Q rows before the T operands are
// released), so the load runs under this item's images.
//   warp 8      TMA of K, Q, V, tensor-memory allocation, and the MMAs from
//               the converged warp: [K; Q] K^T as one M = 128 product (rows
//               0..63 give K K^T, rows 64..127 Q K^T), then
//               W^T = K^T (T diag(beta e^g))^T and Ut^T = V^T (T diag(beta))^T
//               back to back, with K and V read as MN-major A
//               operands straight from their TMA tiles and T split into a
//               bf16 high and low part.
//   warps 0..7  rows of A (tensor-memory lanes 0..63) and of P (lanes
//               64..127, straight to the workspace), warps w and w + 4
//               taking the two halves of a row; then warps 0..3 solve for T
//               (below) while warps 4..7 form K' in the dead Q rows; then all
//               eight write the T operands and the W^T / Ut^T images out of
//               tensor memory.
//
// T = (I + A)^{-1} by recursive doubling (A is strictly lower triangular):
// the four 16 x 16 diagonal blocks by forward substitution (one thread per
// column), then the 32 x 32 diagonal blocks, [[T_0, 0], [-T_1 A_10 T_0, T_1]],
// then the whole, the same formula one level up; each product is spread over
// all four solver warps.  The serial part is 16 dependent rows instead of 64.
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
constexpr int kThreads = 288;  // warps 0..7 rows / solve / images, warp 8 copies and MMAs
constexpr int kWarpCtl = 8;
constexpr long long kWaitCycles = 4000000000LL;
// Shared memory (from a 1024-aligned base).
//   KQ: two [128][64] bf16 slabs (slab h = columns 64h.. of d): rows 0..63 the chunk's K, rows 64..127 its Q
//       (K' is formed over the Q rows once Q K^T is done)
//   V:  two [64][64] slabs
//   A:  fp32 [64][64], 16-byte pieces of row t swizzled by t % 16; later the T operand of Ut
//   Tt: T transposed (row c = column c of T), same layout; later the Ut^T image
//   B:  the T operand of W (high part, low part: [64 s][64 u] bf16 each), later the W^T image; during
//       the solve its scratch: the X blocks of the first merge, row-major copies of the diagonal blocks
//       (rows of 20 floats), the lower-right 32 x 32 block of T row-major (rows of 36), and the X of the
//       second merge (rows of 36, over the first two)
constexpr int kOffKQ = 0, kOffV = 32768, kOffA = 49152, kOffT = 65536, kOffB = 81920;
constexpr int kOffXS = kOffB, kOffTD = kOffB + 2560, kOffT1 = kOffB + 7680, kOffX2 = kOffB;
constexpr int kTD = 20, kT1 = 36;  // row strides (floats) of the padded scratch
constexpr int kSmem = 98304;
constexpr uint32_t kTxKQ = 32768, kTxV = 16384;
// tensor-memory columns (256): [K; Q] K^T, then W^T and Ut^T
constexpr uint32_t kTKQ = 0, kTW = 64, kTU = 128;

constexpr uint32_t kIdescKQ = tc::idesc_bf16(128, 64, 0, 0);  // A, B K-major
constexpr uint32_t kIdescWU = tc::idesc_bf16(128, 64, 1, 1);  // A, B MN-major

struct Prm {
  const int32_t* meta;
  int H;
  const float* alpha;
  const float* beta;
  uint8_t* ws;
  int32_t* status;
};

// byte offset of fp32 element (row, col) of a [64][64] matrix whose 16-byte pieces are swizzled by row % 16
__device__ __forceinline__ uint32_t f32_off(int row, int col) {
  return (uint32_t)(row * 256 + ((((col >> 2) ^ (row & 15))) << 4) + (col & 3) * 4);
}
// four consecutive fp32 of such a matrix at shared address `base` (col4 = the first of them)
__device__ __forceinline__ float4 ld4(uint32_t base, int row, int col4) { return tc::lds_f4(base + f32_off(row, col4)); }
__device__ __forceinline__ void fma4(float (&acc)[4], float a, const float4& b) {
  acc[0] = fmaf(a, b.x, acc[0]);
  acc[1] = fmaf(a, b.y, acc[1]);
  acc[2] = fmaf(a, b.z, acc[2]);
  acc[3] = fmaf(a, b.w, acc[3]);
}
__device__ __forceinline__ float dot4(const float4& a, const float4& b, float acc) {
  return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, fmaf(a.x, b.x, acc))));
}

// No minimum-blocks hint: two CTAs per SM are set by the shared memory and the tensor-memory columns.
__global__ void __launch_bounds__(kThreads, 2)
gdn_chunk_prep_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const Prm p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_kq, bar_v, bar_d, bar_b1, bar_w1, bar_w2;
  __shared__ uint32_t tmem_slot;
  __shared__ float gsh[64], bsh[64], gpart;
  // aligned up to 1024 bytes by pointer arithmetic on the shared array, so every access through smem stays
  // a shared-memory access (an integer round trip would turn them into generic loads and stores)
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);

  Meta M{p.meta};
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    tc::mbar_init(&bar_kq, 1);
    tc::mbar_init(&bar_v, 1);
    tc::mbar_init(&bar_d, 1);
    tc::mbar_init(&bar_b1, 256);
    tc::mbar_init(&bar_w1, 1);
    tc::mbar_init(&bar_w2, 1);
    tc::fence_mbar_init();
  }
  if (warp == kWarpCtl) {
    tc::tmem_alloc(&tmem_slot, 256);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  // (launched with launch_pdl) Everything above reads only the round's metadata, which host copies write;
  // inputs, workspace and state written by the earlier kernels in the stream are touched only after the
  // wait.  The next kernel may start launching only now, once every block of this one holds its tensor
  // memory: a block of the next kernel that took the columns first, then waited here for this kernel, would
  // block this kernel's allocation for good.
  hsd::pdl_trigger();
  hsd::pdl_wait();
  const int n_items = M.h(H_N_CHUNK) * p.H;
  // K, Q, V of item wi into the tiles, completing the next phase of bar_kq / bar_v (lane 0 of the copy warp)
  auto load_item = [&](int wi) {
    const int hq = wi % p.H, r0 = M.chunk(wi / p.H)[C_ROW0];
    tc::mbar_expect_tx(&bar_kq, kTxKQ);
    for (int h = 0; h < 2; ++h) {
      tc::tma_load_3d(smem + kOffKQ + h * 16384, &tm_k, h * 64, hq, r0, &bar_kq);
      tc::tma_load_3d(smem + kOffKQ + h * 16384 + 8192, &tm_q, h * 64, hq, r0, &bar_kq);
    }
    tc::mbar_expect_tx(&bar_v, kTxV);
    for (int h = 0; h < 2; ++h) tc::tma_load_3d(smem + kOffV + h * 8192, &tm_v, h * 64, hq, r0, &bar_v);
  };
  bool ahead = false;  // (copy warp) the next item's loads are in flight
  int it = 0;          // items taken by this CTA: the phases of its barriers
  for (int w = (int)blockIdx.x; w < n_items; w += (int)gridDim.x, ++it) {
  const int c = w / p.H, hh = w % p.H;
  const int32_t* ch = M.chunk(c);
  const int row0 = ch[C_ROW0], len = ch[C_LEN];
  const uint32_t ph = (uint32_t)it & 1u;
  bool item_ok = true;

  if (warp == kWarpCtl) {
    // ------------------------------------------------------- copies and MMAs
    // (copies from lane 0; the MMAs from the converged warp: voted waits, one elected lane issues; the
    // first item's tiles are loaded here, every later one's by the item before)
    if (it == 0 && lane == 0) load_item(w);
    __syncwarp();
    bool ok = __all_sync(~0u, tc::mbar_wait(&bar_kq, ph, kWaitCycles));
    int issued = 0;  // MMA groups committed: [K; Q] K^T, W^T, Ut^T
    if (ok) {
      tc::fence_after_sync();
      const uint64_t dkq = tc::sdesc_sw128(tc::smem_u32(smem + kOffKQ), 16, 1024);
#pragma unroll
      for (int k = 0; k < 8; ++k) {  // [K; Q] K^T over d (16 per step): B = the K rows of the same slabs
        const uint64_t off = (uint64_t)(((k >> 2) * 16384 + (k & 3) * 32) >> 4);
        tc::mma_bf16_ss_w(tmem + kTKQ, dkq + off, dkq + off, kIdescKQ, k > 0 ? 1u : 0u);
      }
      tc::mma_commit_w(&bar_d);
      issued = 1;
    }
    // W^T from the K rows and Ut^T from V, back to back once both T operands are written
    if (ok) ok = __all_sync(~0u, tc::mbar_wait(&bar_b1, ph, kWaitCycles)) &&
                 __all_sync(~0u, tc::mbar_wait(&bar_v, ph, kWaitCycles));
    for (int pass = 0; pass < 2 && ok; ++pass) {
      if (pass == 0) tc::fence_after_sync();
      const uint64_t da = pass == 0 ? tc::sdesc_sw128(tc::smem_u32(smem + kOffKQ), 16384, 1024)
                                    : tc::sdesc_sw128(tc::smem_u32(smem + kOffV), 8192, 1024);
      const uint64_t db = tc::sdesc_sw128(tc::smem_u32(smem + (pass == 0 ? kOffB : kOffA)), 8192, 1024);
#pragma unroll
      for (int part = 0; part < 2; ++part) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // over the chunk's tokens s, 16 per step
          tc::mma_bf16_ss_w(tmem + (pass == 0 ? kTW : kTU), da + (uint64_t)((k * 2048) >> 4),
                            db + (uint64_t)((part * 8192 + k * 2048) >> 4), kIdescWU, (part > 0 || k > 0) ? 1u : 0u);
        }
      }
      tc::mma_commit_w(pass == 0 ? &bar_w1 : &bar_w2);
      issued = 2 + pass;
    }
    if (!ok && lane == 0) hsd::set_status(p.status, HS_DEV_TIMEOUT);
    // drain: every copy into this CTA's shared memory has landed and every MMA issued has completed
    // before the block may exit (bounded as every wait)
    if (lane == 0) {
      tc::mbar_wait(&bar_kq, ph, kWaitCycles);
      tc::mbar_wait(&bar_v, ph, kWaitCycles);
    }
    uint64_t* last = issued == 3 ? &bar_w2 : issued == 2 ? &bar_w1 : issued == 1 ? &bar_d : nullptr;
    if (last) ok = __all_sync(~0u, tc::mbar_wait(last, ph, kWaitCycles)) && ok;
    // the MMAs that read K, V and the K rows are complete, both phases of the tiles' barriers are seen, and
    // the K' stores have read the Q rows (before bar_b1): the next item's tiles may be loaded
    ahead = ok && w + (int)gridDim.x < n_items;
    if (ahead && lane == 0) load_item(w + (int)gridDim.x);
    __syncwarp();
    item_ok = ok;
  } else {
    // -------------------------------------------------------------- rows
    // (shared memory through explicit ld/st.shared on 32-bit addresses: sb = the aligned base)
    const uint32_t sb = tc::smem_u32(smem);
    const int r = threadIdx.x;                     // 0..255
    const int lg = warp & 3, half = warp >> 2;     // TMEM lane group (lanes 32 lg ..), half of the columns
    const int row = 32 * lg + lane;                // this thread's TMEM lane
    const uint32_t lb = (uint32_t)(32 * lg) << 16;
    uint8_t* wsi = p.ws + ((size_t)c * p.H + hh) * gdnws::kBytes;
    // decays: g = inclusive cumulative sum of log alpha over the chunk (a warp scan per 32 tokens)
    if (r < 64) {
      const size_t a = (size_t)(row0 + r) * p.H + hh;
      float gl = r < len ? logf(p.alpha[a]) : 0.f;
      const float b = r < len ? p.beta[a] : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float v = __shfl_up_sync(~0u, gl, o);
        if (lane >= o) gl += v;
      }
      if (r == 31) gpart = gl;
      gsh[r] = gl;
      bsh[r] = b;
    }
    tc::named_sync(1, 256);
    if (r >= 32 && r < 64) gsh[r] += gpart;
    tc::named_sync(1, 256);
    const float gC = gsh[len - 1];
    if (r < 64) {
      float* gd = reinterpret_cast<float*>(wsi + gdnws::kG);
      const float gt = gsh[r];
      gd[r] = r < len ? expf(gt) : 0.f;
      gd[64 + r] = r < len ? expf(gC - gt) : 0.f;
      if (r == 0) gd[128] = expf(gC);
    }
    bool ok = __all_sync(~0u, tc::mbar_wait(&bar_d, ph, kWaitCycles));
    if (ok) {
      // half a row of A (lanes 0..63, fp32, swizzled, in shared memory) or of P (lanes 64..127, bf16, its
      // swizzled 128-byte row of the workspace image)
      tc::fence_after_sync();
      uint32_t d[32];
      tc::tmem_ld32(tmem + lb + kTKQ + 32 * half, d);
      tc::tmem_wait_ld();
      const int t = row & 63;
      const float gt = gsh[t], bt = bsh[t];
      const bool live = t < len;
      if (row < 64) {
#pragma unroll
        for (int s4 = 0; s4 < 8; ++s4) {
          float av[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int s = 32 * half + 4 * s4 + e;
            // e^{g_t - g_s} = 2^{(g_t - g_s) log2 e}, g_t <= g_s (hardware 2^x: relative error ~2^-22)
            av[e] = (live && s < t) ? bt * tc::ex2_approx((gt - gsh[s]) * 1.4426950408889634f) *
                                          __uint_as_float(d[4 * s4 + e])
                                    : 0.f;
          }
          tc::sts_f4(sb + kOffA + f32_off(t, 32 * half + 4 * s4), make_float4(av[0], av[1], av[2], av[3]));
        }
      } else {
        uint8_t* Pi = wsi + gdnws::kP + t * 128;
#pragma unroll
        for (int s8 = 0; s8 < 4; ++s8) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float pv[2];
#pragma unroll
            for (int f = 0; f < 2; ++f) {
              const int s = 32 * half + 8 * s8 + 2 * e + f;
              pv[f] = (live && s <= t) ? tc::ex2_approx((gt - gsh[s]) * 1.4426950408889634f) *
                                             __uint_as_float(d[8 * s8 + 2 * e + f])
                                       : 0.f;
            }
            pk[e] = tc::pack_bf16x2(pv[0], pv[1]);
          }
          *reinterpret_cast<uint4*>(Pi + (((4 * half + s8) ^ (t & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
    }
    tc::named_sync(1, 256);  // A complete
    if (warp < 4) {
      // ================================ T = (I + A)^{-1} (warps 0..3, barrier 2)
      const uint32_t Tt = sb + kOffT, A = sb + kOffA, T1 = sb + kOffT1;
      if (r < 64) {
        // diagonal 16 x 16 blocks: column cc of T_II by forward substitution, x_rr = [rr == cc] - sum_s A_rr,s x_s
        const int I = r >> 4, cc = r & 15;
        float4 arow[16][4];  // the block's rows of A (strictly lower: only pieces left of the diagonal)
#pragma unroll
        for (int rr = 1; rr < 16; ++rr)
#pragma unroll
          for (int s4 = 0; s4 < 4; ++s4)
            if (4 * s4 < rr) arow[rr][s4] = ld4(A, 16 * I + rr, 16 * I + 4 * s4);
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = 0.f;
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
          float acc[4] = {rr == cc ? 1.f : 0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int s4 = 0; s4 < 4; ++s4) {
            if (4 * s4 >= rr) break;
            const float4 a = arow[rr][s4];
            acc[0] = fmaf(-a.x, x[4 * s4], acc[0]);
            acc[1] = fmaf(-a.y, x[4 * s4 + 1], acc[1]);
            acc[2] = fmaf(-a.z, x[4 * s4 + 2], acc[2]);
            acc[3] = fmaf(-a.w, x[4 * s4 + 3], acc[3]);
          }
          x[rr] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)  // column cc of T_II = row 16 I + cc of Tt
          tc::sts_f4(Tt + f32_off(16 * I + cc, 16 * I + 4 * j), make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]));
        const uint32_t td = sb + kOffTD + I * 16 * kTD * 4;
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) tc::sts_f1(td + (rr * kTD + cc) * 4, x[rr]);
        if (I >= 2) {
#pragma unroll
          for (int rr = 0; rr < 16; ++rr) tc::sts_f1(T1 + ((16 * (I - 2) + rr) * kT1 + 16 * (I - 2) + cc) * 4, x[rr]);
        }
      } else {
        // zeros above the diagonal: rows 16 J + c (J >= 1) of Tt, columns [0, 16 J) (96 pieces per c), and
        // the upper-right 16 x 16 block of T1
        for (int i = r - 64; i < 16 * 24; i += 64) {
          const int cc = i / 24, q = i % 24;
          const int J = q < 4 ? 1 : q < 12 ? 2 : 3;
          const int piece = q < 4 ? q : q < 12 ? q - 4 : q - 12;
          tc::sts_f4(Tt + f32_off(16 * J + cc, 4 * piece), make_float4(0.f, 0.f, 0.f, 0.f));
        }
        const int rr = (r - 64) >> 2, c4 = (r - 64) & 3;
        tc::sts_f4(T1 + (rr * kT1 + 16 + 4 * c4) * 4, make_float4(0.f, 0.f, 0.f, 0.f));
      }
      tc::named_sync(2, 128);
      // first merge, blocks P = 0 (rows/columns 0..31) and P = 1 (32..63): T_hi,lo = -T_hi,hi A_hi,lo T_lo,lo.
      // Thread = (row rr, columns 4 cq ..): a warp's lanes cover 16 rows and two column groups, so a load
      // of T is a broadcast and the rows of A fall in different banks.
      {
        const int P = r >> 6, lo = 2 * P, hi = 2 * P + 1, q = r & 63, rr = q & 15, cq = q >> 4;
        float4 a[4], tt[4][4];
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) a[s4] = ld4(A, 16 * hi + rr, 16 * lo + 4 * s4);
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int s4 = 0; s4 < 4; ++s4) tt[j][s4] = ld4(Tt, 16 * lo + 4 * cq + j, 16 * lo + 4 * s4);
        float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4)
#pragma unroll
          for (int j = 0; j < 4; ++j) x[j] = dot4(a[s4], tt[j][s4], x[j]);
        const uint32_t xs = sb + kOffXS + P * 16 * kTD * 4;
        tc::sts_f4(xs + (rr * kTD + 4 * cq) * 4, make_float4(x[0], x[1], x[2], x[3]));
        tc::named_sync(2, 128);
        const uint32_t td = sb + kOffTD + hi * 16 * kTD * 4;
        float4 dd[4], xv[16];
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) dd[s4] = tc::lds_f4(td + (rr * kTD + 4 * s4) * 4);
#pragma unroll
        for (int sr = 0; sr < 16; ++sr) xv[sr] = tc::lds_f4(xs + (sr * kTD + 4 * cq) * 4);
        float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) {
          fma4(y, dd[s4].x, xv[4 * s4]);
          fma4(y, dd[s4].y, xv[4 * s4 + 1]);
          fma4(y, dd[s4].z, xv[4 * s4 + 2]);
          fma4(y, dd[s4].w, xv[4 * s4 + 3]);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) tc::sts_f1(Tt + f32_off(16 * lo + 4 * cq + j, 16 * hi + rr), -y[j]);
        if (P == 1) tc::sts_f4(T1 + ((16 + rr) * kT1 + 4 * cq) * 4, make_float4(-y[0], -y[1], -y[2], -y[3]));
      }
    } else {
      // ================================ K' = diag(e^{g_C - g}) K over the Q rows (warps 4..7, barrier 3)
      // thread = (row t, slab h); the row's eight 16-byte pieces in an order rotated by the row, so the
      // lanes of a warp touch different banks
      ok = ok && __all_sync(~0u, tc::mbar_wait(&bar_kq, ph, kWaitCycles));  // (makes the TMA-written tile visible)
      if (ok) {
        const int t = (r - 128) & 63, h = (r - 128) >> 6;
        const float dk = t < len ? expf(gC - gsh[t]) : 0.f;
        const uint32_t src = sb + kOffKQ + h * 16384 + t * 128;
        const uint32_t dst = src + 8192;  // row 64 + t: the same swizzle phase
        uint4 kv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) kv[i] = tc::lds_u4(src + ((i ^ (t & 7)) << 4));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t w4[4] = {kv[i].x, kv[i].y, kv[i].z, kv[i].w};
          uint32_t o4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            o4[e] = tc::pack_bf16x2(dk * __uint_as_float(w4[e] << 16), dk * __uint_as_float(w4[e] & 0xFFFF0000u));
          tc::sts_u4(dst + ((i ^ (t & 7)) << 4), make_uint4(o4[0], o4[1], o4[2], o4[3]));
        }
      }
      tc::fence_proxy_async_smem();
      tc::named_sync(3, 128);
      if (r == 128 && ok) {
        for (int h = 0; h < 2; ++h)
          tc::bulk_store(wsi + gdnws::kK + h * 8192, smem + kOffKQ + h * 16384 + 8192, 8192);
        tc::bulk_commit();
      }
    }
    tc::named_sync(1, 256);  // T[0:32, 0:32], T1 complete; K' written
    // second merge, all eight warps: T[32:64, 0:32] = -T1 A[32:64, 0:32] T[0:32, 0:32].  Thread = (row rr,
    // columns 4 cg ..): every lane of a warp reads the same row of Tt (a broadcast), the 32 rows of A
    // fall in different banks.
    {
      const uint32_t Tt = sb + kOffT, A = sb + kOffA, T1 = sb + kOffT1, x2 = sb + kOffX2;
      const int rr = r & 31, cg = r >> 5;
      float x[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s8 = 0; s8 < 4; ++s8) {  // eight columns s at a time: 2 + 8 loads, then 32 FMAs
        float4 a[2], tt[4][2];
#pragma unroll
        for (int i = 0; i < 2; ++i) a[i] = ld4(A, 32 + rr, 8 * s8 + 4 * i);
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
          for (int i = 0; i < 2; ++i) tt[j][i] = ld4(Tt, 4 * cg + j, 8 * s8 + 4 * i);  // T[s][c] = Tt[c][s]
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = dot4(a[1], tt[j][1], dot4(a[0], tt[j][0], x[j]));
      }
      tc::sts_f4(x2 + (rr * kT1 + 4 * cg) * 4, make_float4(x[0], x[1], x[2], x[3]));
      tc::named_sync(1, 256);
      float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s8 = 0; s8 < 4; ++s8) {  // eight rows s of X at a time
        const float4 d0 = tc::lds_f4(T1 + (rr * kT1 + 8 * s8) * 4), d1 = tc::lds_f4(T1 + (rr * kT1 + 8 * s8 + 4) * 4);
        float4 xv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) xv[e] = tc::lds_f4(x2 + ((8 * s8 + e) * kT1 + 4 * cg) * 4);
        const float dv[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) fma4(y, dv[e], xv[e]);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) tc::sts_f1(Tt + f32_off(4 * cg + j, 32 + rr), -y[j]);
    }
    tc::named_sync(1, 256);  // T complete
    // ---- the T operands: row s of B = column s of T scaled by beta_s e^{g_s} (for W, in the B region) and by
    // beta_s (for Ut, over A); thread = (s, quarter of u); high and low parts
    {
      const int s = r >> 2, qq = r & 3;
      const float scw = s < len ? bsh[s] * expf(gsh[s]) : 0.f, scu = bsh[s];
      float4 v4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v4[i] = ld4(sb + kOffT, s, 16 * qq + 4 * i);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int c8 = 2 * qq + i;
        const float v[8] = {v4[2 * i].x, v4[2 * i].y, v4[2 * i].z, v4[2 * i].w,
                            v4[2 * i + 1].x, v4[2 * i + 1].y, v4[2 * i + 1].z, v4[2 * i + 1].w};
        const uint32_t off = s * 128 + ((c8 ^ (s & 7)) << 4);
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const float sc = w == 0 ? scw : scu;
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a = v[2 * e] * sc, b = v[2 * e + 1] * sc;
            hi[e] = tc::pack_bf16x2(a, b);
            lo[e] = tc::pack_bf16x2(a - __uint_as_float(hi[e] << 16), b - __uint_as_float(hi[e] & 0xFFFF0000u));
          }
          const uint32_t base = sb + (w == 0 ? kOffB : kOffA);
          tc::sts_u4(base + off, make_uint4(hi[0], hi[1], hi[2], hi[3]));
          tc::sts_u4(base + 8192 + off, make_uint4(lo[0], lo[1], lo[2], lo[3]));
        }
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
    }
    // ---- half a row of a product out of tensor memory (lane = row k of W^T or Ut^T) into its swizzled
    // 128-byte image row
    auto image_out = [&](uint32_t col, int off_img) {
      uint32_t v[32];
      tc::tmem_ld32(tmem + lb + col + 32 * half, v);
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t* w = v + 8 * j;
        uint4 u;
        u.x = tc::pack_bf16x2(__uint_as_float(w[0]), __uint_as_float(w[1]));
        u.y = tc::pack_bf16x2(__uint_as_float(w[2]), __uint_as_float(w[3]));
        u.z = tc::pack_bf16x2(__uint_as_float(w[4]), __uint_as_float(w[5]));
        u.w = tc::pack_bf16x2(__uint_as_float(w[6]), __uint_as_float(w[7]));
        tc::sts_u4(sb + off_img + row * 128 + (((4 * half + j) ^ (row & 7)) << 4), u);
      }
      tc::fence_proxy_async_smem();
    };
    if (r == 128) tc::bulk_wait_read_all();  // the K' stores have read the Q rows: they are the next item's
    tc::mbar_arrive(&bar_b1);
    ok = ok && __all_sync(~0u, tc::mbar_wait(&bar_w1, ph, kWaitCycles));
    if (ok) {
      tc::fence_after_sync();
      image_out(kTW, kOffB);  // W^T image over its (read) operand
    }
    tc::named_sync(1, 256);
    if (r == 0 && ok) {
      tc::bulk_store(wsi + gdnws::kW, smem + kOffB, 16384);
      tc::bulk_commit();
    }
    ok = ok && __all_sync(~0u, tc::mbar_wait(&bar_w2, ph, kWaitCycles));
    if (ok) {
      tc::fence_after_sync();
      image_out(kTU, kOffT);  // Ut^T image over Tt
    }
    tc::named_sync(1, 256);
    if (r == 0) {
      if (ok) {
        tc::bulk_store(wsi + gdnws::kU, smem + kOffT, 16384);
        tc::bulk_commit();
      }
      tc::bulk_wait_read_all();  // the images may be released once read; the writes finish on their own
    }
    if (!ok && lane == 0) hsd::set_status(p.status, HS_DEV_TIMEOUT);
    item_ok = ok;
  }
  // every MMA of the item is complete and its bulk stores have read shared memory (a wait that ran out
  // anywhere stops every thread here, once the copies already issued for the next item have landed)
  tc::fence_before_sync();
  const bool stop = __syncthreads_or(!item_ok);
  tc::fence_after_sync();
  if (stop) {
    if (warp == kWarpCtl && lane == 0 && ahead) {
      tc::mbar_wait(&bar_kq, ph ^ 1u, kWaitCycles);
      tc::mbar_wait(&bar_v, ph ^ 1u, kWaitCycles);
    }
    break;
  }
  }
  if (warp == kWarpCtl) tc::tmem_dealloc(tmem, 256);
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
  static std::atomic<int> sm_count[hsd::kMaxDevices];  // per device, 0 until read
  int n_sm = sm_count[slot].load();
  if (n_sm <= 0) {
    if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, slot) != cudaSuccess || n_sm <= 0)
      return hs::fail(HS_ECUDA, "gdn_chunk_prep_tc: cannot read the SM count");
    sm_count[slot].store(n_sm);
  }
  const long long items = (long long)caps->max_chunks * H;
  const int grid = (int)(items < 2LL * n_sm ? items : 2LL * n_sm);  // persistent: two CTAs per SM
  hsd::launch_pdl(gdn_chunk_prep_tc_kernel, dim3(grid), dim3(kThreads), kSmem + 1024, st, mq, mk, mv, prm);
  HS_LAUNCH_CHECK("gdn_chunk_prep_tc");
  return HS_OK;
}
