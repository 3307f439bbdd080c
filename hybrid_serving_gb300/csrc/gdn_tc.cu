// gdn_tc.cu -- Gated DeltaNet state pass on tcgen05 (bf16 inputs, d_k = d_v = 128).
//
// Flide, "Accelerating Decision Inference with Exact State Forking", section
// 3.2.2 (Eq. 4; children continue from the parent's end state by index),
// section 3.4 (checkpoint = saved end state of the first level), section 3.5
// (every node's chunks start at its first token).
//
// One CTA walks one node's chunks for one head, carrying the whole state S
// (d_v = 128 rows x d_k = 128) with d_v as the MMA M dimension.  For a chunk
// with inputs W, Ut, P and the decay factors (chunk-local pass) and Q, K (the
// stream):
//
//   D1 = S W^T            U  = Ut^T - D1         (U[j][t], j = row of S)
//   D2 = S Q^T
//   D3 = U P^T            O  = D2 diag(e^g) + D3   -> out[t][h][j]
//   D4 = U K'             S <- e^{gC} S + D4,   K' = diag(e^{gC-g}) K
//
// S lives in tensor memory twice: in fp32 as the accumulator of D4 (scaled
// by e^{gC} in place before D4 adds to it) and in bf16 as the A operand of
// D1 and D2; U is a bf16 A operand in tensor memory too, so shared memory
// holds only the chunk inputs, in a 3-stage ring.  Roles:
//
//   warp 8      producer: bulk copies of W^T, Ut^T, P, K' and the decay
//               factors from the workspace, TMA boxes of Q, up to 3 chunks
//               ahead;
//   warp 9      issues the state chain's MMAs (D1, then D4 as soon as U is
//               written), converged, from one elected lane;
//   warp 10     issues the output MMAs the same way, each in a gap of the
//               chain's: D2 once D1 is done (while the rows form U), D3 once
//               D4 is done (while the rows form the bf16 state), so that
//               they never share the tensor pipe with the chain's products;
//   warps 0..3  rows of the state (thread j = TMEM lane j = row j of S):
//               U, the scaling of S, the bf16 copy of S;
//   warps 4..7  outputs: O for chunk c (staged in the chunk's Q buffer, then
//               written out in 16-byte pieces) while the rows work on c + 1.
//
// Operands are bf16, accumulation fp32.  The four hand-offs of the state chain
// (S -> D1 -> U -> D4 -> S) poll their barriers without suspending.  Every
// wait is bounded (HS_DEV_TIMEOUT).
//
// A long node (24 chunks or more) is split into groups of consecutive chunks
// for a two-level scan of the affine chunk map S -> S M_c + N_c: a first pass
// without outputs (the output-less variant: per group its N from the zero
// state and its M from the identity with Ut = 0, two chains in one CTA; and
// the end of group 0), then every group with outputs from its start state
// S_g = (...(S_1 M_1 + N_1)...) M_{g-1} + N_{g-1}, formed on tensor cores.
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
constexpr long long kWaitCycles = 4000000000LL;

// Two variants of the state pass.  With outputs (O = true): rows, outputs, producer, chain MMA and
// output MMA warps, 3 stages of {W^T, Q, K', P, Ut^T, decay block}, all 512 TMEM columns.  Without
// (O = false; the scan's first pass): rows, producer and chain MMA warps, 3 stages of {W^T, K', Ut^T,
// decay block}, and two chains over the same chunks -- the group's N (zero start) and M (identity
// start, Ut = 0) -- in 256 TMEM columns each (U written over the columns of D1 once D1 is read); the
// two chains' steps interleave, so one's products run while the rows work on the other.
template <bool O>
struct Cfg;
template <>
struct Cfg<true> {
  static constexpr int kThreads = 352, kMinBlocks = 1;
  static constexpr int kWarpProd = 8, kWarpMma = 9, kWarpOmma = 10;
  // one stage of chunk inputs (offsets from the stage base)
  static constexpr int kStW = 0, kStQ = 16384, kStK = 32768, kStP = 49152, kStUt = 57344, kStG = 73728;
  static constexpr int kStageBytes = 74752;  // 73728 + the 1 KB decay block
  static constexpr int kStages = 3;
  static constexpr uint32_t kStageTx = 16384 * 4 + 8192 + 1024;
  // tensor-memory columns
  static constexpr uint32_t kTS32 = 0;    // S fp32 [128][128]
  static constexpr uint32_t kTS16 = 128;  // S bf16, two per column (64)
  static constexpr uint32_t kTU = 192;    // U bf16 (32)
  static constexpr uint32_t kTSlo = 192;  // S bf16 low part (64), only while a later group forms its start state
  static constexpr uint32_t kTD1 = 256, kTD2 = 320, kTD3 = 384;  // fp32 [128][64] each
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kEmptyCount = 2 + 8;  // two MMA commits + one arrival per row and output warp
};
template <>
struct Cfg<false> {
  static constexpr int kThreads = 192, kMinBlocks = 1;
  static constexpr int kWarpProd = 4, kWarpMma = 5, kWarpOmma = -1;
  static constexpr int kStW = 0, kStK = 16384, kStUt = 32768, kStG = 49152, kStQ = 0, kStP = 0;
  static constexpr int kStageBytes = 50176;
  static constexpr int kStages = 3;
  static constexpr uint32_t kStageTx = 16384 * 3 + 1024;
  // per chain, from its base column (256 c)
  static constexpr uint32_t kTS32 = 0, kTS16 = 128, kTD1 = 192, kTU = 192, kTD2 = 0, kTD3 = 0;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kEmptyCount = 1 + 4;  // the chain's MMA commit + one arrival per row warp
};
static_assert(Cfg<true>::kStG + (gdnws::kBytes - gdnws::kG) == Cfg<true>::kStageBytes, "stage layout");
static_assert(Cfg<false>::kStG + (gdnws::kBytes - gdnws::kG) == Cfg<false>::kStageBytes, "stage layout");
template <bool O>
constexpr int smem_bytes() { return Cfg<O>::kStages * Cfg<O>::kStageBytes; }

constexpr uint32_t kIdesc64 = tc::idesc_bf16(128, 64, 0, 0);      // D[128x64], B K-major
constexpr uint32_t kIdesc64mn = tc::idesc_bf16(128, 64, 0, 1);    // D[128x64], B N-major
constexpr uint32_t kIdesc128mn = tc::idesc_bf16(128, 128, 0, 1);  // D[128x128], B N-major

// The rows' tensor-memory round trips, two 32-column loads in flight per wait.
// bf16 copy of this lane's 128 fp32 state columns (s32) into 64 packed columns (s16).
__device__ __forceinline__ void state_to_bf16(uint32_t s32, uint32_t s16) {
#pragma unroll
  for (int q2 = 0; q2 < 2; ++q2) {
    uint32_t f[2][32];
    tc::tmem_ld32(s32 + q2 * 64, f[0]);
    tc::tmem_ld32(s32 + q2 * 64 + 32, f[1]);
    tc::tmem_wait_ld();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t b[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) b[i] = tc::pack_bf16x2(__uint_as_float(f[h][2 * i]), __uint_as_float(f[h][2 * i + 1]));
      tc::tmem_st16(s16 + q2 * 32 + h * 16, b);
    }
  }
}
// the 128 fp32 state columns scaled by ec in place
__device__ __forceinline__ void state_scale(uint32_t s32, float ec) {
#pragma unroll
  for (int q2 = 0; q2 < 2; ++q2) {
    uint32_t f[2][32];
    tc::tmem_ld32(s32 + q2 * 64, f[0]);
    tc::tmem_ld32(s32 + q2 * 64 + 32, f[1]);
    tc::tmem_wait_ld();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int e = 0; e < 32; ++e) f[h][e] = __float_as_uint(ec * __uint_as_float(f[h][e]));
      tc::tmem_st32(s32 + q2 * 64 + h * 32, f[h]);
    }
  }
}

struct Prm {
  const int32_t* meta;
  int level, H, n_slots;
  const uint8_t* ws;
  uint8_t* scan;  // per (extra scan group, head) buffers (gdn_ws.h)
  float* state;
  __nv_bfloat16* out;
  int32_t* status;
};

// What one CTA does with its group of chunks.
enum InitKind { kInitSlot, kInitZero, kInitIdentity, kInitScan };
enum EndKind { kEndNone, kEndSlot, kEndScanS, kEndScanN, kEndScanM };

template <bool O>
__global__ void __launch_bounds__(Cfg<O>::kThreads, Cfg<O>::kMinBlocks)
gdn_chain_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const Prm p) {
  using C = Cfg<O>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_full[C::kStages], bar_empty[C::kStages], bar_s, bar_u, bar_of;
  __shared__ uint64_t bar_d1, bar_d4, bar_d2, bar_d23, bar_done, bar_done2, bar_cb[3], bar_ps, bar_pd;
  __shared__ uint64_t bar_sc[2], bar_uc[2], bar_d1c[2], bar_d4c[2];  // per chain (output-less variant)
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  // aligned up to 1024 bytes by pointer arithmetic on the shared array, so every access through smem stays
  // a shared-memory access (an integer round trip would turn them into generic loads and stores)
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);

  Meta M{p.meta};
  if (p.level >= M.h(H_N_LEVEL)) return;
  // The task.  O = false (first pass of the two-level scan): for scan entry e (node, group g >= 1), part 0 =
  // N_g (zero start) and M_g (identity start, Ut = 0) as two chains, part 2 (g = 1 only) = the end state of
  // group 0 (the node's own start).  O = true: task < cap_seg = the node's group 0 (a node without a
  // scan: all of it); past it, scan entry e = group g >= 1 from its start state S_g (formed from the end
  // of group 0 and the (M, N) of groups 1 .. g-1).  Every task with outputs writes the node's end state
  // if it holds the node's last chunk.
  const int n_lev_seg = M.level_off()[p.level + 1] - M.level_off()[p.level];
  const int scan_lo = M.scan_level_off()[p.level];
  const int n_lev_scan = M.scan_level_off()[p.level + 1] - scan_lo;
  const int cap_seg = M.h(H_CAP_SEG), cap_scan = scan_cap(M.h(H_CAP_CHUNK));
  // blockIdx.x = head, blockIdx.y = task: blocks are dispatched x fastest, so every head's copy of a task
  // is placed before the next task, and the tasks that exit at once come after the ones with work (measured:
  // with the tasks of a head contiguous, a fifth of the first pass's CTAs waited for a second wave)
  const int task = (int)blockIdx.y;
  int seg, g = 0, part = 0, e = -1;
  if (!O) {
    // task t < cap_scan: N and M of entry t's group (part 0, two chains); task cap_scan + t: the end of
    // group 0 (part 2, live for one entry per long node), so the tasks with work come first
    part = task < cap_scan ? 0 : 2;
    const int t = task < cap_scan ? task : task - cap_scan;
    if (task >= 2 * cap_scan || t >= n_lev_scan) return;
    e = scan_lo + t;
    seg = M.scan()[2 * e];
    g = M.scan()[2 * e + 1];
    if (part == 2) {
      if (g != 1) return;
      g = 0;
    }
  } else if (task < cap_seg) {
    if (task >= n_lev_seg) return;
    seg = M.level_seg()[M.level_off()[p.level] + task];
  } else {
    const int t = task - cap_seg;
    if (t >= n_lev_scan) return;
    e = scan_lo + t;
    seg = M.scan()[2 * e];
    g = M.scan()[2 * e + 1];
  }
  const int32_t* sg = M.seg(seg);
  const int h = blockIdx.x;
  const int init = sg[S_INIT_SLOT], endslot = sg[S_END_SLOT];
  if (init >= p.n_slots || endslot >= p.n_slots) {
    if (threadIdx.x == 0) hsd::set_status(p.status, HS_DEV_BAD_SLOT);
    return;
  }
  const int n_all = sg[S_N_CHUNK], G = scan_groups(n_all), e1 = sg[S_SCAN1];
  const int c_off = sg[S_CHUNK_OFF] + (int)((long long)g * n_all / G);
  const int n_c = sg[S_CHUNK_OFF] + (int)((long long)(g + 1) * n_all / G) - c_off;
  const bool outputs = O;
  const bool zero_ut = !O && part == 1;
  const InitKind ik = g == 0 ? (init >= 0 ? kInitSlot : kInitZero)
                      : O    ? kInitScan
                             : (part == 0 ? kInitZero : kInitIdentity);
  const EndKind ek = O ? (g == G - 1 && endslot >= 0 ? kEndSlot : kEndNone)
                       : (part == 2 ? kEndScanS : part == 0 ? kEndScanN : kEndScanM);
  const int n_comb = O && g >= 1 ? g - 1 : 0;  // products S <- S M_q + N_q before the chain (groups 1 .. g-1)
  auto scanbuf = [&](int entry) { return p.scan + ((size_t)entry * p.H + h) * gdnws::kScanBytes; };
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int s = 0; s < C::kStages; ++s) {
      tc::mbar_init(&bar_full[s], 1);
      tc::mbar_init(&bar_empty[s], C::kEmptyCount);
    }
    tc::mbar_init(&bar_s, 4);  // (the four row warps, one arrival each; likewise every count of 4 below)
    tc::mbar_init(&bar_u, 4);
    tc::mbar_init(&bar_of, 4);
    tc::mbar_init(&bar_d1, 1);
    for (int c = 0; c < 2; ++c) {
      tc::mbar_init(&bar_sc[c], 4);
      tc::mbar_init(&bar_uc[c], 4);
      tc::mbar_init(&bar_d1c[c], 1);
      tc::mbar_init(&bar_d4c[c], 1);
    }
    tc::mbar_init(&bar_d4, 1);
    tc::mbar_init(&bar_d2, 1);
    tc::mbar_init(&bar_d23, 1);
    tc::mbar_init(&bar_done, 1);
    tc::mbar_init(&bar_done2, 1);
    for (int b = 0; b < 3; ++b) tc::mbar_init(&bar_cb[b], 1);  // combine buffers (M or N images) filled
    tc::mbar_init(&bar_ps, 4);
    tc::mbar_init(&bar_pd, 1);
    tc::fence_mbar_init();
  }
  if (warp == C::kWarpMma) {
    tc::tmem_alloc(&tmem_slot, C::kTmemCols);
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
  auto fail = [&]() {
    hsd::set_status(p.status, HS_DEV_TIMEOUT);
    atomicExch(&abort_flag, 1);
  };
  auto stage = [&](int ci) { return smem + (ci % C::kStages) * C::kStageBytes; };

  if (warp == C::kWarpProd) {
    // ----------------------------------------------------------- producer
    if (lane == 0) {
      tc::prefetch_tmap(&tm_q);
      // the start state of a later group: the images of M_q and N_q, q = 1 .. g-1, as items 2q-2 and 2q-1
      // of a rotation through three 64 KB buffers (the stage regions), up to three items ahead; buffer b is
      // refilled once the combine that read its previous item is done (bar_pd: never two phases ahead,
      // since a later combine needs an item not yet issued)
      bool pro_ok = true;
      for (int i = 0; i < 2 * n_comb && pro_ok; ++i) {
        const int b = i % 3;
        if (i >= 3 && !tc::mbar_wait(&bar_pd, ((i - 3) / 2) & 1, kWaitCycles)) {
          pro_ok = false;
          break;
        }
        const uint8_t* src = scanbuf(e1 + i / 2) + ((i & 1) ? gdnws::kScanN : gdnws::kScanMhi);
        const uint32_t nb = (i & 1) ? 65536u : 32768u;  // N in fp32; the high part of M
        tc::mbar_expect_tx(&bar_cb[b], nb);
        tc::bulk_load(smem + b * C::kStageBytes, src, nb, &bar_cb[b]);
      }
      if (pro_ok && n_comb > 0 && !tc::mbar_wait(&bar_pd, (n_comb - 1) & 1, kWaitCycles)) pro_ok = false;
      if (!pro_ok) fail();
      int issued = 0;
      for (int ci = 0; ci < n_c && pro_ok; ++ci) {
        const int s = ci % C::kStages, n = ci / C::kStages;
        if (n >= 1 && !tc::mbar_wait(&bar_empty[s], (n - 1) & 1, kWaitCycles)) {
          fail();
          break;
        }
        if (*(volatile int*)&abort_flag) break;
        const int row0 = M.chunk(c_off + ci)[C_ROW0];
        const uint8_t* w = p.ws + ((size_t)(c_off + ci) * p.H + h) * gdnws::kBytes;
        uint8_t* sb = stage(ci);
        // a transition (Ut = 0) needs no Ut
        tc::mbar_expect_tx(&bar_full[s], C::kStageTx - (zero_ut ? 16384u : 0u));
        tc::bulk_load(sb + C::kStW, w + gdnws::kW, 16384, &bar_full[s]);
        if (!zero_ut) tc::bulk_load(sb + C::kStUt, w + gdnws::kU, 16384, &bar_full[s]);
        tc::bulk_load(sb + C::kStG, w + gdnws::kG, gdnws::kBytes - gdnws::kG, &bar_full[s]);
        tc::bulk_load(sb + C::kStK, w + gdnws::kK, 16384, &bar_full[s]);
        if (outputs) {
          for (int half = 0; half < 2; ++half)
            tc::tma_load_3d(sb + C::kStQ + half * 8192, &tm_q, half * 64, h, row0, &bar_full[s]);
          tc::bulk_load(sb + C::kStP, w + gdnws::kP, 8192, &bar_full[s]);
        }
        ++issued;
      }
      for (int ci = issued >= C::kStages ? issued - C::kStages : 0; ci < issued; ++ci)
        tc::mbar_wait(&bar_full[ci % C::kStages], (ci / C::kStages) & 1, kWaitCycles);
    }
  } else if (warp == C::kWarpMma) {
    if constexpr (!O) {
      // ---------------------------------- MMA: the N and M chains of a group (or group 0's one chain)
      // (converged warp, voted waits, one elected lane issues); per chunk D1 of each chain, then D4 of each
      const int nch = part == 0 ? 2 : 1;
      bool ok = true;
      for (int ci = 0; ci < n_c && ok; ++ci) {
        const int s = ci % C::kStages;
        const uint32_t sb = tc::smem_u32(stage(ci));
        if (!__all_sync(~0u, tc::mbar_wait(&bar_full[s], (ci / C::kStages) & 1, kWaitCycles))) {
          ok = false;
          break;
        }
        const uint64_t dw = tc::sdesc_sw128(sb + C::kStW, 16384, 1024);
        const uint64_t dk = tc::sdesc_sw128(sb + C::kStK, 8192, 1024);
        for (int c = 0; c < nch && ok; ++c) {
          if (!__all_sync(~0u, tc::mbar_wait_spin(&bar_sc[c], ci & 1, kWaitCycles))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t tb = tmem + 256 * c;
#pragma unroll
          for (int k = 0; k < 8; ++k)  // D1 = S W^T
            tc::mma_bf16_ts_w(tb + C::kTD1, tb + C::kTS16 + 8 * k, dw + (uint64_t)((k * 2048) >> 4), kIdesc64mn,
                              k > 0 ? 1u : 0u);
          tc::mma_commit_w(&bar_d1c[c]);
        }
        for (int c = 0; c < nch && ok; ++c) {
          if (!__all_sync(~0u, tc::mbar_wait_spin(&bar_uc[c], ci & 1, kWaitCycles))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t tb = tmem + 256 * c;
#pragma unroll
          for (int k = 0; k < 4; ++k)  // S += U K'
            tc::mma_bf16_ts_w(tb + C::kTS32, tb + C::kTU + 8 * k, dk + (uint64_t)((k * 2048) >> 4), kIdesc128mn, 1u);
          tc::mma_commit_w(&bar_d4c[c]);
        }
        tc::mma_commit_w(&bar_empty[s]);
        if (*(volatile int*)&abort_flag) ok = false;
      }
      if (!ok && lane == 0) fail();
      tc::mma_commit_w(&bar_done);
      tc::mbar_wait(&bar_done, 0, kWaitCycles);
    } else {
    // ------------------------------------------------ MMA: the state chain
      // (the whole warp, converged: waits are voted and one elected lane issues; descriptors are built once
      // per stage and a K step adds a constant to the start-address field)
      {
        bool ok = true;
        // start state of a later group: S <- S M_q + N_q as D = N_q (placed in the fp32 state columns by the
        // rows) + S_hi M_hi + S_lo M_hi, with S split into bf16 high and low parts and M in bf16
        for (int q = 1; q <= n_comb && ok; ++q) {
          const int im = 2 * q - 2;  // the item of M_q
          if (!__all_sync(~0u, tc::mbar_wait(&bar_cb[im % 3], (im / 3) & 1, kWaitCycles)) ||
              !__all_sync(~0u, tc::mbar_wait_spin(&bar_ps, (q - 1) & 1, kWaitCycles))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint64_t dm = tc::sdesc_sw128(tc::smem_u32(smem) + (im % 3) * C::kStageBytes, 16384, 1024);
#pragma unroll
          for (int pr = 0; pr < 2; ++pr) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              tc::mma_bf16_ts_w(tmem + C::kTS32, tmem + (pr == 0 ? C::kTS16 : C::kTSlo) + 8 * k,
                                dm + (uint64_t)((k * 2048) >> 4), kIdesc128mn, 1u);
          }
          tc::mma_commit_w(&bar_pd);
        }
        for (int ci = 0; ci < n_c && ok; ++ci) {
          const int s = ci % C::kStages;
          const uint32_t sb = tc::smem_u32(stage(ci));
          if (!__all_sync(~0u, tc::mbar_wait(&bar_full[s], (ci / C::kStages) & 1, kWaitCycles)) ||
              !__all_sync(~0u, tc::mbar_wait_spin(&bar_s, ci & 1, kWaitCycles))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint64_t dw = tc::sdesc_sw128(sb + C::kStW, 16384, 1024);
#pragma unroll
          for (int k = 0; k < 8; ++k) {  // D1 = S W^T   (K = d_k, 16 per step; A = bf16 S in TMEM)
            tc::mma_bf16_ts_w(tmem + C::kTD1, tmem + C::kTS16 + 8 * k, dw + (uint64_t)((k * 2048) >> 4), kIdesc64mn,
                              k > 0 ? 1u : 0u);
          }
          tc::mma_commit_w(&bar_d1);
          if (!__all_sync(~0u, tc::mbar_wait_spin(&bar_u, ci & 1, kWaitCycles))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint64_t dk = tc::sdesc_sw128(sb + C::kStK, 8192, 1024);
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // S += U K'   (K = tokens; S already scaled by e^{gC})
            tc::mma_bf16_ts_w(tmem + C::kTS32, tmem + C::kTU + 8 * k, dk + (uint64_t)((k * 2048) >> 4), kIdesc128mn, 1u);
          }
          tc::mma_commit_w(&bar_d4);
          tc::mma_commit_w(&bar_empty[s]);
          if (*(volatile int*)&abort_flag) ok = false;
        }
        if (!ok && lane == 0) fail();
        tc::mma_commit_w(&bar_done);
        tc::mbar_wait(&bar_done, 0, kWaitCycles);
      }
      __syncwarp();
    }
  } else if (O && warp == C::kWarpOmma) {
    // -------------------------------------------------- MMA: the outputs
    // (converged warp, voted waits, one elected lane issues)
    {
      bool ok = true;
      for (int ci = 0; ci < n_c && ok; ++ci) {
        const int s = ci % C::kStages;
        const uint32_t sb = tc::smem_u32(stage(ci));
        // D2 once the chain's D1 is done and D3 once its D4 is done: the output products fill the tensor pipe
        // while the rows form U and the bf16 state, instead of sharing it with the chain's products
        if (!__all_sync(~0u, tc::mbar_wait(&bar_s, ci & 1, kWaitCycles)) ||
            !__all_sync(~0u, tc::mbar_wait(&bar_full[s], (ci / C::kStages) & 1, kWaitCycles)) ||
            (ci >= 1 && !__all_sync(~0u, tc::mbar_wait(&bar_of, (ci - 1) & 1, kWaitCycles))) ||
            !__all_sync(~0u, tc::mbar_wait(&bar_d1, ci & 1, kWaitCycles))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        if (outputs) {
          const uint64_t dq = tc::sdesc_sw128(sb + C::kStQ, 16, 1024);
#pragma unroll
          for (int k = 0; k < 8; ++k) {  // D2 = S Q^T
            tc::mma_bf16_ts_w(tmem + C::kTD2, tmem + C::kTS16 + 8 * k, dq + (uint64_t)(((k >> 2) * 8192 + (k & 3) * 32) >> 4),
                              kIdesc64, k > 0 ? 1u : 0u);
          }
        }
        tc::mma_commit_w(&bar_d2);
        if (!__all_sync(~0u, tc::mbar_wait(&bar_d4, ci & 1, kWaitCycles))) {  // (D4 read U: U is written)
          ok = false;
          break;
        }
        tc::fence_after_sync();
        if (outputs) {
          const uint64_t dp = tc::sdesc_sw128(sb + C::kStP, 16, 1024);
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // D3 = U P^T
            tc::mma_bf16_ts_w(tmem + C::kTD3, tmem + C::kTU + 8 * k, dp + (uint64_t)((k * 32) >> 4), kIdesc64, k > 0 ? 1u : 0u);
          }
        }
        tc::mma_commit_w(&bar_d23);
        tc::mma_commit_w(&bar_empty[s]);
        if (*(volatile int*)&abort_flag) ok = false;
      }
      if (!ok && lane == 0) fail();
      tc::mma_commit_w(&bar_done2);
      tc::mbar_wait(&bar_done2, 0, kWaitCycles);
    }
    __syncwarp();
  } else if (warp < 4) {
    if constexpr (!O) {
      // ------------------------------------- rows of the N and M chains (or of group 0's one chain)
      const int j = threadIdx.x;  // row of S == TMEM lane
      const uint32_t lb = (uint32_t)(warp * 32) << 16;
      const int nch = part == 0 ? 2 : 1;
      bool ok = true;
      // start states: chain 0 from zero (N) or the node's start slot (group 0), chain 1 the identity (M)
      for (int c = 0; c < nch; ++c) {
        const float* src = c == 0 && ik == kInitSlot ? p.state + (((size_t)init * p.H + h) * kD + j) * kD : nullptr;
        const uint32_t tb = tmem + lb + 256 * c;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t f[32], b[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 v = src ? reinterpret_cast<const float4*>(src)[q * 8 + i] : make_float4(0.f, 0.f, 0.f, 0.f);
            f[4 * i] = __float_as_uint(v.x);
            f[4 * i + 1] = __float_as_uint(v.y);
            f[4 * i + 2] = __float_as_uint(v.z);
            f[4 * i + 3] = __float_as_uint(v.w);
          }
          if (c == 1) {
#pragma unroll
            for (int i = 0; i < 32; ++i) f[i] = __float_as_uint(q * 32 + i == j ? 1.f : 0.f);
          }
          tc::tmem_st32(tb + C::kTS32 + q * 32, f);
#pragma unroll
          for (int i = 0; i < 16; ++i) b[i] = tc::pack_bf16x2(__uint_as_float(f[2 * i]), __uint_as_float(f[2 * i + 1]));
          tc::tmem_st16(tb + C::kTS16 + q * 16, b);
        }
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      for (int c = 0; c < nch; ++c) tc::mbar_arrive_warp(&bar_sc[c]);
      for (int ci = 0; ci < n_c && ok; ++ci) {
        const int s = ci % C::kStages;
        const uint8_t* sb = stage(ci);
        if (!__all_sync(~0u, tc::mbar_wait(&bar_full[s], (ci / C::kStages) & 1, kWaitCycles))) {
          ok = false;
          break;
        }
        const float ec = reinterpret_cast<const float*>(sb + C::kStG)[128];  // e^{gC}
        // S <- e^{gC} S in place, both chains (overlaps their D1; D4 adds to it)
        for (int c = 0; c < nch; ++c) state_scale(tmem + lb + 256 * c + C::kTS32, ec);
        // U = Ut^T - D1 (chain 0) and U = -D1 (chain 1, Ut = 0), over the D1 columns once read
        const uint8_t* utj = sb + C::kStUt + j * 128;
        for (int c = 0; c < nch && ok; ++c) {
          if (!__all_sync(~0u, tc::mbar_wait_spin(&bar_d1c[c], ci & 1, kWaitCycles))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t tb = tmem + lb + 256 * c;
          // both halves of D1 in registers before U is written over their columns
          uint32_t d1[2][32];
          tc::tmem_ld32(tb + C::kTD1, d1[0]);
          tc::tmem_ld32(tb + C::kTD1 + 32, d1[1]);
          uint4 uv[8];
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8)
            uv[c8] = c == 1 ? make_uint4(0u, 0u, 0u, 0u) : *reinterpret_cast<const uint4*>(utj + ((c8 ^ (j & 7)) << 4));
          tc::tmem_wait_ld();
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t u2[16];
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              const uint4 w = uv[half * 4 + c4];
              const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int e2 = 0; e2 < 4; ++e2)
                u2[c4 * 4 + e2] = tc::pack_bf16x2(__uint_as_float(w4[e2] << 16) - __uint_as_float(d1[half][c4 * 8 + 2 * e2]),
                                                  __uint_as_float(w4[e2] & 0xFFFF0000u) - __uint_as_float(d1[half][c4 * 8 + 2 * e2 + 1]));
            }
            tc::tmem_st16(tb + C::kTU + half * 16, u2);
          }
          tc::tmem_wait_st();
          tc::fence_before_sync();
          tc::mbar_arrive_warp(&bar_uc[c]);
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bar_empty[s]);  // Ut and the decay block are read
        // the bf16 operand of each new state
        for (int c = 0; c < nch && ok; ++c) {
          if (!__all_sync(~0u, tc::mbar_wait_spin(&bar_d4c[c], ci & 1, kWaitCycles))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          state_to_bf16(tmem + lb + 256 * c + C::kTS32, tmem + lb + 256 * c + C::kTS16);
          tc::tmem_wait_st();
          tc::fence_before_sync();
          tc::mbar_arrive_warp(&bar_sc[c]);
        }
      }
      if (!ok) {
        fail();
      } else {
        for (int c = 0; c < nch; ++c) {
          const EndKind ekc = c == 0 ? ek : kEndScanM;
          const uint32_t tb = tmem + lb + 256 * c;
          if (ekc == kEndScanS) {
            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(scanbuf(e1) + gdnws::kScanS) + j * kD);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t f[32];
              tc::tmem_ld32(tb + C::kTS32 + q * 32, f);
              tc::tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 8; ++i)
                dst[q * 8 + i] = make_float4(__uint_as_float(f[4 * i]), __uint_as_float(f[4 * i + 1]),
                                             __uint_as_float(f[4 * i + 2]), __uint_as_float(f[4 * i + 3]));
            }
          } else if (ekc == kEndScanN) {
            // row j of N in fp32, its 16-byte pieces swizzled by j % 32 (read back row by row from shared
            // memory by the rows of the combine, one row per lane)
            uint8_t* dst = scanbuf(e) + gdnws::kScanN + j * 512;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t f[32];
              tc::tmem_ld32(tb + C::kTS32 + q * 32, f);
              tc::tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 8; ++i)
                *reinterpret_cast<float4*>(dst + (((q * 8 + i) ^ (j & 31)) << 4)) =
                    make_float4(__uint_as_float(f[4 * i]), __uint_as_float(f[4 * i + 1]), __uint_as_float(f[4 * i + 2]),
                                __uint_as_float(f[4 * i + 3]));
            }
          } else {
            // row j of M as the bf16 image of an MN-major B operand: element (j, n) in slab n / 64, 128-byte
            // row j, 16-byte chunk (n % 64) / 8 swizzled by j % 8
            uint8_t* mh = scanbuf(e) + gdnws::kScanMhi;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t f[32];
              tc::tmem_ld32(tb + C::kTS32 + q * 32, f);
              tc::tmem_wait_ld();
#pragma unroll
              for (int c8 = 0; c8 < 4; ++c8) {
                const int n0 = q * 32 + c8 * 8;
                const int off = (n0 >> 6) * 16384 + (j >> 3) * 1024 + (j & 7) * 128 + ((((n0 & 63) >> 3) ^ (j & 7)) << 4);
                uint32_t hw[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  hw[i] = tc::pack_bf16x2(__uint_as_float(f[c8 * 8 + 2 * i]), __uint_as_float(f[c8 * 8 + 2 * i + 1]));
                *reinterpret_cast<uint4*>(mh + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
              }
            }
          }
        }
      }
    } else {
    // ---------------------------------------------------- rows of the state
    const int j = threadIdx.x;  // row of S == TMEM lane
    const uint32_t lb = (uint32_t)(warp * 32) << 16;
    bool ok = true;
    // the initial state into the fp32 columns: a slot, zero, the identity (a transition), or a scan buffer
    {
      const float* src = ik == kInitSlot   ? p.state + (((size_t)init * p.H + h) * kD + j) * kD
                         : ik == kInitScan ? reinterpret_cast<const float*>(scanbuf(e1) + gdnws::kScanS) + j * kD
                                           : nullptr;
#pragma unroll
      for (int q2 = 0; q2 < 2; ++q2) {  // 16 loads in flight, then two stores
        uint32_t f[2][32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float4 v = src ? reinterpret_cast<const float4*>(src)[q2 * 16 + i] : make_float4(0.f, 0.f, 0.f, 0.f);
          f[i >> 3][4 * (i & 7)] = __float_as_uint(v.x);
          f[i >> 3][4 * (i & 7) + 1] = __float_as_uint(v.y);
          f[i >> 3][4 * (i & 7) + 2] = __float_as_uint(v.z);
          f[i >> 3][4 * (i & 7) + 3] = __float_as_uint(v.w);
        }
        if (ik == kInitIdentity) {
#pragma unroll
          for (int i = 0; i < 64; ++i) f[i >> 5][i & 31] = __float_as_uint(q2 * 64 + i == j ? 1.f : 0.f);
        }
        tc::tmem_st32(tmem + lb + C::kTS32 + q2 * 64, f[0]);
        tc::tmem_st32(tmem + lb + C::kTS32 + q2 * 64 + 32, f[1]);
      }
      tc::tmem_wait_st();
    }
    // a later group's start state: S <- S M_q + N_q for q = 1 .. g-1 on tensor cores: the rows split S into
    // bf16 high and low parts, then write row j of N_q (fp32, from its combine buffer) over the fp32 state,
    // and the MMAs add S_hi M_q + S_lo M_q to it
    for (int q = 1; q <= n_comb && ok; ++q) {
#pragma unroll
      for (int q2 = 0; q2 < 2; ++q2) {
        uint32_t f[2][32];
        tc::tmem_ld32(tmem + lb + C::kTS32 + q2 * 64, f[0]);
        tc::tmem_ld32(tmem + lb + C::kTS32 + q2 * 64 + 32, f[1]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t bh[16], bl[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a = __uint_as_float(f[hf][2 * i]), b = __uint_as_float(f[hf][2 * i + 1]);
            bh[i] = tc::pack_bf16x2(a, b);
            bl[i] = tc::pack_bf16x2(a - __uint_as_float(bh[i] << 16), b - __uint_as_float(bh[i] & 0xFFFF0000u));
          }
          tc::tmem_st16(tmem + lb + C::kTS16 + (2 * q2 + hf) * 16, bh);
          tc::tmem_st16(tmem + lb + C::kTSlo + (2 * q2 + hf) * 16, bl);
        }
      }
      const int in = 2 * q - 1;  // the item of N_q
      if (!__all_sync(~0u, tc::mbar_wait(&bar_cb[in % 3], (in / 3) & 1, kWaitCycles))) {
        ok = false;
        break;
      }
      {
        const uint8_t* nrow = smem + (in % 3) * C::kStageBytes + j * 512;  // pieces swizzled by j % 32
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
          uint32_t f[2][32];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float4 v = *reinterpret_cast<const float4*>(nrow + (((q2 * 16 + i) ^ (j & 31)) << 4));
            f[i >> 3][4 * (i & 7)] = __float_as_uint(v.x);
            f[i >> 3][4 * (i & 7) + 1] = __float_as_uint(v.y);
            f[i >> 3][4 * (i & 7) + 2] = __float_as_uint(v.z);
            f[i >> 3][4 * (i & 7) + 3] = __float_as_uint(v.w);
          }
          tc::tmem_st32(tmem + lb + C::kTS32 + q2 * 64, f[0]);
          tc::tmem_st32(tmem + lb + C::kTS32 + q2 * 64 + 32, f[1]);
        }
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      tc::mbar_arrive_warp(&bar_ps);
      if (!__all_sync(~0u, tc::mbar_wait_spin(&bar_pd, (q - 1) & 1, kWaitCycles))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
    }
    // the bf16 operand of the start state
    state_to_bf16(tmem + lb + C::kTS32, tmem + lb + C::kTS16);
    tc::tmem_wait_st();
    tc::fence_before_sync();
    tc::mbar_arrive_warp(&bar_s);
    for (int ci = 0; ci < n_c; ++ci) {
      const int s = ci % C::kStages;
      const uint8_t* sb = stage(ci);
      if (!__all_sync(~0u, tc::mbar_wait(&bar_full[s], (ci / C::kStages) & 1, kWaitCycles))) {
        ok = false;
        break;
      }
      const float* gblk = reinterpret_cast<const float*>(sb + C::kStG);  // e^g [64] | e^{gC-g} [64] | e^{gC}
      // S <- e^{gC} S in place (overlaps D1; D4 adds to it)
      state_scale(tmem + lb + C::kTS32, gblk[128]);
      // D1 done; D3 of the previous chunk (which reads U) done
      if (!__all_sync(~0u, tc::mbar_wait_spin(&bar_d1, ci & 1, kWaitCycles)) ||
          (O && ci >= 1 && !__all_sync(~0u, tc::mbar_wait(&bar_d23, (ci - 1) & 1, kWaitCycles)))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      // U = Ut^T - D1;  row j of Ut^T is one swizzled 128-byte row
      const uint8_t* utj = sb + C::kStUt + j * 128;
      {
        uint32_t d1[2][32];
        tc::tmem_ld32(tmem + lb + C::kTD1, d1[0]);
        tc::tmem_ld32(tmem + lb + C::kTD1 + 32, d1[1]);
        uint4 uv[8];
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8)  // (a transition M runs with Ut = 0)
          uv[c8] = zero_ut ? make_uint4(0u, 0u, 0u, 0u) : *reinterpret_cast<const uint4*>(utj + ((c8 ^ (j & 7)) << 4));
        tc::tmem_wait_ld();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t u2[16];
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const uint4 w = uv[half * 4 + c4];
            const uint32_t w4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              u2[c4 * 4 + e] = tc::pack_bf16x2(__uint_as_float(w4[e] << 16) - __uint_as_float(d1[half][c4 * 8 + 2 * e]),
                                               __uint_as_float(w4[e] & 0xFFFF0000u) - __uint_as_float(d1[half][c4 * 8 + 2 * e + 1]));
          }
          tc::tmem_st16(tmem + lb + C::kTU + half * 16, u2);
        }
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      tc::mbar_arrive_warp(&bar_u);
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar_empty[s]);  // Ut and the decay block are read
      // D4 done (new S), D2 done (the bf16 S may be overwritten)
      if (!__all_sync(~0u, tc::mbar_wait_spin(&bar_d4, ci & 1, kWaitCycles)) ||
          (O && !__all_sync(~0u, tc::mbar_wait(&bar_d2, ci & 1, kWaitCycles)))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      // the bf16 operand of the new state
      state_to_bf16(tmem + lb + C::kTS32, tmem + lb + C::kTS16);
      tc::tmem_wait_st();
      tc::fence_before_sync();
      tc::mbar_arrive_warp(&bar_s);
    }
    if (!ok) {
      fail();
    } else if (ek == kEndSlot || ek == kEndScanS) {
      float4* dst = reinterpret_cast<float4*>(
          ek == kEndSlot ? p.state + (((size_t)endslot * p.H + h) * kD + j) * kD
                         : reinterpret_cast<float*>(scanbuf(e1) + gdnws::kScanS) + j * kD);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t f[32];
        tc::tmem_ld32(tmem + lb + C::kTS32 + q * 32, f);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i)
          dst[q * 8 + i] = make_float4(__uint_as_float(f[4 * i]), __uint_as_float(f[4 * i + 1]),
                                       __uint_as_float(f[4 * i + 2]), __uint_as_float(f[4 * i + 3]));
      }
    }
    }
  } else if (O) {
    // ------------------------------------------------------------- outputs
    const int j = threadIdx.x - 128;  // TMEM lane j
    const uint32_t lb = (uint32_t)((warp - 4) * 32) << 16;
    bool ok = true;
    for (int ci = 0; ci < n_c; ++ci) {
      const int s = ci % C::kStages;
      uint8_t* sb = stage(ci);
      const float* egs = reinterpret_cast<const float*>(sb + C::kStG);
      if (!__all_sync(~0u, tc::mbar_wait(&bar_full[s], (ci / C::kStages) & 1, kWaitCycles)) ||
          !__all_sync(~0u, tc::mbar_wait(&bar_d23, ci & 1, kWaitCycles))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      if (!outputs) {  // no D2, D3 were formed: keep the hand-offs only
        tc::mbar_arrive_warp(&bar_of);
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bar_empty[s]);
        continue;
      }
      const int32_t* ch = M.chunk(c_off + ci);
      const int row0 = ch[C_ROW0], len = ch[C_LEN];
      // D2, D3 and e^g into registers first, so that D2, D3 are released at once and the
      // staging stores below do not wait on loads from the same buffer
      uint32_t d2[64], d3[64];
      tc::tmem_ld32(tmem + lb + C::kTD2, *reinterpret_cast<uint32_t(*)[32]>(d2));
      tc::tmem_ld32(tmem + lb + C::kTD2 + 32, *reinterpret_cast<uint32_t(*)[32]>(d2 + 32));
      tc::tmem_ld32(tmem + lb + C::kTD3, *reinterpret_cast<uint32_t(*)[32]>(d3));
      tc::tmem_ld32(tmem + lb + C::kTD3 + 32, *reinterpret_cast<uint32_t(*)[32]>(d3 + 32));
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      tc::mbar_arrive_warp(&bar_of);  // D2, D3 may be overwritten
      float o[64];
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 e = *reinterpret_cast<const float4*>(egs + 4 * c4);
        o[4 * c4] = fmaf(e.x, __uint_as_float(d2[4 * c4]), __uint_as_float(d3[4 * c4]));
        o[4 * c4 + 1] = fmaf(e.y, __uint_as_float(d2[4 * c4 + 1]), __uint_as_float(d3[4 * c4 + 1]));
        o[4 * c4 + 2] = fmaf(e.z, __uint_as_float(d2[4 * c4 + 2]), __uint_as_float(d3[4 * c4 + 2]));
        o[4 * c4 + 3] = fmaf(e.w, __uint_as_float(d2[4 * c4 + 3]), __uint_as_float(d3[4 * c4 + 3]));
      }
      // O[t][j] into the chunk's Q buffer (D2 has read it), plain [64][128] bf16
      __nv_bfloat16* stg = reinterpret_cast<__nv_bfloat16*>(sb + C::kStQ);
#pragma unroll
      for (int t = 0; t < 64; ++t) stg[t * kD + j] = __float2bfloat16_rn(o[t]);
      tc::named_sync(2, 128);
      __nv_bfloat16* dst = p.out + ((size_t)row0 * p.H + h) * kD;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e = j + 128 * i, t = e >> 4, c16 = e & 15;
        if (t < len)
          *reinterpret_cast<uint4*>(dst + (size_t)t * p.H * kD + c16 * 8) =
              *reinterpret_cast<const uint4*>(sb + C::kStQ + t * 256 + c16 * 16);
      }
      tc::fence_proxy_async_smem();  // the Q buffer is refilled by TMA after this
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar_empty[s]);
    }
    if (!ok) fail();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == C::kWarpMma) tc::tmem_dealloc(tmem, C::kTmemCols);
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

// State passes of every tree level on tensor cores, reading the compact
// workspace written by the chunk-local pass.
hs_status hs_gdn_chain_tc_launch(const hs_round_caps* caps, const int32_t* meta, int H, const void* q,
                                 const uint8_t* ws, uint8_t* scan, float* state, int n_slots, void* out,
                                 int32_t* status, cudaStream_t st) {
  CUtensorMap mq;
  if (!map_rows(&mq, q, H, caps->max_tokens))
    return hs::fail(HS_ECUDA, "gdn: tensor map encoding failed");
  static std::atomic<bool> configured[hsd::kMaxDevices];  // zero-initialised: per device
  const int slot = hsd::device_slot();
  if (slot < 0) return hs::fail(HS_ECUDA, "gdn_chain_tc: no usable CUDA device");
  if (!configured[slot].load()) {
    if (cudaFuncSetAttribute(gdn_chain_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes<true>() + 1024) != cudaSuccess ||
        cudaFuncSetAttribute(gdn_chain_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_bytes<false>() + 1024) != cudaSuccess)
      return hs::fail(HS_ECUDA, "gdn_chain_tc: cannot raise the shared-memory limit");
    configured[slot].store(true);
  }
  // per level: the scan's first pass (group 0's end state and the later groups' N and M, no outputs), then
  // every group of every node with outputs
  const int cap_scan = scan_cap(caps->max_chunks);
  const bool any_scan = caps->max_chunks >= 2 * kScanMinChunks;
  for (int lev = 0; lev < caps->max_levels && caps->max_segments > 0; ++lev) {
    Prm prm{meta, lev, H, n_slots, ws, scan, state, (__nv_bfloat16*)out, status};
    if (any_scan) {
      hsd::launch_pdl(gdn_chain_tc_kernel<false>, dim3(H, 2 * cap_scan), dim3(Cfg<false>::kThreads),
                      smem_bytes<false>() + 1024, st, mq, prm);
      HS_LAUNCH_CHECK("gdn_chain_tc (scan)");
    }
    hsd::launch_pdl(gdn_chain_tc_kernel<true>, dim3(H, caps->max_segments + (any_scan ? cap_scan : 0)),
                    dim3(Cfg<true>::kThreads), smem_bytes<true>() + 1024, st, mq, prm);
    HS_LAUNCH_CHECK("gdn_chain_tc");
  }
  return HS_OK;
}
