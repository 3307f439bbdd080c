// fork_attn_tc.cu -- tensor-core ForkAttention for sm_103a (bf16, d = 128).
//
// Flide, "Accelerating Decision Inference with Exact State Forking":
// section 3.2.1, Eq. 3 (visibility), section 3.3.1 (keys from the shared
// state and the query's own question; fully visible key blocks read without
// a mask, only partial blocks masked), section 3.5 (a question's reductions
// start at the fork and do not depend on the rest of the round).  The scale
// is 1/sqrt(d) (Flex, "Request-Adaptive Execution ...", section 2, Eq. 1).
//
// One CTA = one attention tile (up to 128 consecutive stream rows: a run of
// one node, or sibling nodes packed together) x one query head.  The CTA
// walks the tile's key spans (ancestors first, then the tile's own nodes) in
// blocks of 128 keys starting at each span's first key, so a row's sequence
// of blocks depends only on its own tree path:
//
//   warp 8      TMA producer: Q once; per block K and V pages into a 3-stage
//               ring (one 128-row box per 64-column half when the 8 pages of
//               a block are consecutive, else one 16-row box per page; pages
//               past the span are loaded from out of range, i.e. zeros).  A
//               K stage is refilled once its S has been computed, a V stage
//               once its P.V has.
//   warp 9      allocates TMEM and issues tcgen05.mma from one thread:
//               S_j = Q K_j^T into one of two TMEM buffers, then
//               O_c += P_{j-1,c} V_{j-1,c} for the two key halves c once the
//               softmax has written P_{j-1}, with P read from TMEM.
//   warps 0..7  softmax.  Warp w serves TMEM lanes 32 (w % 4) .. +31 (query
//               rows) and key half c = w / 4 (keys 64 c .. 64 c + 63 of every
//               block): each (row, half) runs its own online softmax over its
//               half of the keys into its own accumulator O_c, with the
//               running max in log2 units, rescaling O_c and l_c only when
//               the max grows by more than 2^8 (a per-(row, half) decision;
//               only then does it wait for the previous P.V).  The exponent
//               is the hardware 2^x approximation (relative error ~2^-22).
//               P_j overwrites S_j in place, split into a bf16 high part (the
//               top 16 bits of p) and a bf16 low part (p - high, rounded),
//               both multiplied into O_c, so P enters the product with ~16
//               significant bits.  At the end the two halves of a
//               row combine (m = max m_c, O = sum 2^(m_c - m) O_c, l likewise,
//               in a fixed order) and write O / l.
//
// TMEM: columns [0,128) and [128,256) = S/P ping-pong (half c of a row: S in
// columns 64c..64c+63, then P high in the first 32 and P low in the next 32),
// [256,384) = O_0, [384,512) = O_1.  Shared memory: Q 32 KB | K 3 x 32 KB |
// V 3 x 32 KB (SW128).  MMAs issued by one thread run in issue order, so S_{j+2}
// overwrites P_j only after P.V_j has read it.  Every wait is bounded; a wait
// that runs out records HS_DEV_TIMEOUT in the status word, and the CTA drains
// its own copies and MMAs before leaving.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "device.cuh"
#include "tc_ptx.cuh"

using namespace hsm;
using hsd::Meta;

namespace {

constexpr int kD = 128;
constexpr int kBlk = 128;                    // keys per block
constexpr int kSlab = 128 * 128;             // bytes of one [128 rows][64 cols] bf16 slab
constexpr int kTile = 2 * kSlab;             // 32 KB: 128 x 128 bf16
constexpr int kStages = 3;                   // K/V ring depth
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTile;
constexpr int kOffV = kOffK + kStages * kTile;
constexpr int kSmemBytes = kOffV + kStages * kTile;  // 224 KB
constexpr int kSoftWarps = 8, kWarpProd = 8, kWarpMma = 9;
constexpr int kThreads = 320;
constexpr uint32_t kTmO = 256;               // O_0 at 256, O_1 at 384
constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz

constexpr uint32_t kIdescQK = tc::idesc_bf16(128, 128, 0, 0);  // A = Q (K-major), B = K (K-major)
constexpr uint32_t kIdescPV = tc::idesc_bf16(128, 128, 0, 1);  // A = P (K-major), B = V (N-major)

struct Params {
  const int32_t* meta;
  int hq, hkv, n_pages;
  float scale_log2e;
  __nv_bfloat16* out;
  int32_t* status;
  int window;      // sliding width W (> 0: a row sees keys t_x - t_y < W), 0 = none
  int bidir_root;  // 1: a root node's rows see the whole root
};

// The key blocks of a tile in the order every role walks them.  Mask variants: with a sliding window the
// blocks that end before the tile's first window start are skipped by every role (they are hidden from every
// row of the tile; each row still masks its own window start); with a bidirectional root the rows of a root
// node see all of it.  A key's position: a shared span's keys follow the earlier shared spans along the path
// (history first, then each ancestor), an own span's start at its node's first position.  kMask = false
// compiles the mask tests out (plain causal attention).
template <bool kMask>
struct CursorT {
  Meta M;
  const int32_t* tspans;
  int n_shared, n_spans, n_own, tile_lo, tile_hi;
  int si, b0, kmax;
  int sp_off, sp_n, owner, own, first_idx;
  int p0, p_shared, lo_min, window, bidir, whole;
  __device__ void init(Meta m, const int32_t* tl, int window_ = 0, int bidir_ = 0) {
    M = m;
    tspans = m.tile_spans() + tl[TL_SPAN_OFF];
    n_shared = tl[TL_N_SHARED];
    n_own = tl[TL_N_OWN];
    n_spans = n_shared + n_own;
    tile_lo = tl[TL_ROW0];
    tile_hi = tl[TL_ROW0] + tl[TL_N_ROWS];
    si = -1;
    b0 = 0;
    kmax = 0;
    p0 = p_shared = 0;
    window = kMask ? window_ : 0;
    bidir = kMask ? bidir_ : 0;
    whole = 0;
    lo_min = -(1 << 30);
    if (kMask && window > 0) {  // the tile's first row has its smallest position
      const int32_t* tk = m.tok(tile_lo);
      lo_min = m.seg(tk[T_SEG])[S_POS0] + tk[T_IDX] - window + 1;
    }
  }
  // advance to the next block; false when the tile has no more
  __device__ bool next() {
    b0 += kBlk;
    while (true) {
      while (b0 >= kmax) {
        if (++si >= n_spans) return false;
        const int32_t* sp = M.span(tspans[si]);
        sp_off = sp[SP_PAGE_REF_OFF];
        sp_n = sp[SP_N_TOK];
        owner = sp[SP_OWNER];
        own = si >= n_shared;
        kmax = sp_n;
        first_idx = 0;
        whole = 0;
        if (own) {
          const int32_t* og = M.seg(owner);
          const int lo = max(tile_lo, og[S_STREAM_OFF]);
          const int hi = min(tile_hi, og[S_STREAM_OFF] + og[S_LEN]);
          whole = kMask && bidir && og[S_LEVEL] == 0;  // a bidirectional root: its rows see the whole node
          kmax = hi > lo ? (whole ? og[S_LEN] : hi - og[S_STREAM_OFF]) : 0;
          first_idx = lo - og[S_STREAM_OFF];
          p0 = og[S_POS0];
        } else {
          p0 = p_shared;
          p_shared += sp_n;
        }
        b0 = 0;
      }
      if (kMask && p0 + b0 + kBlk <= lo_min) {  // wholly before every row's window
        b0 += kBlk;
        continue;
      }
      return true;
    }
  }
  __device__ int valid() const { return min(kBlk, sp_n - b0); }
  // every row of the tile sees every key of the block
  __device__ bool full() const {
    if (kMask && window > 0) return false;
    if (!own) return sp_n - b0 >= kBlk;
    return n_own == 1 && b0 + kBlk <= sp_n && ((kMask && whole) || b0 + kBlk <= first_idx);
  }
};
using Cursor = CursorT<false>;

__device__ __forceinline__ void record(int32_t* status, int* abort_flag, int code) {
  hsd::set_status(status, code);
  atomicExch(abort_flag, 1);
}

__global__ void __launch_bounds__(kThreads, 1)
fork_attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k16,
                    const __grid_constant__ CUtensorMap tm_k128, const __grid_constant__ CUtensorMap tm_v16,
                    const __grid_constant__ CUtensorMap tm_v128, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_q, bar_kf[kStages], bar_vf[kStages], bar_ke[kStages], bar_ve[kStages];
  __shared__ uint64_t bar_sf[2], bar_pf[2], bar_pv[2], bar_done, bar_x;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  Meta M{p.meta};
  // tile-major order: every head of the heaviest tiles first (tiles are sorted by work)
  const int tile = blockIdx.x / p.hq;
  if (tile >= M.h(H_N_TILE)) return;
  const int32_t* tl = M.tile(tile);
  const int h = blockIdx.x % p.hq;
  const int kvh = h / (p.hq / p.hkv);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // aligned up to 1024 bytes by pointer arithmetic on the shared array, so every access through smem stays
  // a shared-memory access (an integer round trip would turn them into generic loads and stores)
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    tc::mbar_init(&bar_q, 1);
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&bar_kf[s], 1);
      tc::mbar_init(&bar_vf[s], 1);
      tc::mbar_init(&bar_ke[s], 1);
      tc::mbar_init(&bar_ve[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bar_sf[b], 1);
      tc::mbar_init(&bar_pf[b], 32 * kSoftWarps);
      tc::mbar_init(&bar_pv[b], 1);
    }
    tc::mbar_init(&bar_done, 1);
    tc::mbar_init(&bar_x, 32 * kSoftWarps);
    tc::fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tc::tmem_alloc(&tmem_slot, 512);
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

  Cursor cur;
  cur.init(M, tl);
  const int n_ref = M.h(H_N_PAGE_REF);
  const int32_t* refs = M.page_ref();

  if (warp == kWarpProd) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tc::prefetch_tmap(&tm_q);
      tc::prefetch_tmap(&tm_k16);
      tc::prefetch_tmap(&tm_v16);
      tc::mbar_expect_tx(&bar_q, kTile);
      tc::tma_load_3d(smem + kOffQ, &tm_q, 0, h, tl[TL_ROW0], &bar_q);
      tc::tma_load_3d(smem + kOffQ + kSlab, &tm_q, 64, h, tl[TL_ROW0], &bar_q);
      const int oob_y = p.hkv * p.n_pages * kPage;  // first row past the pool: zero fill
      int j = 0, s = 0, n = 0;                      // block, its stage, uses of the stage before it
      while (cur.next()) {
        const int npg = (cur.valid() + kPage - 1) / kPage;
        int pg[8];
        bool consecutive = npg == 8;
        for (int i = 0; i < 8; ++i) {
          pg[i] = -1;
          if (i < npg) {
            const int ref = cur.sp_off + cur.b0 / kPage + i;
            const int page = ref < n_ref ? refs[ref] : -1;
            if (page >= 0 && page < p.n_pages) {
              pg[i] = page;
            } else {
              hsd::set_status(p.status, ref < n_ref ? HS_DEV_BAD_PAGE : HS_DEV_BAD_META);
            }
          }
          if (i > 0 && (pg[i] < 0 || pg[i] != pg[i - 1] + 1)) consecutive = false;
        }
        if (pg[0] < 0) consecutive = false;
        uint8_t* ks = smem + kOffK + s * kTile;
        uint8_t* vs = smem + kOffV + s * kTile;
        // K stage s is free once S of block j - kStages is computed
        if (n > 0 && !tc::mbar_wait(&bar_ke[s], (n - 1) & 1, kWaitCycles)) {
          record(p.status, &abort_flag, HS_DEV_TIMEOUT);
          break;
        }
        if (*(volatile int*)&abort_flag) break;
        tc::mbar_expect_tx(&bar_kf[s], kTile);
        if (consecutive) {
          const int y = (kvh * p.n_pages + pg[0]) * kPage;
          for (int half = 0; half < 2; ++half) tc::tma_load_2d(ks + half * kSlab, &tm_k128, half * 64, y, &bar_kf[s]);
        } else {
          for (int i = 0; i < 8; ++i) {
            const int y = pg[i] >= 0 ? (kvh * p.n_pages + pg[i]) * kPage : oob_y;
            for (int half = 0; half < 2; ++half)
              tc::tma_load_2d(ks + half * kSlab + i * 2048, &tm_k16, half * 64, y, &bar_kf[s]);
          }
        }
        // V stage s is free once P.V of block j - kStages is done
        if (n > 0 && !tc::mbar_wait(&bar_ve[s], (n - 1) & 1, kWaitCycles)) {
          record(p.status, &abort_flag, HS_DEV_TIMEOUT);
          ++j;  // the K copy of this block is in flight: drain it below
          break;
        }
        tc::mbar_expect_tx(&bar_vf[s], kTile);
        if (consecutive) {
          const int y = (kvh * p.n_pages + pg[0]) * kPage;
          for (int half = 0; half < 2; ++half) tc::tma_load_2d(vs + half * kSlab, &tm_v128, half * 64, y, &bar_vf[s]);
        } else {
          for (int i = 0; i < 8; ++i) {
            const int y = pg[i] >= 0 ? (kvh * p.n_pages + pg[i]) * kPage : oob_y;
            for (int half = 0; half < 2; ++half)
              tc::tma_load_2d(vs + half * kSlab + i * 2048, &tm_v16, half * 64, y, &bar_vf[s]);
          }
        }
        ++j;
        if (++s == kStages) {
          s = 0;
          ++n;
        }
      }
      // drain: every copy this thread issued has landed before the CTA leaves
      tc::mbar_wait(&bar_q, 0, kWaitCycles);
      for (int i = (j >= kStages ? j - kStages : 0); i < j; ++i) {
        tc::mbar_wait(&bar_kf[i % kStages], (i / kStages) & 1, kWaitCycles);
        tc::mbar_wait(&bar_vf[i % kStages], (i / kStages) & 1, kWaitCycles);
      }
    }
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------------- MMA
    // (the whole warp, converged: waits are voted, one elected lane issues)
    {
      // stage-base descriptors built once; a K or key step adds a constant to the start-address field
      const uint32_t s0 = tc::smem_u32(smem);
      const uint64_t dq = tc::sdesc_sw128(s0 + kOffQ, 16, 1024);
      const uint64_t dk0 = tc::sdesc_sw128(s0 + kOffK, 16, 1024);
      const uint64_t dv0 = tc::sdesc_sw128(s0 + kOffV, kSlab, 1024);
      bool ok = __all_sync(~0u, tc::mbar_wait(&bar_q, 0, kWaitCycles));
      if (!ok && lane == 0) record(p.status, &abort_flag, HS_DEV_TIMEOUT);
      auto pv = [&](int i) -> bool {
        const int si = i % kStages;
        // (polling waits: a suspended MMA thread would notice the softmax late)
        if (!__all_sync(~0u, tc::mbar_wait_spin(&bar_pf[i & 1], (i >> 1) & 1, kWaitCycles)) ||
            !__all_sync(~0u, tc::mbar_wait_spin(&bar_vf[si], (i / kStages) & 1, kWaitCycles)))
          return false;
        tc::fence_after_sync();
        const uint64_t b0 = dv0 + (uint64_t)(si * (kTile >> 4));
        const uint32_t pt = tmem + (uint32_t)(i & 1) * 128;  // P_i sits where S_i was
#pragma unroll
        for (int c = 0; c < 2; ++c) {        // key half c -> accumulator O_c
#pragma unroll
          for (int part = 0; part < 2; ++part) {  // P high part, then low part
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              tc::mma_bf16_ts_w(tmem + kTmO + 128 * c, pt + 64 * c + 32 * part + 8 * k,
                              b0 + (uint64_t)((c * 8192 + k * 2048) >> 4), kIdescPV,
                              (i > 0 || part > 0 || k > 0) ? 1u : 0u);
            }
          }
        }
        tc::mma_commit_w(&bar_pv[i & 1]);
        tc::mma_commit_w(&bar_ve[si]);
        return true;
      };
      int j = 0;
      while (ok && cur.next()) {
        const int s = j % kStages;
        if (!__all_sync(~0u, tc::mbar_wait_spin(&bar_kf[s], (j / kStages) & 1, kWaitCycles))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        if (*(volatile int*)&abort_flag) {
          ok = false;
          break;
        }
        const uint64_t b0 = dk0 + (uint64_t)(s * (kTile >> 4));
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t off = (uint64_t)(((k >> 2) * kSlab + (k & 3) * 32) >> 4);
          tc::mma_bf16_ss_w(tmem + (uint32_t)(j & 1) * 128, dq + off, b0 + off, kIdescQK, k > 0 ? 1u : 0u);
        }
        tc::mma_commit_w(&bar_ke[s]);
        tc::mma_commit_w(&bar_sf[j & 1]);
        if (j >= 1 && !pv(j - 1)) {
          ok = false;
          break;
        }
        ++j;
      }
      if (ok && j >= 1 && !pv(j - 1)) ok = false;
      if (!ok && lane == 0) record(p.status, &abort_flag, HS_DEV_TIMEOUT);
      // every MMA issued by this thread completes before O is read and TMEM is freed
      tc::mma_commit_w(&bar_done);
      tc::mbar_wait(&bar_done, 0, kWaitCycles);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp % 4, hc = warp / 4;  // TMEM lane quarter, key half
    const int t = quarter * 32 + lane;            // row of the tile == TMEM lane
    const int row = tl[TL_ROW0] + t;
    const bool active = t < tl[TL_N_ROWS];
    int my_seg = -1, my_idx = 0;
    if (active) {
      my_seg = M.tok(row)[T_SEG];
      my_idx = M.tok(row)[T_IDX];
    }
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t col_o = kTmO + 128 * hc;
    float m_used = -INFINITY, l = 0.f;
    const float sl2 = p.scale_log2e;
    int j = 0;
    bool ok = true;
    while (cur.next()) {
      const int b = j & 1;
      // tcgen05.ld/st are warp-collective: every branch around them is decided warp-wide
      if (!__all_sync(~0u, tc::mbar_wait(&bar_sf[b], (j >> 1) & 1, kWaitCycles))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t sb = tmem + lane_base + (uint32_t)b * 128 + 64 * hc;
      uint32_t r[2][32];
      tc::tmem_ld32(sb, r[0]);
      tc::tmem_ld32(sb + 32, r[1]);
      tc::tmem_wait_ld();
      float s[64];
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(r[c][i]);
      if (!cur.full()) {
        const int lim = (!active ? 0 : !cur.own ? cur.sp_n - cur.b0 : (cur.owner == my_seg ? my_idx + 1 - cur.b0 : 0)) -
                        64 * hc;
#pragma unroll
        for (int i = 0; i < 64; ++i) s[i] = i < lim ? s[i] : -INFINITY;
      }
      // row max of this half: 8 partial maxima, then a fixed tree
      float mp[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) mp[a] = s[a];
#pragma unroll
      for (int i = 8; i < 64; ++i) mp[i & 7] = fmaxf(mp[i & 7], s[i]);
      const float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])), fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
      const float m_new = fmaxf(m_used, mx * sl2);
      float factor = 1.f;
      const bool rescale = m_new > m_used + 8.f;
      if (rescale) {
        factor = exp2f(m_used - m_new);
        m_used = m_new;
      }
      const float mref = m_used == -INFINITY ? 0.f : m_used;
      float rp[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) rp[a] = 0.f;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        s[i] = tc::ex2_approx(fmaf(s[i], sl2, -mref));
        rp[i & 7] += s[i];
      }
      const float rs = ((rp[0] + rp[1]) + (rp[2] + rp[3])) + ((rp[4] + rp[5]) + (rp[6] + rp[7]));
      l = l * factor + rs;
      // P_j over S_j: keys 2i, 2i+1 of this half in column i (high part), 32 + i (low part)
      uint32_t hi[32], lo[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float a = s[2 * i], c = s[2 * i + 1];
        hi[i] = tc::pack_bf16x2_trunc(a, c);
        lo[i] = tc::pack_bf16x2(a - __uint_as_float(hi[i] << 16), c - __uint_as_float(hi[i] & 0xFFFF0000u));
      }
      tc::tmem_st32(sb, hi);
      tc::tmem_st32(sb + 32, lo);
      // O_c rescaled to the new max once P.V_{j-1} is done; rows of the warp that keep
      // their max multiply by factor = 1, which is exact
      if (j >= 1 && __any_sync(~0u, rescale)) {
        if (!__all_sync(~0u, tc::mbar_wait(&bar_pv[(j - 1) & 1], ((j - 1) >> 1) & 1, kWaitCycles))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tc::tmem_ld32(tmem + lane_base + col_o + c * 32, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * factor);
          tc::tmem_st32(tmem + lane_base + col_o + c * 32, o);
        }
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      tc::mbar_arrive(&bar_pf[b]);
      ++j;
    }
    if (ok && j >= 1) {
      // combine the two halves of the row once every MMA is done (so none still reads Q):
      // exchange (m, l) through the Q buffer
      float* xm = reinterpret_cast<float*>(smem + kOffQ);  // [2][128] maxima, then [2][128] sums
      bool got = __all_sync(~0u, tc::mbar_wait(&bar_done, 0, kWaitCycles));
      if (got) {
        xm[hc * 128 + t] = m_used;
        xm[256 + hc * 128 + t] = l;
        tc::mbar_arrive(&bar_x);
        got = __all_sync(~0u, tc::mbar_wait(&bar_x, 0, kWaitCycles));
      }
      if (got) {
        tc::fence_after_sync();
        const float m0 = xm[t], m1 = xm[128 + t];
        const float m = fmaxf(m0, m1);
        const float c0 = m0 == -INFINITY ? 0.f : exp2f(m0 - m);
        const float c1 = m1 == -INFINITY ? 0.f : exp2f(m1 - m);
        const float inv = 1.f / (c0 * xm[256 + t] + c1 * xm[384 + t]);
        const float w0 = c0 * inv, w1 = c1 * inv;
        __nv_bfloat16* dst = p.out + ((size_t)row * p.hq + h) * kD + 64 * hc;
#pragma unroll
        for (int c = 0; c < 2; ++c) {  // output columns 64 hc + 32 c .. +31
          uint32_t o0[32], o1[32];
          tc::tmem_ld32(tmem + lane_base + kTmO + 64 * hc + 32 * c, o0);
          tc::tmem_ld32(tmem + lane_base + kTmO + 128 + 64 * hc + 32 * c, o1);
          tc::tmem_wait_ld();
          if (active) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e)
                f[e] = fmaf(w0, __uint_as_float(o0[q * 8 + e]), w1 * __uint_as_float(o1[q * 8 + e]));
              uint4 v;
              v.x = tc::pack_bf16x2(f[0], f[1]);
              v.y = tc::pack_bf16x2(f[2], f[3]);
              v.z = tc::pack_bf16x2(f[4], f[5]);
              v.w = tc::pack_bf16x2(f[6], f[7]);
              *reinterpret_cast<uint4*>(dst + c * 32 + q * 8) = v;
            }
          }
        }
      } else {
        ok = false;
      }
    }
    if (!ok) record(p.status, &abort_flag, HS_DEV_TIMEOUT);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == kWarpMma) tc::tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// Two query heads per work item (heads 2p and 2p + 1 of a KV-head group of
// even size share every K and V page): the heads' online softmaxes run in two
// warp groups while the MMA warp alternates between them, so one head's
// softmax overlaps the other head's products and each K/V block is loaded
// once.  One persistent CTA per SM takes items one at a time from a counter
// in the round's metadata (tiles longest first, so this is longest-first
// list scheduling); block counters run across items, the
// next item's Q loads once the current item's S products are done, and its
// first P.V waits until the current item's O has been read out, so the next
// item's first S products and copies overlap the current item's epilogue.
//
//   warp 8      TMA: Q of both heads once; per block K and V into a 2-stage
//               ring (a K stage is refilled once both heads' S are computed,
//               a V stage once both heads' P.V are).
//   warp 9      TMEM (512 columns: S_A, S_B, O_A, O_B) and the MMAs, in the
//               order S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...;
//               S_X(j+1) overwrites P_X(j) only after P.V_X(j) is issued
//               (MMAs of one thread run in issue order).
//   warps 0..3  softmax of head A, warps 4..7 of head B: thread t = query row
//               t = TMEM lane t over all 128 keys of a block (a first pass
//               over the scores for the row max, a second for the
//               exponentials, 32 keys at a time); P overwrites S in place:
//               the 32 score columns of keys 32g .. 32g+31 become 16 columns
//               of P in bf16.  A tile holding a readout row keeps ~16
//               significant bits of P -- the 16 columns hold its high parts
//               (top 16 bits), the next 16 its rounded low parts, and both
//               enter P.V -- because the option distribution at a readout
//               row is sensitive to single-ulp changes of the bf16 output;
//               every other tile rounds P to bf16 (nearest) and issues half
//               the P.V products.
//               Since S_X(j) is computed after P.V_X(j-1) is issued, O_X is
//               final for block j-1 when S_X(j) is seen, so a lazy rescale
//               (running max grown by more than 2^8) never waits.
// ---------------------------------------------------------------------------
namespace pair {
constexpr int kOffQ = 0;                  // Q_A, Q_B: 32 KB each
constexpr int kOffK = 2 * kTile;          // 2 stages
constexpr int kOffV = kOffK + 2 * kTile;  // 2 stages
constexpr int kSmemBytes = kOffV + 2 * kTile;  // 192 KB
constexpr uint32_t kTmS = 0, kTmO = 256;  // S_X[h] at 128 X + 64 h, O_X at 256 + 128 X
constexpr uint32_t kIdescQK = tc::idesc_bf16(128, 64, 0, 0);  // S of 64 keys: A = Q, B = K (K-major)
constexpr int kWarpMmaB = 10, kThreads = 352;  // warp 9: MMAs of head A, warp 10: of head B
constexpr int kRing = 4;                       // items published ahead by the producer
}  // namespace pair

template <bool kMask>
__global__ void __launch_bounds__(pair::kThreads, 1)
fork_attn_tc2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k16,
                     const __grid_constant__ CUtensorMap tm_k128, const __grid_constant__ CUtensorMap tm_v16,
                     const __grid_constant__ CUtensorMap tm_v128, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bar_q, bar_qe, bar_kf[2], bar_vf[2], bar_ke[2], bar_ve[2];
  __shared__ uint64_t bar_sf[2][2], bar_pf[2][2], bar_pv[2], bar_done;
  __shared__ uint64_t bar_rf[pair::kRing], bar_re[pair::kRing];  // item ring: index written / read by all
  __shared__ int ring[pair::kRing];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  Meta M{p.meta};
  const int np = p.hq / 2;
  const int n_items = M.h(H_N_TILE) * np;  // (tile, head pair), heaviest tiles first
  const int n_cta = min((int)gridDim.x, n_items);
  if ((int)blockIdx.x >= n_items) return;
  // Items are handed out in order to whichever CTA asks next (a counter in the round's metadata, longest-
  // first list scheduling): the producer lane takes the CTA's k-th item and publishes it in ring slot
  // k % kRing; the MMA and softmax warps read the same sequence.  -1 ends it.
  int32_t* ctr = const_cast<int32_t*>(p.meta);
  auto item_of = [&](int k) -> int {  // every consumer warp, converged; false from a wait means a timeout
    const int s = k % pair::kRing;
    if (!__all_sync(~0u, tc::mbar_wait(&bar_rf[s], (k / pair::kRing) & 1, kWaitCycles))) return -2;
    const int w = *(volatile int*)&ring[s];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) tc::mbar_arrive(&bar_re[s]);
    return w;
  };
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // aligned up to 1024 bytes by pointer arithmetic on the shared array, so every access through smem stays
  // a shared-memory access (an integer round trip would turn them into generic loads and stores)
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);

  if (threadIdx.x == 0) {
    abort_flag = 0;
    tc::mbar_init(&bar_q, 1);
    tc::mbar_init(&bar_qe, 2);  // both MMA warps
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&bar_kf[s], 1);
      tc::mbar_init(&bar_vf[s], 1);
      tc::mbar_init(&bar_ke[s], 2);  // both MMA warps
      tc::mbar_init(&bar_ve[s], 2);
      for (int h = 0; h < 2; ++h) {
        tc::mbar_init(&bar_sf[s][h], 1);    // [X][h]: S_X of a block's key half h done
        tc::mbar_init(&bar_pf[s][h], 4);  // [X][h]: P_X of key half h written (one arrival per softmax warp)
      }
      tc::mbar_init(&bar_pv[s], 1);   // [X]: P.V_X of a key half done
    }
    tc::mbar_init(&bar_done, 2);
    for (int r = 0; r < pair::kRing; ++r) {
      tc::mbar_init(&bar_rf[r], 1);
      tc::mbar_init(&bar_re[r], 2 + kSoftWarps);  // both MMA warps and the softmax warps
    }
    tc::fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tc::tmem_alloc(&tmem_slot, 512);
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
  const int n_ref = M.h(H_N_PAGE_REF);
  const int32_t* refs = M.page_ref();

  if (warp == kWarpProd) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tc::prefetch_tmap(&tm_q);
      tc::prefetch_tmap(&tm_k16);
      tc::prefetch_tmap(&tm_v16);
      const int oob_y = p.hkv * p.n_pages * kPage;  // first row past the pool: zero fill
      int jg = 0, n_q = 0;                           // blocks and Q tiles (non-empty items) issued
      bool ok = true;
      for (int k = 0; ok; ++k) {
        // take the next item and publish it (ring slot k % kRing once its previous item is read by all)
        const int rs = k % pair::kRing;
        if (k >= pair::kRing && !tc::mbar_wait(&bar_re[rs], (k / pair::kRing - 1) & 1, kWaitCycles)) {
          record(p.status, &abort_flag, HS_DEV_TIMEOUT);
          ok = false;
        }
        int w = -1;
        if (ok && !*(volatile int*)&abort_flag) {
          w = atomicAdd(ctr + H_ATTN_NEXT, 1);
          if (w >= n_items) w = -1;
        }
        *(volatile int*)&ring[rs] = w;
        tc::mbar_arrive(&bar_rf[rs]);
        if (w < 0) break;
        const int32_t* tl = M.tile(w / np);
        const int h0 = 2 * (w % np), kvh = h0 / (p.hq / p.hkv);
        CursorT<kMask> cur;
        cur.init(M, tl, p.window, p.bidir_root);
        if (!cur.next()) continue;  // an item without keys is skipped by every role
        // Q of this item once every S product of the previous item is done
        if (n_q >= 1 && !tc::mbar_wait(&bar_qe, (n_q - 1) & 1, kWaitCycles)) {
          record(p.status, &abort_flag, HS_DEV_TIMEOUT);
          break;
        }
        if (*(volatile int*)&abort_flag) break;
        tc::mbar_expect_tx(&bar_q, 2 * kTile);
        for (int x = 0; x < 2; ++x) {
          tc::tma_load_3d(smem + pair::kOffQ + x * kTile, &tm_q, 0, h0 + x, tl[TL_ROW0], &bar_q);
          tc::tma_load_3d(smem + pair::kOffQ + x * kTile + kSlab, &tm_q, 64, h0 + x, tl[TL_ROW0], &bar_q);
        }
        ++n_q;
        do {
          const int s = jg & 1, n = jg >> 1;
          const int npg = (cur.valid() + kPage - 1) / kPage;
          int pg[8];
          bool consecutive = npg == 8;
          for (int i = 0; i < 8; ++i) {
            pg[i] = -1;
            if (i < npg) {
              const int ref = cur.sp_off + cur.b0 / kPage + i;
              const int page = ref < n_ref ? refs[ref] : -1;
              if (page >= 0 && page < p.n_pages) {
                pg[i] = page;
              } else {
                hsd::set_status(p.status, ref < n_ref ? HS_DEV_BAD_PAGE : HS_DEV_BAD_META);
              }
            }
            if (i > 0 && (pg[i] < 0 || pg[i] != pg[i - 1] + 1)) consecutive = false;
          }
          if (pg[0] < 0) consecutive = false;
          uint8_t* ks = smem + pair::kOffK + s * kTile;
          uint8_t* vs = smem + pair::kOffV + s * kTile;
          if (n > 0 && !tc::mbar_wait(&bar_ke[s], (n - 1) & 1, kWaitCycles)) {
            record(p.status, &abort_flag, HS_DEV_TIMEOUT);
            ok = false;
            break;
          }
          if (*(volatile int*)&abort_flag) {
            ok = false;
            break;
          }
          tc::mbar_expect_tx(&bar_kf[s], kTile);
          if (consecutive) {
            const int y = (kvh * p.n_pages + pg[0]) * kPage;
            for (int half = 0; half < 2; ++half) tc::tma_load_2d(ks + half * kSlab, &tm_k128, half * 64, y, &bar_kf[s]);
          } else {
            for (int i = 0; i < 8; ++i) {
              const int y = pg[i] >= 0 ? (kvh * p.n_pages + pg[i]) * kPage : oob_y;
              for (int half = 0; half < 2; ++half)
                tc::tma_load_2d(ks + half * kSlab + i * 2048, &tm_k16, half * 64, y, &bar_kf[s]);
            }
          }
          if (n > 0 && !tc::mbar_wait(&bar_ve[s], (n - 1) & 1, kWaitCycles)) {
            record(p.status, &abort_flag, HS_DEV_TIMEOUT);
            ++jg;  // the K copy of this block is in flight: drain it below
            ok = false;
            break;
          }
          tc::mbar_expect_tx(&bar_vf[s], kTile);
          if (consecutive) {
            const int y = (kvh * p.n_pages + pg[0]) * kPage;
            for (int half = 0; half < 2; ++half) tc::tma_load_2d(vs + half * kSlab, &tm_v128, half * 64, y, &bar_vf[s]);
          } else {
            for (int i = 0; i < 8; ++i) {
              const int y = pg[i] >= 0 ? (kvh * p.n_pages + pg[i]) * kPage : oob_y;
              for (int half = 0; half < 2; ++half)
                tc::tma_load_2d(vs + half * kSlab + i * 2048, &tm_v16, half * 64, y, &bar_vf[s]);
            }
          }
          ++jg;
        } while (cur.next());
      }
      // drain: every copy this thread issued has landed before the CTA leaves
      if (n_q > 0) tc::mbar_wait(&bar_q, (n_q - 1) & 1, kWaitCycles);
      for (int i = (jg >= 2 ? jg - 2 : 0); i < jg; ++i) {
        tc::mbar_wait(&bar_kf[i & 1], (i >> 1) & 1, kWaitCycles);
        tc::mbar_wait(&bar_vf[i & 1], (i >> 1) & 1, kWaitCycles);
      }
    }
  } else if (warp == kWarpMma || warp == pair::kWarpMmaB) {
    // ---------------------------------------------------------------- MMA
    // One warp per head (head A: warp 9, head B: warp 10, on different SM sub-partitions), each converged:
    // waits are voted and one elected lane issues.  The two streams share the tensor pipe, so one warp's
    // bookkeeping between MMA groups is covered by the other's products.
    const int x = warp == kWarpMma ? 0 : 1;
    // (the whole warp, converged: waits are voted, one elected lane issues)
    {
      bool ok = true;
      int jg = 0, kq = 0;  // blocks issued over all items, non-empty items
      // Descriptors of the stage bases, built once; a K step or a 16-key step adds a constant to the
      // start-address field (addresses below 256 KB: no carry out of the field).  Every operand of an
      // MMA is then one add away, so MMAs issue at the tensor pipe's rate.
      const uint32_t s0 = tc::smem_u32(smem);
      const uint64_t dq0 = tc::sdesc_sw128(s0 + pair::kOffQ, 16, 1024);
      const uint64_t dk0 = tc::sdesc_sw128(s0 + pair::kOffK, 16, 1024);
      const uint64_t dv0 = tc::sdesc_sw128(s0 + pair::kOffV, kSlab, 1024);
      auto s_mma = [&](int x, int jj, int h) {  // S_X(jj, h) = Q_X K_jj[64h .. 64h+63]^T into S_X[h]
        const uint64_t a0 = dq0 + (uint64_t)(x * (kTile >> 4));
        const uint64_t b0 = dk0 + (uint64_t)(((jj & 1) * kTile + h * 8192) >> 4);
        const uint32_t d = tmem + pair::kTmS + 128 * x + 64 * h;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t off = (uint64_t)(((k >> 2) * kSlab + (k & 3) * 32) >> 4);
          tc::mma_bf16_ss_w(d, a0 + off, b0 + off, pair::kIdescQK, k > 0 ? 1u : 0u);
        }
        tc::mma_commit_w(&bar_sf[x][h]);
      };
      // O_X += P_X(jj, h) V_jj[64h .. 64h+63], per 32 keys: the high (or only) part, then (readout tiles)
      // the low part
      auto pv_mma = [&](int x, int jj, int h, bool first, bool precise) {
        const uint64_t b0 = dv0 + (uint64_t)(((jj & 1) * kTile + h * 8192) >> 4);
        const uint32_t pt = tmem + pair::kTmS + 128 * x + 64 * h, d = tmem + pair::kTmO + 128 * x;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            if (part == 1 && !precise) continue;
#pragma unroll
            for (int k = 0; k < 2; ++k) {  // keys 64 h + 32 g + 16 k .. +15
              tc::mma_bf16_ts_w(d, pt + 32 * g + 16 * part + 8 * k, b0 + (uint64_t)((g * 4096 + k * 2048) >> 4),
                              kIdescPV, (!first || g > 0 || part > 0 || k > 0) ? 1u : 0u);
            }
          }
        }
        tc::mma_commit_w(&bar_pv[x]);
      };
      for (int k = 0; ok; ++k) {
        const int w = item_of(k);
        if (w == -2) ok = false;
        if (w < 0) break;
        CursorT<kMask> cur;
        cur.init(M, M.tile(w / np), p.window, p.bidir_root);
        const bool precise = M.tile(w / np)[TL_READOUT] != 0;
        int n_blk = 0;
        while (cur.next()) ++n_blk;  // counted once: the loop needs no cursor
        if (n_blk == 0) continue;
        const int nh = 2 * n_blk;  // key halves of the item
        if (!__all_sync(~0u, tc::mbar_wait(&bar_q, kq & 1, kWaitCycles)) ||
            !__all_sync(~0u, tc::mbar_wait_spin(&bar_kf[jg & 1], (jg >> 1) & 1, kWaitCycles))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        // S of the item's first block, both halves: the buffers hold the previous item's last P, whose P.V is issued
        s_mma(x, jg, 0);
        s_mma(x, jg, 1);
        tc::mma_commit_w(&bar_ke[jg & 1]);
        if (n_blk == 1) tc::mma_commit_w(&bar_qe);
        for (int v = 0; ok && v < nh; ++v) {
          const int h = v & 1, jb = jg + (v >> 1);  // key half v: half h of block jb
          const int v2 = v + 2, jb2 = jg + (v2 >> 1);  // the half whose S goes into buffer h next
          {
            // (polling waits: a suspended MMA thread would notice the softmax late)
            if (!__all_sync(~0u, tc::mbar_wait_spin(&bar_pf[x][h], jb & 1, kWaitCycles)) ||
                (h == 0 && !__all_sync(~0u, tc::mbar_wait_spin(&bar_vf[jb & 1], (jb >> 1) & 1, kWaitCycles)))) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            pv_mma(x, jb, h, v == 0, precise);  // (the item's first P.V_X starts O_X afresh)
            if (h == 1) tc::mma_commit_w(&bar_ve[jb & 1]);
            if (v2 < nh) {
              if (h == 0 && !__all_sync(~0u, tc::mbar_wait_spin(&bar_kf[jb2 & 1], (jb2 >> 1) & 1, kWaitCycles))) {
                ok = false;
                break;
              }
              tc::fence_after_sync();
              s_mma(x, jb2, h);  // S_X[h] is overwritten after the P.V_X that reads it (issue order)
              if (h == 1) {
                tc::mma_commit_w(&bar_ke[jb2 & 1]);
                if (v2 == nh - 1) tc::mma_commit_w(&bar_qe);  // the item's last S products are issued
              }
            }
            if (*(volatile int*)&abort_flag) {  // (checked after the issue: off the P -> P.V path)
              ok = false;
              break;
            }
          }
        }
        jg += n_blk;
        ++kq;
      }
      if (!ok && lane == 0) record(p.status, &abort_flag, HS_DEV_TIMEOUT);
      // every MMA issued by the elected lane completes before O is read and TMEM is freed
      tc::mma_commit_w(&bar_done);
      tc::mbar_wait(&bar_done, 0, kWaitCycles);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int x = warp / 4;                      // head A or B
    const int t = (warp % 4) * 32 + lane;        // row of the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp % 4) * 32) << 16;
    const uint32_t sbuf = tmem + lane_base + pair::kTmS + 128 * x, obuf = tmem + lane_base + pair::kTmO + 128 * x;
    const float sl2 = p.scale_log2e;
    int jg = 0;  // blocks over all items
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int w = item_of(k);
      if (w == -2) ok = false;
      if (w < 0) break;
      const int32_t* tl = M.tile(w / np);
      const int h0 = 2 * (w % np);
      CursorT<kMask> cur;
      cur.init(M, tl, p.window, p.bidir_root);
      const int row = tl[TL_ROW0] + t;
      const bool active = t < tl[TL_N_ROWS];
      const bool precise = tl[TL_READOUT] != 0;
      int my_seg = -1, my_idx = 0, my_pos = 0, my_whole = 0;
      if (active) {
        my_seg = M.tok(row)[T_SEG];
        my_idx = M.tok(row)[T_IDX];
        my_pos = M.seg(my_seg)[S_POS0] + my_idx;
        my_whole = kMask && p.bidir_root && M.seg(my_seg)[S_LEVEL] == 0;
      }
      float m_used = -INFINITY, l = 0.f;
      int j = 0, n_blk = 0;
      {
        CursorT<kMask> c2 = cur;
        while (c2.next()) ++n_blk;
      }
      while (ok && cur.next()) {
        const int lim = cur.full() ? kBlk
                                   : (!active ? 0 : !cur.own ? cur.sp_n - cur.b0
                                                             : (cur.owner == my_seg ? (kMask && my_whole ? cur.sp_n : my_idx + 1) - cur.b0
                                                                                    : 0));
        // a window: this row's keys start at position my_pos - W + 1
        const int lo_in = (kMask && p.window > 0 && active) ? my_pos - p.window + 1 - (cur.p0 + cur.b0) : -(1 << 30);
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {  // key half h of the block: S_X[h]
          const int u = 2 * jg + h;    // key halves over all items (phases of bar_pv[x])
          const uint32_t sb = sbuf + 64 * h;
          const int lh = lim - 64 * h;  // this row's visible keys in the half: [lo_h, lh)
          const int lo_h = lo_in - 64 * h;
          // tcgen05.ld/st are warp-collective: every branch around them is decided warp-wide
          if (!__all_sync(~0u, tc::mbar_wait(&bar_sf[x][h], jg & 1, kWaitCycles))) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          // the half's 64 scores in registers (one load, one wait; scores past the row's visible keys read as
          // -inf), then pass 1: the row max
          const bool masked = __any_sync(~0u, lh < 64 || lo_h > 0);
          uint32_t sr[2][32];
          tc::tmem_ld32(sb, sr[0]);
          tc::tmem_ld32(sb + 32, sr[1]);
          tc::tmem_wait_ld();
          float mx = -INFINITY;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            if (masked) {
#pragma unroll
              for (int i = 0; i < 32; ++i) sr[c][i] = (32 * c + i < lh && 32 * c + i >= lo_h) ? sr[c][i] : 0xFF800000u;
            }
            float m2[2] = {mx, -INFINITY};
#pragma unroll
            for (int i = 0; i < 16; ++i)
              m2[i & 1] = tc::max3(m2[i & 1], __uint_as_float(sr[c][2 * i]), __uint_as_float(sr[c][2 * i + 1]));
            mx = fmaxf(m2[0], m2[1]);
          }
          const float m_new = fmaxf(m_used, mx * sl2);
          float factor = 1.f;
          const bool rescale = m_new > m_used + 8.f;
          if (rescale) {
            factor = exp2f(m_used - m_new);
            m_used = m_new;
          }
          const float mref = m_used == -INFINITY ? 0.f : m_used;
          // O_X rescaled before this half's P.V_X: it must first hold the previous half's P.V_X.  When this
          // S_X was seen, every P.V_X up to half u - 2 was complete, so the parity of half u - 1 is unambiguous.
          // Rows of the warp that keep their max multiply by factor = 1, which is exact.  The item's first half
          // never rescales (its P.V starts O_X afresh).
          if ((j > 0 || h > 0) && __any_sync(~0u, rescale)) {
            if (!__all_sync(~0u, tc::mbar_wait(&bar_pv[x], (u - 1) & 1, kWaitCycles))) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t o[32];
              tc::tmem_ld32(obuf + c * 32, o);
              tc::tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * factor);
              tc::tmem_st32(obuf + c * 32, o);
            }
          }
          // pass 2, 32 keys at a time: P = 2^(s log2e scale - m) over S in place; pairs of keys in fp32x2
          const uint64_t sc2 = tc::f2_pack(sl2, sl2), mm2 = tc::f2_pack(-mref, -mref);
          uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int g = 0; g < 2; ++g) {  // keys 64 h + 32 g .. +31: P words in the same 32 columns (16 high, 16 low)
            const uint32_t* r = sr[g];
            uint32_t hi[16], lo[16];
            if (precise) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float ya, yb;
                tc::f2_unpack(tc::f2_fma(tc::f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), sc2, mm2), ya, yb);
                const float a = tc::ex2_approx(ya), b = tc::ex2_approx(yb);
                const uint64_t ab = tc::f2_pack(a, b);
                acc2[i & 3] = tc::f2_add(acc2[i & 3], ab);
                hi[i] = tc::pack_bf16x2_trunc(a, b);
                float da, db;
                tc::f2_unpack(tc::f2_sub(ab, tc::f2_pack(__uint_as_float(hi[i] << 16), __uint_as_float(hi[i] & 0xFFFF0000u))), da, db);
                lo[i] = tc::pack_bf16x2(da, db);
              }
              tc::tmem_st16(sb + 32 * g, hi);
              tc::tmem_st16(sb + 32 * g + 16, lo);
            } else {
              // P rounded to bf16
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                float ya, yb;
                tc::f2_unpack(tc::f2_fma(tc::f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), sc2, mm2), ya, yb);
                const float a = tc::ex2_approx(ya), b = tc::ex2_approx(yb);
                acc2[i & 3] = tc::f2_add(acc2[i & 3], tc::f2_pack(a, b));
                hi[i] = tc::pack_bf16x2(a, b);
              }
              tc::tmem_st16(sb + 32 * g, hi);
            }
          }
          float rp[8];
#pragma unroll
          for (int a = 0; a < 4; ++a) tc::f2_unpack(acc2[a], rp[2 * a], rp[2 * a + 1]);
          const float rs = ((rp[0] + rp[1]) + (rp[2] + rp[3])) + ((rp[4] + rp[5]) + (rp[6] + rp[7]));
          l = l * factor + rs;
          // Waits on bar_pv[x] are for half u - 1 and come before this half's P is released, so the barrier is
          // never two phases past the one waited for.  The item's last half waits here for half u - 1, which
          // leaves the epilogue one phase (its own) to wait for.
          if (j == n_blk - 1 && h == 1 && !__all_sync(~0u, tc::mbar_wait(&bar_pv[x], (u - 1) & 1, kWaitCycles))) {
            ok = false;
            break;
          }
          tc::tmem_wait_st();
          tc::fence_before_sync();
          tc::mbar_arrive_warp(&bar_pf[x][h]);
        }
        ++j;
        ++jg;
      }
      if (!ok) break;
      if (j == 0) continue;
      // O_X / l once the item's last P.V_X is done (the one before it was waited for); then O_X may be
      // overwritten by the next item
      if (!__all_sync(~0u, tc::mbar_wait(&bar_pv[x], (2 * jg - 1) & 1, kWaitCycles))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const float inv = 1.f / l;
      __nv_bfloat16* dst = p.out + ((size_t)row * p.hq + h0 + x) * kD;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tc::tmem_ld32(obuf + c * 32, o);
        tc::tmem_wait_ld();
        if (active) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v;
            v.x = tc::pack_bf16x2(__uint_as_float(o[q * 8 + 0]) * inv, __uint_as_float(o[q * 8 + 1]) * inv);
            v.y = tc::pack_bf16x2(__uint_as_float(o[q * 8 + 2]) * inv, __uint_as_float(o[q * 8 + 3]) * inv);
            v.z = tc::pack_bf16x2(__uint_as_float(o[q * 8 + 4]) * inv, __uint_as_float(o[q * 8 + 5]) * inv);
            v.w = tc::pack_bf16x2(__uint_as_float(o[q * 8 + 6]) * inv, __uint_as_float(o[q * 8 + 7]) * inv);
            *reinterpret_cast<uint4*>(dst + c * 32 + q * 8) = v;
          }
        }
      }
    }
    if (!ok) record(p.status, &abort_flag, HS_DEV_TIMEOUT);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == kWarpMma) tc::tmem_dealloc(tmem, 512);
  // the last CTA to finish sets the counters back to zero for the next launch on this metadata (every CTA's
  // last take from H_ATTN_NEXT precedes its increment of H_ATTN_DONE)
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(ctr + H_ATTN_DONE, 1) == n_cta - 1) {
      atomicExch(ctr + H_ATTN_NEXT, 0);
      atomicExch(ctr + H_ATTN_DONE, 0);
      __threadfence();
    }
  }
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

bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
              const cuuint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Runs the tensor-core kernel when it applies (bf16, d = 128); returns
// HS_EUNSUPPORTED otherwise so the caller takes the CUDA-core kernel.
hs_status hs_fork_attn_tc_launch(const hs_round_caps* caps, const void* meta, int hq, int hkv, int d, float scale,
                                 const void* q, const void* kp, const void* vp, int n_pages, void* out,
                                 int32_t* status, cudaStream_t st, int window, int bidir_root) {
  if (d != kD) return HS_EUNSUPPORTED;
  if (caps->max_tiles <= 0) return HS_OK;
  // the pool rows must be addressable by 32-bit TMA coordinates
  if ((long long)hkv * n_pages * kPage + kPage >= (1LL << 31)) return HS_EUNSUPPORTED;
  const long long T = caps->max_tokens;
  CUtensorMap m_q, m_k16, m_k128, m_v16, m_v128;
  {
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)hq, (cuuint64_t)(T > 0 ? T : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)hq * kD * 2};
    cuuint32_t box[3] = {64, 1, 128};
    if (!make_map(&m_q, q, 3, dims, strides, box)) return hs::fail(HS_ECUDA, "tensor map for q");
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)hkv * n_pages * kPage};
    cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    cuuint32_t b16[2] = {64, 16}, b128[2] = {64, 128};
    if (!make_map(&m_k16, kp, 2, dims, strides, b16) || !make_map(&m_k128, kp, 2, dims, strides, b128) ||
        !make_map(&m_v16, vp, 2, dims, strides, b16) || !make_map(&m_v128, vp, 2, dims, strides, b128))
      return hs::fail(HS_ECUDA, "tensor map for the page pools");
  }
  static std::atomic<bool> configured[hsd::kMaxDevices];  // zero-initialised: per device
  const int slot = hsd::device_slot();
  if (slot < 0) return hs::fail(HS_ECUDA, "fork_attn_tc: no usable CUDA device");
  if (!configured[slot].load()) {
    if (cudaFuncSetAttribute(fork_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes + 1024) !=
            cudaSuccess ||
        cudaFuncSetAttribute(fork_attn_tc2_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             pair::kSmemBytes + 1024) != cudaSuccess ||
        cudaFuncSetAttribute(fork_attn_tc2_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             pair::kSmemBytes + 1024) != cudaSuccess)
      return hs::fail(HS_ECUDA, "fork_attn_tc: cannot raise the shared-memory limit");
    configured[slot].store(true);
  }
  Params prm{(const int32_t*)meta, hq, hkv, n_pages, scale * 1.4426950408889634f, (__nv_bfloat16*)out, status,
             window, bidir_root};
  if ((window > 0 || bidir_root) && (hq / hkv) % 2 != 0) return HS_EUNSUPPORTED;  // (masks: the paired kernel)
  if ((hq / hkv) % 2 == 0) {  // two query heads that share a KV head per CTA, one persistent CTA per SM
    static std::atomic<int> sm_count[hsd::kMaxDevices];  // per device, 0 until read
    int n_sm = sm_count[slot].load();
    if (n_sm <= 0) {
      if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, slot) != cudaSuccess || n_sm <= 0)
        return hs::fail(HS_ECUDA, "fork_attn_tc: cannot read the SM count");
      sm_count[slot].store(n_sm);
    }
    const int items = caps->max_tiles * (hq / 2);
    const dim3 grid(items < n_sm ? items : n_sm);
    if (window > 0 || bidir_root)
      hsd::launch_pdl(fork_attn_tc2_kernel<true>, grid, dim3(pair::kThreads), pair::kSmemBytes + 1024, st, m_q,
                      m_k16, m_k128, m_v16, m_v128, prm);
    else
      hsd::launch_pdl(fork_attn_tc2_kernel<false>, grid, dim3(pair::kThreads), pair::kSmemBytes + 1024, st, m_q,
                      m_k16, m_k128, m_v16, m_v128, prm);
  } else {
    hsd::launch_pdl(fork_attn_tc_kernel, dim3(caps->max_tiles * hq), dim3(kThreads), kSmemBytes + 1024, st,
                    m_q, m_k16, m_k128, m_v16, m_v128, prm);
  }
  HS_LAUNCH_CHECK("fork_attn_tc");
  return HS_OK;
}
