// fork_attn.cu -- ForkAttention prefill: KV page write + paged tree attention.
//
// Flide, "Accelerating Decision Inference with Exact State Forking":
//   section 3.2.1, Eq. 3 -- a token x sees y iff same request, y's node is
//     x's node or an ancestor, and t_y <= t_x;
//   section 3.3.1 -- keys come from two sources (the shared state and the
//     query's own question), other requests are skipped, full key blocks are
//     read without a mask and only partial blocks are masked;
//   section 3.4 -- a resumed state's cached keys precede the new ones;
//   section 3.5 -- a question's reductions start at the fork and do not
//     depend on the rest of the round.
// ForkServe README, "Copy-on-write context tree": writes go to a node's own
// pages only; children read their ancestors' pages in place.
//
// Two attention paths share the metadata: a bf16 d=128 tensor-core kernel
// (fork_attn_tc.cu) and the CUDA-core kernel here (fp32 inputs, d=64, and
// any shape the tensor-core kernel does not take).
#include <cuda_bf16.h>

#include "device.cuh"

using namespace hsm;
using hsd::Meta;

namespace {

// ---------------------------------------------------------------------------
// K1: write the stream's K/V into each node's own pages.  The thread block
// of a node's last token also zeroes the unused rows of that node's last
// page, so every page row a key block can touch holds finite values.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256)
kv_page_write_kernel(const int32_t* __restrict__ meta, int hkv, int d, const T* __restrict__ k_new,
                     const T* __restrict__ v_new, T* __restrict__ kp, T* __restrict__ vp, int n_pages,
                     int32_t* status) {
  hsd::pdl_wait();  // (launched with launch_pdl: nothing global before this)
  hsd::pdl_trigger();
  Meta M{meta};
  const int n_tok = M.h(H_N_TOK);
  const int n_seg = M.h(H_N_SEG);
  const int n_ref = M.h(H_N_PAGE_REF);
  constexpr int VEC = 16 / sizeof(T);
  const int vpt = hkv * d / VEC;  // 16-byte vectors per token, per tensor
  // one token per warp: the eight warps' metadata lookups (token -> node -> page) are in flight together
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (int t = blockIdx.x * 8 + warp; t < n_tok; t += gridDim.x * 8) {
    const int32_t* tk = M.tok(t);
    const int seg = tk[T_SEG], idx = tk[T_IDX];
    if (seg < 0 || seg >= n_seg) { hsd::set_status(status, HS_DEV_BAD_META); continue; }
    const int32_t* sg = M.seg(seg);
    const int ref = sg[S_PAGE_REF_OFF] + idx / kPage;
    if (idx < 0 || idx >= sg[S_LEN] || ref >= n_ref) { hsd::set_status(status, HS_DEV_BAD_META); continue; }
    const int page = M.page_ref()[ref];
    if (page < 0 || page >= n_pages) { hsd::set_status(status, HS_DEV_BAD_PAGE); continue; }
    const int row = idx % kPage;
    const bool last = idx == sg[S_LEN] - 1;
    for (int j = lane; j < 2 * vpt; j += 32) {
      const int which = j >= vpt;
      const int jj = which ? j - vpt : j;
      const int e = jj * VEC;
      const int h = e / d, c = e % d;
      const T* src = (which ? v_new : k_new) + (size_t)t * hkv * d + e;
      T* dst = (which ? vp : kp) + (((size_t)h * n_pages + page) * kPage + row) * d + c;
      *reinterpret_cast<float4*>(dst) = *reinterpret_cast<const float4*>(src);
      if (last)
        for (int rr = row + 1; rr < kPage; ++rr)
          *reinterpret_cast<float4*>(dst + (size_t)(rr - row) * d) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// ---------------------------------------------------------------------------
// K2 (CUDA cores): one warp per query row, 16 rows per thread block, key
// blocks of 32 staged in shared memory in fp32.  Each row walks the tile's
// spans in order (shared spans, then own spans) in blocks of 32 keys from
// each span's start and skips blocks where it sees no key, so its sequence
// of online-softmax steps depends on its own visible keys only.
// ---------------------------------------------------------------------------
constexpr int kSimtRows = 16;
constexpr int kSimtKeys = 32;

template <typename T, int D>
__global__ void __launch_bounds__(kSimtRows * 32)
fork_attn_simt_kernel(const int32_t* __restrict__ meta, int hq, int hkv, float scale_log2e,
                      const T* __restrict__ q, const T* __restrict__ kp, const T* __restrict__ vp, int n_pages,
                      T* __restrict__ out, int32_t* status, int window, int bidir_root) {
  constexpr int DP = D + 1;
  constexpr int CPL = D / 32;  // output columns per lane
  __shared__ float q_s[kSimtRows][D];
  __shared__ float k_s[kSimtKeys][DP];
  __shared__ float v_s[kSimtKeys][D];

  Meta M{meta};
  const int tile_id = blockIdx.x / (kTileRows / kSimtRows);
  const int sub = blockIdx.x % (kTileRows / kSimtRows);
  if (tile_id >= M.h(H_N_TILE)) return;
  const int32_t* tl = M.tile(tile_id);
  const int row0 = tl[TL_ROW0], n_rows = tl[TL_N_ROWS];
  if (sub * kSimtRows >= n_rows) return;
  const int sub_lo = row0 + sub * kSimtRows;
  const int sub_hi = row0 + min(n_rows, (sub + 1) * kSimtRows);  // exclusive
  const int h = blockIdx.y;
  const int kvh = h / (hq / hkv);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int row = sub_lo + warp;
  const bool active = row < sub_hi;
  const int n_ref = M.h(H_N_PAGE_REF);
  const int32_t* refs = M.page_ref();

  int my_seg = -1, my_idx = 0, my_pos = 0, my_whole = 0;
  if (active) {
    my_seg = M.tok(row)[T_SEG];
    my_idx = M.tok(row)[T_IDX];
    my_pos = M.seg(my_seg)[S_POS0] + my_idx;
    my_whole = bidir_root && M.seg(my_seg)[S_LEVEL] == 0;  // a bidirectional root: its rows see all of it
  }
  // stage this warp's query row, pre-scaled so that exp2 gives e^(scale s)
  for (int c = lane; c < D; c += 32)
    q_s[warp][c] = active ? hsd::to_f(q[((size_t)row * hq + h) * D + c]) * scale_log2e : 0.f;

  float o[CPL];
#pragma unroll
  for (int i = 0; i < CPL; ++i) o[i] = 0.f;
  float m = -INFINITY, l = 0.f;

  const int n_shared = tl[TL_N_SHARED], n_spans = n_shared + tl[TL_N_OWN];
  const int32_t* tspans = M.tile_spans() + tl[TL_SPAN_OFF];
  int p_shared = 0;  // position of the next shared span's first key (shared spans follow the path in order)
  for (int si = 0; si < n_spans; ++si) {
    const int32_t* sp = M.span(tspans[si]);
    const int sp_off = sp[SP_PAGE_REF_OFF], sp_n = sp[SP_N_TOK], owner = sp[SP_OWNER];
    const bool own = si >= n_shared;
    int kmax = sp_n;  // keys this thread block needs from the span
    int p0 = p_shared;  // position of the span's first key
    if (own) {
      const int32_t* og = M.seg(owner);
      const int lo = max(sub_lo, og[S_STREAM_OFF]);
      const int hi = min(sub_hi, og[S_STREAM_OFF] + og[S_LEN]);
      const bool whole = bidir_root && og[S_LEVEL] == 0;
      kmax = hi > lo ? (whole ? og[S_LEN] : hi - og[S_STREAM_OFF]) : 0;
      p0 = og[S_POS0];
    } else {
      p_shared += sp_n;
    }
    // keys of this span the row sees: [my_lo, my_n) -- all (shared), up to itself (own; all of a
    // bidirectional root), none (sibling); a window starts them at position my_pos - W + 1
    const int my_n = !active ? 0 : !own ? sp_n : (owner == my_seg ? (my_whole ? sp_n : my_idx + 1) : 0);
    const int my_lo = (window > 0 && active) ? max(0, my_pos - window + 1 - p0) : 0;
    for (int b0 = 0; b0 < kmax; b0 += kSimtKeys) {
      __syncthreads();
      const int nb = min(kSimtKeys, kmax - b0);
      for (int e = threadIdx.x; e < kSimtKeys * (D / 4); e += blockDim.x) {
        const int r = e / (D / 4), c4 = (e % (D / 4)) * 4;
        float kv[4] = {0.f, 0.f, 0.f, 0.f}, vv[4] = {0.f, 0.f, 0.f, 0.f};
        if (r < nb) {
          const int key = b0 + r;
          const int ref = sp_off + key / kPage;
          const int page = ref < n_ref ? refs[ref] : -1;
          if (page >= 0 && page < n_pages) {
            const size_t base = (((size_t)kvh * n_pages + page) * kPage + key % kPage) * D + c4;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              kv[i] = hsd::to_f(kp[base + i]);
              vv[i] = hsd::to_f(vp[base + i]);
            }
          } else {
            hsd::set_status(status, ref < n_ref ? HS_DEV_BAD_PAGE : HS_DEV_BAD_META);
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          k_s[r][c4 + i] = kv[i];
          v_s[r][c4 + i] = vv[i];
        }
      }
      __syncthreads();
      const int nvis = min(kSimtKeys, my_n - b0), nlo = max(0, my_lo - b0);
      if (nvis <= nlo) continue;  // this row sees nothing in the block
      float s = -INFINITY;
      if (lane < nvis && lane >= nlo) {
        float acc = 0.f;
#pragma unroll 8
        for (int c = 0; c < D; ++c) acc = fmaf(q_s[warp][c], k_s[lane][c], acc);
        s = acc;
      }
      const float m_new = fmaxf(m, hsd::warp_max(s));
      const float corr = exp2f(m - m_new);
      const float p = (lane < nvis && lane >= nlo) ? exp2f(s - m_new) : 0.f;
      l = l * corr + hsd::warp_sum(p);
#pragma unroll
      for (int i = 0; i < CPL; ++i) o[i] *= corr;
      for (int j = 0; j < nvis; ++j) {
        const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
        for (int i = 0; i < CPL; ++i) o[i] = fmaf(pj, v_s[j][lane + 32 * i], o[i]);
      }
      m = m_new;
    }
  }
  if (active) {
    const float inv = 1.f / l;
#pragma unroll
    for (int i = 0; i < CPL; ++i) out[((size_t)row * hq + h) * D + lane + 32 * i] = hsd::from_f<T>(o[i] * inv);
  }
}

template <typename T>
hs_status launch_attn_simt(const hs_round_caps* caps, const void* meta, int hq, int hkv, int d, float scale,
                           const void* q, const void* kp, const void* vp, int n_pages, void* out, int32_t* status,
                           cudaStream_t st, int window, int bidir_root) {
  dim3 grid(caps->max_tiles * (kTileRows / kSimtRows), hq);
  const float sl2 = scale * 1.4426950408889634f;
  if (grid.x == 0) return HS_OK;
  if (d == 128)
    fork_attn_simt_kernel<T, 128><<<grid, kSimtRows * 32, 0, st>>>(
        (const int32_t*)meta, hq, hkv, sl2, (const T*)q, (const T*)kp, (const T*)vp, n_pages, (T*)out, status,
        window, bidir_root);
  else
    fork_attn_simt_kernel<T, 64><<<grid, kSimtRows * 32, 0, st>>>(
        (const int32_t*)meta, hq, hkv, sl2, (const T*)q, (const T*)kp, (const T*)vp, n_pages, (T*)out, status,
        window, bidir_root);
  HS_LAUNCH_CHECK("fork_attn_simt");
  return HS_OK;
}

template <typename T>
hs_status launch_kv_write(const hs_round_caps* caps, const void* meta, int hkv, int d, const void* k_new,
                          const void* v_new, void* kp, void* vp, int n_pages, int32_t* status, cudaStream_t st) {
  const int want = (caps->max_tokens + 7) / 8;  // eight tokens per block
  const int grid = want < 152 * 8 ? want : 152 * 8;
  if (grid <= 0) return HS_OK;
  hsd::launch_pdl(kv_page_write_kernel<T>, dim3(grid), dim3(256), 0, st, (const int32_t*)meta, hkv, d,
                  (const T*)k_new, (const T*)v_new, (T*)kp, (T*)vp, n_pages, status);
  HS_LAUNCH_CHECK("kv_page_write");
  return HS_OK;
}

}  // namespace

// tensor-core path (fork_attn_tc.cu); returns HS_EUNSUPPORTED when it does not apply
hs_status hs_fork_attn_tc_launch(const hs_round_caps* caps, const void* meta, int hq, int hkv, int d, float scale,
                                 const void* q, const void* kp, const void* vp, int n_pages, void* out,
                                 int32_t* status, cudaStream_t st, int window, int bidir_root);

static bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

static hs_status check_common(const hs_round_caps* caps, const void* meta, hs_dtype dt, int hkv, int d,
                              int n_pages) {
  HS_CHECK_ARG(caps && meta, "null argument");
  HS_CHECK_ARG(hkv > 0, "hkv must be > 0");
  HS_CHECK_ARG(n_pages > 0, "n_pages must be > 0");
  if (d != 64 && d != 128) return hs::fail(HS_EUNSUPPORTED, "head size %d (built: 64, 128)", d);
  if (dt != HS_F32 && dt != HS_BF16) return hs::fail(HS_EUNSUPPORTED, "dtype %d", (int)dt);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return hs::fail(HS_ECUDA, "no CUDA device");
  return HS_OK;
}

extern "C" hs_status hs_kv_page_write(const hs_round_caps* caps, const void* dev_meta, hs_dtype dt, int32_t hkv,
                                      int32_t d, const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                                      int32_t n_pages, int32_t* dev_status, void* stream) {
  HS_CHECK_ARG(k_new && v_new && k_pages && v_pages, "null argument");
  HS_CHECK_ARG(aligned16(k_new) && aligned16(v_new) && aligned16(k_pages) && aligned16(v_pages),
               "tensors must be 16-byte aligned");
  hs_status s = check_common(caps, dev_meta, dt, hkv, d, n_pages);
  if (s != HS_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  if (dt == HS_BF16)
    return launch_kv_write<__nv_bfloat16>(caps, dev_meta, hkv, d, k_new, v_new, k_pages, v_pages, n_pages,
                                          dev_status, st);
  return launch_kv_write<float>(caps, dev_meta, hkv, d, k_new, v_new, k_pages, v_pages, n_pages, dev_status, st);
}

extern "C" hs_status hs_fork_attn_masked(const hs_round_caps* caps, const void* dev_meta, hs_dtype dt, int32_t hq,
                                         int32_t hkv, int32_t d, float scale, const hs_attn_mask* mask, const void* q,
                                         const void* k_pages, const void* v_pages, int32_t n_pages, void* out,
                                         int32_t* dev_status, void* stream) {
  HS_CHECK_ARG(q && k_pages && v_pages && out, "null argument");
  HS_CHECK_ARG(hq > 0 && hkv > 0 && hq % hkv == 0, "hq=%d must be a positive multiple of hkv=%d", hq, hkv);
  HS_CHECK_ARG(scale > 0.f && scale < 1e30f, "bad scale");
  HS_CHECK_ARG(aligned16(q) && aligned16(k_pages) && aligned16(v_pages) && aligned16(out),
               "tensors must be 16-byte aligned");
  const int window = mask ? mask->window : 0, bidir = mask ? mask->bidirectional_root : 0;
  HS_CHECK_ARG(window >= 0, "window %d must be >= 0 (0 = none)", window);
  HS_CHECK_ARG(bidir == 0 || bidir == 1, "bidirectional_root must be 0 or 1");
  hs_status s = check_common(caps, dev_meta, dt, hkv, d, n_pages);
  if (s != HS_OK) return s;
  cudaStream_t st = (cudaStream_t)stream;
  if (dt == HS_BF16) {
    s = hs_fork_attn_tc_launch(caps, dev_meta, hq, hkv, d, scale, q, k_pages, v_pages, n_pages, out, dev_status, st,
                               window, bidir);
    if (s != HS_EUNSUPPORTED) return s;
    return launch_attn_simt<__nv_bfloat16>(caps, dev_meta, hq, hkv, d, scale, q, k_pages, v_pages, n_pages, out,
                                           dev_status, st, window, bidir);
  }
  return launch_attn_simt<float>(caps, dev_meta, hq, hkv, d, scale, q, k_pages, v_pages, n_pages, out, dev_status, st,
                                 window, bidir);
}

extern "C" hs_status hs_fork_attn(const hs_round_caps* caps, const void* dev_meta, hs_dtype dt, int32_t hq,
                                  int32_t hkv, int32_t d, float scale, const void* q, const void* k_pages,
                                  const void* v_pages, int32_t n_pages, void* out, int32_t* dev_status, void* stream) {
  return hs_fork_attn_masked(caps, dev_meta, dt, hq, hkv, d, scale, nullptr, q, k_pages, v_pages, n_pages, out,
                             dev_status, stream);
}

extern "C" hs_status hs_fork_attn_prefill(const hs_round_caps* caps, const void* dev_meta, hs_dtype dt, int32_t hq,
                                          int32_t hkv, int32_t d, float scale, const void* q, const void* k_new,
                                          const void* v_new, void* k_pages, void* v_pages, int32_t n_pages, void* out,
                                          int32_t* dev_status, void* stream) {
  HS_CHECK_ARG(hq > 0 && hkv > 0 && hq % hkv == 0, "hq=%d must be a positive multiple of hkv=%d", hq, hkv);
  HS_CHECK_ARG(q && out && scale > 0.f && scale < 1e30f, "bad query, output or scale");
  hs_status s = hs_kv_page_write(caps, dev_meta, dt, hkv, d, k_new, v_new, k_pages, v_pages, n_pages, dev_status,
                                 stream);
  if (s != HS_OK) return s;
  return hs_fork_attn(caps, dev_meta, dt, hq, hkv, d, scale, q, k_pages, v_pages, n_pages, out, dev_status, stream);
}
