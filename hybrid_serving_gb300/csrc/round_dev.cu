// round_dev.cu -- parts of a round's metadata built on the GPU from the
// segment table already in device memory.
//
// Flide, "Accelerating Decision Inference with Exact State Forking", section
// 3.3.1 (the metadata that fixed-shape launches read is GPU-resident; the GDN
// layers iterate over a fixed-length chunk list), section 3.5 (every node
// starts a chunk at its first token).
//
// The chunk list: the nodes in stream order (Eq. 2: increasing stream
// offset), each cut into chunks of 64 tokens from its first token, the last
// one possibly shorter; record {node, first stream row, length, index within
// the node}.  A node's first chunk is the number of chunks of the nodes that
// start before it in the stream.  One CTA: the nodes' (stream offset, chunk
// count) pairs are staged in shared memory a tile at a time, and each thread
// counts, for its own nodes, the chunks of every node earlier in the stream --
// then writes its nodes' records and chunk fields.  The result is the host
// round builder's, word for word.
#include <cuda_runtime.h>

#include "device.cuh"

using namespace hsm;
using hsd::Meta;

namespace {

constexpr int kThreads = 512;
constexpr int kTileSeg = 2048;

__global__ void __launch_bounds__(kThreads) build_chunks_kernel(int32_t* meta, int32_t* status) {
  __shared__ int32_t s_off[kTileSeg], s_nc[kTileSeg];
  __shared__ int32_t s_tot, s_max;
  const int n_seg = meta[H_N_SEG];
  const int cap_chunk = meta[H_CAP_CHUNK];
  int32_t* seg = meta + meta[H_OFF_SEG];
  int32_t* chunk = meta + meta[H_OFF_CHUNK];
  if (threadIdx.x == 0) {
    s_tot = 0;
    s_max = 0;
  }
  __syncthreads();
  // per thread: its nodes i = threadIdx.x, + kThreads, ...  -- their chunk offsets accumulate over all tiles
  constexpr int kMine = 8;  // up to kThreads * kMine nodes
  int32_t first[kMine];
#pragma unroll
  for (int m = 0; m < kMine; ++m) first[m] = 0;
  for (int t0 = 0; t0 < n_seg; t0 += kTileSeg) {
    const int nt = min(kTileSeg, n_seg - t0);
    for (int j = threadIdx.x; j < nt; j += kThreads) {
      const int32_t* g = seg + (size_t)(t0 + j) * kSegWords;
      s_off[j] = g[S_STREAM_OFF];
      s_nc[j] = (g[S_LEN] + kChunk - 1) / kChunk;
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < kMine; ++m) {
      const int i = threadIdx.x + m * kThreads;
      if (i >= n_seg) break;
      const int my_off = seg[(size_t)i * kSegWords + S_STREAM_OFF];
      int acc = 0;
      for (int j = 0; j < nt; ++j) acc += s_off[j] < my_off ? s_nc[j] : 0;
      first[m] += acc;
    }
    __syncthreads();
  }
  int tot = 0, mx = 0;
#pragma unroll
  for (int m = 0; m < kMine; ++m) {
    const int i = threadIdx.x + m * kThreads;
    if (i >= n_seg) break;
    int32_t* g = seg + (size_t)i * kSegWords;
    const int off = g[S_STREAM_OFF], len = g[S_LEN], nc = (len + kChunk - 1) / kChunk;
    if (first[m] + nc > cap_chunk) {
      hsd::set_status(status, HS_DEV_BAD_META);
      continue;
    }
    g[S_CHUNK_OFF] = first[m];
    g[S_N_CHUNK] = nc;
    for (int c = 0; c < nc; ++c) {
      int32_t* rec = chunk + (size_t)(first[m] + c) * kChunkWords;
      rec[C_SEG] = i;
      rec[C_ROW0] = off + c * kChunk;
      rec[C_LEN] = min(kChunk, len - c * kChunk);
      rec[C_IDX] = c;
    }
    tot += nc;
    mx = max(mx, nc);
  }
  atomicAdd(&s_tot, tot);
  atomicMax(&s_max, mx);
  __syncthreads();
  if (threadIdx.x == 0) {
    meta[H_N_CHUNK] = s_tot;
    meta[H_MAX_SEG_CHUNKS] = s_max;
  }
}

// ------------------------------------------------------------------ tile table
// The attention tiles (Flide section 3.3.1; section 3.5: tiles start at the node), as the host round builder
// forms them: in stream order, a root or a node of more than 128 tokens gets one tile per 128 rows; a run of
// consecutive siblings (same parent, each <= 128 rows) is packed into tiles of at most 128 rows.  A tile's
// span list: the root's history spans, each ancestor's own span (root first), then the own spans of the
// tile's nodes; its work = key blocks of 128 over those spans (a single node's own span counted up to the
// tile's last row); READOUT = a readout row among its rows (packed: a member with a readout).  Tiles are
// then ordered by cost = work x (readout ? 7 : 5), heaviest first, ties in generation order.
constexpr int kMaxTileSeg = 4096;  // nodes ranked in shared memory
constexpr int kSegMine = kMaxTileSeg / kThreads;  // nodes per thread in the ranking
constexpr int kTileMine = 8;       // tiles per thread in the final permutation

__device__ __forceinline__ int blocks128(int keys) { return (keys + kTileRows - 1) / kTileRows; }

// the ancestor spans of node id (history of its root, then every ancestor's own span, root first) into out;
// returns their number (out may be null: count only)
// (the walk stops after max_depth parents: -1 then means inconsistent metadata)
__device__ int ancestor_spans(const int32_t* seg, int id, int32_t* out, int max_depth) {
  int d = 0, top = id;
  for (int p = seg[(size_t)id * kSegWords + S_PARENT]; p >= 0; p = seg[(size_t)p * kSegWords + S_PARENT]) {
    if (++d > max_depth) return -1;
    top = p;
  }
  const int32_t hist = seg[(size_t)top * kSegWords + S_HIST];
  const int h0 = hist & ((1 << kHistShift) - 1), nh = hist >> kHistShift;
  if (out) {
    for (int k = 0; k < nh; ++k) out[k] = h0 + k;
    int pos = nh + d - 1;
    for (int p = seg[(size_t)id * kSegWords + S_PARENT]; p >= 0; p = seg[(size_t)p * kSegWords + S_PARENT])
      out[pos--] = seg[(size_t)p * kSegWords + S_OWN_SPAN];
  }
  return nh + d;
}

__global__ void __launch_bounds__(kThreads) build_tiles_kernel(int32_t* meta, int32_t* status) {
  __shared__ int32_t s_order[kMaxTileSeg], s_cost[kMaxTileSeg], s_off[kTileSeg];
  __shared__ int32_t s_ntile, s_nspan, s_bad;
  const int n_seg = meta[H_N_SEG];
  const int cap_tile = meta[H_CAP_TILE], cap_tspan = meta[H_CAP_TILE_SPAN], max_depth = meta[H_CAP_LEVEL];
  if (n_seg > kMaxTileSeg || n_seg > meta[H_CAP_SEG]) {
    if (threadIdx.x == 0) hsd::set_status(status, HS_DEV_BAD_META);
    return;
  }
  const int32_t* seg = meta + meta[H_OFF_SEG];
  const int32_t* span = meta + meta[H_OFF_SPAN];
  int32_t* tile = meta + meta[H_OFF_TILE];
  int32_t* tspan = meta + meta[H_OFF_TILE_SPAN];
  // 1. stream order: node i goes to the rank of its stream offset (offsets are distinct: no node is empty)
  int rank[kSegMine];
#pragma unroll
  for (int m = 0; m < kSegMine; ++m) rank[m] = 0;
  for (int t0 = 0; t0 < n_seg; t0 += kTileSeg) {
    const int nt = min(kTileSeg, n_seg - t0);
    for (int j = threadIdx.x; j < nt; j += kThreads) s_off[j] = seg[(size_t)(t0 + j) * kSegWords + S_STREAM_OFF];
    __syncthreads();
#pragma unroll
    for (int m = 0; m < kSegMine; ++m) {
      const int i = threadIdx.x + m * kThreads;
      if (i >= n_seg) break;
      const int my_off = seg[(size_t)i * kSegWords + S_STREAM_OFF];
      int acc = 0;
      for (int j = 0; j < nt; ++j) acc += s_off[j] < my_off;
      rank[m] += acc;
    }
    __syncthreads();
  }
#pragma unroll
  for (int m = 0; m < kSegMine; ++m) {
    const int i = threadIdx.x + m * kThreads;
    if (i < n_seg) s_order[rank[m]] = i;
  }
  __syncthreads();
  // 2. the tiles in generation order, straight into the tile table and the tile span lists (one thread)
  if (threadIdx.x == 0) {
    int nt = 0, ns = 0;
    bool bad = false;
    auto emit = [&](int row0, int rows, int n_shared, int n_own, int work, int seg0, int ro) {
      if (nt >= cap_tile || nt >= kMaxTileSeg) {
        bad = true;
        return;
      }
      int32_t* r = tile + (size_t)nt * kTileWords;
      r[TL_ROW0] = row0;
      r[TL_N_ROWS] = rows;
      r[TL_SPAN_OFF] = ns - n_shared - n_own;
      r[TL_N_SHARED] = n_shared;
      r[TL_N_OWN] = n_own;
      r[TL_WORK] = work;
      r[TL_SEG0] = seg0;
      r[TL_READOUT] = ro;
      s_cost[nt] = work * (ro ? 7 : 5);
      ++nt;
    };
    for (int oi = 0; oi < n_seg && !bad;) {
      const int id = s_order[oi];
      const int32_t* g = seg + (size_t)id * kSegWords;
      const int n_anc = ancestor_spans(seg, id, nullptr, max_depth);
      int anc_work = 0;
      if (n_anc < 0 || ns + n_anc > cap_tspan) {
        bad = true;
        break;
      }
      ancestor_spans(seg, id, tspan + ns, max_depth);  // (written again for every tile of the node below)
      for (int k = 0; k < n_anc; ++k) anc_work += blocks128(span[(size_t)tspan[ns + k] * kSpanWords + SP_N_TOK]);
      const int len = g[S_LEN], off = g[S_STREAM_OFF], ro_row = g[S_READOUT_ROW];
      if (len > kTileRows || g[S_PARENT] < 0) {
        for (int r0 = 0; r0 < len && !bad; r0 += kTileRows) {
          const int nr = min(kTileRows, len - r0);
          if (ns + n_anc + 1 > cap_tspan) {
            bad = true;
            break;
          }
          ancestor_spans(seg, id, tspan + ns, max_depth);
          tspan[ns + n_anc] = g[S_OWN_SPAN];
          ns += n_anc + 1;
          emit(off + r0, nr, n_anc, 1, anc_work + blocks128(r0 + nr), id, ro_row >= off + r0 && ro_row < off + r0 + nr);
        }
        ++oi;
        continue;
      }
      // consecutive siblings, each <= 128 rows, while they fit
      int oj = oi, rows = 0, work = anc_work, ro = 0;
      const int parent = g[S_PARENT];
      while (oj < n_seg) {
        const int32_t* t = seg + (size_t)s_order[oj] * kSegWords;
        if (t[S_PARENT] != parent || t[S_LEN] > kTileRows || rows + t[S_LEN] > kTileRows) break;
        if (ns + n_anc + (oj - oi) + 1 > cap_tspan) {
          bad = true;
          break;
        }
        tspan[ns + n_anc + (oj - oi)] = t[S_OWN_SPAN];
        rows += t[S_LEN];
        work += blocks128(t[S_LEN]);
        ro |= t[S_READOUT_ROW] >= 0;
        ++oj;
      }
      if (bad) break;
      ns += n_anc + (oj - oi);
      emit(off, rows, n_anc, oj - oi, work, id, ro);
      oi = oj;
    }
    s_ntile = nt;
    s_nspan = ns;
    s_bad = bad;
    if (bad) hsd::set_status(status, HS_DEV_BAD_META);
  }
  __syncthreads();
  if (s_bad) return;
  const int nt = s_ntile;
  // 3. heaviest first, ties in generation order: each thread ranks its tiles, then all move them at once
  int32_t rec[kTileMine][kTileWords];
  int dst[kTileMine];
#pragma unroll
  for (int m = 0; m < kTileMine; ++m) {
    const int i = threadIdx.x + m * kThreads;
    dst[m] = -1;
    if (i >= nt) continue;
    const int c = s_cost[i];
    int r = 0;
    for (int j = 0; j < nt; ++j) r += s_cost[j] > c || (s_cost[j] == c && j < i);
    dst[m] = r;
#pragma unroll
    for (int w = 0; w < kTileWords; ++w) rec[m][w] = tile[(size_t)i * kTileWords + w];
  }
  __syncthreads();
#pragma unroll
  for (int m = 0; m < kTileMine; ++m) {
    if (dst[m] < 0) continue;
#pragma unroll
    for (int w = 0; w < kTileWords; ++w) tile[(size_t)dst[m] * kTileWords + w] = rec[m][w];
  }
  if (threadIdx.x == 0) {
    meta[H_N_TILE] = nt;
    meta[H_N_TILE_SPAN] = s_nspan;
  }
}

}  // namespace

extern "C" hs_status hs_round_build_tiles(const hs_round_caps* caps, void* dev_meta, int32_t* dev_status,
                                          void* stream) {
  HS_CHECK_ARG(caps && dev_meta, "null argument");
  HS_CHECK_ARG(caps->max_segments <= kMaxTileSeg && caps->max_tiles <= kThreads * kTileMine,
               "max_segments %d / max_tiles %d above the %d / %d this call supports", caps->max_segments,
               caps->max_tiles, kMaxTileSeg, kThreads * kTileMine);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return hs::fail(HS_ECUDA, "no CUDA device");
  build_tiles_kernel<<<1, kThreads, 0, (cudaStream_t)stream>>>((int32_t*)dev_meta, dev_status);
  HS_LAUNCH_CHECK("round_build_tiles");
  return HS_OK;
}

extern "C" hs_status hs_round_build_chunks(const hs_round_caps* caps, void* dev_meta, int32_t* dev_status,
                                           void* stream) {
  HS_CHECK_ARG(caps && dev_meta, "null argument");
  HS_CHECK_ARG(caps->max_segments <= kThreads * 8, "max_segments %d above the %d this call supports",
               caps->max_segments, kThreads * 8);
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return hs::fail(HS_ECUDA, "no CUDA device");
  build_chunks_kernel<<<1, kThreads, 0, (cudaStream_t)stream>>>((int32_t*)dev_meta, dev_status);
  HS_LAUNCH_CHECK("round_build_chunks");
  return HS_OK;
}
