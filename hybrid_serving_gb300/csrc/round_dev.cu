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

}  // namespace

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
