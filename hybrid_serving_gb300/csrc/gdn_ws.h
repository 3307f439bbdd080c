// gdn_ws.h -- compact per-(chunk, head) GDN workspace shared by the
// chunk-local pass and the tensor-core state pass (bf16 inputs, d = 128).
//
//   W   bf16, the 128-byte-swizzled image of W^T: row k (128 rows, d_k) holds
//       W[t][k] for the 64 tokens t (one [128][64] slab) -- the MN-major
//       B operand of S W^T, and one row per thread for the writer
//   U   bf16, Ut^T in the same layout: row j (d_v) holds Ut[t][j]
//   P   [64][64] bf16, swizzled K-major image (one slab)
//   K'  bf16, diag(e^{g_C - g}) K: [64 tokens][128] as two swizzled [64][64]
//       slabs (the image a TMA box of K would give), the MN-major B operand
//       of the state update
//   G   decay factors, fp32: e^{g_t} [64] | e^{g_C - g_t} [64] | e^{g_C} [1],
//       padded to 1 KB (g = cumulative log-decay inside the chunk, C = its
//       last token; zero past the chunk's length)
#pragma once

namespace gdnws {
constexpr int kW = 0;
constexpr int kU = 16384;
constexpr int kP = 32768;
constexpr int kK = 40960;
constexpr int kG = 57344;
constexpr int kBytes = 58368;  // per (chunk, head); multiple of 1024
constexpr int kFloats = kBytes / 4;

// Per (extra scan group, head) buffers of the two-level state scan, after the
// per-chunk blocks: the end state of the node's first group S (fp32
// [128][128], rows d_v; in the entry of group 1), the group's zero-start end
// state N (fp32 [128][128], row j's 16-byte pieces swizzled by j % 32) and
// its transition M (d_k x d_k) as the bf16 image of an MN-major B operand
// (two [128][64] slabs: row k holds M[k][n]).
constexpr int kScanS = 0;
constexpr int kScanN = 65536;
constexpr int kScanMhi = 131072;
constexpr int kScanBytes = 163840;

// Byte offset of bf16 element (row, col) in a 128-byte-swizzled K-major image
// made of [rows][64]-element slabs (one slab per 64 columns): 16-byte chunk c
// of a 128-byte row lands at chunk c ^ (row % 8).
__host__ __device__ inline int sw128_off(int row, int col, int rows) {
  const int slab = col >> 6, c = col & 63;
  return slab * rows * 128 + row * 128 + (((c >> 3) ^ (row & 7)) << 4) + (c & 7) * 2;
}
}  // namespace gdnws
