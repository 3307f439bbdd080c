// meta.h -- layout of the GPU-resident round metadata (one int32 blob).
//
// Flide, section 3.3.1: every quantity fixed by the round composition
// (segment lengths, positions, key ranges, state indices, the chunk list,
// readout rows) lives in compact device buffers filled before the launches;
// every kernel derives its work from them.  The blob's array offsets depend
// only on the capacities, so rounds with equal capacities share one layout.
#pragma once
#include <stdint.h>

#ifdef __CUDACC__
#define HSM_HD __host__ __device__
#else
#define HSM_HD
#endif

namespace hsm {

constexpr int32_t kMagic = 0x48534d31;  // "HSM1"
constexpr int kPage = 16;               // tokens per KV page
constexpr int kTileRows = 128;          // query rows per attention tile
constexpr int kChunk = 64;              // GDN chunk length
constexpr int kHeaderWords = 64;

// header word indices
enum : int {
  H_MAGIC = 0,
  H_N_TOK,
  H_N_SEG,
  H_N_SPAN,
  H_N_TILE,
  H_N_TILE_SPAN,
  H_N_CHUNK,
  H_N_READOUT,
  H_N_LEVEL,
  H_N_PAGE_REF,
  // offsets (in int32 words from the blob start)
  H_OFF_SEG,
  H_OFF_TOK,
  H_OFF_SPAN,
  H_OFF_TILE,
  H_OFF_TILE_SPAN,
  H_OFF_CHUNK,
  H_OFF_READOUT,
  H_OFF_LEVEL,      // [max_levels + 1] prefix offsets into LEVEL_SEG
  H_OFF_LEVEL_SEG,  // segment ids grouped by level
  H_OFF_PAGE_REF,
  // capacities (copied from hs_round_caps)
  H_CAP_TOK,
  H_CAP_SEG,
  H_CAP_SPAN,
  H_CAP_TILE,
  H_CAP_TILE_SPAN,
  H_CAP_CHUNK,
  H_CAP_READOUT,
  H_CAP_LEVEL,
  H_CAP_PAGE_REF,
  H_TOTAL_WORDS,
  H_MAX_SEG_CHUNKS,  // largest number of chunks in one segment
  H_OFF_PRED,        // per token: kConvTaps-1 predecessor rows for the causal conv
  H_N_SCAN,          // extra scan groups (group 1 and up of the long nodes), all levels
  H_OFF_SCAN,        // [segment, group] per extra scan group, grouped by level
  H_OFF_SCAN_LEVEL,  // [max_levels + 1] prefix offsets into SCAN
  // the paired-head attention kernel's work counters: the next (tile, head pair) item to hand out and the
  // CTAs done; zero as uploaded, and set back to zero by the kernel's last CTA
  H_ATTN_NEXT,
  H_ATTN_DONE,
};

// The GDN state chain of a long node is split into groups of consecutive
// chunks that run side by side (a two-level scan of the affine chunk map
// S -> S M_c + N_c): group g of a node with n chunks holds chunks
// [g n / G, (g + 1) n / G).  G depends on the node's own length only.
constexpr int kScanMinChunks = 12;
constexpr int kScanMaxGroups = 9;
HSM_HD inline int32_t scan_groups(int32_t n_chunks) {
  if (n_chunks < 2 * kScanMinChunks) return 1;
  const int32_t g = n_chunks / kScanMinChunks;
  return g < kScanMaxGroups ? g : kScanMaxGroups;
}
// bound on the number of extra groups of a round with cap_chunk chunks
HSM_HD inline int32_t scan_cap(int32_t cap_chunk) { return cap_chunk / kScanMinChunks + 1; }

// segment record
constexpr int kSegWords = 16;
enum : int {
  S_STREAM_OFF = 0,  // first stream row
  S_LEN,             // tokens in the stream
  S_POS0,            // position of the first token (history length for a resumed root)
  S_REQUEST,
  S_PARENT,          // -1 for a root
  S_LEVEL,           // depth in the tree
  S_OWN_SPAN,        // index of the node's own key span
  S_INIT_SLOT,       // GDN state slot read at the start (-1 = zero state)
  S_END_SLOT,        // GDN state slot written at the end (-1 = none)
  S_CHUNK_OFF,       // first chunk of the node
  S_N_CHUNK,
  S_READOUT_ROW,     // stream row of the readout (-1 = none)
  S_PAGE_REF_OFF,    // first own page in the page-ref array
  S_N_PAGES,
  S_SCAN1,           // scan-table entry of the node's group 1 (-1 = one group); groups 2.. follow it
  S_HIST,            // a resumed root's history spans: first span | count << kHistShift (0: none)
};
constexpr int kHistShift = 20;  // history spans of one root: first < 2^20, count < 2^11

// Causal-conv predecessors of a token (Flide section 3.2.2: the convolution
// reads a token's predecessors through an index, so a question's first tokens
// see its state's last tokens).  pred[k-1] = the token k steps back in the
// isolated sequence: >= 0 a stream row; -1 none (before the sequence);
// <= -2 row (-2 - value) of the caller's conv-window buffer (a resumed root).
constexpr int kConvTaps = 4;
constexpr int kPredWords = kConvTaps - 1;

// token record: the node a stream row belongs to and its index inside it
constexpr int kTokWords = 2;
enum : int { T_SEG = 0, T_IDX = 1 };

// key span: n_tok keys on consecutive page-ref entries starting at PAGE_REF_OFF,
// key i at page refs[off + i/16], row i%16.  OWNER = owning segment (-1: history).
constexpr int kSpanWords = 4;
enum : int { SP_PAGE_REF_OFF = 0, SP_N_TOK, SP_OWNER, SP_PAD };

// attention tile: n_rows consecutive stream rows (all children of one parent,
// or one segment), whose keys are the n_shared spans visible to every row
// followed by n_own own spans (each visible causally to its owner's rows only).
// READOUT = 1 when one of its rows is a readout row (the option head reads it).
constexpr int kTileWords = 8;
enum : int { TL_ROW0 = 0, TL_N_ROWS, TL_SPAN_OFF, TL_N_SHARED, TL_N_OWN, TL_WORK, TL_SEG0, TL_READOUT };

// GDN chunk: len <= 64 rows starting at stream row ROW0, inside segment SEG
constexpr int kChunkWords = 4;
enum : int { C_SEG = 0, C_ROW0, C_LEN, C_IDX };

struct Layout {
  int32_t off_seg, off_tok, off_span, off_tile, off_tile_span, off_chunk, off_readout, off_level,
      off_level_seg, off_page_ref, off_pred, off_scan, off_scan_level, total_words;
};

inline int32_t align16(int32_t x) { return (x + 15) & ~15; }

// Array offsets from capacities (words; each array starts on a 64-byte boundary).
inline Layout layout_for(int32_t cap_tok, int32_t cap_seg, int32_t cap_span, int32_t cap_tile,
                         int32_t cap_tile_span, int32_t cap_chunk, int32_t cap_readout,
                         int32_t cap_level, int32_t cap_page_ref) {
  Layout L;
  int32_t o = kHeaderWords;
  L.off_seg = o;        o = align16(o + cap_seg * kSegWords);
  L.off_tok = o;        o = align16(o + cap_tok * kTokWords);
  L.off_span = o;       o = align16(o + cap_span * kSpanWords);
  L.off_tile = o;       o = align16(o + cap_tile * kTileWords);
  L.off_tile_span = o;  o = align16(o + cap_tile_span);
  L.off_chunk = o;      o = align16(o + cap_chunk * kChunkWords);
  L.off_readout = o;    o = align16(o + cap_readout);
  L.off_level = o;      o = align16(o + cap_level + 1);
  L.off_level_seg = o;  o = align16(o + cap_seg);
  L.off_page_ref = o;   o = align16(o + cap_page_ref);
  L.off_pred = o;       o = align16(o + cap_tok * kPredWords);
  L.off_scan = o;       o = align16(o + scan_cap(cap_chunk) * 2);
  L.off_scan_level = o; o = align16(o + cap_level + 1);
  L.total_words = o;
  return L;
}

}  // namespace hsm
