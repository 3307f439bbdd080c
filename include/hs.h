/*
 * hs.h -- C ABI of the GB300 tree-prefill library (libhsfork.so).
 *
 * Exact tree-structured (forked) prefill: one or more requests, each a tree
 * of a shared trunk and its question branches (or deeper residuals), packed
 * into ONE flat token stream; two token mixers run over the stream:
 *
 *   - ForkAttention: paged causal attention in which a token sees its own
 *     node's earlier tokens and every token of its ancestors, never a
 *     sibling's (Flide, "Accelerating Decision Inference with Exact State
 *     Forking", section 3.2.1, Eq. 3).  Children alias their ancestors' KV
 *     pages without copying (ForkServe README, "Copy-on-write context tree").
 *   - Gated DeltaNet fork prefill: the gated delta rule (Flide section 3.2.2,
 *     Eq. 4) in chunks; each child continues from its parent's end state
 *     through a state-slot index, never a copy (Flide section 3.2.2, "two
 *     calls"), and a root may resume from a state saved by an earlier pass
 *     (Flide section 3.4).
 *
 * Conventions
 *   - Every call returns hs_status: 0 (HS_OK) or a negative code.  The message
 *     of the last failure on the calling thread is hs_last_error().
 *   - The CALLER owns all device memory (inputs, outputs, KV page pools,
 *     state pools, workspaces, the metadata buffer, the status word).  No call
 *     allocates device memory.  Host objects (page pool, round) are opaque
 *     handles with create/destroy.
 *   - Device calls enqueue work on the given cudaStream_t (passed as void*;
 *     NULL = the legacy default stream) and never synchronise.
 *   - Kernels never trap.  A kernel that meets inconsistent metadata writes a
 *     nonzero code into the caller's int32 device status word (first error
 *     wins) and skips the offending work; read it back after a sync and pass
 *     the host copy to hs_check_status().
 *   - There is no CPU fallback: without a usable CUDA device, device calls
 *     fail with HS_ECUDA.
 *   - Layouts are row-major, last index fastest.  T = stream tokens.
 */
#ifndef HS_H_
#define HS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t hs_status;
#define HS_OK 0
#define HS_EINVAL (-1)        /* bad argument or tree (cycle, unknown parent, empty node, bad slot) */
#define HS_ECAPACITY (-2)     /* a round exceeds one of its hs_round_caps */
#define HS_EUNSUPPORTED (-3)  /* dtype / head size / chunk size not built */
#define HS_ECUDA (-4)         /* a CUDA runtime call failed (including: no device) */
#define HS_EDEVICE (-5)       /* the device status word reports an error */
#define HS_ENOPAGES (-6)      /* page pool exhausted (refcounts are left unchanged) */

typedef enum { HS_F32 = 0, HS_BF16 = 1 } hs_dtype;

/* Device status codes (values of the int32 status word). */
#define HS_DEV_OK 0
#define HS_DEV_BAD_PAGE 1     /* a page id outside [0, n_pages) */
#define HS_DEV_BAD_SLOT 2     /* a state slot outside [0, n_slots) */
#define HS_DEV_BAD_META 3     /* counts above capacity or inconsistent records */
#define HS_DEV_TIMEOUT 4      /* a bounded wait inside a kernel ran out (the call's outputs are invalid) */

/* ------------------------------------------------------------------------ */
/* Fixed capacities of a round.  They size the device metadata buffer and   */
/* every launch grid, so rounds with the same caps reuse the same launch    */
/* shapes (Flide section 3.3.2: launches fixed by capacity, the tree lives  */
/* in GPU-resident metadata).                                               */
/* Every device call below takes the caps of the round whose metadata sits  */
/* in dev_meta: grids and the GDN workspace are sized from them, and the    */
/* kernels trust the metadata's counts up to them.  Passing other caps is   */
/* a caller error the host cannot detect.                                   */
/* ------------------------------------------------------------------------ */
typedef struct {
  int32_t max_tokens;      /* stream tokens T */
  int32_t max_segments;    /* tree nodes over all requests */
  int32_t max_hist_spans;  /* KV history spans of resumed roots */
  int32_t max_tiles;       /* attention query tiles (128 rows each) */
  int32_t max_tile_spans;  /* total span references over all tiles */
  int32_t max_chunks;      /* GDN chunks (64 tokens, per segment) */
  int32_t max_readouts;    /* readout rows */
  int32_t max_page_refs;   /* page-table entries (own pages + history pages) */
  int32_t max_levels;      /* tree depth + 1 */
} hs_round_caps;

/* Capacities sufficient for a round of the given totals (tokens, segments,
 * tree depth, history spans and history pages). */
hs_status hs_round_caps_for(int32_t n_tokens, int32_t n_segments, int32_t n_levels,
                            int32_t n_hist_spans, int32_t n_hist_pages, int32_t page_size,
                            hs_round_caps* out);

/* ------------------------------------------------------------------------ */
/* KV page pool (host bookkeeping of a caller-owned device page pool).       */
/* ForkServe README, "Copy-on-write context tree": a node's writes allocate  */
/* pages for its own tokens; children alias ancestors' pages; abort decrefs. */
/* Device pools are K and V arrays [Hkv][n_pages][page_size][d].             */
/* Allocation takes the lowest free page ids, in ascending order, whatever   */
/* order pages were freed in: a node's pages are consecutive wherever the    */
/* free pages are, which the attention kernel's block copies rely on for     */
/* speed (never for correctness).                                            */
/* ------------------------------------------------------------------------ */
typedef struct hs_page_pool hs_page_pool;

hs_status hs_page_pool_create(int32_t n_pages, int32_t page_size, hs_page_pool** out);
void hs_page_pool_destroy(hs_page_pool* pool);
/* number of free pages and of pages with refcount > 0 */
hs_status hs_page_pool_stats(const hs_page_pool* pool, int32_t* n_free, int32_t* n_live);
hs_status hs_page_pool_refcount(const hs_page_pool* pool, int32_t page, int32_t* ref);
/* Drop one reference per listed page (pages reaching 0 return to the free
 * list).  A page may be listed k times if it holds >= k references; any
 * invalid entry fails the whole call with HS_EINVAL before anything changes. */
hs_status hs_page_pool_decref(hs_page_pool* pool, const int32_t* pages, int32_t n);

/* ------------------------------------------------------------------------ */
/* Round: a set of request trees flattened into one stream (Flide Eq. 2).    */
/* ------------------------------------------------------------------------ */
typedef struct hs_round hs_round;

#define HS_SEG_READOUT 1       /* the node's last token is a readout row (default for leaves) */
#define HS_SEG_NO_READOUT 2    /* suppress the default readout of a leaf */

hs_status hs_round_create(const hs_round_caps* caps, hs_round** out);
/* Frees the host object only: page references a finalized round holds stay
 * until hs_round_release drops them. */
void hs_round_destroy(hs_round* r);

/* Add a node.  parent_seg = -1 starts a new request (its trunk).  Nodes of
 * one request must be added after their parent.  save_slot >= 0 persists the
 * node's end-of-node GDN state into that state slot (a checkpoint, Flide
 * section 3.4); -1 = no persistent save.  The new node's id (dense, in add
 * order) is written to *seg_out. */
hs_status hs_round_add_segment(hs_round* r, int32_t parent_seg, int32_t n_tokens, int32_t flags,
                               int32_t save_slot, int32_t* seg_out);

/* Add n nodes in one call, as n calls of hs_round_add_segment would: node j
 * gets id first + j, where first (written to *first_id) is the number of
 * nodes added before; parent[j] is -1 or an id below first + j.  flags and
 * save_slot may be NULL (0 and -1 for every node).  Every entry is checked
 * first: on an error nothing is added. */
hs_status hs_round_add_segments(hs_round* r, int32_t n, const int32_t* parent, const int32_t* n_tokens,
                                const int32_t* flags, const int32_t* save_slot, int32_t* first_id);

/* Resume a ROOT node from a checkpoint (Flide section 3.4): its first stream
 * token sits at position ckpt_pos and its GDN state starts from ckpt_slot. */
hs_status hs_gdn_state_resume(hs_round* r, int32_t seg, int32_t ckpt_slot, int32_t ckpt_pos);

/* Attach the cached KV history of a resumed root: n_spans spans, span i
 * holding ntok[i] tokens on ceil(ntok[i]/page_size) pages taken in order
 * from `pages`.  The spans precede the root's own keys (Flide section 3.4:
 * cached keys and values precede new ones).  sum(ntok) must equal ckpt_pos.
 * The round takes one reference on each page and drops it at release. */
hs_status hs_round_attach_history(hs_round* r, int32_t seg, int32_t n_spans, const int32_t* ntok,
                                  const int32_t* pages);

/* Give a resumed ROOT the causal-conv window it continues from: its
 * kConvTaps-1 = 3 predecessor tokens (oldest first) are rows
 * window_row0 .. window_row0+2 of the caller's conv-window buffer passed to
 * hs_gdn_prep (Flide section 3.4: a checkpoint keeps the convolution window).
 * Without a window, a root's first tokens see zeros before them. */
hs_status hs_round_set_conv_window(hs_round* r, int32_t seg, int32_t window_row0);

/* Lay out the stream, allocate each node's own KV pages from `pool` (may be
 * NULL for GDN-only rounds), assign temporary GDN state slots
 * [temp_slot0, temp_slot0 + n_temp_slots) to inner nodes, and build the
 * metadata.  Errors leave the pool unchanged, and a finalize retried after an
 * error (e.g. with more temporary slots) starts again from the nodes as added. */
hs_status hs_round_finalize(hs_round* r, hs_page_pool* pool, int32_t temp_slot0, int32_t n_temp_slots);

/* Bytes of the device metadata buffer for these caps (fixed per caps). */
size_t hs_round_meta_bytes(const hs_round_caps* caps);
/* Copy the packed metadata (int32 words) into a host buffer. */
hs_status hs_round_pack(const hs_round* r, void* host, size_t bytes);
/* One cudaMemcpyAsync of the packed metadata into the device buffer. */
hs_status hs_round_upload(const hs_round* r, void* dev_meta, size_t bytes, void* stream);

typedef struct {
  int32_t n_tokens, n_segments, n_tiles, n_chunks, n_readouts, n_levels, n_pages_allocated;
  int32_t n_spans, n_tile_spans, n_page_refs;
} hs_round_info;
hs_status hs_round_get_info(const hs_round* r, hs_round_info* out);

typedef struct {
  int32_t stream_off, n_tokens, pos0, request, parent, level;
  int32_t init_slot, end_slot, readout_row, n_pages;
} hs_segment_info;
hs_status hs_round_segment(const hs_round* r, int32_t seg, hs_segment_info* out);
/* the node's own pages (cap entries at most; *n = count) */
hs_status hs_round_segment_pages(const hs_round* r, int32_t seg, int32_t* pages, int32_t cap, int32_t* n);
/* the readout rows in readout order (stream row of each readout node's last token) */
hs_status hs_round_readout_rows(const hs_round* r, int32_t* rows, int32_t cap, int32_t* n);

/* Commit/abort (ForkServe README: commit keeps one path, abort decrefs the
 * residuals).  Drops the round's page references for every node NOT listed
 * in keep_segs and for the history pages; kept nodes' own pages stay live
 * (one reference each, now owned by the caller).  `pool` must be the pool the
 * round was finalized with (NULL if it was finalized without one). */
hs_status hs_round_release(hs_round* r, hs_page_pool* pool, const int32_t* keep_segs, int32_t n_keep);

/* The GDN chunk list built on the GPU (Flide section 3.3.1: GPU-resident
 * metadata for the fixed-shape launches; section 3.5: every node starts a
 * chunk): from the segment table already in dev_meta (each node's stream
 * offset and length), rewrites in place the chunk list -- the nodes in
 * stream order, each cut into 64-token chunks from its first token, record
 * {node, first row, length, index} -- each node's first-chunk and
 * chunk-count fields, and the header's chunk count and largest per-node
 * count: word for word what the host round build writes.  One small launch
 * on `stream`; a chunk list beyond caps->max_chunks sets HS_DEV_BAD_META.
 * Supports caps->max_segments <= 4096 (HS_EINVAL above). */
hs_status hs_round_build_chunks(const hs_round_caps* caps, void* dev_meta, int32_t* dev_status, void* stream);
/* The attention tile table built on the GPU (Flide section 3.3.1: a tile
 * table in GPU-resident metadata; section 3.5: tiles start at the node):
 * from the segment table (stream offsets, lengths, parents, own spans, each
 * root's history spans, readout rows) and the span lengths already in
 * dev_meta, rewrites in place the tile records, the tile span lists and the
 * header's tile and tile-span counts -- word for word what the host round
 * build writes: in stream order a root or a node of more than 128 tokens
 * gets one tile per 128 rows, a run of consecutive siblings of at most 128
 * rows each is packed into tiles of at most 128 rows; a tile's spans are the
 * root's history, every ancestor's own span (root first) and its nodes' own
 * spans; tiles ordered by work x (7 with a readout row, else 5), heaviest
 * first, ties in that order.  One small launch on `stream`; a table beyond
 * the caps (or inconsistent parents) sets HS_DEV_BAD_META.  Supports
 * caps->max_segments <= 4096 and caps->max_tiles <= 4096 (HS_EINVAL above). */
hs_status hs_round_build_tiles(const hs_round_caps* caps, void* dev_meta, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------ */
/* Hot path                                                                  */
/* ------------------------------------------------------------------------ */

/* ForkAttention prefill (Flide section 3.2.1, Eq. 3; scaled dot-product
 * attention, Flex "Request-Adaptive Execution ..." section 2, Eq. 1).
 * Writes the stream's new K/V into each node's own pages, then for every
 * stream row and query head h computes
 *   out[t,h] = sum_{y visible to t} softmax(scale * q[t,h].k[y,g]) v[y,g],
 * g = h / (hq/hkv), the visible keys being the resumed history, every
 * ancestor's tokens and the row's own node up to itself.
 *   q      [Tcap, hq, d]  dt        k_new, v_new [Tcap, hkv, d] dt
 *   (Tcap = caps->max_tokens: buffers are sized by capacity; rows past the
 *   round's stream are read as padding and never written)
 *   k_pages, v_pages [hkv, n_pages, page_size, d] dt (head-major: one head's
 *                    pages are contiguous; written: own pages only; every
 *                    row must hold finite values -- zero the pools once)
 *   out    [Tcap, hq, d]  dt        (bf16 outputs are round-to-nearest-even)
 * Supported: dt in {HS_F32, HS_BF16}; d in {64, 128}; hq % hkv == 0;
 * page_size 16.  Inputs must be 16-byte aligned.  Accumulation is fp32;
 * the result of a row does not depend on what else is in the round.
 * Precision (bf16, d = 128): P = softmax weights enter P.V rounded to bf16,
 * except on attention tiles holding a readout row, where P keeps ~16
 * significant bits (a bf16 high part and low part) because the option
 * distribution read there is sensitive to single-ulp output changes.
 * dev_meta is read, except for two header words (the bf16 d = 128 kernel's
 * work counter: items are handed to CTAs in order, longest first): they are
 * zero as the round uploads them and the kernel sets them back to zero
 * before it completes, so launches on one metadata buffer must run one at a
 * time (stream order or graph order), never concurrently. */
hs_status hs_fork_attn_prefill(const hs_round_caps* caps, const void* dev_meta, hs_dtype dt,
                               int32_t hq, int32_t hkv, int32_t d, float scale, const void* q,
                               const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                               int32_t n_pages, void* out, int32_t* dev_status, void* stream);

/* The two halves of hs_fork_attn_prefill, for callers that write the pages
 * themselves or time the halves apart:
 *   hs_kv_page_write -- k_new/v_new rows into each node's own pages (and
 *     zeroes the unused rows of each node's last page);
 *   hs_fork_attn     -- the attention over pages already written.
 * Arguments as for hs_fork_attn_prefill. */
hs_status hs_kv_page_write(const hs_round_caps* caps, const void* dev_meta, hs_dtype dt, int32_t hkv, int32_t d,
                           const void* k_new, const void* v_new, void* k_pages, void* v_pages, int32_t n_pages,
                           int32_t* dev_status, void* stream);
hs_status hs_fork_attn(const hs_round_caps* caps, const void* dev_meta, hs_dtype dt, int32_t hq, int32_t hkv,
                       int32_t d, float scale, const void* q, const void* k_pages, const void* v_pages,
                       int32_t n_pages, void* out, int32_t* dev_status, void* stream);

/* Mask variants of ForkAttention (Flide section 3.2.1: a sliding window adds
 * t_x - t_y < W to Eq. 3; Appendix H: models that read their state both
 * ways see it as a block).  Positions are along the row's own path (a
 * resumed history, every ancestor, the node): the trunk's tokens count
 * from 0 (or from the history's length), a child's from its parent's end.
 *   window              > 0: a row sees only keys with t_x - t_y < window;
 *                       0: no window
 *   bidirectional_root  1: a root node's rows see every token of the root
 *                       (and its history), later ones included; every
 *                       other node stays causal; 0: plain Eq. 3 */
typedef struct {
  int32_t window;
  int32_t bidirectional_root;
} hs_attn_mask;

/* hs_fork_attn with a mask (NULL = none, the same as hs_fork_attn).  The
 * bf16 d = 128 tensor-core kernel takes masks when a KV head's query-head
 * group has an even size; other shapes run the CUDA-core kernel.  Blocks a
 * window hides from every row of a tile are skipped. */
hs_status hs_fork_attn_masked(const hs_round_caps* caps, const void* dev_meta, hs_dtype dt, int32_t hq,
                              int32_t hkv, int32_t d, float scale, const hs_attn_mask* mask, const void* q,
                              const void* k_pages, const void* v_pages, int32_t n_pages, void* out,
                              int32_t* dev_status, void* stream);

/* Workspace bytes hs_gdn_fork_prefill needs for these caps and shapes. */
size_t hs_gdn_workspace_bytes(const hs_round_caps* caps, int32_t h, int32_t dk, int32_t dv);

/* Gated DeltaNet fork prefill (Flide section 3.2.2, Eq. 4):
 *   S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,  o_t = S_t q_t
 * per head, over chunks of `chunk` tokens that start at every node's first
 * token.  Level by level: a root starts from zero (or its resume slot), a
 * child from its parent's end state (read through the slot index), and
 * every node that has children or a save slot writes its end state.
 *   q, k   [Tcap, h, dk] dt    v [Tcap, h, dv] dt    alpha, beta [Tcap, h] fp32
 *   (Tcap = caps->max_tokens rows, contiguous; rows past the stream are padding)
 *   state_pool [n_slots, h, dv, dk] fp32 (read: init slots; written: end slots)
 *   out    [Tcap, h, dv] dt (only the stream's rows are written)
 *   ws     >= hs_gdn_workspace_bytes(), 256-byte aligned, contents scratch
 * Supported: dt in {HS_F32, HS_BF16}; dk == dv in {64, 128}; chunk == 64. */
hs_status hs_gdn_fork_prefill(const hs_round_caps* caps, const void* dev_meta, hs_dtype dt, int32_t h,
                              int32_t dk, int32_t dv, int32_t chunk, const void* q, const void* k,
                              const void* v, const float* alpha, const float* beta, float* state_pool,
                              int32_t n_slots, void* out, void* ws, size_t ws_bytes, int32_t* dev_status,
                              void* stream);

/* Gated DeltaNet fork prefill for callers that cannot allocate device memory.
 * (The pages have no counterpart: this is a library convenience.)  Some
 * callers have no allocator to hand a workspace from -- code running where
 * cudaMalloc is forbidden or unavailable, e.g. inside a host framework that
 * owns all device memory, or a plug-in that may only touch the buffers it
 * is given.  This entry point takes the same arguments as
 * hs_gdn_fork_prefill minus the workspace and uses a scratch array compiled
 * into the library instead: HS_GDN_NOALLOC_SCRATCH_BYTES of device memory
 * that every GPU loading the library holds until the process exits.
 *   - A round whose hs_gdn_workspace_bytes() exceeds that size is rejected
 *     with HS_ECAPACITY before anything is launched.
 *   - It allocates nothing: no cudaMalloc / cudaFree, no allocating library.
 *   - The first call on a device looks up that device's scratch address
 *     (cudaGetSymbolAddress, with the device current); make that first call
 *     before any stream capture.
 *   - All calls share the one array and it keeps the last call's contents;
 *     the kernels fully rewrite every entry they read, so nothing needs
 *     clearing, but calls that overlap on the GPU (other streams, other
 *     threads) race on it: serialise them. */
#define HS_GDN_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
hs_status hs_gdn_fork_prefill_noalloc(const hs_round_caps* caps, const void* dev_meta, hs_dtype dt, int32_t h,
                                      int32_t dk, int32_t dv, int32_t chunk, const void* q, const void* k,
                                      const void* v, const float* alpha, const float* beta, float* state_pool,
                                      int32_t n_slots, void* out, int32_t* dev_status, void* stream);

/* Snapshot one GDN state slot into another (Flide section 3.4, checkpoint):
 * state_pool[dst] = state_pool[src], [h, dv, dk] fp32 each. */
hs_status hs_gdn_state_checkpoint(float* state_pool, int32_t n_slots, int32_t src_slot, int32_t dst_slot,
                                  int32_t h, int32_t dk, int32_t dv, void* stream);

/* Option log-probabilities at the readout rows (Flide section 3.1, Eq. 1;
 * section 3.3.3, selective readout through an index buffer):
 *   logprobs[i, o] = log softmax_o( option_rows[o] . hidden[row_i] )
 *   hidden      [Tcap, hidden_dim] dt with row stride hidden_stride elements
 *               (only the readout rows are read)
 *   option_rows [n_opt, hidden_dim] fp32
 *   logprobs    [n_readouts, n_opt] fp32
 * Dot products accumulate in fp32 in a fixed order.  n_opt <= 32. */
hs_status hs_choice_logprobs(const hs_round_caps* caps, const void* dev_meta, hs_dtype dt,
                             const void* hidden, int64_t hidden_stride, int32_t hidden_dim,
                             const float* option_rows, int32_t n_opt, float* logprobs,
                             int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------ */
/* Building blocks of a hybrid attention / Gated DeltaNet stack (the        */
/* per-token parts; Flide section 3.2: pointwise work ignores the tree).     */
/* All bf16 tensors are row-major with the given leading dimension          */
/* (elements); every row is computed alone, in a fixed reduction order.     */
/* ------------------------------------------------------------------------ */

/* C[M,N] = A[M,K] . B[N,K]^T (+ R[M,N]), A and B bf16, fp32 accumulation in
 * a fixed order for any M (128x256 output tiles walked by persistent CTAs,
 * the same K steps for every tile, no split-K; Flide section 3.5); C and R in
 * c_dtype (HS_BF16, rounded to nearest even, or HS_F32: a residual stream
 * kept in fp32).  N % 128 == 0, K % 64 == 0, leading dimensions % 8 == 0,
 * 16-byte aligned pointers.  R may be NULL; R may alias C.
 * HS_EUNSUPPORTED: another c_dtype or shape. */
hs_status hs_gemm_bf16(int32_t M, int32_t N, int32_t K, const void* A, int64_t lda, const void* B, int64_t ldb,
                       void* C, int64_t ldc, const void* R, int64_t ldr, hs_dtype c_dtype, int32_t* dev_status,
                       void* stream);
/* The gate/up projection of a SwiGLU MLP with the activation applied in the
 * GEMM's epilogue:
 *   C[M, N2/2] = silu(A . Bg^T) * (A . Bu^T),   silu(x) = x / (1 + e^-x)
 * B [N2, K] bf16 holds the two weight matrices interleaved in blocks of 128
 * rows: rows 256j .. 256j+127 are Bg's rows 128j .. 128j+127 and rows
 * 256j+128 .. 256j+255 are Bu's same rows.  Both products accumulate in fp32
 * exactly as hs_gemm_bf16's do; silu and the product are taken in fp32 and
 * rounded to bf16 once.  N2 % 256 == 0, K % 64 == 0, ldc >= N2/2; the other
 * rules as for hs_gemm_bf16.  HS_EUNSUPPORTED: another shape. */
hs_status hs_gemm_bf16_swiglu(int32_t M, int32_t N2, int32_t K, const void* A, int64_t lda, const void* B,
                              int64_t ldb, void* C, int64_t ldc, int32_t* dev_status, void* stream);
/* out[t] = table[ids[t]], table bf16 [vocab, dim], out in out_dtype (HS_BF16
 * or HS_F32) [T, dim] (ids: device int32 [T]; an id outside [0,vocab)
 * gives a zero row and HS_DEV_BAD_META). */
hs_status hs_embed(const int32_t* ids, int32_t T, const void* table, int32_t vocab, int32_t dim, void* out,
                   hs_dtype out_dtype, int32_t* dev_status, void* stream);
/* out = x / sqrt(mean(x^2) + eps) * w   (w bf16 [dim] or NULL for ones);
 * x in x_dtype and out in out_dtype, each HS_BF16 or HS_F32 (sums of
 * squares in fp32, a fixed lane-strided order and butterfly per row). */
hs_status hs_rmsnorm(const void* x, int64_t ldx, hs_dtype x_dtype, int32_t T, int32_t dim, const void* w, float eps,
                     void* out, int64_t ldo, hs_dtype out_dtype, void* stream);
/* Host: cos/sin table [max_pos][d/2][2] fp32 of angle p * theta^(-2i/d),
 * computed in double. */
hs_status hs_rope_table(float* host_table, int32_t max_pos, int32_t d, double theta);
/* In place: rotate-half rotary embedding of n_heads heads of width d at
 * column col0 of x [Tcap, ldx], each token at its standalone position
 * (node pos0 + index; Flide section 3.2).  table: device copy of
 * hs_rope_table (8-byte aligned); a position outside [0, max_pos) sets
 * HS_DEV_BAD_META and leaves the token unrotated. */
hs_status hs_rope_apply(const hs_round_caps* caps, const void* dev_meta, void* x, int64_t ldx, int32_t col0,
                        int32_t n_heads, int32_t d, const float* table, int32_t max_pos, int32_t* dev_status,
                        void* stream);
/* Gated DeltaNet front end per token: proj [Tcap, ldp] holds q | k | v
 * (h*d columns each) then a | b (h columns each).  The q, k, v channels go
 * through a depthwise causal convolution of 4 taps, y_t = sum_k w[ch][k] x_{t-k},
 * whose predecessors come from the round metadata (across the fork; from
 * `window` rows [n_window_rows, ldw] for a resumed root), then SiLU; q and k
 * heads are L2-normalised (eps 1e-6).  alpha = exp(-0.1 softplus(a)),
 * beta = sigmoid(b).  conv_w bf16 [3*h*d][4]; q, k, v bf16 [Tcap, h, d];
 * alpha, beta fp32 [Tcap, h]. */
hs_status hs_gdn_prep(const hs_round_caps* caps, const void* dev_meta, const void* proj, int64_t ldp,
                      const void* window, int64_t ldw, int32_t n_window_rows, const void* conv_w, int32_t h, int32_t d,
                      void* q, void* k, void* v, float* alpha, float* beta, int32_t* dev_status, void* stream);
/* out[t, i] = silu(gu[t, i]) * gu[t, F + i]; bf16, F, ldg, ldo multiples
 * of 8, gu and out 16-byte aligned.  (The activation over a stored gate | up
 * tensor; hs_gemm_bf16_swiglu applies it inside the projection instead.) */
hs_status hs_swiglu(const void* gu, int64_t ldg, int32_t T, int32_t F, void* out, int64_t ldo, void* stream);
/* dst row dst_rows[i] = src row src_rows[i] (device int32 row lists; row
 * strides lds, ldd and width_bytes in BYTES, multiples of 16; src and dst
 * 16-byte aligned; a checkpoint's convolution window, for instance).  The
 * row lists are device data the host cannot check: each entry must index a
 * row inside its buffer. */
hs_status hs_copy_rows(const void* src, int64_t lds, const int32_t* src_rows, void* dst, int64_t ldd,
                       const int32_t* dst_rows, int32_t n, int32_t width_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Status and diagnostics                                                    */
/* ------------------------------------------------------------------------ */
/* Failure detection of the bounded device waits.  Every wait of a tcgen05
 * kernel on a shared-memory barrier gives up after a cycle limit: the kernel
 * records HS_DEV_TIMEOUT in the status word, lets its own copies in flight
 * land, frees its tensor memory and returns, so the context stays usable and
 * the host learns of the failure from the status word.  This call takes that
 * path on purpose on one CTA: holding 32 tensor-memory columns and a 1 KB
 * bulk copy in flight, two warps wait on barriers that nothing ever completes
 * -- one with the suspending try_wait poll, one with the spinning test_wait
 * poll -- for wait_cycles SM clocks each (1 .. 2^31); then the copy is
 * waited for and the columns freed.  *dev_status (device int32) receives
 * HS_DEV_TIMEOUT; dev_elapsed (device int64[2], or NULL) the clocks each
 * wait lasted.  Asynchronous on `stream`.  HS_EINVAL: a null status word or
 * wait_cycles outside the range. */
hs_status hs_debug_wait_timeout(int64_t wait_cycles, int32_t* dev_status, int64_t* dev_elapsed, void* stream);
/* Map a host copy of the device status word to HS_OK / HS_EDEVICE. */
hs_status hs_check_status(const int32_t* host_status_word);
/* Thread-local message of the last failing call on this thread. */
const char* hs_last_error(void);
/* Number of kernels this library has launched in this process. */
int64_t hs_launch_count(void);
/* Library version string. */
const char* hs_version(void);

#ifdef __cplusplus
}
#endif
#endif /* HS_H_ */
