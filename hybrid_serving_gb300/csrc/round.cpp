// round.cpp -- host side of the tree-prefill library: the KV page pool, the
// round builder that flattens request trees into one stream, and the packing
// of the GPU-resident metadata.
//
// Sources:
//  * Flide, "Accelerating Decision Inference with Exact State Forking",
//    section 3.2 (Eq. 2: trunks first, then the branches of each request; a
//    branch's positions continue from its parent), section 3.2.1 (Eq. 3:
//    the keys of a token are its ancestors' tokens and its own node up to
//    itself), section 3.2.2 (two GDN calls: children start from the parent's
//    end state by index), section 3.3.1 (GPU-resident metadata, a tile table
//    with unmasked full key blocks, a fixed-length chunk list), section 3.4
//    (checkpoint = state saved at a node boundary; resumed history precedes
//    the new keys), section 3.5 (every question gets tiles and chunks of its
//    own that start at the fork).
//  * ForkServe README, "Copy-on-write context tree": fork aliases the parent
//    page table and alias length and allocates nothing; writes allocate the
//    node's own pages; abort decrefs.
#include <cuda_runtime.h>
#include <string.h>

#include <algorithm>
#include <functional>
#include <string>
#include <vector>

#include "common.h"
#include "meta.h"

using namespace hsm;

namespace hs {

static thread_local std::string g_err;
static std::atomic<int64_t> g_launches{0};

hs_status fail(hs_status code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

}  // namespace hs

extern "C" const char* hs_last_error(void) { return hs::g_err.c_str(); }
extern "C" int64_t hs_launch_count(void) { return hs::g_launches.load(); }
extern "C" const char* hs_version(void) { return "hsfork 0.1 (sm_103a)"; }

extern "C" hs_status hs_check_status(const int32_t* w) {
  if (!w) return hs::fail(HS_EINVAL, "null status word");
  if (*w == HS_DEV_OK) return HS_OK;
  return hs::fail(HS_EDEVICE, "device status %d (%s)", *w,
                  *w == HS_DEV_BAD_PAGE   ? "page id out of range"
                  : *w == HS_DEV_BAD_SLOT ? "state slot out of range"
                  : *w == HS_DEV_BAD_META ? "inconsistent metadata"
                  : *w == HS_DEV_TIMEOUT  ? "a bounded wait in a kernel ran out"
                                          : "unknown");
}

// ---------------------------------------------------------------------------
// page pool
// ---------------------------------------------------------------------------
struct hs_page_pool {
  int32_t n_pages = 0, page_size = 0;
  std::vector<int32_t> ref;
  // Free pages, highest id first, so that an allocation takes the lowest free ids in ascending order: a
  // node's pages form ascending runs wherever the free pages do, and the attention kernel moves a 128-key
  // block of consecutive pages as one box.  Pages freed since the last allocation wait in `returned` and
  // are merged in (sorted) before the next one.
  std::vector<int32_t> free_list;
  std::vector<int32_t> returned;

  int32_t n_free() const { return (int32_t)(free_list.size() + returned.size()); }
  void settle() {
    if (returned.empty()) return;
    std::sort(returned.begin(), returned.end(), std::greater<int32_t>());
    std::vector<int32_t> merged(free_list.size() + returned.size());
    std::merge(free_list.begin(), free_list.end(), returned.begin(), returned.end(), merged.begin(),
               std::greater<int32_t>());
    free_list.swap(merged);
    returned.clear();
  }
  bool alloc(int32_t n, std::vector<int32_t>& out) {
    if (n_free() < n) return false;
    settle();
    for (int32_t i = 0; i < n; ++i) {
      int32_t p = free_list.back();
      free_list.pop_back();
      ref[p] = 1;
      out.push_back(p);
    }
    return true;
  }
  void decref(int32_t p) {
    if (p < 0 || p >= n_pages || ref[p] <= 0) return;
    if (--ref[p] == 0) returned.push_back(p);
  }
};

extern "C" hs_status hs_page_pool_create(int32_t n_pages, int32_t page_size, hs_page_pool** out) {
  HS_CHECK_ARG(out, "null out");
  HS_CHECK_ARG(n_pages > 0, "n_pages must be > 0");
  if (page_size != kPage) return hs::fail(HS_EUNSUPPORTED, "page_size %d (built for %d)", page_size, kPage);
  auto* p = new hs_page_pool;
  p->n_pages = n_pages;
  p->page_size = page_size;
  p->ref.assign(n_pages, 0);
  p->free_list.reserve(n_pages);
  for (int32_t i = n_pages - 1; i >= 0; --i) p->free_list.push_back(i);
  *out = p;
  return HS_OK;
}

extern "C" void hs_page_pool_destroy(hs_page_pool* p) { delete p; }

extern "C" hs_status hs_page_pool_stats(const hs_page_pool* p, int32_t* n_free, int32_t* n_live) {
  HS_CHECK_ARG(p, "null pool");
  if (n_free) *n_free = p->n_free();
  if (n_live) *n_live = p->n_pages - p->n_free();
  return HS_OK;
}

extern "C" hs_status hs_page_pool_refcount(const hs_page_pool* p, int32_t page, int32_t* ref) {
  HS_CHECK_ARG(p && ref, "null argument");
  HS_CHECK_ARG(page >= 0 && page < p->n_pages, "page %d out of range", page);
  *ref = p->ref[page];
  return HS_OK;
}

extern "C" hs_status hs_page_pool_decref(hs_page_pool* p, const int32_t* pages, int32_t n) {
  HS_CHECK_ARG(p && n >= 0 && (pages || n == 0), "null argument");
  for (int32_t i = 0; i < n; ++i) {
    HS_CHECK_ARG(pages[i] >= 0 && pages[i] < p->n_pages && p->ref[pages[i]] > 0,
                 "page %d is not live", pages[i]);
  }
  // a page listed k times must hold at least k references (checked before any change)
  std::vector<int32_t> sorted(pages, pages + n);
  std::sort(sorted.begin(), sorted.end());
  for (int32_t i = 0; i < n;) {
    int32_t j = i;
    while (j < n && sorted[j] == sorted[i]) ++j;
    HS_CHECK_ARG(j - i <= p->ref[sorted[i]], "page %d listed %d times but holds %d references", sorted[i], j - i,
                 p->ref[sorted[i]]);
    i = j;
  }
  for (int32_t i = 0; i < n; ++i) p->decref(pages[i]);
  return HS_OK;
}

// ---------------------------------------------------------------------------
// round
// ---------------------------------------------------------------------------
namespace {

struct Seg {
  int32_t parent = -1, n_tok = 0, flags = 0, save_slot = -1, request = 0;
  int32_t resume_slot = -1, resume_pos = -1, conv_window = -1;
  std::vector<int32_t> hist_ntok, hist_pages;
  std::vector<int32_t> children;
  // computed at finalize
  int32_t level = 0, stream_off = 0, pos0 = 0, own_span = -1, init_slot = -1, end_slot = -1;
  int32_t chunk_off = 0, n_chunk = 0, readout_row = -1, page_ref_off = 0, n_pages = 0;
  std::vector<int32_t> hist_spans;  // span ids of the history (roots only)
  std::vector<int32_t> pages;       // own pages
};

}  // namespace

struct hs_round {
  hs_round_caps caps{};
  Layout L{};
  std::vector<Seg> segs;
  int32_t n_requests = 0;
  bool finalized = false;
  bool released = false;
  hs_page_pool* pool = nullptr;  // the pool finalize allocated from (NULL: none)
  std::vector<int32_t> blob;
  hs_round_info info{};
  std::vector<int32_t> readouts;
  std::vector<int32_t> hist_refs;  // history pages the round holds a reference on
};

static Layout layout_of(const hs_round_caps& c) {
  return layout_for(c.max_tokens, c.max_segments, c.max_segments + c.max_hist_spans, c.max_tiles,
                    c.max_tile_spans, c.max_chunks, c.max_readouts, c.max_levels, c.max_page_refs);
}

extern "C" hs_status hs_round_caps_for(int32_t n_tokens, int32_t n_segments, int32_t n_levels,
                                       int32_t n_hist_spans, int32_t n_hist_pages, int32_t page_size,
                                       hs_round_caps* out) {
  HS_CHECK_ARG(out, "null out");
  HS_CHECK_ARG(n_tokens >= 0 && n_segments >= 0 && n_levels >= 1 && n_hist_spans >= 0 && n_hist_pages >= 0,
               "negative size");
  if (page_size != kPage) return hs::fail(HS_EUNSUPPORTED, "page_size %d (built for %d)", page_size, kPage);
  hs_round_caps c;
  c.max_tokens = n_tokens;
  c.max_segments = n_segments;
  c.max_hist_spans = n_hist_spans;
  c.max_tiles = n_tokens / kTileRows + n_segments + 1;
  c.max_tile_spans = c.max_tiles * (n_levels + n_hist_spans) + 1;
  c.max_chunks = n_tokens / kChunk + n_segments + 1;
  c.max_readouts = n_segments;
  c.max_page_refs = n_tokens / kPage + n_segments + n_hist_pages + 1;
  c.max_levels = n_levels;
  *out = c;
  return HS_OK;
}

extern "C" size_t hs_round_meta_bytes(const hs_round_caps* caps) {
  if (!caps) return 0;
  return (size_t)layout_of(*caps).total_words * 4;
}

extern "C" hs_status hs_round_create(const hs_round_caps* caps, hs_round** out) {
  HS_CHECK_ARG(caps && out, "null argument");
  const hs_round_caps& c = *caps;
  HS_CHECK_ARG(c.max_tokens >= 0 && c.max_segments >= 0 && c.max_hist_spans >= 0 && c.max_tiles >= 0 &&
                   c.max_tile_spans >= 0 && c.max_chunks >= 0 && c.max_readouts >= 0 &&
                   c.max_page_refs >= 0 && c.max_levels >= 1,
               "negative capacity");
  int64_t words = (int64_t)kHeaderWords + (int64_t)c.max_segments * kSegWords + (int64_t)c.max_tokens * kTokWords +
                  (int64_t)(c.max_segments + c.max_hist_spans) * kSpanWords + (int64_t)c.max_tiles * kTileWords +
                  c.max_tile_spans + (int64_t)c.max_chunks * kChunkWords + c.max_readouts + c.max_levels +
                  c.max_segments + c.max_page_refs + (int64_t)c.max_tokens * kPredWords + 200;
  HS_CHECK_ARG(words < (int64_t)1 << 30, "capacities too large");
  auto* r = new hs_round;
  r->caps = c;
  r->L = layout_of(c);
  *out = r;
  return HS_OK;
}

extern "C" void hs_round_destroy(hs_round* r) { delete r; }

extern "C" hs_status hs_round_add_segment(hs_round* r, int32_t parent, int32_t n_tokens, int32_t flags,
                                          int32_t save_slot, int32_t* seg_out) {
  HS_CHECK_ARG(r, "null round");
  HS_CHECK_ARG(!r->finalized, "round already finalized");
  HS_CHECK_ARG(n_tokens >= 1, "a node needs at least one token (got %d)", n_tokens);
  HS_CHECK_ARG(parent >= -1 && parent < (int32_t)r->segs.size(), "unknown parent %d", parent);
  HS_CHECK_ARG(save_slot >= -1, "bad save slot %d", save_slot);
  HS_CHECK_ARG((flags & ~(HS_SEG_READOUT | HS_SEG_NO_READOUT)) == 0, "unknown flags %d", flags);
  if ((int32_t)r->segs.size() >= r->caps.max_segments)
    return hs::fail(HS_ECAPACITY, "more than max_segments=%d nodes", r->caps.max_segments);
  Seg s;
  s.parent = parent;
  s.n_tok = n_tokens;
  s.flags = flags;
  s.save_slot = save_slot;
  if (parent < 0) {
    s.request = r->n_requests++;
  } else {
    s.request = r->segs[parent].request;
    r->segs[parent].children.push_back((int32_t)r->segs.size());
  }
  r->segs.push_back(std::move(s));
  if (seg_out) *seg_out = (int32_t)r->segs.size() - 1;
  return HS_OK;
}

extern "C" hs_status hs_round_add_segments(hs_round* r, int32_t n, const int32_t* parent, const int32_t* n_tokens,
                                           const int32_t* flags, const int32_t* save_slot, int32_t* first_id) {
  HS_CHECK_ARG(r, "null round");
  HS_CHECK_ARG(!r->finalized, "round already finalized");
  HS_CHECK_ARG(n >= 0 && (n == 0 || (parent && n_tokens)), "bad node arrays");
  const int32_t base = (int32_t)r->segs.size();
  if ((int64_t)base + n > r->caps.max_segments)
    return hs::fail(HS_ECAPACITY, "more than max_segments=%d nodes", r->caps.max_segments);
  // every entry is checked before any node is added
  for (int32_t j = 0; j < n; ++j) {
    HS_CHECK_ARG(n_tokens[j] >= 1, "node %d needs at least one token (got %d)", base + j, n_tokens[j]);
    HS_CHECK_ARG(parent[j] >= -1 && parent[j] < base + j, "node %d: unknown parent %d", base + j, parent[j]);
    const int32_t f = flags ? flags[j] : 0, sv = save_slot ? save_slot[j] : -1;
    HS_CHECK_ARG((f & ~(HS_SEG_READOUT | HS_SEG_NO_READOUT)) == 0, "node %d: unknown flags %d", base + j, f);
    HS_CHECK_ARG(sv >= -1, "node %d: bad save slot %d", base + j, sv);
  }
  r->segs.reserve(base + n);
  for (int32_t j = 0; j < n; ++j) {
    Seg s;
    s.parent = parent[j];
    s.n_tok = n_tokens[j];
    s.flags = flags ? flags[j] : 0;
    s.save_slot = save_slot ? save_slot[j] : -1;
    if (s.parent < 0) {
      s.request = r->n_requests++;
    } else {
      s.request = r->segs[s.parent].request;
      r->segs[s.parent].children.push_back(base + j);
    }
    r->segs.push_back(std::move(s));
  }
  if (first_id) *first_id = base;
  return HS_OK;
}

extern "C" hs_status hs_gdn_state_resume(hs_round* r, int32_t seg, int32_t ckpt_slot, int32_t ckpt_pos) {
  HS_CHECK_ARG(r, "null round");
  HS_CHECK_ARG(!r->finalized, "round already finalized");
  HS_CHECK_ARG(seg >= 0 && seg < (int32_t)r->segs.size(), "unknown node %d", seg);
  HS_CHECK_ARG(r->segs[seg].parent < 0, "only a root can resume (node %d has a parent)", seg);
  HS_CHECK_ARG(ckpt_slot >= 0, "bad checkpoint slot %d", ckpt_slot);
  HS_CHECK_ARG(ckpt_pos >= 0, "bad checkpoint position %d", ckpt_pos);
  r->segs[seg].resume_slot = ckpt_slot;
  r->segs[seg].resume_pos = ckpt_pos;
  return HS_OK;
}

extern "C" hs_status hs_round_set_conv_window(hs_round* r, int32_t seg, int32_t window_row0) {
  HS_CHECK_ARG(r, "null round");
  HS_CHECK_ARG(!r->finalized, "round already finalized");
  HS_CHECK_ARG(seg >= 0 && seg < (int32_t)r->segs.size(), "unknown node %d", seg);
  HS_CHECK_ARG(r->segs[seg].parent < 0, "only a root has a conv window (node %d has a parent)", seg);
  HS_CHECK_ARG(window_row0 >= 0, "bad window row %d", window_row0);
  r->segs[seg].conv_window = window_row0;
  return HS_OK;
}

extern "C" hs_status hs_round_attach_history(hs_round* r, int32_t seg, int32_t n_spans, const int32_t* ntok,
                                             const int32_t* pages) {
  HS_CHECK_ARG(r, "null round");
  HS_CHECK_ARG(!r->finalized, "round already finalized");
  HS_CHECK_ARG(seg >= 0 && seg < (int32_t)r->segs.size(), "unknown node %d", seg);
  HS_CHECK_ARG(r->segs[seg].parent < 0, "only a root has history (node %d has a parent)", seg);
  HS_CHECK_ARG(n_spans >= 0 && (n_spans == 0 || (ntok && pages)), "bad history spans");
  Seg& s = r->segs[seg];
  int64_t np = 0;
  for (int32_t i = 0; i < n_spans; ++i) {
    HS_CHECK_ARG(ntok[i] >= 1, "history span %d is empty", i);
    np += (ntok[i] + kPage - 1) / kPage;
  }
  HS_CHECK_ARG(np < ((int64_t)1 << 30), "history of %lld pages is too long", (long long)np);
  s.hist_ntok.assign(ntok, ntok + n_spans);
  s.hist_pages.assign(pages, pages + np);
  return HS_OK;
}

static hs_status build(hs_round* r, hs_page_pool* pool, int32_t temp0, int32_t n_temp,
                       std::vector<int32_t>& allocated) {
  const hs_round_caps& C = r->caps;
  std::vector<Seg>& S = r->segs;
  const int32_t n = (int32_t)S.size();
  HS_CHECK_ARG(n > 0, "empty round");
  for (auto& s : S) {  // a finalize retried after an error starts again from the nodes as added
    s.hist_spans.clear();
    s.pages.clear();
  }

  // levels (parents precede children by construction)
  int32_t n_levels = 0;
  for (int32_t i = 0; i < n; ++i) {
    S[i].level = S[i].parent < 0 ? 0 : S[S[i].parent].level + 1;
    n_levels = std::max(n_levels, S[i].level + 1);
  }
  if (n_levels > C.max_levels) return hs::fail(HS_ECAPACITY, "tree depth %d > max_levels %d", n_levels, C.max_levels);

  // Eq. 2 stream order: level, then request, then node id
  std::vector<int32_t> order(n);
  for (int32_t i = 0; i < n; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
    if (S[a].level != S[b].level) return S[a].level < S[b].level;
    if (S[a].request != S[b].request) return S[a].request < S[b].request;
    return a < b;
  });
  int64_t T = 0;
  for (int32_t id : order) {
    S[id].stream_off = (int32_t)T;
    T += S[id].n_tok;
  }
  if (T > C.max_tokens) return hs::fail(HS_ECAPACITY, "stream of %lld tokens > max_tokens %d", (long long)T, C.max_tokens);

  // positions
  for (int32_t i = 0; i < n; ++i) {
    Seg& s = S[i];
    if (s.parent >= 0) {
      s.pos0 = S[s.parent].pos0 + S[s.parent].n_tok;
    } else {
      int64_t hist = 0;
      for (int32_t t : s.hist_ntok) hist += t;
      if (!s.hist_ntok.empty() && s.resume_pos >= 0 && hist != s.resume_pos)
        return hs::fail(HS_EINVAL, "node %d: history holds %lld tokens but resumes at %d", i, (long long)hist,
                        s.resume_pos);
      if (hist >= ((int64_t)1 << 31)) return hs::fail(HS_EINVAL, "node %d: history too long", i);
      s.pos0 = s.resume_pos >= 0 ? s.resume_pos : (int32_t)hist;
    }
    if ((int64_t)s.pos0 + s.n_tok >= ((int64_t)1 << 31)) return hs::fail(HS_EINVAL, "node %d: positions overflow", i);
  }

  // pages: history pages are referenced, own pages allocated
  int32_t n_hist_spans = 0, n_hist_pages = 0;
  for (auto& s : S) {
    n_hist_spans += (int32_t)s.hist_ntok.size();
    n_hist_pages += (int32_t)s.hist_pages.size();
  }
  if (n_hist_spans > C.max_hist_spans)
    return hs::fail(HS_ECAPACITY, "%d history spans > max_hist_spans %d", n_hist_spans, C.max_hist_spans);
  if (n_hist_spans >= (1 << kHistShift))
    return hs::fail(HS_ECAPACITY, "%d history spans (at most %d)", n_hist_spans, (1 << kHistShift) - 1);
  for (const auto& s : S)
    if (s.hist_ntok.size() >= (size_t)1 << (31 - kHistShift))
      return hs::fail(HS_ECAPACITY, "a root with %d history spans (at most %d)", (int)s.hist_ntok.size(),
                      (1 << (31 - kHistShift)) - 1);
  int64_t n_own_pages = 0;
  if (pool)
    for (auto& s : S) n_own_pages += (s.n_tok + kPage - 1) / kPage;
  if (n_hist_pages + n_own_pages > C.max_page_refs)
    return hs::fail(HS_ECAPACITY, "%lld page refs > max_page_refs %d", (long long)(n_hist_pages + n_own_pages),
                    C.max_page_refs);
  if (n_hist_pages > 0 && !pool) return hs::fail(HS_EINVAL, "history pages need a page pool");
  if (pool) {
    for (auto& s : S)
      for (int32_t p : s.hist_pages)
        if (p < 0 || p >= pool->n_pages || pool->ref[p] <= 0)
          return hs::fail(HS_EINVAL, "history page %d is not live in the pool", p);
    if (n_own_pages > (int64_t)pool->n_free())
      return hs::fail(HS_ENOPAGES, "need %lld pages, %d free", (long long)n_own_pages, (int)pool->n_free());
  }

  std::vector<int32_t> page_ref;
  std::vector<int32_t> spans;  // kSpanWords each
  auto add_span = [&](int32_t off, int32_t ntok, int32_t owner) {
    spans.push_back(off);
    spans.push_back(ntok);
    spans.push_back(owner);
    spans.push_back(0);
    return (int32_t)spans.size() / kSpanWords - 1;
  };
  // history spans of roots (in node order), then own spans in stream order
  for (int32_t i = 0; i < n; ++i) {
    Seg& s = S[i];
    int32_t pi = 0;
    for (int32_t t : s.hist_ntok) {
      int32_t np = (t + kPage - 1) / kPage;
      int32_t off = (int32_t)page_ref.size();
      for (int32_t k = 0; k < np; ++k) page_ref.push_back(s.hist_pages[pi + k]);
      pi += np;
      s.hist_spans.push_back(add_span(off, t, -1));
    }
  }
  for (int32_t id : order) {
    Seg& s = S[id];
    s.page_ref_off = (int32_t)page_ref.size();
    s.pages.clear();
    if (pool) {
      int32_t np = (s.n_tok + kPage - 1) / kPage;
      pool->alloc(np, s.pages);  // capacity checked above
      allocated.insert(allocated.end(), s.pages.begin(), s.pages.end());
      page_ref.insert(page_ref.end(), s.pages.begin(), s.pages.end());
    }
    s.n_pages = (int32_t)s.pages.size();
    s.own_span = add_span(s.page_ref_off, s.n_tok, id);
  }

  // ancestor spans (visible to every row of a node): history, then each ancestor's own span
  std::vector<std::vector<int32_t>> anc(n);
  for (int32_t i = 0; i < n; ++i) {  // parents precede children
    if (S[i].parent < 0) {
      anc[i] = S[i].hist_spans;
    } else {
      anc[i] = anc[S[i].parent];
      anc[i].push_back(S[S[i].parent].own_span);
    }
  }

  // readouts (section 3.3.3): the last token of each readout node, in node order
  r->readouts.clear();
  for (int32_t i = 0; i < n; ++i) {
    Seg& s = S[i];
    bool ro = (s.flags & HS_SEG_READOUT) || (s.children.empty() && !(s.flags & HS_SEG_NO_READOUT));
    s.readout_row = ro ? s.stream_off + s.n_tok - 1 : -1;
    if (ro) r->readouts.push_back(s.readout_row);
  }
  if ((int32_t)r->readouts.size() > C.max_readouts)
    return hs::fail(HS_ECAPACITY, "%d readouts > max_readouts %d", (int)r->readouts.size(), C.max_readouts);

  // attention tiles (section 3.3.1 tile table; section 3.5: tiles start at the node)
  std::vector<int32_t> tiles, tile_spans;
  auto blocks = [](int32_t keys) { return (keys + kTileRows - 1) / kTileRows; };
  for (size_t oi = 0; oi < order.size();) {
    int32_t id = order[oi];
    Seg& s = S[id];
    if (s.n_tok > kTileRows || s.parent < 0) {
      for (int32_t r0 = 0; r0 < s.n_tok; r0 += kTileRows) {
        int32_t nr = std::min(kTileRows, s.n_tok - r0);
        int32_t work = 0;
        for (int32_t sp : anc[id]) work += blocks(spans[sp * kSpanWords + SP_N_TOK]);
        work += blocks(r0 + nr);
        int32_t off = (int32_t)tile_spans.size();
        tile_spans.insert(tile_spans.end(), anc[id].begin(), anc[id].end());
        tile_spans.push_back(s.own_span);
        const int32_t ro = s.readout_row >= s.stream_off + r0 && s.readout_row < s.stream_off + r0 + nr;
        int32_t rec[kTileWords] = {s.stream_off + r0, nr, off, (int32_t)anc[id].size(), 1, work, id, ro};
        tiles.insert(tiles.end(), rec, rec + kTileWords);
      }
      ++oi;
      continue;
    }
    // pack consecutive siblings (same parent, each <= 128 rows) into one tile
    size_t oj = oi;
    int32_t rows = 0;
    std::vector<int32_t> members;
    while (oj < order.size()) {
      Seg& t = S[order[oj]];
      if (t.parent != s.parent || t.n_tok > kTileRows || rows + t.n_tok > kTileRows) break;
      rows += t.n_tok;
      members.push_back(order[oj]);
      ++oj;
    }
    int32_t work = 0;
    for (int32_t sp : anc[id]) work += blocks(spans[sp * kSpanWords + SP_N_TOK]);
    for (int32_t m : members) work += blocks(S[m].n_tok);
    int32_t off = (int32_t)tile_spans.size();
    tile_spans.insert(tile_spans.end(), anc[id].begin(), anc[id].end());
    for (int32_t m : members) tile_spans.push_back(S[m].own_span);
    int32_t ro = 0;
    for (int32_t m : members) ro |= S[m].readout_row >= 0;
    int32_t rec[kTileWords] = {s.stream_off, rows, off, (int32_t)anc[id].size(), (int32_t)members.size(), work, id, ro};
    tiles.insert(tiles.end(), rec, rec + kTileWords);
    oi = oj;
  }
  int32_t n_tiles = (int32_t)tiles.size() / kTileWords;
  if (n_tiles > C.max_tiles) return hs::fail(HS_ECAPACITY, "%d tiles > max_tiles %d", n_tiles, C.max_tiles);
  if ((int32_t)tile_spans.size() > C.max_tile_spans)
    return hs::fail(HS_ECAPACITY, "%d tile spans > max_tile_spans %d", (int)tile_spans.size(), C.max_tile_spans);
  // heaviest tiles first: the paired-head attention kernel hands its (tile, head pair) items out in this
  // order to whichever CTA asks next, i.e. longest-first list scheduling
  {
    std::vector<int32_t> idx(n_tiles);
    for (int32_t i = 0; i < n_tiles; ++i) idx[i] = i;
    // (a tile with a readout row costs ~1.4x per key block: its P.V products carry P's low part too)
    auto cost = [&](int32_t i) { return (int64_t)tiles[i * kTileWords + TL_WORK] * (tiles[i * kTileWords + TL_READOUT] ? 7 : 5); };
    std::stable_sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) { return cost(a) > cost(b); });
    std::vector<int32_t> sorted(tiles.size());
    for (int32_t i = 0; i < n_tiles; ++i)
      memcpy(&sorted[i * kTileWords], &tiles[idx[i] * kTileWords], kTileWords * 4);
    tiles.swap(sorted);
  }

  // GDN chunks (section 3.3.1 chunk list; section 3.5: each node starts a chunk)
  std::vector<int32_t> chunks;
  int32_t max_seg_chunks = 0;
  for (int32_t id : order) {
    Seg& s = S[id];
    s.chunk_off = (int32_t)chunks.size() / kChunkWords;
    int32_t c = 0;
    for (int32_t r0 = 0; r0 < s.n_tok; r0 += kChunk, ++c) {
      int32_t rec[kChunkWords] = {id, s.stream_off + r0, std::min(kChunk, s.n_tok - r0), c};
      chunks.insert(chunks.end(), rec, rec + kChunkWords);
    }
    s.n_chunk = c;
    max_seg_chunks = std::max(max_seg_chunks, c);
  }
  int32_t n_chunks = (int32_t)chunks.size() / kChunkWords;
  if (n_chunks > C.max_chunks) return hs::fail(HS_ECAPACITY, "%d chunks > max_chunks %d", n_chunks, C.max_chunks);

  // GDN state slots (section 3.2.2: children read the parent's end state by index)
  std::vector<int32_t> user_slots;
  for (int32_t i = 0; i < n; ++i) {
    if (S[i].save_slot >= 0) user_slots.push_back(S[i].save_slot);
  }
  {
    std::vector<int32_t> u = user_slots;
    std::sort(u.begin(), u.end());
    if (std::adjacent_find(u.begin(), u.end()) != u.end()) return hs::fail(HS_EINVAL, "two nodes save into one slot");
  }
  for (int32_t i = 0; i < n; ++i) {
    int32_t rs = S[i].resume_slot;
    if (rs < 0) continue;
    for (int32_t j = 0; j < n; ++j)
      if (j != i && S[j].save_slot == rs)
        return hs::fail(HS_EINVAL, "node %d saves into slot %d that node %d resumes from", j, rs, i);
  }
  int32_t next_temp = 0;
  for (int32_t id : order) {
    Seg& s = S[id];
    if (s.save_slot >= 0) {
      s.end_slot = s.save_slot;
    } else if (!s.children.empty()) {
      if (next_temp >= n_temp) return hs::fail(HS_ECAPACITY, "more inner nodes than the %d temporary slots", n_temp);
      s.end_slot = temp0 + next_temp++;
      for (int32_t i = 0; i < n; ++i)
        if (S[i].save_slot == s.end_slot || S[i].resume_slot == s.end_slot)
          return hs::fail(HS_EINVAL, "temporary slot %d collides with a save/resume slot", s.end_slot);
    } else {
      s.end_slot = -1;
    }
    s.init_slot = s.parent >= 0 ? S[s.parent].end_slot : s.resume_slot;
  }

  // ---- pack ----
  const Layout& L = r->L;
  std::vector<int32_t>& B = r->blob;
  B.assign(L.total_words, 0);
  int32_t* h = B.data();
  h[H_MAGIC] = kMagic;
  h[H_N_TOK] = (int32_t)T;
  h[H_N_SEG] = n;
  h[H_N_SPAN] = (int32_t)spans.size() / kSpanWords;
  h[H_N_TILE] = n_tiles;
  h[H_N_TILE_SPAN] = (int32_t)tile_spans.size();
  h[H_N_CHUNK] = n_chunks;
  h[H_N_READOUT] = (int32_t)r->readouts.size();
  h[H_N_LEVEL] = n_levels;
  h[H_N_PAGE_REF] = (int32_t)page_ref.size();
  h[H_OFF_SEG] = L.off_seg;
  h[H_OFF_TOK] = L.off_tok;
  h[H_OFF_SPAN] = L.off_span;
  h[H_OFF_TILE] = L.off_tile;
  h[H_OFF_TILE_SPAN] = L.off_tile_span;
  h[H_OFF_CHUNK] = L.off_chunk;
  h[H_OFF_READOUT] = L.off_readout;
  h[H_OFF_LEVEL] = L.off_level;
  h[H_OFF_LEVEL_SEG] = L.off_level_seg;
  h[H_OFF_PAGE_REF] = L.off_page_ref;
  h[H_OFF_SCAN] = L.off_scan;
  h[H_OFF_SCAN_LEVEL] = L.off_scan_level;
  h[H_CAP_TOK] = C.max_tokens;
  h[H_CAP_SEG] = C.max_segments;
  h[H_CAP_SPAN] = C.max_segments + C.max_hist_spans;
  h[H_CAP_TILE] = C.max_tiles;
  h[H_CAP_TILE_SPAN] = C.max_tile_spans;
  h[H_CAP_CHUNK] = C.max_chunks;
  h[H_CAP_READOUT] = C.max_readouts;
  h[H_CAP_LEVEL] = C.max_levels;
  h[H_CAP_PAGE_REF] = C.max_page_refs;
  h[H_TOTAL_WORDS] = L.total_words;
  h[H_MAX_SEG_CHUNKS] = max_seg_chunks;
  for (int32_t i = 0; i < n; ++i) {
    const Seg& s = S[i];
    int32_t* g = h + L.off_seg + i * kSegWords;
    g[S_STREAM_OFF] = s.stream_off;
    g[S_LEN] = s.n_tok;
    g[S_POS0] = s.pos0;
    g[S_REQUEST] = s.request;
    g[S_PARENT] = s.parent;
    g[S_LEVEL] = s.level;
    g[S_OWN_SPAN] = s.own_span;
    g[S_INIT_SLOT] = s.init_slot;
    g[S_END_SLOT] = s.end_slot;
    g[S_CHUNK_OFF] = s.chunk_off;
    g[S_N_CHUNK] = s.n_chunk;
    g[S_READOUT_ROW] = s.readout_row;
    g[S_PAGE_REF_OFF] = s.page_ref_off;
    g[S_N_PAGES] = s.n_pages;
    g[S_HIST] = s.hist_spans.empty() ? 0 : s.hist_spans[0] | ((int32_t)s.hist_spans.size() << kHistShift);
    for (int32_t u = 0; u < s.n_tok; ++u) {
      int32_t* t = h + L.off_tok + (s.stream_off + u) * kTokWords;
      t[T_SEG] = i;
      t[T_IDX] = u;
    }
  }
  memcpy(h + L.off_span, spans.data(), spans.size() * 4);
  memcpy(h + L.off_tile, tiles.data(), tiles.size() * 4);
  memcpy(h + L.off_tile_span, tile_spans.data(), tile_spans.size() * 4);
  memcpy(h + L.off_chunk, chunks.data(), chunks.size() * 4);
  memcpy(h + L.off_readout, r->readouts.data(), r->readouts.size() * 4);
  memcpy(h + L.off_page_ref, page_ref.data(), page_ref.size() * 4);
  h[H_OFF_PRED] = L.off_pred;
  // conv predecessors: a node's first kPredWords tokens walk back through the node, then its ancestors'
  // last tokens; every later token's predecessors are simply the stream rows before it
  for (int32_t i = 0; i < n; ++i) {
    const Seg& s = S[i];
    const int32_t head = std::min(s.n_tok, (int32_t)kPredWords);
    int32_t* pn = h + L.off_pred + s.stream_off * kPredWords;
    for (int32_t u = head; u < s.n_tok; ++u)
      for (int32_t k = 1; k <= kPredWords; ++k) pn[u * kPredWords + k - 1] = s.stream_off + u - k;
    for (int32_t u = 0; u < head; ++u) {
      int32_t* pr = pn + u * kPredWords;
      for (int32_t k = 1; k <= kPredWords; ++k) {
        int32_t node = i, idx = u - k, val = -1;
        while (idx < 0 && S[node].parent >= 0) {
          node = S[node].parent;
          idx += S[node].n_tok;
        }
        if (idx >= 0) {
          val = S[node].stream_off + idx;
        } else if (S[node].conv_window >= 0) {  // idx in [-kPredWords, -1] of a resumed root
          if (idx >= -kPredWords) val = -2 - (S[node].conv_window + kPredWords + idx);
        }
        pr[k - 1] = val;
      }
    }
  }
  {
    // a level's nodes, most chunks first (stream order among equals): the state pass hands its CTAs out
    // in this order, so when a level needs more than one wave the short nodes fill the last one
    int32_t k = 0;
    std::vector<int32_t> lev_ids;
    for (int32_t lev = 0; lev < n_levels; ++lev) {
      h[L.off_level + lev] = k;
      lev_ids.clear();
      for (int32_t id : order)
        if (S[id].level == lev) lev_ids.push_back(id);
      std::stable_sort(lev_ids.begin(), lev_ids.end(),
                       [&](int32_t a, int32_t b) { return S[a].n_chunk > S[b].n_chunk; });
      for (int32_t id : lev_ids) h[L.off_level_seg + k++] = id;
    }
    for (int32_t lev = n_levels; lev <= C.max_levels; ++lev) h[L.off_level + lev] = k;
  }
  {  // extra scan groups of the long nodes, by level, in segment order then group order
    int32_t k = 0;
    for (int32_t lev = 0; lev < n_levels; ++lev) {
      h[L.off_scan_level + lev] = k;
      for (int32_t id : order) {
        if (S[id].level != lev) continue;
        const int32_t G = scan_groups(S[id].n_chunk);
        h[L.off_seg + id * kSegWords + S_SCAN1] = G > 1 ? k : -1;
        for (int32_t g = 1; g < G; ++g) {
          if (k >= scan_cap(C.max_chunks)) return hs::fail(HS_ECAPACITY, "scan group table full");
          h[L.off_scan + 2 * k] = id;
          h[L.off_scan + 2 * k + 1] = g;
          ++k;
        }
      }
    }
    for (int32_t lev = n_levels; lev <= C.max_levels; ++lev) h[L.off_scan_level + lev] = k;
    h[H_N_SCAN] = k;
  }

  hs_round_info& I = r->info;
  I.n_tokens = (int32_t)T;
  I.n_segments = n;
  I.n_tiles = n_tiles;
  I.n_chunks = n_chunks;
  I.n_readouts = (int32_t)r->readouts.size();
  I.n_levels = n_levels;
  I.n_pages_allocated = (int32_t)n_own_pages;
  I.n_spans = h[H_N_SPAN];
  I.n_tile_spans = (int32_t)tile_spans.size();
  I.n_page_refs = (int32_t)page_ref.size();
  return HS_OK;
}

extern "C" hs_status hs_round_finalize(hs_round* r, hs_page_pool* pool, int32_t temp_slot0, int32_t n_temp_slots) {
  HS_CHECK_ARG(r, "null round");
  HS_CHECK_ARG(!r->finalized, "round already finalized");
  HS_CHECK_ARG(temp_slot0 >= 0 && n_temp_slots >= 0, "bad temporary slot range");
  std::vector<int32_t> allocated;
  hs_status st = build(r, pool, temp_slot0, n_temp_slots, allocated);
  if (st != HS_OK) {
    if (pool)  // (the free list is kept sorted: it returns to its old order)
      for (int32_t pg : allocated) pool->decref(pg);
    for (auto& s : r->segs) s.pages.clear();
    return st;
  }
  if (pool) {
    for (auto& s : r->segs)
      for (int32_t p : s.hist_pages) {
        pool->ref[p]++;
        r->hist_refs.push_back(p);
      }
  }
  r->pool = pool;
  r->finalized = true;
  return HS_OK;
}

extern "C" hs_status hs_round_pack(const hs_round* r, void* host, size_t bytes) {
  HS_CHECK_ARG(r && host, "null argument");
  HS_CHECK_ARG(r->finalized, "round not finalized");
  size_t need = r->blob.size() * 4;
  HS_CHECK_ARG(bytes >= need, "buffer of %zu bytes < %zu", bytes, need);
  memcpy(host, r->blob.data(), need);
  return HS_OK;
}

extern "C" hs_status hs_round_upload(const hs_round* r, void* dev_meta, size_t bytes, void* stream) {
  HS_CHECK_ARG(r && dev_meta, "null argument");
  HS_CHECK_ARG(r->finalized, "round not finalized");
  size_t need = r->blob.size() * 4;
  HS_CHECK_ARG(bytes >= need, "device buffer of %zu bytes < %zu", bytes, need);
  cudaError_t e = cudaMemcpyAsync(dev_meta, r->blob.data(), need, cudaMemcpyHostToDevice, (cudaStream_t)stream);
  if (e != cudaSuccess) return hs::fail(HS_ECUDA, "metadata upload: %s", cudaGetErrorString(e));
  return HS_OK;
}

extern "C" hs_status hs_round_get_info(const hs_round* r, hs_round_info* out) {
  HS_CHECK_ARG(r && out, "null argument");
  HS_CHECK_ARG(r->finalized, "round not finalized");
  *out = r->info;
  return HS_OK;
}

extern "C" hs_status hs_round_segment(const hs_round* r, int32_t seg, hs_segment_info* out) {
  HS_CHECK_ARG(r && out, "null argument");
  HS_CHECK_ARG(r->finalized, "round not finalized");
  HS_CHECK_ARG(seg >= 0 && seg < (int32_t)r->segs.size(), "unknown node %d", seg);
  const Seg& s = r->segs[seg];
  out->stream_off = s.stream_off;
  out->n_tokens = s.n_tok;
  out->pos0 = s.pos0;
  out->request = s.request;
  out->parent = s.parent;
  out->level = s.level;
  out->init_slot = s.init_slot;
  out->end_slot = s.end_slot;
  out->readout_row = s.readout_row;
  out->n_pages = s.n_pages;
  return HS_OK;
}

extern "C" hs_status hs_round_segment_pages(const hs_round* r, int32_t seg, int32_t* pages, int32_t cap, int32_t* n) {
  HS_CHECK_ARG(r && n, "null argument");
  HS_CHECK_ARG(r->finalized, "round not finalized");
  HS_CHECK_ARG(seg >= 0 && seg < (int32_t)r->segs.size(), "unknown node %d", seg);
  const Seg& s = r->segs[seg];
  *n = (int32_t)s.pages.size();
  if (pages)
    for (int32_t i = 0; i < std::min(cap, *n); ++i) pages[i] = s.pages[i];
  return HS_OK;
}

extern "C" hs_status hs_round_readout_rows(const hs_round* r, int32_t* rows, int32_t cap, int32_t* n) {
  HS_CHECK_ARG(r && n, "null argument");
  HS_CHECK_ARG(r->finalized, "round not finalized");
  *n = (int32_t)r->readouts.size();
  if (rows)
    for (int32_t i = 0; i < std::min(cap, *n); ++i) rows[i] = r->readouts[i];
  return HS_OK;
}

extern "C" hs_status hs_round_release(hs_round* r, hs_page_pool* pool, const int32_t* keep, int32_t n_keep) {
  HS_CHECK_ARG(r, "null round");
  HS_CHECK_ARG(r->finalized, "round not finalized");
  HS_CHECK_ARG(!r->released, "round already released");
  HS_CHECK_ARG(pool == r->pool || (!r->pool && !pool), "not the pool the round was finalized with");
  HS_CHECK_ARG(n_keep >= 0 && (n_keep == 0 || keep), "bad keep list");
  std::vector<char> kept(r->segs.size(), 0);
  for (int32_t i = 0; i < n_keep; ++i) {
    HS_CHECK_ARG(keep[i] >= 0 && keep[i] < (int32_t)r->segs.size(), "unknown node %d", keep[i]);
    kept[keep[i]] = 1;
  }
  if (pool) {
    for (size_t i = 0; i < r->segs.size(); ++i)
      if (!kept[i])
        for (int32_t p : r->segs[i].pages) pool->decref(p);
    for (int32_t p : r->hist_refs) pool->decref(p);
  }
  r->hist_refs.clear();
  r->released = true;
  return HS_OK;
}
