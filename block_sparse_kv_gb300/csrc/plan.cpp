// Host-side plans: validation of the CSR index arrays and the per-CTA work lists.
//
// Plans are pure host code (no CUDA call). They turn the caller's index arrays into
// int32 metadata that the kernels read from the caller's int workspace:
//   * decode and MLA: a linear split-KV partition. The units (one per request and kv
//     head, or per query token and latent half) are cut into tiles; the tile sequence
//     of all units is divided into contiguous ranges, one per worker (equal ranges, or for
//     the page-major decode ranges of equal cost, a piece published mid-stream or a merge at
//     a worker's end costing a few tiles); a unit that falls into several ranges is computed
//     in pieces whose partial states are merged.
//   * BSR: longest-processing-time assignment of (row block, kv head) units to
//     persistent CTAs, heaviest unit first.
// The rules are deterministic given num_sms, so the metadata is reproducible bit for bit.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <queue>
#include <utility>

#include "internal.h"

namespace bskv {

namespace {

struct Chunk {
  int32_t unit, a, b, c;  // meaning per plan kind
};

size_t align_words(size_t n) { return (n + 3) & ~size_t(3); }

// Lay out header + sections.
void assemble(bskv_plan* p, int32_t kind, int32_t units, const std::vector<int32_t>& worker_ptr,
              const std::vector<Chunk>& chunks, int32_t slots,
              const std::vector<int32_t>& merges /* 3 per item */, int32_t tile,
              const int32_t* aux0, size_t n_aux0, const int32_t* aux1, size_t n_aux1,
              int32_t grid, int32_t variant) {
  size_t off = H_COUNT;
  const size_t off_workers = off;
  off = align_words(off + worker_ptr.size());
  const size_t off_chunks = off;
  off = align_words(off + 4 * chunks.size());
  const size_t off_merges = off;
  off = align_words(off + merges.size());
  const size_t off_aux0 = off;
  off = align_words(off + n_aux0);
  const size_t off_aux1 = off;
  off = align_words(off + n_aux1);
  std::vector<int32_t>& m = p->meta;
  m.assign(off, 0);
  m[H_MAGIC] = kMetaMagic;
  m[H_KIND] = kind;
  m[H_UNITS] = units;
  m[H_WORKERS] = int32_t(worker_ptr.empty() ? 0 : worker_ptr.size() - 1);
  m[H_CHUNKS] = int32_t(chunks.size());
  m[H_SLOTS] = slots;
  m[H_MERGES] = int32_t(merges.size() / 3);
  m[H_TILE] = tile;
  m[H_OFF_WORKERS] = int32_t(off_workers);
  m[H_OFF_CHUNKS] = int32_t(off_chunks);
  m[H_OFF_MERGES] = int32_t(off_merges);
  m[H_OFF_AUX0] = int32_t(off_aux0);
  m[H_OFF_AUX1] = int32_t(off_aux1);
  m[H_GRID] = grid;
  m[H_TOTAL] = int32_t(off);
  m[H_VARIANT] = variant;
  std::copy(worker_ptr.begin(), worker_ptr.end(), m.begin() + off_workers);
  for (size_t i = 0; i < chunks.size(); ++i) {
    m[off_chunks + 4 * i + 0] = chunks[i].unit;
    m[off_chunks + 4 * i + 1] = chunks[i].a;
    m[off_chunks + 4 * i + 2] = chunks[i].b;
    m[off_chunks + 4 * i + 3] = chunks[i].c;
  }
  std::copy(merges.begin(), merges.end(), m.begin() + off_merges);
  if (n_aux0) std::memcpy(m.data() + off_aux0, aux0, n_aux0 * sizeof(int32_t));
  if (n_aux1) std::memcpy(m.data() + off_aux1, aux1, n_aux1 * sizeof(int32_t));
}

// Linear split-KV partition. unit_len[u] tokens per unit, `tile` tokens per tile, at most
// `max_workers` workers. Chunks: (unit, tok_begin, tok_end, slot); slot = -1 when the
// unit is computed by a single chunk (written straight to the output), else the index
// of its partial state. Merge items: (unit, first_slot, count) for units with 0 chunks
// (zero-filled) or >= 2 chunks (merged), in unit order.
void linear_partition(const std::vector<int64_t>& unit_len, int64_t tile, int64_t max_workers,
                      std::vector<int32_t>& worker_ptr, std::vector<Chunk>& chunks,
                      int32_t& slots, std::vector<int32_t>& merges) {
  const size_t U = unit_len.size();
  std::vector<int64_t> tiles(U), tile_start(U + 1, 0);
  for (size_t u = 0; u < U; ++u) {
    tiles[u] = (unit_len[u] + tile - 1) / tile;
    tile_start[u + 1] = tile_start[u] + tiles[u];
  }
  const int64_t NT = tile_start[U];
  const int64_t P = std::min<int64_t>(max_workers, NT);
  worker_ptr.assign(size_t(P) + 1, 0);
  chunks.clear();
  std::vector<int32_t> nchunks(U, 0);
  size_t u = 0;
  for (int64_t w = 0; w < P; ++w) {
    const int64_t t0 = (w * NT) / P;
    const int64_t t1 = ((w + 1) * NT) / P;
    worker_ptr[size_t(w)] = int32_t(chunks.size());
    int64_t t = t0;
    while (t < t1) {
      while (tile_start[u + 1] <= t) ++u;  // unit holding global tile t
      const int64_t e = std::min(t1, tile_start[u + 1]);
      const int64_t lb = (t - tile_start[u]) * tile;
      const int64_t le = std::min((e - tile_start[u]) * tile, unit_len[u]);
      chunks.push_back(Chunk{int32_t(u), int32_t(lb), int32_t(le), -1});
      nchunks[u] += 1;
      t = e;
    }
  }
  worker_ptr[size_t(P)] = int32_t(chunks.size());
  slots = 0;
  std::vector<int32_t> first_slot(U, -1);
  for (Chunk& c : chunks) {
    if (nchunks[size_t(c.unit)] >= 2) {
      if (first_slot[size_t(c.unit)] < 0) first_slot[size_t(c.unit)] = slots;
      c.c = slots++;
    }
  }
  merges.clear();
  for (size_t v = 0; v < U; ++v) {
    if (nchunks[v] == 1) continue;
    merges.push_back(int32_t(v));
    merges.push_back(first_slot[v]);
    merges.push_back(nchunks[v]);
  }
}

// Slots (one per piece of a unit cut into several, in chunk order) and merge items
// (unit, first slot, pieces) of units with other than one piece.
void assign_slots(size_t U, std::vector<Chunk>& chunks, int32_t& slots,
                  std::vector<int32_t>& merges) {
  std::vector<int32_t> nchunks(U, 0), first_slot(U, -1);
  for (const Chunk& c : chunks) nchunks[size_t(c.unit)] += 1;
  slots = 0;
  for (Chunk& c : chunks) {
    if (nchunks[size_t(c.unit)] >= 2) {
      if (first_slot[size_t(c.unit)] < 0) first_slot[size_t(c.unit)] = slots;
      c.c = slots++;
    }
  }
  merges.clear();
  for (size_t v = 0; v < U; ++v) {
    if (nchunks[v] == 1) continue;
    merges.push_back(int32_t(v));
    merges.push_back(first_slot[v]);
    merges.push_back(nchunks[v]);
  }
}

// Greedy left-to-right fill of the unit tile sequence: a worker takes tiles while its cost
// stays within T. Its cost is its tiles plus: `whole` for every chunk after its first;
// `merge` once it holds two chunks and its first is the tail piece of a unit begun by an
// earlier worker (walked last: its merge lands at the worker's end); `pub` for a last chunk
// that is the head piece of a unit continued by a later worker (walked first and published
// mid-stream). Returns the number of workers; with `out`, appends their chunks (unit, first
// tile, end tile) and worker starts.
struct FillCosts {
  int64_t pub, merge, whole;
};
int64_t fill_workers(const std::vector<int64_t>& tiles, int64_t T, const FillCosts& bc,
                     std::vector<int32_t>* worker_ptr, std::vector<Chunk>* out) {
  const size_t U = tiles.size();
  size_t u = 0;
  int64_t off = 0, workers = 0;
  while (u < U && tiles[u] == 0) ++u;
  while (u < U) {
    ++workers;
    if (worker_ptr) worker_ptr->push_back(int32_t(out->size()));
    int64_t cost = 0, n = 0;
    const bool first_tail = off > 0;
    while (u < U) {
      if (tiles[u] == 0) { ++u; continue; }
      const int64_t add = n == 0 ? 0 : bc.whole + (n == 1 && first_tail ? bc.merge : 0);
      const int64_t rem = tiles[u] - off;
      if (cost + add + rem <= T) {
        if (out) out->push_back(Chunk{int32_t(u), int32_t(off), int32_t(tiles[u]), -1});
        cost += add + rem;
        ++n;
        ++u;
        off = 0;
        continue;
      }
      const int64_t take = T - cost - add - (n > 0 ? bc.pub : 0);
      if (take > 0) {
        if (out) out->push_back(Chunk{int32_t(u), int32_t(off), int32_t(off + take), -1});
        off += take;
        ++n;
      }
      break;
    }
  }
  return workers;
}

// Contiguous partition with the worker costs of fill_workers: the smallest bound T whose
// greedy fill needs at most max_workers workers, each filled up to T. Chunks are in tokens
// like linear_partition's.
void linear_partition_cost(const std::vector<int64_t>& unit_len, int64_t tile,
                           int64_t max_workers, const FillCosts& bc, std::vector<int32_t>& worker_ptr,
                           std::vector<Chunk>& chunks, int32_t& slots,
                           std::vector<int32_t>& merges) {
  std::vector<int64_t> tiles(unit_len.size());
  int64_t NT = 0;
  for (size_t u = 0; u < unit_len.size(); ++u) {
    tiles[u] = (unit_len[u] + tile - 1) / tile;
    NT += tiles[u];
  }
  if (NT == 0) {
    linear_partition(unit_len, tile, max_workers, worker_ptr, chunks, slots, merges);
    return;
  }
  int64_t lo = std::max<int64_t>(1, (NT + max_workers - 1) / max_workers);
  int64_t hi = NT + (bc.pub + bc.merge + bc.whole) * (int64_t(tiles.size()) + 1);
  while (lo < hi) {
    const int64_t mid = (lo + hi) / 2;
    if (fill_workers(tiles, mid, bc, nullptr, nullptr) <= max_workers) hi = mid;
    else lo = mid + 1;
  }
  worker_ptr.clear();
  chunks.clear();
  fill_workers(tiles, lo, bc, &worker_ptr, &chunks);
  worker_ptr.push_back(int32_t(chunks.size()));
  for (Chunk& c : chunks) {
    const int64_t L = unit_len[size_t(c.unit)];
    c.a = int32_t(int64_t(c.a) * tile);
    c.b = int32_t(std::min(int64_t(c.b) * tile, L));
  }
  assign_slots(unit_len.size(), chunks, slots, merges);
}

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

std::vector<std::vector<int32_t>> lpt_assign(const std::vector<int64_t>& cost, int32_t G);

// MLA partition: units (query tokens or requests) of unit_len rows in tiles of `tile`, on at
// most max_workers cluster workers. Whole units by longest processing time (units of more
// tiles first; no slots; units without rows become zero-fill merge items) when the busiest
// worker's tiles stay within kMlaSplitPenaltyTiles of the linear split partition's; else the
// linear split partition.
void mla_partition(const std::vector<int64_t>& unit_len, int64_t tile, int64_t max_workers,
                   std::vector<int32_t>& worker_ptr, std::vector<Chunk>& chunks,
                   int32_t& slots, std::vector<int32_t>& merges) {
  std::vector<int64_t> tiles(unit_len.size());
  std::vector<int32_t> live;
  int64_t NT = 0;
  for (size_t u = 0; u < unit_len.size(); ++u) {
    tiles[u] = (unit_len[u] + tile - 1) / tile;
    NT += tiles[u];
    if (tiles[u] > 0) live.push_back(int32_t(u));
  }
  linear_partition(unit_len, tile, max_workers, worker_ptr, chunks, slots, merges);
  if (NT == 0) return;
  const int64_t P = std::min<int64_t>(max_workers, NT);
  const int64_t split_max = (NT + P - 1) / P;
  const int32_t G = int32_t(std::min<int64_t>(max_workers, int64_t(live.size())));
  std::vector<int64_t> cost(live.size());
  for (size_t i = 0; i < live.size(); ++i) cost[i] = tiles[size_t(live[i])];
  const std::vector<std::vector<int32_t>> lists = lpt_assign(cost, G);
  int64_t whole_max = 0;
  for (const auto& l : lists) {
    int64_t load = 0;
    for (int32_t i : l) load += cost[size_t(i)];
    whole_max = std::max(whole_max, load);
  }
  if (whole_max > split_max + kMlaSplitPenaltyTiles) return;
  worker_ptr.assign(size_t(G) + 1, 0);
  chunks.clear();
  for (int32_t w = 0; w < G; ++w) {
    worker_ptr[size_t(w)] = int32_t(chunks.size());
    for (int32_t i : lists[size_t(w)]) {
      const int32_t u = live[size_t(i)];
      chunks.push_back(Chunk{u, 0, int32_t(unit_len[size_t(u)]), -1});
    }
  }
  worker_ptr[size_t(G)] = int32_t(chunks.size());
  slots = 0;
  merges.clear();
  for (size_t u = 0; u < unit_len.size(); ++u)
    if (tiles[u] == 0) merges.insert(merges.end(), {int32_t(u), -1, 0});
}

// Longest-processing-time assignment of units with costs `cost` to G workers: units taken by
// cost, largest first (stable), each given to the worker of least load so far (ties: the
// lowest worker index). Returns every worker's units in assignment order.
std::vector<std::vector<int32_t>> lpt_assign(const std::vector<int64_t>& cost, int32_t G) {
  std::vector<int32_t> order(cost.size());
  for (size_t u = 0; u < cost.size(); ++u) order[u] = int32_t(u);
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t a, int32_t b) { return cost[size_t(a)] > cost[size_t(b)]; });
  using Item = std::pair<int64_t, int32_t>;  // (load, worker), smallest first
  std::priority_queue<Item, std::vector<Item>, std::greater<Item>> heap;
  for (int32_t c = 0; c < G; ++c) heap.push(Item(0, c));
  std::vector<std::vector<int32_t>> lists(static_cast<size_t>(G));
  for (int32_t u : order) {
    Item it = heap.top();
    heap.pop();
    lists[size_t(it.second)].push_back(u);
    it.first += cost[size_t(u)];
    heap.push(it);
  }
  return lists;
}

// Worker pointers and chunks of an assignment whose unit u is chunk units[u].
void lists_to_chunks(const std::vector<std::vector<int32_t>>& lists,
                     const std::vector<Chunk>& units, std::vector<int32_t>& worker_ptr,
                     std::vector<Chunk>& chunks) {
  worker_ptr.assign(lists.size() + 1, 0);
  chunks.clear();
  chunks.reserve(units.size());
  for (size_t c = 0; c < lists.size(); ++c) {
    worker_ptr[c] = int32_t(chunks.size());
    for (int32_t u : lists[c]) chunks.push_back(units[size_t(u)]);
  }
  worker_ptr[lists.size()] = int32_t(chunks.size());
}

// Tensor-core list plans: unit descriptors and chunks from per-unit step ranges. A unit is a
// 64-token row tile {first token, valid tokens, first step, end step, key limit}, served for
// one kv head; cost in quarter steps of the tensor-core kernel: 2 for its start and
// epilogue, 4 per step of more than 64 keys, 3 per step of at most 64 (1 without steps).
// Units are placed by the longest-processing-time rule on at most num_sms CTAs.
struct TcListPlan {
  std::vector<int32_t> desc;   // kBsrTcUnitWords per descriptor
  std::vector<Chunk> units;    // (descriptor, 0, kv head, 0)
  std::vector<int64_t> cost;
};

int64_t tc_unit_cost(const std::vector<int32_t>& steps, int32_t words, int32_t tb, int32_t te) {
  if (te == tb) return 1;
  int64_t c = 2;
  for (int32_t t = tb; t < te; ++t) {
    const int32_t n = steps[size_t(t) * words + 1] - steps[size_t(t) * words];
    c += n > 64 ? 4 : 3;
  }
  return c;
}

// Unit descriptors of the 64-token row tiles of [tok0, tok0 + ntok), whose keys are the steps
// [tb, te) (in key order); with causal, a tile keeps the steps that start at or before the
// last key its last token sees (limit0 + valid - 1). One unit per tile and kv head.
void tc_list_units(TcListPlan& pl, const std::vector<int32_t>& steps, int32_t words,
                   int32_t tok0, int32_t ntok, int32_t tb, int32_t te, int32_t limit_first,
                   bool causal, const std::vector<int32_t>& heads) {
  for (int32_t r0 = 0; r0 < ntok; r0 += 64) {
    const int32_t valid = std::min(64, ntok - r0);
    const int32_t lim = limit_first + r0;
    int32_t end = te;
    if (causal) {
      end = tb;
      while (end < te && int64_t(steps[size_t(end) * words]) <= int64_t(lim) + valid - 1) ++end;
    }
    const int32_t d = int32_t(pl.desc.size() / kBsrTcUnitWords);
    pl.desc.insert(pl.desc.end(), {tok0 + r0, valid, tb, end, lim});
    const int64_t c = tc_unit_cost(steps, words, tb, end);
    for (int32_t h : heads) {
      pl.units.push_back(Chunk{d, 0, h, 0});
      pl.cost.push_back(c);
    }
  }
}

// Assemble a tensor-core list plan (variant BSR_VARIABLE_TC or BSR_PAGED_PREFILL_TC).
void tc_list_assemble(bskv_plan* p, const TcListPlan& pl, const std::vector<int32_t>& steps,
                      int32_t num_sms, int32_t variant) {
  const int64_t U = int64_t(pl.units.size());
  const int32_t G = int32_t(std::min<int64_t>(num_sms, std::max<int64_t>(U, 1)));
  std::vector<int32_t> worker_ptr, no_merges;
  std::vector<Chunk> chunks;
  lists_to_chunks(lpt_assign(pl.cost, G), pl.units, worker_ptr, chunks);
  assemble(p, KIND_BSR, int32_t(U), worker_ptr, chunks, 0, no_merges, 64, pl.desc.data(),
           pl.desc.size(), steps.data(), steps.size(), U > 0 ? G : 0, variant);
}

// One line per plan on stderr when BSKV_LOGLEVEL >= 1 (plus the spread of work items over
// the workers at level 2), taken from the metadata the kernels will read.
void log_plan(const char* name, const bskv_plan* p) {
  const int lvl = log_level();
  if (lvl < 1) return;
  const std::vector<int32_t>& m = p->meta;
  const char* kernel = "?";
  switch (m[H_KIND]) {
    case KIND_DECODE:
      kernel = m[H_VARIANT] == DECODE_GROUP ? "decode_group_kernel (page-major CTAs)"
                                            : "decode_kernel (one worker per warp)";
      break;
    case KIND_BSR:
      kernel = m[H_VARIANT] == BSR_TCGEN05 ? "bsr_tc_kernel (tcgen05)"
               : m[H_VARIANT] == BSR_VARIABLE_TC ? "bsr_tc_kernel (tcgen05, variable blocks)"
               : m[H_VARIANT] == BSR_PAGED_PREFILL_TC ? "bsr_tc_kernel (tcgen05, paged prefill)"
               : m[H_VARIANT] == BSR_VARIABLE ? "bsr_generic_kernel (variable blocks)"
               : m[H_VARIANT] == BSR_PAGED_PREFILL ? "bsr_generic_kernel (paged prefill)"
                                                   : "bsr_generic_kernel";
      break;
    case KIND_MLA:
      kernel = p->mla_variant == MLA_PAGED ? "mla_kernel (rows from the page table)"
                                           : "mla_kernel (sparse rows)";
      break;
    default:
      break;
  }
  const size_t int_ws = merge_counter_offset(m.size()) + p->counter_words * 4;
  std::fprintf(stderr,
               "[bskv] %s: kernel %s; units %d, workers %d, work items %d, split pieces %d, "
               "merged units %d, grid %d CTAs; int workspace %zu B, float workspace %zu B\n",
               name, kernel, m[H_UNITS], m[H_WORKERS], m[H_CHUNKS], m[H_SLOTS], m[H_MERGES],
               m[H_GRID], int_ws, p->float_ws_bytes);
  if (lvl >= 2 && m[H_WORKERS] > 0) {
    const int32_t* wp = m.data() + m[H_OFF_WORKERS];
    int32_t lo = wp[1] - wp[0], hi = lo;
    for (int32_t w = 1; w < m[H_WORKERS]; ++w) {
      lo = std::min(lo, wp[w + 1] - wp[w]);
      hi = std::max(hi, wp[w + 1] - wp[w]);
    }
    std::fprintf(stderr, "[bskv] %s: work items per worker min %d, mean %.2f, max %d\n", name, lo,
                 double(m[H_CHUNKS]) / m[H_WORKERS], hi);
  }
}

}  // namespace

int log_level() {
  const char* e = std::getenv("BSKV_LOGLEVEL");
  return e ? std::atoi(e) : 0;
}

}  // namespace bskv

using namespace bskv;

extern "C" bskv_status bskv_plan_decode(const int32_t* kv_indptr, const int32_t* kv_indices,
                                        const int32_t* kv_last_page_len, int32_t batch,
                                        int32_t num_pages, int32_t page_size,
                                        int32_t num_qo_heads, int32_t num_kv_heads,
                                        int32_t head_dim, int32_t dtype, int32_t num_sms,
                                        int32_t max_workers, bskv_plan** out_plan) {
  if (!out_plan) { set_error("plan_decode: out_plan is NULL"); return BSKV_ERR_INVALID_ARG; }
  *out_plan = nullptr;
  if (batch < 0 || num_pages < 0 || page_size < 1 || num_sms < 1 || max_workers < 0) {
    set_error("plan_decode: batch=%d num_pages=%d page_size=%d num_sms=%d max_workers=%d",
              batch, num_pages, page_size, num_sms, max_workers);
    return BSKV_ERR_INVALID_ARG;
  }
  if (num_qo_heads < 1 || num_kv_heads < 1 || num_qo_heads % num_kv_heads != 0) {
    set_error("plan_decode: num_qo_heads (%d) must be a positive multiple of num_kv_heads (%d)",
              num_qo_heads, num_kv_heads);
    return BSKV_ERR_INVALID_ARG;
  }
  if (batch > 0 && (!kv_indptr || !kv_last_page_len)) {
    set_error("plan_decode: NULL index array"); return BSKV_ERR_INVALID_ARG;
  }
  const int32_t group = num_qo_heads / num_kv_heads;
  if (group > 16) { set_error("plan_decode: %d query heads per kv head (max 16)", group); return BSKV_ERR_UNSUPPORTED; }
  if (head_dim != 64 && head_dim != 128) { set_error("plan_decode: head_dim %d not in {64,128}", head_dim); return BSKV_ERR_UNSUPPORTED; }
  if (dtype != BSKV_BF16 && dtype != BSKV_FP16) { set_error("plan_decode: dtype %s unsupported", dtype_name(dtype)); return BSKV_ERR_UNSUPPORTED; }
  if (batch > 0 && kv_indptr[0] != 0) { set_error("plan_decode: kv_indptr[0] must be 0"); return BSKV_ERR_INVALID_ARG; }
  const int32_t G = decode_group_heads(num_kv_heads, page_size);
  const int32_t variant = G > 0 ? DECODE_GROUP : DECODE_WARP;
  const int32_t upb = variant == DECODE_GROUP ? num_kv_heads / G : num_kv_heads;  // units per request
  std::vector<int64_t> len(size_t(batch) * size_t(upb));
  int64_t total_tokens = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const int64_t n = int64_t(kv_indptr[b + 1]) - kv_indptr[b];
    if (n < 0) { set_error("plan_decode: kv_indptr decreases at %d", b); return BSKV_ERR_INVALID_ARG; }
    int64_t L = 0;
    if (n > 0) {
      const int32_t lp = kv_last_page_len[b];
      if (lp < 1 || lp > page_size) {
        set_error("plan_decode: kv_last_page_len[%d] = %d outside [1, %d]", b, lp, page_size);
        return BSKV_ERR_INVALID_ARG;
      }
      L = (n - 1) * page_size + lp;
    }
    total_tokens += L;
    for (int32_t h = 0; h < upb; ++h) len[size_t(b) * upb + h] = L;
  }
  const int64_t nnz = batch > 0 ? kv_indptr[batch] : 0;
  if (nnz > 0 && !kv_indices) { set_error("plan_decode: kv_indices is NULL"); return BSKV_ERR_INVALID_ARG; }
  for (int64_t i = 0; i < nnz; ++i) {
    if (kv_indices[i] < 0 || kv_indices[i] >= num_pages) {
      set_error("plan_decode: kv_indices[%lld] = %d outside [0, %d)", (long long)i, kv_indices[i], num_pages);
      return BSKV_ERR_INVALID_ARG;
    }
  }
  if (total_tokens * num_kv_heads > INT32_MAX / 2) { set_error("plan_decode: too many tokens"); return BSKV_ERR_UNSUPPORTED; }
  const int64_t workers_cap = max_workers > 0 ? max_workers
                              : variant == DECODE_GROUP ? int64_t(num_sms)
                                                        : int64_t(num_sms) * kDecodeWarps;
  std::vector<int32_t> worker_ptr, merges;
  std::vector<Chunk> chunks;
  int32_t slots = 0;
  if (variant == DECODE_GROUP)
    linear_partition_cost(len, kDecodeTile, workers_cap,
                          FillCosts{kDecodePublishTiles, kDecodeMergeTiles, kDecodeBoundaryTiles},
                          worker_ptr, chunks, slots, merges);
  else
    linear_partition(len, kDecodeTile, workers_cap, worker_ptr, chunks, slots, merges);
  const int32_t P = int32_t(worker_ptr.size() - 1);
  const int32_t grid = variant == DECODE_GROUP ? P : (P + kDecodeWarps - 1) / kDecodeWarps;
  const int32_t slot_rows = num_qo_heads / upb;  // query heads of one unit
  bskv_plan* p = new bskv_plan();
  p->kind = KIND_DECODE;
  p->batch = batch; p->num_pages = num_pages; p->page_size = page_size;
  p->num_qo_heads = num_qo_heads; p->num_kv_heads = num_kv_heads; p->head_dim = head_dim;
  p->dtype = dtype;
  assemble(p, KIND_DECODE, int32_t(len.size()), worker_ptr, chunks, slots, merges, kDecodeTile,
           kv_indptr, batch > 0 ? size_t(batch) + 1 : 0, kv_indices, size_t(nnz), grid, variant);
  if (variant == DECODE_GROUP) {
    // start records: the first chunk of each worker's walk (its last chunk when it has
    // several, the order in which the kernel walks them) and the first page ids it reads
    std::vector<int32_t>& m = p->meta;
    p->decode_starts = int32_t(m.size());
    for (int32_t w = 0; w < P; ++w) {
      int32_t rec[kDecodeStartWords] = {};
      const int32_t w0 = worker_ptr[size_t(w)], w1 = worker_ptr[size_t(w) + 1];
      if (w1 > w0) {
        const Chunk& c = chunks[size_t(w1 - w0 >= 2 ? w1 - 1 : w0)];
        const int32_t b = c.unit / upb;
        const int32_t pbase = kv_indptr[b], npages = kv_indptr[b + 1] - pbase;
        const int32_t first = c.a / page_size;
        const int32_t n = std::min(kDecodeStartPages, npages - first);
        rec[0] = c.unit; rec[1] = c.a; rec[2] = c.b; rec[3] = c.c;
        rec[4] = pbase; rec[5] = npages; rec[6] = n;
        for (int32_t i = 0; i < n; ++i) rec[8 + i] = kv_indices[pbase + first + i];
      }
      m.insert(m.end(), rec, rec + kDecodeStartWords);
    }
    m[H_TOTAL] = int32_t(m.size());
  }
  p->float_ws_bytes = slots == 0 ? 0
      : align256(size_t(slots) * slot_rows * head_dim * 4) + align256(size_t(slots) * slot_rows * 4);
  p->counter_words = merges.size() / 3 * size_t(num_kv_heads / upb);
  for (size_t i = 2; i < merges.size(); i += 3) p->max_merge_count = std::max(p->max_merge_count, merges[i]);
  *out_plan = p;
  log_plan("bskv_plan_decode", p);
  return BSKV_OK;
}

namespace {

// BSR plan; `masked`: a per-block token mask comes with every run (no causal flag then).
bskv_status plan_bsr(const int32_t* indptr, const int32_t* indices, int32_t M, int32_t N,
                     int32_t R, int32_t C, int32_t num_qo_heads, int32_t num_kv_heads,
                     int32_t head_dim, int32_t causal, int32_t dtype, int32_t num_sms,
                     bool masked, bskv_plan** out_plan) {
  if (!out_plan) { set_error("plan_bsr: out_plan is NULL"); return BSKV_ERR_INVALID_ARG; }
  *out_plan = nullptr;
  if (M < 0 || N < 0 || R < 1 || C < 1 || num_sms < 1) {
    set_error("plan_bsr: M=%d N=%d R=%d C=%d num_sms=%d", M, N, R, C, num_sms);
    return BSKV_ERR_INVALID_ARG;
  }
  if (N % C != 0) { set_error("plan_bsr: N (%d) must be divisible by C (%d)", N, C); return BSKV_ERR_INVALID_ARG; }
  if (num_qo_heads < 1 || num_kv_heads < 1 || num_qo_heads % num_kv_heads != 0) {
    set_error("plan_bsr: num_qo_heads (%d) must be a positive multiple of num_kv_heads (%d)",
              num_qo_heads, num_kv_heads);
    return BSKV_ERR_INVALID_ARG;
  }
  if (head_dim != 64 && head_dim != 128) { set_error("plan_bsr: head_dim %d not in {64,128}", head_dim); return BSKV_ERR_UNSUPPORTED; }
  if (dtype != BSKV_BF16 && dtype != BSKV_FP16) { set_error("plan_bsr: dtype %s unsupported", dtype_name(dtype)); return BSKV_ERR_UNSUPPORTED; }
  const int32_t MB = (M + R - 1) / R, NB = N / C;
  if (!indptr) { set_error("plan_bsr: indptr is NULL"); return BSKV_ERR_INVALID_ARG; }
  if (indptr[0] != 0) { set_error("plan_bsr: indptr[0] must be 0"); return BSKV_ERR_INVALID_ARG; }
  for (int32_t i = 0; i < MB; ++i) {
    if (indptr[i + 1] < indptr[i]) { set_error("plan_bsr: indptr decreases at %d", i); return BSKV_ERR_INVALID_ARG; }
  }
  const int32_t nnz = indptr[MB];
  if (nnz > 0 && !indices) { set_error("plan_bsr: indices is NULL"); return BSKV_ERR_INVALID_ARG; }
  std::vector<int32_t> seen(size_t(NB), -1);
  for (int32_t i = 0; i < MB; ++i) {
    for (int32_t e = indptr[i]; e < indptr[i + 1]; ++e) {
      const int32_t j = indices[e];
      if (j < 0 || j >= NB) { set_error("plan_bsr: indices[%d] = %d outside [0, %d)", e, j, NB); return BSKV_ERR_INVALID_ARG; }
      if (seen[size_t(j)] == i) { set_error("plan_bsr: column block %d listed twice in row block %d", j, i); return BSKV_ERR_INVALID_ARG; }
      seen[size_t(j)] = i;
    }
  }
  const int32_t group = num_qo_heads / num_kv_heads;
  const bool tc = (R == 64 && C == 64 && head_dim == 128 && (R * group == 128 || R * group == 256));
  const int32_t rows_per_unit = tc ? R * group : kBsrGenericRows;
  const int32_t row_tiles = (R * group + rows_per_unit - 1) / rows_per_unit;
  const int64_t U = int64_t(MB) * num_kv_heads * row_tiles;
  if (U > INT32_MAX / 4) { set_error("plan_bsr: too many units"); return BSKV_ERR_UNSUPPORTED; }
  // Longest-processing-time assignment. Cost of a tensor-core unit with n blocks, in
  // quarters of a step of its kernel: 4 per pair of blocks, 3 for a last single block (its
  // QK takes as long as a pair's), 2 for the unit's start and epilogue (1 with no blocks);
  // of a general unit: 1 + n.
  std::vector<int64_t> cost(static_cast<size_t>(U));
  std::vector<Chunk> units(static_cast<size_t>(U));
  for (int64_t u = 0; u < U; ++u) {
    const int32_t i = int32_t(u / (int64_t(num_kv_heads) * row_tiles));
    const int64_t n = indptr[i + 1] - indptr[i];
    cost[size_t(u)] = tc ? (n > 0 ? 2 + 4 * (n / 2) + 3 * (n % 2) : 1) : 1 + n;
    units[size_t(u)] = Chunk{int32_t(u), i, int32_t((u / row_tiles) % num_kv_heads),
                             int32_t(u % row_tiles)};
  }
  const int64_t cap = tc ? num_sms : int64_t(num_sms) * kBsrGenericCtasPerSm;
  const int32_t G = int32_t(std::min<int64_t>(cap, U));
  std::vector<int32_t> worker_ptr;
  std::vector<Chunk> chunks;
  lists_to_chunks(lpt_assign(cost, G), units, worker_ptr, chunks);
  bskv_plan* p = new bskv_plan();
  p->kind = KIND_BSR;
  p->M = M; p->N = N; p->R = R; p->C = C; p->causal = causal ? 1 : 0;
  p->num_qo_heads = num_qo_heads; p->num_kv_heads = num_kv_heads; p->head_dim = head_dim;
  p->dtype = dtype;
  std::vector<int32_t> no_merges;
  assemble(p, KIND_BSR, int32_t(U), worker_ptr, chunks, 0, no_merges, rows_per_unit, indptr,
           size_t(MB) + 1, indices, size_t(nnz), G, tc ? BSR_TCGEN05 : BSR_GENERIC);
  p->float_ws_bytes = 0;
  p->masked = masked ? 1 : 0;
  *out_plan = p;
  log_plan(masked ? "bskv_plan_bsr_masked" : "bskv_plan_bsr", p);
  return BSKV_OK;
}

}  // namespace

extern "C" bskv_status bskv_plan_bsr(const int32_t* indptr, const int32_t* indices, int32_t M,
                                     int32_t N, int32_t R, int32_t C, int32_t num_qo_heads,
                                     int32_t num_kv_heads, int32_t head_dim, int32_t causal,
                                     int32_t dtype, int32_t num_sms, bskv_plan** out_plan) {
  return plan_bsr(indptr, indices, M, N, R, C, num_qo_heads, num_kv_heads, head_dim, causal,
                  dtype, num_sms, false, out_plan);
}

extern "C" bskv_status bskv_plan_bsr_variable(const uint8_t* block_mask_map,
                                              const int32_t* block_row_sz,
                                              const int32_t* block_col_sz, int32_t MB, int32_t NB,
                                              int32_t num_qo_heads, int32_t num_kv_heads,
                                              int32_t head_dim, int32_t causal, int32_t dtype,
                                              int32_t num_sms, bskv_plan** out_plan) {
  if (!out_plan) { set_error("plan_bsr_variable: out_plan is NULL"); return BSKV_ERR_INVALID_ARG; }
  *out_plan = nullptr;
  if (MB < 1 || NB < 1 || num_sms < 1 || !block_mask_map || !block_row_sz || !block_col_sz) {
    set_error("plan_bsr_variable: MB=%d NB=%d num_sms=%d or a NULL array", MB, NB, num_sms);
    return BSKV_ERR_INVALID_ARG;
  }
  if (num_qo_heads < 1 || num_kv_heads < 1 || num_qo_heads % num_kv_heads != 0) {
    set_error("plan_bsr_variable: num_qo_heads (%d) must be a positive multiple of num_kv_heads (%d)",
              num_qo_heads, num_kv_heads);
    return BSKV_ERR_INVALID_ARG;
  }
  if (head_dim != 64 && head_dim != 128) { set_error("plan_bsr_variable: head_dim %d not in {64,128}", head_dim); return BSKV_ERR_UNSUPPORTED; }
  if (dtype != BSKV_BF16 && dtype != BSKV_FP16) { set_error("plan_bsr_variable: dtype %s unsupported", dtype_name(dtype)); return BSKV_ERR_UNSUPPORTED; }
  const int32_t H = num_kv_heads, g = num_qo_heads / num_kv_heads;
  int64_t qo_len = -1, kv_len = -1;
  for (int32_t h = 0; h < H; ++h) {
    int64_t sr = 0, sc = 0;
    for (int32_t a = 0; a < MB; ++a) {
      const int32_t r = block_row_sz[int64_t(h) * MB + a];
      if (r < 1) { set_error("plan_bsr_variable: block_row_sz[%d][%d] = %d must be positive", h, a, r); return BSKV_ERR_INVALID_ARG; }
      sr += r;
    }
    for (int32_t c = 0; c < NB; ++c) {
      const int32_t w = block_col_sz[int64_t(h) * NB + c];
      if (w < 1) { set_error("plan_bsr_variable: block_col_sz[%d][%d] = %d must be positive", h, c, w); return BSKV_ERR_INVALID_ARG; }
      sc += w;
    }
    if ((qo_len >= 0 && sr != qo_len) || (kv_len >= 0 && sc != kv_len)) {
      set_error("plan_bsr_variable: kv head %d covers %lld query / %lld key tokens, head 0 %lld / %lld",
                h, (long long)sr, (long long)sc, (long long)qo_len, (long long)kv_len);
      return BSKV_ERR_INVALID_ARG;
    }
    qo_len = sr;
    kv_len = sc;
  }
  if (qo_len > INT32_MAX / 2 || kv_len > INT32_MAX / 2 || qo_len * g > INT32_MAX / 2) { set_error("plan_bsr_variable: sequence too long"); return BSKV_ERR_UNSUPPORTED; }
  if (bsr_tc_list_shape(head_dim, num_qo_heads, num_kv_heads)) {
    // Tensor-core kernel: per (kv head h, row block a) the runs of visible column blocks cut
    // into steps of at most 128 keys; units are the row block's 64-token tiles.
    std::vector<int32_t> steps;
    TcListPlan pl;
    const int32_t shift = int32_t(kv_len - qo_len);
    for (int32_t h = 0; h < H; ++h) {
      std::vector<int32_t> cs(static_cast<size_t>(NB));
      int32_t acc = 0;
      for (int32_t c = 0; c < NB; ++c) { cs[size_t(c)] = acc; acc += block_col_sz[int64_t(h) * NB + c]; }
      int32_t row = 0;
      for (int32_t a = 0; a < MB; ++a) {
        const uint8_t* mrow = block_mask_map + (int64_t(h) * MB + a) * NB;
        const int32_t tb = int32_t(steps.size() / 2);
        for (int32_t c = 0; c < NB;) {
          if (!mrow[c]) { ++c; continue; }
          const int32_t s0 = cs[size_t(c)];
          int32_t e = s0;
          while (c < NB && mrow[c]) { e += block_col_sz[int64_t(h) * NB + c]; ++c; }
          for (int32_t t = s0; t < e; t += kBsrTcStep) {
            steps.push_back(t);
            steps.push_back(std::min(t + kBsrTcStep, e));
          }
          if (steps.size() > size_t(INT32_MAX) / 2) { set_error("plan_bsr_variable: too many key steps"); return BSKV_ERR_UNSUPPORTED; }
        }
        const int32_t nrow = block_row_sz[int64_t(h) * MB + a];
        tc_list_units(pl, steps, 2, row, nrow, tb, int32_t(steps.size() / 2), row + shift,
                      causal != 0, {h});
        row += nrow;
      }
    }
    bskv_plan* p = new bskv_plan();
    p->kind = KIND_BSR;
    p->M = int32_t(qo_len); p->N = int32_t(kv_len); p->R = 0; p->C = 0; p->causal = causal ? 1 : 0;
    p->num_qo_heads = num_qo_heads; p->num_kv_heads = num_kv_heads; p->head_dim = head_dim;
    p->dtype = dtype;
    tc_list_assemble(p, pl, steps, num_sms, BSR_VARIABLE_TC);
    p->float_ws_bytes = 0;
    *out_plan = p;
    log_plan("bskv_plan_bsr_variable", p);
    return BSKV_OK;
  }
  // Per (kv head h, row block a): its query rows and the 16-token tiles of the key ranges it
  // sees (adjacent selected column blocks merged into one range).
  std::vector<int32_t> desc(size_t(H) * MB * 4), tiles;
  std::vector<int32_t> cstart(static_cast<size_t>(NB));
  for (int32_t h = 0; h < H; ++h) {
    int32_t acc = 0;
    for (int32_t c = 0; c < NB; ++c) { cstart[size_t(c)] = acc; acc += block_col_sz[int64_t(h) * NB + c]; }
    int32_t row = 0;
    for (int32_t a = 0; a < MB; ++a) {
      const uint8_t* mrow = block_mask_map + (int64_t(h) * MB + a) * NB;
      const size_t d = (size_t(h) * MB + a) * 4;
      desc[d] = row;
      desc[d + 1] = block_row_sz[int64_t(h) * MB + a];
      desc[d + 2] = int32_t(tiles.size() / 2);
      for (int32_t c = 0; c < NB;) {
        if (!mrow[c]) { ++c; continue; }
        const int32_t s0 = cstart[size_t(c)];
        int32_t e = s0;
        while (c < NB && mrow[c]) { e += block_col_sz[int64_t(h) * NB + c]; ++c; }
        for (int32_t t = s0; t < e; t += kBsrVarTile) { tiles.push_back(t); tiles.push_back(e); }
        if (tiles.size() > size_t(INT32_MAX) / 2) { set_error("plan_bsr_variable: too many key tiles"); return BSKV_ERR_UNSUPPORTED; }
      }
      desc[d + 3] = int32_t(tiles.size() / 2);
      row += desc[d + 1];
    }
  }
  // Units (h, a, row tile of 64 grouped rows), h-major; longest processing time first on at
  // most 4 CTAs per SM, cost 1 + tiles.
  std::vector<Chunk> units;
  std::vector<int64_t> cost;
  for (int32_t h = 0; h < H; ++h)
    for (int32_t a = 0; a < MB; ++a) {
      const size_t d = (size_t(h) * MB + a) * 4;
      const int32_t rts = (desc[d + 1] * g + kBsrGenericRows - 1) / kBsrGenericRows;
      for (int32_t rt = 0; rt < rts; ++rt) {
        units.push_back(Chunk{h * MB + a, a, h, rt});
        cost.push_back(1 + desc[d + 3] - desc[d + 2]);
      }
    }
  const int64_t U = int64_t(units.size());
  const int32_t G = int32_t(std::min<int64_t>(int64_t(num_sms) * kBsrGenericCtasPerSm, std::max<int64_t>(U, 1)));
  std::vector<int32_t> worker_ptr;
  std::vector<Chunk> chunks;
  lists_to_chunks(lpt_assign(cost, G), units, worker_ptr, chunks);
  bskv_plan* p = new bskv_plan();
  p->kind = KIND_BSR;
  p->M = int32_t(qo_len); p->N = int32_t(kv_len); p->R = 0; p->C = 0; p->causal = causal ? 1 : 0;
  p->num_qo_heads = num_qo_heads; p->num_kv_heads = num_kv_heads; p->head_dim = head_dim;
  p->dtype = dtype;
  std::vector<int32_t> no_merges;
  assemble(p, KIND_BSR, int32_t(U), worker_ptr, chunks, 0, no_merges, kBsrGenericRows,
           desc.data(), desc.size(), tiles.data(), tiles.size(), U > 0 ? G : 0, BSR_VARIABLE);
  p->float_ws_bytes = 0;
  *out_plan = p;
  log_plan("bskv_plan_bsr_variable", p);
  return BSKV_OK;
}

extern "C" bskv_status bskv_plan_prefill_paged(const int32_t* qo_indptr, const int32_t* kv_indptr,
                                               const int32_t* kv_indices,
                                               const int32_t* kv_last_page_len, int32_t batch,
                                               int32_t num_pages, int32_t page_size,
                                               int32_t num_qo_heads, int32_t num_kv_heads,
                                               int32_t head_dim, int32_t causal, int32_t dtype,
                                               int32_t num_sms, bskv_plan** out_plan) {
  if (!out_plan) { set_error("plan_prefill_paged: out_plan is NULL"); return BSKV_ERR_INVALID_ARG; }
  *out_plan = nullptr;
  if (batch < 0 || num_pages < 1 || page_size < 1 || num_sms < 1) {
    set_error("plan_prefill_paged: batch=%d num_pages=%d page_size=%d num_sms=%d", batch,
              num_pages, page_size, num_sms);
    return BSKV_ERR_INVALID_ARG;
  }
  if (num_qo_heads < 1 || num_kv_heads < 1 || num_qo_heads % num_kv_heads != 0) {
    set_error("plan_prefill_paged: num_qo_heads (%d) must be a positive multiple of num_kv_heads (%d)",
              num_qo_heads, num_kv_heads);
    return BSKV_ERR_INVALID_ARG;
  }
  if (head_dim != 64 && head_dim != 128) { set_error("plan_prefill_paged: head_dim %d not in {64,128}", head_dim); return BSKV_ERR_UNSUPPORTED; }
  if (dtype != BSKV_BF16 && dtype != BSKV_FP16) { set_error("plan_prefill_paged: dtype %s unsupported", dtype_name(dtype)); return BSKV_ERR_UNSUPPORTED; }
  if (batch > 0 && (!qo_indptr || !kv_indptr || !kv_last_page_len)) { set_error("plan_prefill_paged: NULL index array"); return BSKV_ERR_INVALID_ARG; }
  if (batch > 0 && (qo_indptr[0] != 0 || kv_indptr[0] != 0)) { set_error("plan_prefill_paged: qo_indptr[0] and kv_indptr[0] must be 0"); return BSKV_ERR_INVALID_ARG; }
  const int32_t g = num_qo_heads / num_kv_heads;
  if (bsr_tc_list_shape(head_dim, num_qo_heads, num_kv_heads) && bsr_tc_page_size(page_size)) {
    // Tensor-core kernel: per request its keys in steps of 128 (whole pages, the step's page
    // ids listed after its key range); units are 64-token tiles of its queries, for every
    // kv head.
    const int32_t ppk = kBsrTcStep / page_size, words = 2 + ppk;
    std::vector<int32_t> steps, heads(static_cast<size_t>(num_kv_heads));
    for (int32_t h = 0; h < num_kv_heads; ++h) heads[size_t(h)] = h;
    TcListPlan pl;
    for (int32_t b = 0; b < batch; ++b) {
      const int64_t nq = int64_t(qo_indptr[b + 1]) - qo_indptr[b];
      const int64_t n = int64_t(kv_indptr[b + 1]) - kv_indptr[b];
      if (nq < 0 || n < 0) { set_error("plan_prefill_paged: qo_indptr or kv_indptr decreases at %d", b); return BSKV_ERR_INVALID_ARG; }
      int64_t L = 0;
      if (n > 0) {
        const int32_t lp = kv_last_page_len[b];
        if (lp < 1 || lp > page_size) {
          set_error("plan_prefill_paged: kv_last_page_len[%d] = %d outside [1, %d]", b, lp, page_size);
          return BSKV_ERR_INVALID_ARG;
        }
        L = (n - 1) * page_size + lp;
      }
      if (L > INT32_MAX / 2 || nq * g > INT32_MAX / 2) { set_error("plan_prefill_paged: request %d too long", b); return BSKV_ERR_UNSUPPORTED; }
      for (int64_t i = kv_indptr[b]; i < kv_indptr[b + 1]; ++i) {
        if (!kv_indices || kv_indices[i] < 0 || kv_indices[i] >= num_pages) {
          set_error("plan_prefill_paged: kv_indices[%lld] outside [0, %d)", (long long)i, num_pages);
          return BSKV_ERR_INVALID_ARG;
        }
      }
      const int32_t tb = int32_t(steps.size() / size_t(words));
      for (int64_t t = 0; t < L; t += kBsrTcStep) {
        const int64_t e = std::min<int64_t>(t + kBsrTcStep, L);
        steps.push_back(int32_t(t));
        steps.push_back(int32_t(e));
        for (int32_t k = 0; k < ppk; ++k) {
          const int64_t k0 = t + int64_t(k) * page_size;
          steps.push_back(k0 < e ? kv_indices[kv_indptr[b] + k0 / page_size] : -1);
        }
        if (steps.size() > size_t(INT32_MAX) / 2) { set_error("plan_prefill_paged: too many key steps"); return BSKV_ERR_UNSUPPORTED; }
      }
      tc_list_units(pl, steps, words, qo_indptr[b], int32_t(nq), tb,
                    int32_t(steps.size() / size_t(words)), int32_t(L - nq), causal != 0, heads);
    }
    const int64_t total_qo = batch > 0 ? qo_indptr[batch] : 0;
    if (total_qo > INT32_MAX / 2) { set_error("plan_prefill_paged: too many query tokens"); return BSKV_ERR_UNSUPPORTED; }
    bskv_plan* p = new bskv_plan();
    p->kind = KIND_BSR;
    p->batch = batch; p->num_pages = num_pages; p->page_size = page_size;
    p->M = int32_t(total_qo); p->N = 0; p->R = 0; p->C = 0; p->causal = causal ? 1 : 0;
    p->num_qo_heads = num_qo_heads; p->num_kv_heads = num_kv_heads; p->head_dim = head_dim;
    p->dtype = dtype;
    tc_list_assemble(p, pl, steps, num_sms, BSR_PAGED_PREFILL_TC);
    p->float_ws_bytes = 0;
    *out_plan = p;
    log_plan("bskv_plan_prefill_paged", p);
    return BSKV_OK;
  }
  std::vector<int32_t> desc(size_t(batch) * 5), tiles;
  for (int32_t b = 0; b < batch; ++b) {
    const int64_t nq = int64_t(qo_indptr[b + 1]) - qo_indptr[b];
    const int64_t n = int64_t(kv_indptr[b + 1]) - kv_indptr[b];
    if (nq < 0 || n < 0) { set_error("plan_prefill_paged: qo_indptr or kv_indptr decreases at %d", b); return BSKV_ERR_INVALID_ARG; }
    int64_t L = 0;
    if (n > 0) {
      const int32_t lp = kv_last_page_len[b];
      if (lp < 1 || lp > page_size) {
        set_error("plan_prefill_paged: kv_last_page_len[%d] = %d outside [1, %d]", b, lp, page_size);
        return BSKV_ERR_INVALID_ARG;
      }
      L = (n - 1) * page_size + lp;
    }
    if (L > INT32_MAX / 2 || nq * g > INT32_MAX / 2) { set_error("plan_prefill_paged: request %d too long", b); return BSKV_ERR_UNSUPPORTED; }
    for (int64_t i = kv_indptr[b]; i < kv_indptr[b + 1]; ++i) {
      if (!kv_indices || kv_indices[i] < 0 || kv_indices[i] >= num_pages) {
        set_error("plan_prefill_paged: kv_indices[%lld] outside [0, %d)", (long long)i, num_pages);
        return BSKV_ERR_INVALID_ARG;
      }
    }
    const size_t d = size_t(b) * 5;
    desc[d] = qo_indptr[b];
    desc[d + 1] = int32_t(nq);
    desc[d + 2] = int32_t(tiles.size() / 4);
    // tiles of up to 32 keys that never cross a page
    for (int64_t t = 0; t < L;) {
      const int64_t pi = t / page_size;
      const int64_t e = std::min({t + kBsrVarTile, (pi + 1) * page_size, L});
      tiles.push_back(int32_t(t));
      tiles.push_back(int32_t(e));
      tiles.push_back(kv_indices[kv_indptr[b] + pi]);
      tiles.push_back(int32_t(t - pi * page_size));
      t = e;
      if (tiles.size() > size_t(INT32_MAX) / 2) { set_error("plan_prefill_paged: too many key tiles"); return BSKV_ERR_UNSUPPORTED; }
    }
    desc[d + 3] = int32_t(tiles.size() / 4);
    desc[d + 4] = int32_t(L - nq);
  }
  const int64_t total_qo = batch > 0 ? qo_indptr[batch] : 0;
  if (total_qo > INT32_MAX / 2) { set_error("plan_prefill_paged: too many query tokens"); return BSKV_ERR_UNSUPPORTED; }
  // Units (request b, kv head h, row tile of 64 grouped rows), b-major; the same longest-
  // processing-time rule as the variable-block plans, cost 1 + tiles.
  std::vector<Chunk> units;
  std::vector<int64_t> cost;
  for (int32_t b = 0; b < batch; ++b) {
    const size_t d = size_t(b) * 5;
    const int32_t rts = (desc[d + 1] * g + kBsrGenericRows - 1) / kBsrGenericRows;
    for (int32_t h = 0; h < num_kv_heads; ++h)
      for (int32_t rt = 0; rt < rts; ++rt) {
        units.push_back(Chunk{b, b, h, rt});
        cost.push_back(1 + desc[d + 3] - desc[d + 2]);
      }
  }
  const int64_t U = int64_t(units.size());
  const int32_t G = int32_t(std::min<int64_t>(int64_t(num_sms) * kBsrGenericCtasPerSm, std::max<int64_t>(U, 1)));
  std::vector<int32_t> worker_ptr;
  std::vector<Chunk> chunks;
  lists_to_chunks(lpt_assign(cost, G), units, worker_ptr, chunks);
  bskv_plan* p = new bskv_plan();
  p->kind = KIND_BSR;
  p->batch = batch; p->num_pages = num_pages; p->page_size = page_size;
  p->M = int32_t(total_qo); p->N = 0; p->R = 0; p->C = 0; p->causal = causal ? 1 : 0;
  p->num_qo_heads = num_qo_heads; p->num_kv_heads = num_kv_heads; p->head_dim = head_dim;
  p->dtype = dtype;
  std::vector<int32_t> no_merges;
  assemble(p, KIND_BSR, int32_t(U), worker_ptr, chunks, 0, no_merges, kBsrGenericRows,
           desc.data(), desc.size(), tiles.data(), tiles.size(), U > 0 ? G : 0,
           BSR_PAGED_PREFILL);
  p->float_ws_bytes = 0;
  *out_plan = p;
  log_plan("bskv_plan_prefill_paged", p);
  return BSKV_OK;
}

extern "C" bskv_status bskv_plan_bsr_masked(const int32_t* indptr, const int32_t* indices,
                                            int32_t M, int32_t N, int32_t R, int32_t C,
                                            int32_t num_qo_heads, int32_t num_kv_heads,
                                            int32_t head_dim, int32_t dtype, int32_t num_sms,
                                            bskv_plan** out_plan) {
  return plan_bsr(indptr, indices, M, N, R, C, num_qo_heads, num_kv_heads, head_dim, 0, dtype,
                  num_sms, true, out_plan);
}

extern "C" bskv_status bskv_plan_mla_sparse(const int32_t* seq_lens, int32_t batch, int32_t q_len,
                                            int32_t num_heads, int32_t top_k, int32_t num_sms,
                                            bskv_plan** out_plan) {
  if (!out_plan) { set_error("plan_mla_sparse: out_plan is NULL"); return BSKV_ERR_INVALID_ARG; }
  *out_plan = nullptr;
  if (batch < 0 || q_len < 1 || num_sms < 1 || (batch > 0 && !seq_lens)) {
    set_error("plan_mla_sparse: batch=%d q_len=%d num_sms=%d", batch, q_len, num_sms);
    return BSKV_ERR_INVALID_ARG;
  }
  if (top_k < 64 || top_k % 64 != 0) { set_error("plan_mla_sparse: top_k (%d) must be divisible by 64 and at least 64", top_k); return BSKV_ERR_INVALID_ARG; }
  if (num_heads < 1 || num_heads > 128) { set_error("plan_mla_sparse: num_heads %d outside [1,128]", num_heads); return BSKV_ERR_UNSUPPORTED; }
  // One unit per query token; a worker is a pair of CTAs (a cluster), one per latent half.
  std::vector<int64_t> len;
  len.reserve(size_t(batch) * q_len);
  for (int32_t b = 0; b < batch; ++b) {
    if (seq_lens[b] < 0 || seq_lens[b] > top_k) {
      set_error("plan_mla_sparse: seq_lens[%d] = %d outside [0, top_k=%d]", b, seq_lens[b], top_k);
      return BSKV_ERR_INVALID_ARG;
    }
    for (int32_t t = 0; t < q_len; ++t) len.push_back(seq_lens[b]);
  }
  std::vector<int32_t> worker_ptr, merges;
  std::vector<Chunk> chunks;
  int32_t slots = 0;
  mla_partition(len, kMlaTile, std::max(1, num_sms / kMlaVSplit), worker_ptr, chunks, slots,
                merges);
  const int32_t P = int32_t(worker_ptr.size() - 1);
  bskv_plan* p = new bskv_plan();
  p->kind = KIND_MLA;
  p->batch = batch; p->q_len = q_len; p->num_qo_heads = num_heads; p->top_k = top_k;
  p->head_dim = 576; p->dtype = BSKV_E4M3;
  assemble(p, KIND_MLA, int32_t(len.size()), worker_ptr, chunks, slots, merges, kMlaTile,
           nullptr, 0, nullptr, 0, P * kMlaVSplit, 0);
  // a slot holds one piece of a unit for both latent halves
  p->float_ws_bytes = slots == 0 ? 0
      : align256(size_t(slots) * kMlaVSplit * 128 * kMlaVDim * 4) +
            align256(size_t(slots) * kMlaVSplit * 128 * 4);
  *out_plan = p;
  log_plan("bskv_plan_mla_sparse", p);
  return BSKV_OK;
}

extern "C" bskv_status bskv_plan_mla_paged(const int32_t* kv_indptr, const int32_t* kv_indices,
                                           const int32_t* kv_last_page_len, int32_t batch,
                                           int32_t num_pages, int32_t page_size,
                                           int32_t num_heads, int32_t num_sms,
                                           bskv_plan** out_plan) {
  if (!out_plan) { set_error("plan_mla_paged: out_plan is NULL"); return BSKV_ERR_INVALID_ARG; }
  *out_plan = nullptr;
  if (batch < 0 || num_sms < 1 || page_size < 1 || num_pages < 1) {
    set_error("plan_mla_paged: batch=%d num_pages=%d page_size=%d num_sms=%d", batch, num_pages,
              page_size, num_sms);
    return BSKV_ERR_INVALID_ARG;
  }
  if (num_heads < 1 || num_heads > 128) { set_error("plan_mla_paged: num_heads %d outside [1,128]", num_heads); return BSKV_ERR_UNSUPPORTED; }
  if (int64_t(num_pages) * page_size > INT32_MAX) { set_error("plan_mla_paged: num_pages * page_size exceeds int32 row ids"); return BSKV_ERR_UNSUPPORTED; }
  if (batch > 0 && (!kv_indptr || !kv_last_page_len)) { set_error("plan_mla_paged: NULL index array"); return BSKV_ERR_INVALID_ARG; }
  if (batch > 0 && kv_indptr[0] != 0) { set_error("plan_mla_paged: kv_indptr[0] must be 0"); return BSKV_ERR_INVALID_ARG; }
  std::vector<int64_t> len(size_t(batch), 0);
  int64_t longest = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const int64_t n = int64_t(kv_indptr[b + 1]) - kv_indptr[b];
    if (n < 0) { set_error("plan_mla_paged: kv_indptr decreases at %d", b); return BSKV_ERR_INVALID_ARG; }
    if (n > 0) {
      const int32_t lp = kv_last_page_len[b];
      if (lp < 1 || lp > page_size) {
        set_error("plan_mla_paged: kv_last_page_len[%d] = %d outside [1, %d]", b, lp, page_size);
        return BSKV_ERR_INVALID_ARG;
      }
      len[size_t(b)] = (n - 1) * page_size + lp;
    }
    longest = std::max(longest, len[size_t(b)]);
  }
  const int64_t nnz = batch > 0 ? kv_indptr[batch] : 0;
  if (nnz > 0 && !kv_indices) { set_error("plan_mla_paged: kv_indices is NULL"); return BSKV_ERR_INVALID_ARG; }
  for (int64_t i = 0; i < nnz; ++i) {
    if (kv_indices[i] < 0 || kv_indices[i] >= num_pages) {
      set_error("plan_mla_paged: kv_indices[%lld] = %d outside [0, %d)", (long long)i, kv_indices[i], num_pages);
      return BSKV_ERR_INVALID_ARG;
    }
  }
  const int64_t stride = std::max<int64_t>(64, (longest + 63) / 64 * 64);
  if (stride > INT32_MAX / 2) { set_error("plan_mla_paged: a request of %lld tokens is too long", (long long)longest); return BSKV_ERR_UNSUPPORTED; }
  // One unit per request, partitioned like the sparse decode.
  std::vector<int32_t> worker_ptr, merges;
  std::vector<Chunk> chunks;
  int32_t slots = 0;
  mla_partition(len, kMlaTile, std::max(1, num_sms / kMlaVSplit), worker_ptr, chunks, slots,
                merges);
  const int32_t P = int32_t(worker_ptr.size() - 1);
  bskv_plan* p = new bskv_plan();
  p->kind = KIND_MLA;
  p->mla_variant = MLA_PAGED;
  p->batch = batch; p->q_len = 1; p->num_qo_heads = num_heads; p->top_k = int32_t(stride);
  p->num_pages = num_pages; p->page_size = page_size;
  p->head_dim = 576; p->dtype = BSKV_E4M3;
  assemble(p, KIND_MLA, int32_t(len.size()), worker_ptr, chunks, slots, merges, kMlaTile,
           kv_indptr, batch > 0 ? size_t(batch) + 1 : 0, kv_indices, size_t(nnz), P * kMlaVSplit,
           MLA_PAGED);
  p->float_ws_bytes = slots == 0 ? 0
      : align256(size_t(slots) * kMlaVSplit * 128 * kMlaVDim * 4) +
            align256(size_t(slots) * kMlaVSplit * 128 * 4);
  *out_plan = p;
  log_plan("bskv_plan_mla_paged", p);
  return BSKV_OK;
}

extern "C" bskv_status bskv_plan_destroy(bskv_plan* plan) {
  delete plan;
  return BSKV_OK;
}

extern "C" bskv_status bskv_plan_metadata(const bskv_plan* plan, const int32_t** meta,
                                          int64_t* num_words) {
  if (!plan || !meta || !num_words) { set_error("plan_metadata: NULL argument"); return BSKV_ERR_INVALID_ARG; }
  *meta = plan->meta.data();
  *num_words = int64_t(plan->meta.size());
  return BSKV_OK;
}

extern "C" bskv_status bskv_plan_workspace_sizes(const bskv_plan* plan, size_t* int_ws_bytes,
                                                 size_t* float_ws_bytes) {
  if (!plan) { set_error("plan_workspace_sizes: NULL plan"); return BSKV_ERR_INVALID_ARG; }
  // metadata, then the int32 merge counters (zeroed by bskv_plan_upload)
  if (int_ws_bytes)
    *int_ws_bytes = merge_counter_offset(plan->meta.size()) + plan->counter_words * sizeof(int32_t);
  if (float_ws_bytes) *float_ws_bytes = plan->float_ws_bytes;
  return BSKV_OK;
}
