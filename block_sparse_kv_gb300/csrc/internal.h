// Internal declarations shared by the host core and the kernel launchers of libbskv.
#pragma once

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/bskv.h"

namespace bskv {

// ---- plan metadata: int32 words, header then 16-byte aligned sections ----------------
constexpr int32_t kMetaMagic = 0x766b7362;  // "bskv"
enum Kind : int32_t { KIND_DECODE = 1, KIND_BSR = 2, KIND_MLA = 3 };
enum Header : int {
  H_MAGIC = 0,
  H_KIND,
  H_UNITS,
  H_WORKERS,
  H_CHUNKS,
  H_SLOTS,
  H_MERGES,
  H_TILE,
  H_OFF_WORKERS,
  H_OFF_CHUNKS,
  H_OFF_MERGES,
  H_OFF_AUX0,
  H_OFF_AUX1,
  H_GRID,
  H_TOTAL,
  H_VARIANT,
  H_COUNT
};

// ---- kernel shape constants the plans depend on ----------------------------------------
constexpr int kDecodeTile = 16;        // tokens per pipeline stage of a decode worker
constexpr int kDecodeWarps = 8;        // decode workers (warps) per CTA, one CTA per SM
constexpr int kBsrGenericRows = 64;    // packed (token, head) rows per general-BSR unit
constexpr int kBsrGenericCtasPerSm = 4;
constexpr int kMlaTile = 128;          // sparse rows per MLA tile
// An MLA plan assigns whole query tokens (no split-KV pieces, no merge kernel) when the
// busiest worker then has at most this many tiles more than under the balanced split
// partition: splitting costs about that much (each piece writes fp32 partial states of both
// latent halves and loads its query again, and the merge is a second launch; measured on the
// 128-query sparse decode as 98.9 us split on 76 workers against 92.2 us whole on 64).
constexpr int kMlaSplitPenaltyTiles = 7;
constexpr int kMlaVSplit = 2;          // the 512 latent output values split in halves
constexpr int kMlaVDim = 512 / kMlaVSplit;

constexpr int kDecodeGroupMax = 8;     // kv heads per CTA in the page-major decode variant
constexpr int kDecodeGroupMaxPage = 16; // largest page_size that takes the page-major variant
// Page-major decode plans charge a worker, in 16-token tiles: a piece it publishes mid-stream
// (kDecodePublishTiles), a merge at its end (kDecodeMergeTiles), each whole-unit boundary
// (kDecodeBoundaryTiles). Measured per CTA: workers holding two split pieces finished ~6 us
// after those holding one (~3.7 us publishing mid-stream, ~2.4 us more merging at the end);
// the charges were then chosen by timing the headline decode (2 and 2 ran best).
constexpr int kDecodePublishTiles = 2;
constexpr int kDecodeMergeTiles = 2;
constexpr int kDecodeBoundaryTiles = 0;
// A page-major decode plan ends with one record per worker describing the first chunk of its
// walk: {unit, first token, end token, slot, kv_indptr[b], pages of b, n, 0, the ids of the
// chunk's first n <= 8 pages}, so that a worker's first copies wait on one round trip.
constexpr int kDecodeStartWords = 16;
constexpr int kDecodeStartPages = 8;
// bskv_run_decode merges inside the attention kernel when no unit is cut into more pieces
// than this; beyond it one warp would merge many pieces serially at the kernel's tail, and
// the separate merge kernel (more warps per unit) is faster.
constexpr int kFusedMergeMaxPieces = 8;

// BSR_VARIABLE: per-kv-head variable block sizes; the general kernel walks, per unit, the
// query row range and the 32-token key tiles listed in the metadata (aux0: per (kv head,
// row block) {row start, row count, first tile, end tile}; aux1: tiles {key start, range end}).
// BSR_PAGED_PREFILL: batch prefill over a paged KV cache on the general kernel; aux0: per
// request {first query token, query tokens, first tile, end tile, causal shift L_b - qo_len_b};
// aux1: tiles {first key, tile end, page, first slot}, never crossing a page.
// BSR_VARIABLE_TC / BSR_PAGED_PREFILL_TC: the same two rows on the tensor-core kernel (head_dim
// 128, 2 or 4 query heads per kv head; paged: page_size 8, 16, 32, 64 or 128). aux0: per unit
// (64-token row tile) {first query token, valid tokens (<= 64), first step, end step, key
// limit of the tile's first token (causal: key j visible to tile row t iff j <= limit + t)};
// aux1: steps of up to 128 keys {key start, key end} (variable blocks: within one run of
// visible column blocks; paged: within one request, from a multiple of 128, followed by the
// 128 / page_size page ids the step covers, -1 past the request's last page).
enum BsrVariant : int32_t { BSR_GENERIC = 0, BSR_TCGEN05 = 1, BSR_VARIABLE = 2,
                            BSR_PAGED_PREFILL = 3, BSR_VARIABLE_TC = 4, BSR_PAGED_PREFILL_TC = 5 };
constexpr int kBsrVarTile = 32;  // key tokens per tile of a variable-block plan
constexpr int kBsrTcStep = 128;  // key tokens per step of the tensor-core list plans
constexpr int kBsrTcUnitWords = 5;

// The tensor-core kernel serves a list plan of this shape.
inline bool bsr_tc_list_shape(int32_t head_dim, int32_t num_qo_heads, int32_t num_kv_heads) {
  const int32_t g = num_kv_heads > 0 ? num_qo_heads / num_kv_heads : 0;
  return head_dim == 128 && (g == 2 || g == 4);
}
inline bool bsr_tc_page_size(int32_t page_size) {
  return page_size == 8 || page_size == 16 || page_size == 32 || page_size == 64 ||
         page_size == 128;
}
// MLA_SPARSE: row lists given by the caller. MLA_PAGED: rows read from the page table in
// the metadata (aux0 = kv_indptr, aux1 = kv_indices) by the gather itself.
enum MlaVariant : int32_t { MLA_SPARSE = 0, MLA_PAGED = 1 };
// DECODE_WARP: one worker per warp, units (request, kv head).
// DECODE_GROUP: one worker per CTA, units (request, group of G kv heads), G = Hkv when
// Hkv <= 8, else 8 (Hkv a multiple of 8); every page piece is read for all G heads at once.
enum DecodeVariant : int32_t { DECODE_WARP = 0, DECODE_GROUP = 1 };

// kv heads per page-major group for a decode shape, 0 when the variant does not apply.
inline int32_t decode_group_heads(int32_t num_kv_heads, int32_t page_size) {
  if (page_size > kDecodeGroupMaxPage) return 0;
  if (num_kv_heads <= kDecodeGroupMax) return num_kv_heads;
  return num_kv_heads % kDecodeGroupMax == 0 ? kDecodeGroupMax : 0;
}

// Byte offset in the int workspace of the merge counters (after the metadata).
inline size_t merge_counter_offset(size_t meta_words) { return ((meta_words * 4 + 255) / 256) * 256; }

// Softmax scale of a run: the caller's value, or for 0 the pages' default 1/sqrt(head_dim)
// ("flashinfer.sparse", BlockSparseAttentionWrapper.plan: sm_scale defaults to
// 1/sqrt(head_dim)), as log2(e) * scale for the kernels' exp2 arithmetic.
inline float sm_scale_log2(float sm_scale, int32_t head_dim) {
  const float s = sm_scale == 0.f ? float(1.0 / std::sqrt(double(head_dim))) : sm_scale;
  return s * 1.4426950408889634f;
}

// NVTX range around one public call (its launches show up under the call's name in a
// profiler timeline; without a profiler attached the push and pop return at once).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
#define BSKV_NVTX_RANGE(name) ::bskv::NvtxRange bskv_nvtx_range_(name)

// BSKV_LOGLEVEL from the environment (0 when unset): 1 = one line per plan, 2 = more.
int log_level();

void set_error(const char* fmt, ...);
const char* dtype_name(int32_t dt);

}  // namespace bskv

struct bskv_plan {
  int32_t kind = 0;
  std::vector<int32_t> meta;
  // decode
  int32_t batch = 0, num_pages = 0, page_size = 0;
  // shared
  int32_t num_qo_heads = 0, num_kv_heads = 0, head_dim = 0, dtype = 0;
  // bsr (masked: runs take a per-block token mask, the general kernel serves them)
  int32_t M = 0, N = 0, R = 0, C = 0, causal = 0, masked = 0;
  // mla (paged: batch, num_pages and page_size as for decode; top_k is the longest request
  // rounded up to 64)
  int32_t q_len = 0, top_k = 0, mla_variant = 0;
  size_t float_ws_bytes = 0;
  // int32 merge counters after the metadata in the int workspace (decode: one per merge
  // item and kv head of the unit)
  size_t counter_words = 0;
  int32_t max_merge_count = 0;  // most pieces of one split unit
  // page-major decode: word offset in the metadata of the per-worker start records
  // (kDecodeStartWords each), or -1
  int32_t decode_starts = -1;
  // set by bskv_plan_upload
  const int32_t* meta_dev = nullptr;
  int32_t* counters_dev = nullptr;  // one merge counter per merge item, zero between runs
};
