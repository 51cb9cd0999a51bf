// Internal declarations shared by the host core and the kernel launchers of libbskv.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

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
constexpr int kMlaTile = 64;           // sparse rows per MLA chunk
constexpr int kMlaVSplit = 2;          // the 512 latent output values split in halves
constexpr int kMlaVDim = 512 / kMlaVSplit;

enum BsrVariant : int32_t { BSR_GENERIC = 0, BSR_TCGEN05 = 1 };

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
  // bsr
  int32_t M = 0, N = 0, R = 0, C = 0, causal = 0;
  // mla
  int32_t q_len = 0, top_k = 0;
  size_t float_ws_bytes = 0;
  // set by bskv_plan_upload
  const int32_t* meta_dev = nullptr;
};
