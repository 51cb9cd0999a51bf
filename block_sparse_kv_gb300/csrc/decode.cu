// Paged-KV batch decode with split-KV, and the LSE merge of attention states.
//
// Method: "FlashInfer" agent-skill summary, KV-Cache Formats (paged KV-cache: kv_cache
// (num_pages, 2, num_kv_heads, page_size, head_dim), kv_indptr, kv_indices,
// kv_last_page_len); "flashinfer.sparse" BlockSparseAttentionWrapper.__init__ (a float
// workspace holds the intermediate results of the split-k algorithm); FlashInfer
// cascade.rst (merge_state / merge_states).
//
// GB300 design. Decode reads every K/V byte once (O(1) flop per byte), so the kernel is an
// HBM stream, and its efficiency follows from how large the contiguous pieces it asks
// HBM for are. Two variants, chosen by the plan:
//   * group (pages of 8 or 16 tokens): one CTA per SM, a producer warp, one consumer warp
//     per kv head of a group of up to 8, and a lookup warp. Each 16-token tile is copied by
//     TMA for all heads of the group at once, so with the contiguous layout a page's K (and
//     V) for 8 heads is one 32 KB piece instead of eight 4 KB ones. A 3-stage ring (64 KB
//     stages for 8 heads of 128 dims) holds up to 192 KB in flight per SM; the producer
//     starts from the plan's start record of its worker (first chunk, page range, first
//     page ids) and then reads the page ids of 32 pages at a time, and the lookup warp finds
//     the merge items of the worker's first and last chunks while the KV streams.
//   * warp (larger pages, or head counts that do not group): 8 independent worker warps
//     per CTA, each with a private 3-stage ring over its own (request, kv head) range;
//     a page of 64 tokens is already a 16 KB piece per head.
// In both, the up-to-16 query heads that share a kv head form the M=16 rows of mma.sync
// m16n8k16 (bf16/fp16 in, fp32 accumulate): S = Q K^T, online softmax in registers
// (exp2), O += P V with P reused from the S accumulators. The work is the plan's linear
// split-KV partition; a unit split over several workers leaves normalised partial states
// and LSE in the float workspace, and the worker that finishes the unit's last piece
// (an atomic counter per unit in the int workspace) merges them in the same launch.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "launch.h"

namespace bskv {
namespace {

using namespace dev;

constexpr int kTile = kDecodeTile;  // 16 tokens per stage
constexpr int kStages = 3;
constexpr int kWarps = kDecodeWarps;
constexpr int kPanelBytes = kTile * 128;  // 16 rows x 64 elements of 16 bits
// Group kernel warps: 8 consumers (one per kv head of the unit), then the producer, then the
// lookup warp.
constexpr int kGroupProducerWarp = kDecodeGroupMax;
constexpr int kGroupLookupWarp = kDecodeGroupMax + 1;
constexpr int kGroupThreads = (kDecodeGroupMax + 2) * 32;
constexpr uint32_t kGroupRingBytes = 196608;                // ring budget of the group kernel
// The group kernel's 10 warps put 3 on one SM sub-partition, which caps a thread at 168
// registers; its merges keep fewer loads in flight than the 8-warp kernels' (4 x 4).
constexpr int kGroupMergeSlots = 2, kGroupMergeRows = 2;

struct DecodeParams {
  const int32_t* meta;
  const void* q;
  int64_t q_s0, q_s1;
  void* out;
  int64_t o_s0, o_s1;
  float* lse;
  float* ws_o;
  float* ws_lse;
  int* counters;  // non-null: the last worker to finish a split unit merges it
  int num_kv_heads, group, page_size, num_qo_heads;
  int heads_per_unit;  // kv heads of one unit: 1 (warp variant) or G (group variant)
  int stages;          // ring depth of the group variant
  // word offsets of the metadata's sections and the merge count (the header's values,
  // passed by value so that a worker's first loads do not wait on the header)
  int off_workers, off_chunks, off_merges, off_aux0, off_aux1, num_merges;
  int off_starts;  // page-major plans: the per-worker start records, else -1
  float scale_log2;
  StatusArgs st;
};

template <int D>
__host__ __device__ constexpr int tile_bytes() {
  return (D / 64) * kPanelBytes;
}

// Where one head's 16 K and V rows of a stage sit in shared memory. Row r of 64-column
// half hf starts at base + hf * half + (r / 8) * blk8 + (r % 8) * 128; every group of 8
// rows starts on a 1024-byte boundary, so the 128-byte swizzle of the TMA copy is
// chunk ^ (r % 8).
struct KvRows {
  uint32_t k, v, half, blk8;
};

__device__ __forceinline__ uint32_t kv_row(const KvRows& g, uint32_t base, int row, int hf) {
  return base + hf * g.half + (row >> 3) * g.blk8 + (row & 7) * 128;
}

// One 16-token tile for the (up to 16) query heads of one kv head: S = Q K^T on the
// tensor cores (mma.sync m16n8k16), online softmax in base 2 on rows r0 = lane/4 and
// r1 = r0 + 8, O += P V with P taken from the S accumulators.
template <typename T, int D>
__device__ __forceinline__ void decode_tile(const KvRows& kv, int valid, float scale_log2,
                                            int lane, const uint32_t (&qa)[D / 16][4],
                                            float (&o)[D / 8][4], float& m0, float& m1,
                                            float& l0, float& l1) {
  using Mma = MmaOp<T>;
  const int cq = lane & 3;
  if (valid < kTile) {
    // Rows past the unit's end hold whatever the pages hold there (or stale data); zero
    // the V rows so that 0 * garbage cannot reach the output.
    const int per_half = (kTile - valid) * 8;
    for (int i = lane; i < per_half * (D / 64); i += 32) {
      const int hf = i / per_half, rem = i % per_half;
      sts128(kv_row(kv, kv.v, valid + rem / 8, hf) + (rem % 8) * 16, make_uint4(0, 0, 0, 0));
    }
    __syncwarp();
  }
  float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  {
    const int mi = lane >> 3;
    const int trow = (mi >> 1) * 8 + (lane & 7);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int dim = kk * 16 + (mi & 1) * 8;
      const uint32_t addr =
          kv_row(kv, kv.k, trow, dim / 64) + ((((dim % 64) / 8) ^ (trow & 7)) << 4);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(addr, b0, b1, b2, b3);
      Mma::run(s[0], qa[kk], b0, b1);
      Mma::run(s[1], qa[kk], b2, b3);
    }
  }
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int col = nt * 8 + 2 * cq + (e & 1);
      const float x = s[nt][e] * scale_log2;
      s[nt][e] = col < valid ? x : -INFINITY;
    }
    mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
    mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
  }
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
  const float a0 = fast_exp2(m0 - mn0), a1 = fast_exp2(m1 - mn1);
  m0 = mn0;
  m1 = mn1;
  float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    s[nt][0] = fast_exp2(s[nt][0] - mn0);
    s[nt][1] = fast_exp2(s[nt][1] - mn0);
    s[nt][2] = fast_exp2(s[nt][2] - mn1);
    s[nt][3] = fast_exp2(s[nt][3] - mn1);
    ps0 += s[nt][0] + s[nt][1];
    ps1 += s[nt][2] + s[nt][3];
  }
  l0 = l0 * a0 + ps0;
  l1 = l1 * a1 + ps1;
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    o[n][0] *= a0;
    o[n][1] *= a0;
    o[n][2] *= a1;
    o[n][3] *= a1;
  }
  uint32_t pa[4];
  pa[0] = Mma::pack(s[0][0], s[0][1]);
  pa[1] = Mma::pack(s[0][2], s[0][3]);
  pa[2] = Mma::pack(s[1][0], s[1][1]);
  pa[3] = Mma::pack(s[1][2], s[1][3]);
  {
    const int mi = lane >> 3;
    const int trow = (mi & 1) * 8 + (lane & 7);
#pragma unroll
    for (int dd = 0; dd < D / 16; ++dd) {
      const int dim = dd * 16 + (mi >> 1) * 8;
      const uint32_t addr =
          kv_row(kv, kv.v, trow, dim / 64) + ((((dim % 64) / 8) ^ (trow & 7)) << 4);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(addr, b0, b1, b2, b3);
      Mma::run(o[2 * dd], pa, b0, b1);
      Mma::run(o[2 * dd + 1], pa, b2, b3);
    }
  }
}

// Query rows r0, r1 (< g) of kv head `kvh` of request b into the A fragments.
template <typename T, int D>
__device__ __forceinline__ void load_q(const DecodeParams& p, int b, int kvh, int lane,
                                       uint32_t (&qa)[D / 16][4]) {
  const int g = p.group, r0 = lane >> 2, r1 = r0 + 8, cq = lane & 3;
  const T* qb = static_cast<const T*>(p.q) + b * p.q_s0 + int64_t(kvh) * g * p.q_s1;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int d0 = kk * 16 + 2 * cq;
    qa[kk][0] = r0 < g ? *reinterpret_cast<const uint32_t*>(qb + r0 * p.q_s1 + d0) : 0u;
    qa[kk][1] = r1 < g ? *reinterpret_cast<const uint32_t*>(qb + r1 * p.q_s1 + d0) : 0u;
    qa[kk][2] = r0 < g ? *reinterpret_cast<const uint32_t*>(qb + r0 * p.q_s1 + d0 + 8) : 0u;
    qa[kk][3] = r1 < g ? *reinterpret_cast<const uint32_t*>(qb + r1 * p.q_s1 + d0 + 8) : 0u;
  }
}

// Normalise a finished chunk of kv head `kvh` and write it: straight to out/lse when the
// unit is one chunk (slot < 0), else as partial state row (slot, row0 + r).
template <typename T, int D>
__device__ __forceinline__ void finish_chunk(const DecodeParams& p, int b, int kvh, int slot,
                                             int slot_rows, int row0, int lane,
                                             const float (&o)[D / 8][4], float m0, float m1,
                                             float l0, float l1) {
  using Mma = MmaOp<T>;
  const int g = p.group, r0 = lane >> 2, r1 = r0 + 8, cq = lane & 3;
  float lt0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
  lt0 += __shfl_xor_sync(0xffffffffu, lt0, 2);
  float lt1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
  lt1 += __shfl_xor_sync(0xffffffffu, lt1, 2);
  const float inv0 = 1.f / lt0, inv1 = 1.f / lt1;
  const float lse0 = (m0 + __log2f(lt0)) * kLn2, lse1 = (m1 + __log2f(lt1)) * kLn2;
  if (slot < 0) {
    T* ob = static_cast<T*>(p.out) + b * p.o_s0 + int64_t(kvh) * g * p.o_s1;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      const int d = n * 8 + 2 * cq;
      if (r0 < g)
        *reinterpret_cast<uint32_t*>(ob + r0 * p.o_s1 + d) = Mma::pack(o[n][0] * inv0, o[n][1] * inv0);
      if (r1 < g)
        *reinterpret_cast<uint32_t*>(ob + r1 * p.o_s1 + d) = Mma::pack(o[n][2] * inv1, o[n][3] * inv1);
    }
    if (p.lse && cq == 0) {
      float* lb = p.lse + int64_t(b) * p.num_qo_heads + kvh * g;
      if (r0 < g) lb[r0] = lse0;
      if (r1 < g) lb[r1] = lse1;
    }
  } else {
    const int64_t base = int64_t(slot) * slot_rows + row0;
    float* wo = p.ws_o + base * D;
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      const int d = n * 8 + 2 * cq;
      if (r0 < g) *reinterpret_cast<float2*>(wo + r0 * D + d) = make_float2(o[n][0] * inv0, o[n][1] * inv0);
      if (r1 < g) *reinterpret_cast<float2*>(wo + r1 * D + d) = make_float2(o[n][2] * inv1, o[n][3] * inv1);
    }
    if (cq == 0) {
      if (r0 < g) p.ws_lse[base + r0] = lse0;
      if (r1 < g) p.ws_lse[base + r1] = lse1;
    }
  }
}

// Merge `count` partial states of output rows row0..row0+nrows-1 (of slots
// first..first+count-1, slot_rows rows per slot) into out0 + r * out_stride and lse0[r];
// count == 0 writes zeros and -inf. One warp; a lane covers 4 values of every (128 / D)-th
// row, NI rows (2 NI for D = 64) per pass. The slots are loaded B at a time (all in flight
// together) and combined one by one in slot order (the result depends on neither B nor NI):
//   m' = max(m, lse_c), s = exp(m - m'), w = exp(lse_c - m'),
//   l' = l s + w, acc' = acc s + w o_c;  out = acc / l, lse = m + log(l),
// the log-sum-exp merge of attention states. Partials written by other SMs in the same
// launch are read through L2 (ld.global.cg).
template <typename T, int D, int B = 4, int NI = 4>
__device__ __forceinline__ void merge_rows(int lane, const float* ws_o, const float* ws_lse,
                                           int first, int count, int slot_rows, int row0,
                                           int nrows, T* out0, int64_t out_stride, float* lse0) {
  constexpr int RS = 128 / D;  // rows covered by one pass of the warp
  const int dl = (lane * 4) % D, rl = (lane * 4) / D;
  for (int rb = 0; rb < nrows; rb += NI * RS) {
    float m[NI], tot[NI];
    float4 acc[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      m[i] = -INFINITY;
      tot[i] = 0.f;
      acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int c0 = 0; c0 < count; c0 += B) {
      float bl[B][NI];
      float4 bx[B][NI];
#pragma unroll
      for (int j = 0; j < B; ++j) {
        const int64_t base = int64_t(first + c0 + j) * slot_rows + row0 + rb + rl;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          if (c0 + j < count && rb + rl + RS * i < nrows) {
            bl[j][i] = __ldcg(ws_lse + base + RS * i);
            bx[j][i] = __ldcg(reinterpret_cast<const float4*>(ws_o + (base + RS * i) * D + dl));
          }
        }
      }
#pragma unroll
      for (int j = 0; j < B; ++j) {
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          if (c0 + j >= count || rb + rl + RS * i >= nrows) continue;
          const float mn = fmaxf(m[i], bl[j][i]);
          const float sc = m[i] == -INFINITY ? 0.f : expf(m[i] - mn);
          const float w = expf(bl[j][i] - mn);
          tot[i] = tot[i] * sc + w;
          acc[i].x = acc[i].x * sc + w * bx[j][i].x;
          acc[i].y = acc[i].y * sc + w * bx[j][i].y;
          acc[i].z = acc[i].z * sc + w * bx[j][i].z;
          acc[i].w = acc[i].w * sc + w * bx[j][i].w;
          m[i] = mn;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < NI; ++i) {
      const int r = rb + rl + RS * i;
      if (r >= nrows) continue;
      const float inv = count > 0 ? 1.f / tot[i] : 0.f;
      // two 4-byte stores: output strides need only be multiples of 2 elements
      uint32_t* dst = reinterpret_cast<uint32_t*>(out0 + r * out_stride + dl);
      dst[0] = MmaOp<T>::pack(acc[i].x * inv, acc[i].y * inv);
      dst[1] = MmaOp<T>::pack(acc[i].z * inv, acc[i].w * inv);
      if (lse0 && dl == 0) lse0[r] = count > 0 ? m[i] + logf(tot[i]) : -INFINITY;
    }
  }
}

// The order in which a worker walks its chunks c0..c1-1: its last chunk first, then the
// others in order. A unit cut between workers w and w+1 is the last chunk of w and the
// first of w+1, so both pieces are computed early and its merge is off the kernel's tail.
__device__ __forceinline__ int chunk_at(int c0, int c1, int k) {
  return c1 - c0 >= 2 ? (k == 0 ? c1 - 1 : c0 + k - 1) : c0 + k;
}

// Merge item (unit, first_slot, count) of `unit`; items are sorted by unit.
__device__ __forceinline__ int find_merge_item(const int32_t* merges, int n, int unit) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (merges[3 * mid] < unit) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Output row h*g + r of unit (b, u): rows of kv head u * heads_per_unit + h.
template <typename T>
__device__ __forceinline__ T* out_row(const DecodeParams& p, int b, int head) {
  return static_cast<T*>(p.out) + b * p.o_s0 + int64_t(head) * p.o_s1;
}
__device__ __forceinline__ float* lse_row(const DecodeParams& p, int b, int head) {
  return p.lse ? p.lse + int64_t(b) * p.num_qo_heads + head : nullptr;
}

// ---------------------------------------------------------------------------------------
// warp variant: 8 independent workers per CTA, each with a private TMA ring
// ---------------------------------------------------------------------------------------

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32, 1)
    decode_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p) {
  constexpr int kTileBytes = tile_bytes<D>();
  constexpr int kStageBytes = 2 * kTileBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  uint8_t* ring = smem + warp * (kStages * kStageBytes);
  uint64_t* bars =
      reinterpret_cast<uint64_t*>(smem + kWarps * kStages * kStageBytes) + warp * kStages;

  const int32_t* hdr = p.meta;
  const int P = hdr[H_WORKERS];
  const int w = blockIdx.x * kWarps + warp;
  if (w >= P) return;
  const int32_t* wptr = hdr + hdr[H_OFF_WORKERS];
  const int4* chunks = reinterpret_cast<const int4*>(hdr + hdr[H_OFF_CHUNKS]);
  const int32_t* merges = hdr + hdr[H_OFF_MERGES];
  const int NM = hdr[H_MERGES];
  const int32_t* kv_indptr = hdr + hdr[H_OFF_AUX0];
  const int32_t* kv_indices = hdr + hdr[H_OFF_AUX1];
  const int c0 = wptr[w], c1 = wptr[w + 1];

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
    prefetch_tensormap(&kv_map);
  }
  __syncwarp();

  const bool forced = forced_timeout(p.st);
  const int Hkv = p.num_kv_heads, g = p.group, ps = p.page_size;
  const int box_rows = ps < kTile ? ps : kTile;
  const uint32_t piece_bytes = uint32_t(box_rows) * 128u;

  const uint64_t stream_policy = l2_evict_first_policy();  // KV is read once
  // Issue the TMA copies of tile `t` of chunk `c` into `stage` (lane 0 only).
  auto issue = [&](int stage, int c, int t) {
    const int4 ch = chunks[c];
    const int b = ch.x / Hkv, kvh = ch.x % Hkv;
    const int tok = ch.y + t * kTile;
    const int pbase = kv_indptr[b];
    uint8_t* kdst = ring + stage * kStageBytes;
    uint8_t* vdst = kdst + kTileBytes;
    uint32_t bytes = 0;
    if (ps >= kTile) {
      const int page = kv_indices[pbase + tok / ps];
      const int s = tok % ps;
      bytes = 2u * (D / 64) * piece_bytes;
      mbar_arrive_expect_tx(&bars[stage], bytes);
#pragma unroll
      for (int hf = 0; hf < D / 64; ++hf) {
        tma_load_5d_hint(kdst + hf * kPanelBytes, &kv_map, hf * 64, s, kvh, 0, page, &bars[stage],
                         stream_policy);
        tma_load_5d_hint(vdst + hf * kPanelBytes, &kv_map, hf * 64, s, kvh, 1, page, &bars[stage],
                         stream_policy);
      }
    } else {
      const int npages = kv_indptr[b + 1] - pbase;
      const int first = tok / ps;
      int pieces = kTile / ps;
      if (first + pieces > npages) pieces = npages - first;
      bytes = 2u * (D / 64) * piece_bytes * uint32_t(pieces);
      mbar_arrive_expect_tx(&bars[stage], bytes);
      for (int k = 0; k < pieces; ++k) {
        const int page = kv_indices[pbase + first + k];
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf) {
          tma_load_5d_hint(kdst + hf * kPanelBytes + k * piece_bytes, &kv_map, hf * 64, 0, kvh,
                           0, page, &bars[stage], stream_policy);
          tma_load_5d_hint(vdst + hf * kPanelBytes + k * piece_bytes, &kv_map, hf * 64, 0, kvh,
                           1, page, &bars[stage], stream_policy);
        }
      }
    }
  };
  auto ntiles = [&](int c) {
    const int4 ch = chunks[c];
    return (ch.z - ch.y + kTile - 1) / kTile;
  };

  // Fused merge: units without tokens are zero-filled by the workers in turn.
  if (p.counters) {
    for (int i = w; i < NM; i += P) {
      if (merges[3 * i + 2] != 0) continue;
      const int unit = merges[3 * i], b = unit / Hkv, kvh = unit % Hkv;
      merge_rows<T, D>(lane, p.ws_o, p.ws_lse, 0, 0, g, 0, g, out_row<T>(p, b, kvh * g), p.o_s1,
                       lse_row(p, b, kvh * g));
    }
  }

  // Producer cursor (pk, pt) runs kStages tiles ahead of the consumer cursor (ck, ct);
  // k counts chunks in the order chunk_at gives.
  const int nck = c1 - c0;
  int pk = 0, pt = 0;
  auto advance = [&](int& k, int& t) {
    if (++t == ntiles(chunk_at(c0, c1, k))) {
      ++k;
      t = 0;
    }
  };
  uint32_t issued = 0, consumed = 0;
  for (int s = 0; s < kStages && pk < nck; ++s) {
    if (lane == 0) issue(s, chunk_at(c0, c1, pk), pt);
    ++issued;
    advance(pk, pt);
  }

  uint32_t qa[D / 16][4];
  float o[D / 8][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  bool ok = true;
  int ck = 0, ct = 0;
  while (ck < nck) {
    const int cc = chunk_at(c0, c1, ck);
    const int4 ch = chunks[cc];
    const int b = ch.x / Hkv, kvh = ch.x % Hkv;
    if (ct == 0) {
      load_q<T, D>(p, b, kvh, lane, qa);
#pragma unroll
      for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
    }
    const int stage = consumed % kStages;
    if (!warp_wait(&bars[stage], (consumed / kStages) & 1u, p.st, forced)) {
      ok = false;
      break;
    }
    const uint32_t kt = smem_u32(ring + stage * kStageBytes);
    const KvRows kv{kt, kt + uint32_t(kTileBytes), uint32_t(kPanelBytes), 1024u};
    const int tok0 = ch.y + ct * kTile;
    decode_tile<T, D>(kv, min(kTile, ch.z - tok0), p.scale_log2, lane, qa, o, m0, m1, l0, l1);
    ++consumed;
    __syncwarp();
    if (pk < nck) {
      if (lane == 0) {
        fence_proxy_async_smem();
        issue(stage, chunk_at(c0, c1, pk), pt);
      }
      ++issued;
      advance(pk, pt);
    }
    if (++ct == ntiles(cc)) {
      const int slot = ch.w;
      finish_chunk<T, D>(p, b, kvh, slot, g, 0, lane, o, m0, m1, l0, l1);
      if (slot >= 0 && p.counters) {
        // The last of the unit's chunks to finish merges all of them (release / acquire
        // through lane 0's atomic, as in the group kernel).
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          const int item = find_merge_item(merges, NM, ch.x);
          const int old = atomic_add_acq_rel(p.counters + item, 1);
          last = old == merges[3 * item + 2] - 1 ? item + 1 : 0;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
          const int item = last - 1;
          merge_rows<T, D>(lane, p.ws_o, p.ws_lse, merges[3 * item + 1], merges[3 * item + 2], g,
                           0, g, out_row<T>(p, b, kvh * g), p.o_s1, lse_row(p, b, kvh * g));
          if (lane == 0) p.counters[item] = 0;  // ready for the next run
        }
      }
      ++ck;
      ct = 0;
    }
  }
  if (!ok) {
    // Drain the copies still in flight before the warp leaves (bounded, not forcible).
    for (uint32_t k = consumed; k < issued; ++k)
      mbar_wait(&bars[k % kStages], (k / kStages) & 1u, p.st, false);
  }
}

// ---------------------------------------------------------------------------------------
// group variant: one worker per CTA; a producer warp copies each 16-token tile of all G
// kv heads of a unit (page-contiguous pieces of G * page_size * 256 bytes) into a shared
// ring, consumer warp h computes kv head h of the group.
// ---------------------------------------------------------------------------------------

template <int D>
__host__ __device__ constexpr uint32_t group_stage_bytes(int G) {
  return 2u * (D / 64) * uint32_t(G) * kPanelBytes;
}

// Bounded wait that also gives up when the CTA's abort flag is raised.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity,
                                              const StatusArgs& st, bool give_up,
                                              const volatile int* abort_flag) {
  if (give_up) {
    record_error(st, BSKV_ERR_TIMEOUT);
    return false;
  }
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(a, parity)) return true;
    if ((i & 63u) == 63u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        record_error(st, BSKV_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Merge of one kv head's g query rows of a split unit (pieces first..first+cnt-1) into the
// output, for the group kernel. Not inlined: the consumers' main loop then keeps its
// registers (inlined after the loop, the kernel spills at its 168-register cap).
template <typename T, int D>
__device__ __noinline__ void group_merge_head(const DecodeParams& p, int lane, int first, int cnt,
                                              int slot_rows, int h, int b, int head) {
  merge_rows<T, D, kGroupMergeSlots, kGroupMergeRows>(lane, p.ws_o, p.ws_lse, first, cnt,
                                                      slot_rows, h * p.group, p.group,
                                                      out_row<T>(p, b, head), p.o_s1,
                                                      lse_row(p, b, head));
}

template <typename T, int D>
__global__ void __launch_bounds__(kGroupThreads, 1)
    decode_group_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.heads_per_unit, ns = p.stages;
  const int ps = p.page_size, box_rows = ps < kTile ? ps : kTile;
  const uint32_t head_bytes = uint32_t(box_rows) * 128u;    // one head, one half, one piece
  const uint32_t piece_bytes = uint32_t(G) * head_bytes;     // all G heads
  const uint32_t half_bytes = uint32_t(G) * kPanelBytes;     // 16 rows of all G heads
  const uint32_t kv_bytes = (D / 64) * half_bytes;           // K (or V) of one stage
  const uint32_t stage_bytes = 2u * kv_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ns * stage_bytes);
  uint64_t* empty = full + ns;
  uint64_t* items_ready = empty + ns;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(items_ready + 1);
  int* items = reinterpret_cast<int*>(items_ready + 1) + 1;  // [0]: first chunk, [1]: last

  const int32_t* hdr = p.meta;
  const int w = blockIdx.x;
  const int32_t* wptr = hdr + p.off_workers;
  const int4* chunks = reinterpret_cast<const int4*>(hdr + p.off_chunks);
  const int32_t* merges = hdr + p.off_merges;
  const int NM = p.num_merges;
  const int32_t* kv_indptr = hdr + p.off_aux0;
  const int32_t* kv_indices = hdr + p.off_aux1;
  const int c0 = wptr[w], c1 = wptr[w + 1];
  const int HG = p.num_kv_heads / G, g = p.group, SR = G * g;

  if (threadIdx.x == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], uint32_t(G));
    }
    mbar_init(items_ready, 2);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&kv_map);
  }
  __syncthreads();
  const bool forced = forced_timeout(p.st);
  auto ntiles = [&](const int4& ch) { return (ch.z - ch.y + kTile - 1) / kTile; };

  if (warp == kGroupProducerWarp) {
    // Producer: lane 0 issues every copy, then waits for its own copies to land. The warp's
    // lanes read the ids of 32 consecutive pages of the request at once and lane 0 takes them
    // by shuffle, so a copy never waits on a page-table read.
    const uint64_t stream_policy = l2_evict_first_policy();  // KV is read once
    uint32_t it = 0;
    bool ok = true;
    for (int k = 0; k < c1 - c0 && ok; ++k) {
      int4 ch;
      int pbase, npages;
      // lane j holds the id of page win + j of the request, for j < wsize
      int win = -(1 << 30), wsize = 32, pid = 0;
      if (k == 0 && p.off_starts >= 0) {
        // the walk's first chunk, its request's pages and their first ids from the worker's
        // start record: words that do not depend on one another, one round trip
        const int v = lane < kDecodeStartWords ? hdr[p.off_starts + kDecodeStartWords * w + lane] : 0;
        ch = make_int4(__shfl_sync(0xffffffffu, v, 0), __shfl_sync(0xffffffffu, v, 1),
                       __shfl_sync(0xffffffffu, v, 2), __shfl_sync(0xffffffffu, v, 3));
        pbase = __shfl_sync(0xffffffffu, v, 4);
        npages = __shfl_sync(0xffffffffu, v, 5);
        wsize = __shfl_sync(0xffffffffu, v, 6);
        pid = __shfl_sync(0xffffffffu, v, 8 + (lane & (kDecodeStartPages - 1)));
        win = ch.y / ps;
      } else {
        ch = chunks[chunk_at(c0, c1, k)];
        const int b = ch.x / HG;
        pbase = kv_indptr[b];
        npages = kv_indptr[b + 1] - pbase;
      }
      const int hg = ch.x % HG;
      const int nt = ntiles(ch);
      for (int t = 0; t < nt; ++t, ++it) {
        const int stage = int(it % uint32_t(ns));
        const int tok = ch.y + t * kTile;
        const int first = tok / ps;
        const int pieces = ps >= kTile ? 1 : min(kTile / ps, npages - first);
        if (first + pieces > win + wsize) {
          win = first;
          wsize = 32;
          pid = win + lane < npages ? kv_indices[pbase + win + lane] : 0;
        }
        if (it >= uint32_t(ns)) {
          int good = 1;
          if (lane == 0)
            good = wait_or_abort(&empty[stage], ((it / ns) & 1u) ^ 1u, p.st, forced, abort_flag);
          if (!__shfl_sync(0xffffffffu, good, 0)) {
            if (lane == 0) *abort_flag = 1;
            ok = false;
            break;
          }
        }
        uint8_t* kdst = smem + stage * stage_bytes;
        uint8_t* vdst = kdst + kv_bytes;
        if (ps >= kTile) {
          const int page = __shfl_sync(0xffffffffu, pid, first - win);
          const int s = tok % ps;
          if (lane == 0) {
            mbar_arrive_expect_tx(&full[stage], 2u * (D / 64) * piece_bytes);
#pragma unroll
            for (int hf = 0; hf < D / 64; ++hf) {
              tma_load_5d_hint(kdst + hf * half_bytes, &kv_map, hf * 64, s, hg * G, 0, page,
                               &full[stage], stream_policy);
              tma_load_5d_hint(vdst + hf * half_bytes, &kv_map, hf * 64, s, hg * G, 1, page,
                               &full[stage], stream_policy);
            }
          }
        } else {
          if (lane == 0)
            mbar_arrive_expect_tx(&full[stage], 2u * (D / 64) * piece_bytes * uint32_t(pieces));
          for (int q = 0; q < pieces; ++q) {
            const int page = __shfl_sync(0xffffffffu, pid, first + q - win);
            if (lane == 0) {
#pragma unroll
              for (int hf = 0; hf < D / 64; ++hf) {
                tma_load_5d_hint(kdst + hf * half_bytes + q * piece_bytes, &kv_map, hf * 64, 0,
                                 hg * G, 0, page, &full[stage], stream_policy);
                tma_load_5d_hint(vdst + hf * half_bytes + q * piece_bytes, &kv_map, hf * 64, 0,
                                 hg * G, 1, page, &full[stage], stream_policy);
              }
            }
          }
        }
      }
    }
    // Every copy issued must land before the CTA may exit (bounded, not forcible).
    if (lane == 0)
      for (uint32_t k = it > uint32_t(ns) ? it - ns : 0; k < it; ++k)
        mbar_wait(&full[k % ns], (k / ns) & 1u, p.st, false);
    return;
  }
  if (warp == kGroupLookupWarp) {
    // Lookup warp: finds the merge items of the first and the last chunk of the worker's walk
    // (lanes 0 and 1, in parallel) while the KV streams, so that the consumers publish those
    // pieces without searching the merge list (a linear partition puts a worker's pieces
    // only there; a search costs several dependent round trips while HBM is saturated).
    if (lane < 2 && p.counters && c1 > c0) {
      const int4 ch = chunks[chunk_at(c0, c1, lane == 0 ? 0 : c1 - c0 - 1)];
      items[lane] = ch.w >= 0 ? find_merge_item(merges, NM, ch.x) : -1;
      mbar_arrive(items_ready);
    }
    return;
  }
  if (warp >= G) return;

  // Consumer warp h: kv head hg * G + h of each chunk's unit. After a failed wait it
  // skips the arithmetic (and the stage releases) of the rest of its work.
  const int h = warp;
  if (p.counters) {
    for (int i = w; i < NM; i += gridDim.x) {
      if (merges[3 * i + 2] != 0) continue;
      const int unit = merges[3 * i], b = unit / HG, hg = unit % HG;
      const int head = (hg * G + h) * g;
      merge_rows<T, D, kGroupMergeSlots, kGroupMergeRows>(lane, p.ws_o, p.ws_lse, 0, 0, SR, h * g, g, out_row<T>(p, b, head), p.o_s1,
                       lse_row(p, b, head));
    }
  }
  uint32_t qa[D / 16][4];
  float o[D / 8][4];
  float m0, m1, l0, l1;
  bool ok = true;
  uint32_t it = 0;
  for (int k = 0; k < c1 - c0; ++k) {
    const int4 ch = chunks[chunk_at(c0, c1, k)];
    const int b = ch.x / HG, hg = ch.x % HG, kvh = hg * G + h;
    load_q<T, D>(p, b, kvh, lane, qa);
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    m0 = m1 = -INFINITY;
    l0 = l1 = 0.f;
    const int nt = ntiles(ch);
    for (int t = 0; t < nt; ++t, ++it) {
      const int stage = int(it % uint32_t(ns));
      if (ok) ok = warp_wait(&full[stage], (it / ns) & 1u, p.st, forced, abort_flag);
      if (!ok) {
        if (lane == 0) *abort_flag = 1;
        continue;
      }
      const uint32_t kt = smem_u32(smem + stage * stage_bytes) + uint32_t(h) * head_bytes;
      const KvRows kv{kt, kt + kv_bytes, half_bytes, box_rows == kTile ? 1024u : piece_bytes};
      const int valid = min(kTile, ch.z - (ch.y + t * kTile));
      decode_tile<T, D>(kv, valid, p.scale_log2, lane, qa, o, m0, m1, l0, l1);
      if (valid < kTile) fence_proxy_async_smem();  // zeroed rows before the next copy
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }
    const int slot = ch.w;
    if (!ok) continue;
    finish_chunk<T, D>(p, b, kvh, slot, SR, h * g, lane, o, m0, m1, l0, l1);
    if (slot >= 0 && p.counters) {
      // Per kv head: the last warp to finish a piece of the unit merges that head's rows.
      // The warp's partial-state writes are ordered before lane 0's release (the
      // __syncwarp), and the merging warp reads the other pieces after its acquire.
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        int item;
        if ((k == 0 || k + 1 == c1 - c0) && mbar_wait(items_ready, 0, p.st, false))
          item = items[k == 0 ? 0 : 1];
        else
          item = find_merge_item(merges, NM, ch.x);
        const int old = atomic_add_acq_rel(p.counters + item * G + h, 1);
        last = old == merges[3 * item + 2] - 1 ? item + 1 : 0;
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      __syncwarp();
      if (last) {
        const int item = last - 1;
        group_merge_head<T, D>(p, lane, merges[3 * item + 1], merges[3 * item + 2], SR, h, b,
                               kvh * g);
        if (lane == 0) p.counters[item * G + h] = 0;  // ready for the next run
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// merge of split-KV partial states (decode path) and the public merge_states
// ---------------------------------------------------------------------------------------

struct MergeParams {
  const int32_t* meta;
  float* ws_o;
  float* ws_lse;
  void* out;
  int64_t o_s0, o_s1;
  float* lse;
  int units_per_request, slot_rows, num_qo_heads;
};

// One warp per (merge item, group of 4 rows of the unit; 8 for head_dim 64).
template <int D, typename T>
__global__ void __launch_bounds__(128) decode_merge_kernel(const MergeParams p) {
  const int32_t* hdr = p.meta;
  const int NM = hdr[H_MERGES];
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  constexpr int RPW = 4 * (128 / D);  // rows per warp
  const int SR = p.slot_rows, nchunk = (SR + RPW - 1) / RPW;
  if (gw >= NM * nchunk) return;
  const int item = gw / nchunk, r0 = (gw % nchunk) * RPW;
  const int32_t* mi = hdr + hdr[H_OFF_MERGES] + 3 * item;
  const int unit = mi[0];
  const int b = unit / p.units_per_request, u = unit % p.units_per_request;
  const int head = u * SR + r0;
  T* dst = static_cast<T*>(p.out) + b * p.o_s0 + head * p.o_s1;
  merge_rows<T, D>(lane, p.ws_o, p.ws_lse, mi[1], mi[2], SR, r0, min(RPW, SR - r0), dst, p.o_s1,
                   p.lse ? p.lse + int64_t(b) * p.num_qo_heads + head : nullptr);
}

template <typename TO>
__device__ __forceinline__ void put(TO* dst, float x);
template <>
__device__ __forceinline__ void put<float>(float* dst, float x) { *dst = x; }
template <>
__device__ __forceinline__ void put<__nv_bfloat16>(__nv_bfloat16* dst, float x) {
  *dst = __float2bfloat16_rn(x);
}
template <>
__device__ __forceinline__ void put<__half>(__half* dst, float x) { *dst = __float2half_rn(x); }

// One warp per (sequence position, head); lanes stride over head_dim in float4 steps.
template <typename TO>
__global__ void __launch_bounds__(128)
    merge_states_kernel(const float* __restrict__ v, const float* __restrict__ s, int64_t seq_len,
                        int num_states, int num_heads, int head_dim, TO* __restrict__ v_out,
                        float* __restrict__ s_out) {
  const int64_t gw = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= seq_len * num_heads) return;
  const int64_t i = gw / num_heads;
  const int h = int(gw % num_heads);
  const float* sp = s + i * num_states * num_heads + h;
  float mx = -INFINITY;
  for (int c = lane; c < num_states; c += 32) mx = fmaxf(mx, sp[int64_t(c) * num_heads]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  const bool live = mx > -INFINITY;
  float tot = 0.f;
  if (live)
    for (int c = 0; c < num_states; ++c) tot += expf(sp[int64_t(c) * num_heads] - mx);
  const float inv = live ? 1.f / tot : 0.f;
  TO* dst = v_out + (i * num_heads + h) * head_dim;
  for (int d = lane * 4; d < head_dim; d += 128) {
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    if (live) {
      for (int c = 0; c < num_states; ++c) {
        const float wgt = expf(sp[int64_t(c) * num_heads] - mx) * inv;
        const float4 x = *reinterpret_cast<const float4*>(
            v + ((i * num_states + c) * num_heads + h) * head_dim + d);
        a[0] += wgt * x.x; a[1] += wgt * x.y; a[2] += wgt * x.z; a[3] += wgt * x.w;
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) put<TO>(dst + d + e, a[e]);
  }
  if (s_out && lane == 0) s_out[i * num_heads + h] = live ? mx + logf(tot) : -INFINITY;
}

template <typename T, int D>
bskv_status launch_decode_t(const bskv_plan* plan, const CUtensorMap& map, DecodeParams& dp,
                            cudaStream_t stream) {
  const int grid = meta_word(plan, H_GRID);
  if (grid <= 0) return BSKV_OK;
  if (meta_word(plan, H_VARIANT) == DECODE_GROUP) {
    const uint32_t sb = group_stage_bytes<D>(dp.heads_per_unit);
    dp.stages = int(kGroupRingBytes / sb) < 8 ? int(kGroupRingBytes / sb) : 8;
    const size_t smem = size_t(dp.stages) * sb + 1024 +
                        size_t(2 * dp.stages + 1) * 8 + 16;
    auto kern = decode_group_kernel<T, D>;
    if (bskv_status s = cuda_check(
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)),
            "decode: cudaFuncSetAttribute"))
      return s;
    kern<<<grid, kGroupThreads, smem, stream>>>(map, dp);
  } else {
    const size_t smem = size_t(kWarps) * kStages * 2 * tile_bytes<D>() + 1024 +
                        size_t(kWarps) * kStages * sizeof(uint64_t);
    auto kern = decode_kernel<T, D>;
    if (bskv_status s = cuda_check(
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)),
            "decode: cudaFuncSetAttribute"))
      return s;
    kern<<<grid, kWarps * 32, smem, stream>>>(map, dp);
  }
  return cuda_check(cudaGetLastError(), "decode kernel launch");
}

template <typename T, int D>
bskv_status launch_merge_t(const bskv_plan* plan, const MergeParams& mp, cudaStream_t stream) {
  const int nm = meta_word(plan, H_MERGES);
  if (nm == 0) return BSKV_OK;
  const int rpw = 4 * (128 / D);
  const int warps = nm * ((mp.slot_rows + rpw - 1) / rpw);
  decode_merge_kernel<D, T><<<(warps + 3) / 4, 128, 0, stream>>>(mp);
  return cuda_check(cudaGetLastError(), "decode merge launch");
}

bskv_status launch_decode_any(const bskv_plan* plan, const CUtensorMap& map, DecodeParams& dp,
                              cudaStream_t st) {
  const bool bf = plan->dtype == BSKV_BF16;
  if (plan->head_dim == 128)
    return bf ? launch_decode_t<__nv_bfloat16, 128>(plan, map, dp, st)
              : launch_decode_t<__half, 128>(plan, map, dp, st);
  return bf ? launch_decode_t<__nv_bfloat16, 64>(plan, map, dp, st)
            : launch_decode_t<__half, 64>(plan, map, dp, st);
}

bskv_status launch_merge_any(const bskv_plan* plan, const MergeParams& mp, cudaStream_t st) {
  const bool bf = plan->dtype == BSKV_BF16;
  if (plan->head_dim == 128)
    return bf ? launch_merge_t<__nv_bfloat16, 128>(plan, mp, st) : launch_merge_t<__half, 128>(plan, mp, st);
  return bf ? launch_merge_t<__nv_bfloat16, 64>(plan, mp, st) : launch_merge_t<__half, 64>(plan, mp, st);
}

// Units per request and query heads per unit (= rows of one partial-state slot).
struct DecodeShape {
  int heads_per_unit, units_per_request, slot_rows;
};

DecodeShape decode_shape(const bskv_plan* plan) {
  const int Hkv = plan->num_kv_heads;
  const int G = meta_word(plan, H_VARIANT) == DECODE_GROUP
                    ? decode_group_heads(Hkv, plan->page_size) : 1;
  return DecodeShape{G, Hkv / G, G * (plan->num_qo_heads / Hkv)};
}

// Float-workspace pointers of a decode plan (partial outputs, then their LSE).
void decode_ws(const bskv_plan* plan, void* float_ws, float** ws_o, float** ws_lse) {
  const int rows = decode_shape(plan).slot_rows;
  const int slots = meta_word(plan, H_SLOTS);
  *ws_o = static_cast<float*>(float_ws);
  *ws_lse = slots ? reinterpret_cast<float*>(static_cast<uint8_t*>(float_ws) +
                                             ((size_t(slots) * rows * plan->head_dim * 4 + 255) &
                                              ~size_t(255)))
                  : nullptr;
}

bskv_status check_decode_ws(const bskv_plan* plan, void* float_ws, size_t float_ws_bytes) {
  if (float_ws_bytes < plan->float_ws_bytes || (plan->float_ws_bytes && !float_ws)) {
    set_error("decode: float workspace of %zu bytes, %zu needed", float_ws_bytes,
              plan->float_ws_bytes);
    return BSKV_ERR_WORKSPACE_TOO_SMALL;
  }
  if (float_ws && !aligned16(float_ws)) {
    set_error("decode: float workspace must be 16-byte aligned");
    return BSKV_ERR_INVALID_ARG;
  }
  return BSKV_OK;
}

// Argument checks shared by the decode entry points, then the kernel parameters and the
// KV tensor map (box: 64 elements x min(page_size, 16) tokens x the unit's kv heads).
bskv_status prepare_decode(const char* who, const bskv_plan* plan, const int32_t* meta,
                           const void* q, const int64_t* q_strides, const void* kv_cache,
                           const int64_t* kv_strides, void* out, const int64_t* out_strides,
                           float* lse, float sm_scale, void* ws, DecodeParams* dp,
                           CUtensorMap* map) {
  if (!q_strides || !kv_strides || !out_strides) { set_error("%s: NULL strides", who); return BSKV_ERR_INVALID_ARG; }
  const int ps = plan->page_size;
  if (!(ps == 8 || ps % 16 == 0)) {
    set_error("%s: page_size %d unsupported (8 or a multiple of 16)", who, ps);
    return BSKV_ERR_UNSUPPORTED;
  }
  const int esz = 2;
  const int Hkv = plan->num_kv_heads, D = plan->head_dim;
  for (int i = 0; i < 4; ++i) {
    if (kv_strides[i] <= 0 || (kv_strides[i] * esz) % 16 != 0) {
      set_error("%s: kv stride %d (%lld elements) must be positive and 16-byte aligned", who, i,
                (long long)kv_strides[i]);
      return BSKV_ERR_INVALID_ARG;
    }
  }
  if ((q_strides[0] * esz) % 4 || (q_strides[1] * esz) % 4 || (out_strides[0] * esz) % 4 ||
      (out_strides[1] * esz) % 4) {
    set_error("%s: q/out strides must be multiples of 2 elements", who);
    return BSKV_ERR_INVALID_ARG;
  }
  if (!q || !kv_cache || !out) { set_error("%s: NULL tensor", who); return BSKV_ERR_INVALID_ARG; }
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out)) { set_error("%s: tensors must be 16-byte aligned", who); return BSKV_ERR_INVALID_ARG; }
  const DecodeShape sh = decode_shape(plan);
  *dp = DecodeParams{};
  dp->meta = meta;
  dp->q = q; dp->q_s0 = q_strides[0]; dp->q_s1 = q_strides[1];
  dp->out = out; dp->o_s0 = out_strides[0]; dp->o_s1 = out_strides[1];
  dp->lse = lse;
  decode_ws(plan, ws, &dp->ws_o, &dp->ws_lse);
  dp->num_kv_heads = Hkv; dp->group = plan->num_qo_heads / Hkv; dp->page_size = ps;
  dp->num_qo_heads = plan->num_qo_heads;
  dp->heads_per_unit = sh.heads_per_unit;
  dp->off_workers = meta_word(plan, H_OFF_WORKERS);
  dp->off_chunks = meta_word(plan, H_OFF_CHUNKS);
  dp->off_merges = meta_word(plan, H_OFF_MERGES);
  dp->off_aux0 = meta_word(plan, H_OFF_AUX0);
  dp->off_aux1 = meta_word(plan, H_OFF_AUX1);
  dp->num_merges = meta_word(plan, H_MERGES);
  dp->off_starts = plan->decode_starts;
  dp->scale_log2 = sm_scale_log2(sm_scale, plan->head_dim);
  if (bskv_status s = status_args(&dp->st)) return s;
  const uint64_t dims[5] = {uint64_t(D), uint64_t(ps), uint64_t(Hkv), 2, uint64_t(plan->num_pages)};
  const uint64_t strides[4] = {uint64_t(kv_strides[3]) * esz, uint64_t(kv_strides[2]) * esz,
                               uint64_t(kv_strides[1]) * esz, uint64_t(kv_strides[0]) * esz};
  const uint32_t box[5] = {64, uint32_t(ps < kTile ? ps : kTile), uint32_t(sh.heads_per_unit), 1, 1};
  const CUtensorMapDataType dt =
      plan->dtype == BSKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return encode_tiled(map, dt, 5, kv_cache, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

MergeParams merge_params(const bskv_plan* plan, const int32_t* meta, const DecodeParams& dp) {
  const DecodeShape sh = decode_shape(plan);
  MergeParams mp{};
  mp.meta = meta;
  mp.ws_o = dp.ws_o; mp.ws_lse = dp.ws_lse;
  mp.out = dp.out; mp.o_s0 = dp.o_s0; mp.o_s1 = dp.o_s1;
  mp.lse = dp.lse;
  mp.units_per_request = sh.units_per_request;
  mp.slot_rows = sh.slot_rows;
  mp.num_qo_heads = plan->num_qo_heads;
  return mp;
}

}  // namespace
}  // namespace bskv

using namespace bskv;

extern "C" bskv_status bskv_run_decode_partial(const bskv_plan* plan, const void* q,
                                       const int64_t* q_strides, const void* kv_cache,
                                       const int64_t* kv_strides, void* out,
                                       const int64_t* out_strides, float* lse, float sm_scale,
                                       void* float_ws, size_t float_ws_bytes, void* stream) {
  BSKV_NVTX_RANGE("bskv_run_decode_partial");
  if (!plan || plan->kind != KIND_DECODE) { set_error("run_decode: not a decode plan"); return BSKV_ERR_INVALID_ARG; }
  if (!plan->meta_dev) { set_error("run_decode: plan not uploaded (bskv_plan_upload)"); return BSKV_ERR_INVALID_ARG; }
  if (bskv_status s = check_decode_ws(plan, float_ws, float_ws_bytes)) return s;
  if (plan->batch == 0) return BSKV_OK;
  DecodeParams dp;
  CUtensorMap map;
  if (bskv_status s = prepare_decode("run_decode", plan, plan->meta_dev, q, q_strides, kv_cache,
                                     kv_strides, out, out_strides, lse, sm_scale, float_ws, &dp, &map))
    return s;
  return launch_decode_any(plan, map, dp, static_cast<cudaStream_t>(stream));
}

extern "C" bskv_status bskv_decode_merge(const bskv_plan* plan, void* out,
                                         const int64_t* out_strides, float* lse,
                                         void* float_ws, size_t float_ws_bytes, void* stream) {
  BSKV_NVTX_RANGE("bskv_decode_merge");
  if (!plan || plan->kind != KIND_DECODE) { set_error("decode_merge: not a decode plan"); return BSKV_ERR_INVALID_ARG; }
  if (!plan->meta_dev) { set_error("decode_merge: plan not uploaded (bskv_plan_upload)"); return BSKV_ERR_INVALID_ARG; }
  if (!out_strides) { set_error("decode_merge: NULL strides"); return BSKV_ERR_INVALID_ARG; }
  if (bskv_status s = check_decode_ws(plan, float_ws, float_ws_bytes)) return s;
  if (meta_word(plan, H_MERGES) == 0) return BSKV_OK;
  if (!out || !aligned16(out)) { set_error("decode_merge: out must be a 16-byte aligned tensor"); return BSKV_ERR_INVALID_ARG; }
  if ((out_strides[0] * 2) % 4 || (out_strides[1] * 2) % 4) { set_error("decode_merge: out strides must be multiples of 2 elements"); return BSKV_ERR_INVALID_ARG; }
  DecodeParams dp{};
  decode_ws(plan, float_ws, &dp.ws_o, &dp.ws_lse);
  dp.out = out; dp.o_s0 = out_strides[0]; dp.o_s1 = out_strides[1];
  dp.lse = lse;
  return launch_merge_any(plan, merge_params(plan, plan->meta_dev, dp),
                          static_cast<cudaStream_t>(stream));
}

extern "C" bskv_status bskv_run_decode(const bskv_plan* plan, const void* q,
                                       const int64_t* q_strides, const void* kv_cache,
                                       const int64_t* kv_strides, void* out,
                                       const int64_t* out_strides, float* lse, float sm_scale,
                                       void* float_ws, size_t float_ws_bytes, void* stream) {
  BSKV_NVTX_RANGE("bskv_run_decode");
  if (!plan || plan->kind != KIND_DECODE) { set_error("run_decode: not a decode plan"); return BSKV_ERR_INVALID_ARG; }
  if (!plan->meta_dev) { set_error("run_decode: plan not uploaded (bskv_plan_upload)"); return BSKV_ERR_INVALID_ARG; }
  if (bskv_status s = check_decode_ws(plan, float_ws, float_ws_bytes)) return s;
  if (plan->batch == 0) return BSKV_OK;
  DecodeParams dp;
  CUtensorMap map;
  if (bskv_status s = prepare_decode("run_decode", plan, plan->meta_dev, q, q_strides, kv_cache,
                                     kv_strides, out, out_strides, lse, sm_scale, float_ws, &dp, &map))
    return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool merges = meta_word(plan, H_MERGES) > 0;
  if (meta_word(plan, H_GRID) == 0)  // no tokens at all: only zero-filling is left
    return merges ? launch_merge_any(plan, merge_params(plan, plan->meta_dev, dp), st) : BSKV_OK;
  if (merges && plan->max_merge_count > kFusedMergeMaxPieces) {
    // many pieces per unit: the attention kernel, then the merge kernel
    if (bskv_status s = launch_decode_any(plan, map, dp, st)) return s;
    return launch_merge_any(plan, merge_params(plan, plan->meta_dev, dp), st);
  }
  if (merges) {
    if (!plan->counters_dev) { set_error("run_decode: plan has no merge counters (bskv_plan_upload)"); return BSKV_ERR_INVALID_ARG; }
    dp.counters = plan->counters_dev;  // split units are merged inside the decode kernel
  }
  return launch_decode_any(plan, map, dp, st);
}

extern "C" bskv_status bskv_merge_states(const float* v, const float* s, int64_t seq_len,
                                         int32_t num_states, int32_t num_heads,
                                         int32_t head_dim, void* v_out, int32_t out_dtype,
                                         float* s_out, void* stream) {
  BSKV_NVTX_RANGE("bskv_merge_states");
  if (seq_len < 0 || num_states < 1 || num_heads < 1 || head_dim < 4 || head_dim % 4) {
    set_error("merge_states: seq_len=%lld num_states=%d num_heads=%d head_dim=%d", (long long)seq_len, num_states, num_heads, head_dim);
    return BSKV_ERR_INVALID_ARG;
  }
  if (seq_len == 0) return BSKV_OK;
  if (!v || !s || !v_out) { set_error("merge_states: NULL tensor"); return BSKV_ERR_INVALID_ARG; }
  if (!aligned16(v)) { set_error("merge_states: v must be 16-byte aligned"); return BSKV_ERR_INVALID_ARG; }
  const int64_t warps = seq_len * num_heads;
  const int64_t blocks = (warps + 3) / 4;
  if (blocks > INT32_MAX) { set_error("merge_states: too large"); return BSKV_ERR_UNSUPPORTED; }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (out_dtype) {
    case BSKV_FP32:
      merge_states_kernel<float><<<unsigned(blocks), 128, 0, st>>>(v, s, seq_len, num_states, num_heads, head_dim, static_cast<float*>(v_out), s_out);
      break;
    case BSKV_BF16:
      merge_states_kernel<__nv_bfloat16><<<unsigned(blocks), 128, 0, st>>>(v, s, seq_len, num_states, num_heads, head_dim, static_cast<__nv_bfloat16*>(v_out), s_out);
      break;
    case BSKV_FP16:
      merge_states_kernel<__half><<<unsigned(blocks), 128, 0, st>>>(v, s, seq_len, num_states, num_heads, head_dim, static_cast<__half*>(v_out), s_out);
      break;
    default:
      set_error("merge_states: out dtype %s unsupported", dtype_name(out_dtype));
      return BSKV_ERR_UNSUPPORTED;
  }
  return cuda_check(cudaGetLastError(), "merge_states launch");
}

// ---------------------------------------------------------------------------------------
// Allocation-free paged decode
//
// For callers that cannot allocate device memory: code embedded in a host framework that
// hands it only tensors and a stream (no allocator of its own), processes whose device
// memory is fully reserved by another allocator, and latency-critical loops where a
// cudaMalloc/cudaFree (which can synchronise the device) is not acceptable. The plan
// metadata and the split-KV partial states live in two file-scope device arrays instead
// of caller workspaces. Every GPU that loads the library keeps them (9 MiB) until exit.
// ---------------------------------------------------------------------------------------
namespace bskv {
namespace {

constexpr size_t kNoAllocMetaWords = size_t(1) << 18;     // 1 MiB of plan metadata
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB of split-KV partials
static __device__ __align__(256) int32_t g_noalloc_meta[kNoAllocMetaWords];
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocPtrs {
  int32_t* meta = nullptr;
  uint8_t* scratch = nullptr;
};
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
NoAllocPtrs g_noalloc_ptrs[kNoAllocMaxDevices];

// Device addresses of the two arrays on the current device, looked up once per device.
// In host code the arrays' names are host-side stand-ins, never device addresses.
bskv_status noalloc_ptrs(NoAllocPtrs* out) {
  int d = 0;
  if (bskv_status s = cuda_check(cudaGetDevice(&d), "cudaGetDevice")) return s;
  if (d < 0 || d >= kNoAllocMaxDevices) {
    set_error("run_decode_noalloc: device ordinal %d too large", d);
    return BSKV_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocPtrs& p = g_noalloc_ptrs[d];
  if (!p.meta) {
    void* m = nullptr;
    void* s = nullptr;
    if (bskv_status e = cuda_check(cudaGetSymbolAddress(&m, g_noalloc_meta),
                                   "run_decode_noalloc: cudaGetSymbolAddress(meta)"))
      return e;
    if (bskv_status e = cuda_check(cudaGetSymbolAddress(&s, g_noalloc_scratch),
                                   "run_decode_noalloc: cudaGetSymbolAddress(scratch)"))
      return e;
    p.meta = static_cast<int32_t*>(m);
    p.scratch = static_cast<uint8_t*>(s);
  }
  *out = p;
  return BSKV_OK;
}

}  // namespace
}  // namespace bskv

extern "C" bskv_status bskv_run_decode_noalloc(const bskv_plan* plan, const void* q,
                                               const int64_t* q_strides, const void* kv_cache,
                                               const int64_t* kv_strides, void* out,
                                               const int64_t* out_strides, float* lse,
                                               float sm_scale, void* stream) {
  BSKV_NVTX_RANGE("bskv_run_decode_noalloc");
  if (!plan || plan->kind != KIND_DECODE) { set_error("run_decode_noalloc: not a decode plan"); return BSKV_ERR_INVALID_ARG; }
  const size_t meta_words = plan->meta.size();
  if (meta_words > kNoAllocMetaWords || plan->float_ws_bytes > kNoAllocScratchBytes) {
    set_error("run_decode_noalloc: plan needs %zu metadata bytes and %zu scratch bytes; the "
              "static arrays hold %zu and %zu (use bskv_run_decode with caller workspaces)",
              meta_words * 4, plan->float_ws_bytes, kNoAllocMetaWords * 4, kNoAllocScratchBytes);
    return BSKV_ERR_UNSUPPORTED;
  }
  if (plan->batch == 0) return BSKV_OK;
  NoAllocPtrs st_ptrs;
  if (bskv_status s = noalloc_ptrs(&st_ptrs)) return s;
  DecodeParams dp;
  CUtensorMap map;
  if (bskv_status s = prepare_decode("run_decode_noalloc", plan, st_ptrs.meta, q, q_strides,
                                     kv_cache, kv_strides, out, out_strides, lse, sm_scale,
                                     st_ptrs.scratch, &dp, &map))
    return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The metadata is copied into the static array on the caller's stream; nothing in the
  // scratch array has to start at zero (every partial state is written before it is read).
  if (bskv_status s = cuda_check(cudaMemcpyAsync(st_ptrs.meta, plan->meta.data(), meta_words * 4,
                                                 cudaMemcpyHostToDevice, st),
                                 "run_decode_noalloc: metadata copy"))
    return s;
  bskv_status s = launch_decode_any(plan, map, dp, st);
  if (s == BSKV_OK) s = launch_merge_any(plan, merge_params(plan, st_ptrs.meta, dp), st);
  return s;
}
