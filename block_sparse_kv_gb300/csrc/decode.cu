// Paged-KV batch decode with split-KV, and the LSE merge of attention states.
//
// Method: "FlashInfer" agent-skill summary, KV-Cache Formats (paged KV-cache: kv_cache
// (num_pages, 2, num_kv_heads, page_size, head_dim), kv_indptr, kv_indices,
// kv_last_page_len); "flashinfer.sparse" BlockSparseAttentionWrapper.__init__ (a float
// workspace holds the intermediate results of the split-k algorithm); FlashInfer
// cascade.rst (merge_state / merge_states).
//
// GB300 design. Decode reads every K/V byte once (O(1) flop per byte), so the kernel is an
// HBM stream: one CTA per SM with 8 independent worker warps. Each warp owns a contiguous
// range of 16-token tiles (the plan's linear split-KV partition) and a private 3-stage ring
// in shared memory filled by TMA tensor copies (128-byte swizzle) straight from the pages;
// lane 0 issues the copies, the whole warp waits on the stage's mbarrier. The up-to-16
// query heads that share a kv head form the M=16 rows of mma.sync m16n8k16 (bf16/fp16 in,
// fp32 accumulate): S = Q K^T, online softmax in registers (exp2), O += P V with P reused
// from the S accumulators. A unit that is split over several workers writes its normalised
// partial output and LSE to the float workspace; the merge kernel then combines them.
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

struct DecodeParams {
  const int32_t* meta;
  const void* q;
  int64_t q_s0, q_s1;
  void* out;
  int64_t o_s0, o_s1;
  float* lse;
  float* ws_o;
  float* ws_lse;
  int num_kv_heads, group, page_size, num_qo_heads;
  float scale_log2;
  StatusArgs st;
};

template <int D>
__host__ __device__ constexpr int tile_bytes() {
  return (D / 64) * kPanelBytes;
}

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
        tma_load_5d(kdst + hf * kPanelBytes, &kv_map, hf * 64, s, kvh, 0, page, &bars[stage]);
        tma_load_5d(vdst + hf * kPanelBytes, &kv_map, hf * 64, s, kvh, 1, page, &bars[stage]);
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
          tma_load_5d(kdst + hf * kPanelBytes + k * piece_bytes, &kv_map, hf * 64, 0, kvh, 0,
                      page, &bars[stage]);
          tma_load_5d(vdst + hf * kPanelBytes + k * piece_bytes, &kv_map, hf * 64, 0, kvh, 1,
                      page, &bars[stage]);
        }
      }
    }
  };
  auto ntiles = [&](int c) {
    const int4 ch = chunks[c];
    return (ch.z - ch.y + kTile - 1) / kTile;
  };

  // Producer cursor (pc, pt) runs kStages tiles ahead of the consumer cursor (cc, ct).
  int pc = c0, pt = 0;
  auto advance = [&](int& c, int& t) {
    if (++t == ntiles(c)) {
      ++c;
      t = 0;
    }
  };
  uint32_t issued = 0, consumed = 0;
  for (int s = 0; s < kStages && pc < c1; ++s) {
    if (lane == 0) issue(s, pc, pt);
    ++issued;
    advance(pc, pt);
  }

  using Mma = MmaOp<T>;
  const int r0 = lane >> 2, r1 = r0 + 8, cq = lane & 3;
  uint32_t qa[D / 16][4];
  float o[D / 8][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  bool ok = true;
  int cc = c0, ct = 0;
  while (cc < c1) {
    const int4 ch = chunks[cc];
    const int b = ch.x / Hkv, kvh = ch.x % Hkv;
    if (ct == 0) {
      const T* qb = static_cast<const T*>(p.q) + b * p.q_s0 + int64_t(kvh) * g * p.q_s1;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int d0 = kk * 16 + 2 * cq;
        qa[kk][0] = r0 < g ? *reinterpret_cast<const uint32_t*>(qb + r0 * p.q_s1 + d0) : 0u;
        qa[kk][1] = r1 < g ? *reinterpret_cast<const uint32_t*>(qb + r1 * p.q_s1 + d0) : 0u;
        qa[kk][2] = r0 < g ? *reinterpret_cast<const uint32_t*>(qb + r0 * p.q_s1 + d0 + 8) : 0u;
        qa[kk][3] = r1 < g ? *reinterpret_cast<const uint32_t*>(qb + r1 * p.q_s1 + d0 + 8) : 0u;
      }
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
    uint8_t* kt = ring + stage * kStageBytes;
    uint8_t* vt = kt + kTileBytes;
    const int tok0 = ch.y + ct * kTile;
    const int valid = min(kTile, ch.z - tok0);
    if (valid < kTile) {
      // Rows past the unit's end hold whatever the pages hold there (or stale data);
      // zero the V rows so that 0 * garbage cannot reach the output.
      for (int i = lane; i < (kTile - valid) * (D / 64) * 8; i += 32) {
        const int hf = i / ((kTile - valid) * 8);
        const int rem = i % ((kTile - valid) * 8);
        const int row = valid + rem / 8;
        *reinterpret_cast<uint4*>(vt + hf * kPanelBytes + row * 128 + (rem % 8) * 16) =
            make_uint4(0, 0, 0, 0);
      }
      __syncwarp();
    }
    // S = Q K^T over the tile's 16 tokens (two n8 tiles).
    float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int mi = lane >> 3;
      const int trow = (mi >> 1) * 8 + (lane & 7);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int dim = kk * 16 + (mi & 1) * 8;
        const uint32_t addr =
            smem_u32(kt + (dim / 64) * kPanelBytes) + swz(trow, (dim % 64) / 8, 128);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(addr, b0, b1, b2, b3);
        Mma::run(s[0], qa[kk], b0, b1);
        Mma::run(s[1], qa[kk], b2, b3);
      }
    }
    // Online softmax (base 2) on rows r0 and r1.
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int col = nt * 8 + 2 * cq + (e & 1);
        const float x = s[nt][e] * p.scale_log2;
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
    // O += P V.
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
            smem_u32(vt + (dim / 64) * kPanelBytes) + swz(trow, (dim % 64) / 8, 128);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(addr, b0, b1, b2, b3);
        Mma::run(o[2 * dd], pa, b0, b1);
        Mma::run(o[2 * dd + 1], pa, b2, b3);
      }
    }
    ++consumed;
    __syncwarp();
    if (pc < c1) {
      if (lane == 0) {
        fence_proxy_async_smem();
        issue(stage, pc, pt);
      }
      ++issued;
      advance(pc, pt);
    }
    if (++ct == ntiles(cc)) {
      // Finish the chunk: normalise and write the output rows or the partial state.
      float lt0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
      lt0 += __shfl_xor_sync(0xffffffffu, lt0, 2);
      float lt1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
      lt1 += __shfl_xor_sync(0xffffffffu, lt1, 2);
      const float inv0 = 1.f / lt0, inv1 = 1.f / lt1;
      const float lse0 = (m0 + __log2f(lt0)) * kLn2, lse1 = (m1 + __log2f(lt1)) * kLn2;
      const int slot = ch.w;
      if (slot < 0) {
        T* ob = static_cast<T*>(p.out) + b * p.o_s0 + int64_t(kvh) * g * p.o_s1;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
          const int d = n * 8 + 2 * cq;
          if (r0 < g)
            *reinterpret_cast<uint32_t*>(ob + r0 * p.o_s1 + d) =
                Mma::pack(o[n][0] * inv0, o[n][1] * inv0);
          if (r1 < g)
            *reinterpret_cast<uint32_t*>(ob + r1 * p.o_s1 + d) =
                Mma::pack(o[n][2] * inv1, o[n][3] * inv1);
        }
        if (p.lse && cq == 0) {
          float* lb = p.lse + int64_t(b) * p.num_qo_heads + kvh * g;
          if (r0 < g) lb[r0] = lse0;
          if (r1 < g) lb[r1] = lse1;
        }
      } else {
        float* wo = p.ws_o + int64_t(slot) * g * D;
#pragma unroll
        for (int n = 0; n < D / 8; ++n) {
          const int d = n * 8 + 2 * cq;
          if (r0 < g)
            *reinterpret_cast<float2*>(wo + r0 * D + d) = make_float2(o[n][0] * inv0, o[n][1] * inv0);
          if (r1 < g)
            *reinterpret_cast<float2*>(wo + r1 * D + d) = make_float2(o[n][2] * inv1, o[n][3] * inv1);
        }
        if (cq == 0) {
          if (r0 < g) p.ws_lse[slot * g + r0] = lse0;
          if (r1 < g) p.ws_lse[slot * g + r1] = lse1;
        }
      }
      ++cc;
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
// merge of split-KV partial states (decode path) and the public merge_states
// ---------------------------------------------------------------------------------------

struct MergeParams {
  const int32_t* meta;
  float* ws_o;
  float* ws_lse;
  void* out;
  int64_t o_s0, o_s1;
  float* lse;
  int num_kv_heads, group, num_qo_heads;
};

template <int D, typename T>
__global__ void __launch_bounds__(128) decode_merge_kernel(const MergeParams p) {
  const int32_t* hdr = p.meta;
  const int NM = hdr[H_MERGES];
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int g = p.group;
  if (gw >= NM * g) return;
  const int item = gw / g, r = gw % g;
  const int32_t* mi = hdr + hdr[H_OFF_MERGES] + 3 * item;
  const int unit = mi[0], first = mi[1], count = mi[2];
  const int b = unit / p.num_kv_heads, kvh = unit % p.num_kv_heads;
  const int head = kvh * g + r;
  constexpr int V = D / 32;  // values per lane
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  float lse_out = -INFINITY;
  if (count > 0) {
    float mx = -INFINITY;
    for (int c = lane; c < count; c += 32) mx = fmaxf(mx, p.ws_lse[(first + c) * g + r]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float tot = 0.f;
    for (int c = 0; c < count; ++c) {
      const float wgt = expf(p.ws_lse[(first + c) * g + r] - mx);
      tot += wgt;
      const float* src = p.ws_o + (int64_t(first + c) * g + r) * D + lane * V;
      if constexpr (V == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        acc[0] += wgt * x.x; acc[1] += wgt * x.y; acc[2] += wgt * x.z; acc[3] += wgt * x.w;
      } else {
        const float2 x = *reinterpret_cast<const float2*>(src);
        acc[0] += wgt * x.x; acc[1] += wgt * x.y;
      }
    }
    const float inv = 1.f / tot;
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] *= inv;
    lse_out = mx + logf(tot);
  }
  T* dst = static_cast<T*>(p.out) + b * p.o_s0 + head * p.o_s1 + lane * V;
#pragma unroll
  for (int i = 0; i < V; i += 2)
    *reinterpret_cast<uint32_t*>(dst + i) = MmaOp<T>::pack(acc[i], acc[i + 1]);
  if (p.lse && lane == 0) p.lse[int64_t(b) * p.num_qo_heads + head] = lse_out;
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
  const size_t smem = size_t(kWarps) * kStages * 2 * tile_bytes<D>() + 1024 +
                      size_t(kWarps) * kStages * sizeof(uint64_t);
  if (grid > 0) {
    auto kern = decode_kernel<T, D>;
    if (bskv_status s = cuda_check(
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)),
            "decode: cudaFuncSetAttribute"))
      return s;
    kern<<<grid, kWarps * 32, smem, stream>>>(map, dp);
    if (bskv_status s = cuda_check(cudaGetLastError(), "decode kernel launch")) return s;
  }
  return BSKV_OK;
}

template <typename T, int D>
bskv_status launch_merge_t(const bskv_plan* plan, const MergeParams& mp, cudaStream_t stream) {
  const int nm = meta_word(plan, H_MERGES);
  if (nm == 0) return BSKV_OK;
  const int warps = nm * mp.group;
  decode_merge_kernel<D, T><<<(warps + 3) / 4, 128, 0, stream>>>(mp);
  return cuda_check(cudaGetLastError(), "decode merge launch");
}

// Float-workspace pointers of a decode plan (partial outputs, then their LSE).
void decode_ws(const bskv_plan* plan, void* float_ws, float** ws_o, float** ws_lse) {
  const int g = plan->num_qo_heads / plan->num_kv_heads;
  const int slots = meta_word(plan, H_SLOTS);
  *ws_o = static_cast<float*>(float_ws);
  *ws_lse = slots ? reinterpret_cast<float*>(static_cast<uint8_t*>(float_ws) +
                                             ((size_t(slots) * g * plan->head_dim * 4 + 255) &
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

}  // namespace
}  // namespace bskv

using namespace bskv;

extern "C" bskv_status bskv_run_decode_partial(const bskv_plan* plan, const void* q,
                                       const int64_t* q_strides, const void* kv_cache,
                                       const int64_t* kv_strides, void* out,
                                       const int64_t* out_strides, float* lse, float sm_scale,
                                       void* float_ws, size_t float_ws_bytes, void* stream) {
  if (!plan || plan->kind != KIND_DECODE) { set_error("run_decode: not a decode plan"); return BSKV_ERR_INVALID_ARG; }
  if (!plan->meta_dev) { set_error("run_decode: plan not uploaded (bskv_plan_upload)"); return BSKV_ERR_INVALID_ARG; }
  if (!q_strides || !kv_strides || !out_strides) { set_error("run_decode: NULL strides"); return BSKV_ERR_INVALID_ARG; }
  const int ps = plan->page_size;
  if (!(ps == 8 || ps % 16 == 0)) {
    set_error("run_decode: page_size %d unsupported (8 or a multiple of 16)", ps);
    return BSKV_ERR_UNSUPPORTED;
  }
  const int esz = 2;
  const int Hkv = plan->num_kv_heads, D = plan->head_dim;
  const int64_t* ks = kv_strides;
  for (int i = 0; i < 4; ++i) {
    if (ks[i] <= 0 || (ks[i] * esz) % 16 != 0) {
      set_error("run_decode: kv stride %d (%lld elements) must be positive and 16-byte aligned", i, (long long)ks[i]);
      return BSKV_ERR_INVALID_ARG;
    }
  }
  if ((q_strides[0] * esz) % 4 || (q_strides[1] * esz) % 4 || (out_strides[0] * esz) % 4 ||
      (out_strides[1] * esz) % 4) {
    set_error("run_decode: q/out strides must be multiples of 2 elements");
    return BSKV_ERR_INVALID_ARG;
  }
  if (plan->batch > 0 && (!q || !kv_cache || !out)) { set_error("run_decode: NULL tensor"); return BSKV_ERR_INVALID_ARG; }
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out)) { set_error("run_decode: tensors must be 16-byte aligned"); return BSKV_ERR_INVALID_ARG; }
  if (bskv_status s = check_decode_ws(plan, float_ws, float_ws_bytes)) return s;
  if (plan->batch == 0) return BSKV_OK;
  DecodeParams dp{};
  dp.meta = plan->meta_dev;
  dp.q = q; dp.q_s0 = q_strides[0]; dp.q_s1 = q_strides[1];
  dp.out = out; dp.o_s0 = out_strides[0]; dp.o_s1 = out_strides[1];
  dp.lse = lse;
  const int g = plan->num_qo_heads / Hkv;
  decode_ws(plan, float_ws, &dp.ws_o, &dp.ws_lse);
  dp.num_kv_heads = Hkv; dp.group = g; dp.page_size = ps; dp.num_qo_heads = plan->num_qo_heads;
  dp.scale_log2 = sm_scale * 1.4426950408889634f;
  if (bskv_status s = status_args(&dp.st)) return s;
  CUtensorMap map;
  const uint64_t dims[5] = {uint64_t(D), uint64_t(ps), uint64_t(Hkv), 2, uint64_t(plan->num_pages)};
  const uint64_t strides[4] = {uint64_t(ks[3]) * esz, uint64_t(ks[2]) * esz, uint64_t(ks[1]) * esz,
                               uint64_t(ks[0]) * esz};
  const uint32_t box[5] = {64, uint32_t(ps < kTile ? ps : kTile), 1, 1, 1};
  const CUtensorMapDataType dt =
      plan->dtype == BSKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (bskv_status s = encode_tiled(&map, dt, 5, kv_cache, dims, strides, box,
                                   CU_TENSOR_MAP_SWIZZLE_128B))
    return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (plan->dtype == BSKV_BF16) {
    return D == 128 ? launch_decode_t<__nv_bfloat16, 128>(plan, map, dp, st)
                    : launch_decode_t<__nv_bfloat16, 64>(plan, map, dp, st);
  }
  return D == 128 ? launch_decode_t<__half, 128>(plan, map, dp, st)
                  : launch_decode_t<__half, 64>(plan, map, dp, st);
}

extern "C" bskv_status bskv_decode_merge(const bskv_plan* plan, void* out,
                                         const int64_t* out_strides, float* lse,
                                         void* float_ws, size_t float_ws_bytes, void* stream) {
  if (!plan || plan->kind != KIND_DECODE) { set_error("decode_merge: not a decode plan"); return BSKV_ERR_INVALID_ARG; }
  if (!plan->meta_dev) { set_error("decode_merge: plan not uploaded (bskv_plan_upload)"); return BSKV_ERR_INVALID_ARG; }
  if (!out_strides) { set_error("decode_merge: NULL strides"); return BSKV_ERR_INVALID_ARG; }
  if (bskv_status s = check_decode_ws(plan, float_ws, float_ws_bytes)) return s;
  if (meta_word(plan, H_MERGES) == 0) return BSKV_OK;
  if (!out || !aligned16(out)) { set_error("decode_merge: out must be a 16-byte aligned tensor"); return BSKV_ERR_INVALID_ARG; }
  if ((out_strides[0] * 2) % 4 || (out_strides[1] * 2) % 4) { set_error("decode_merge: out strides must be multiples of 2 elements"); return BSKV_ERR_INVALID_ARG; }
  MergeParams mp{};
  mp.meta = plan->meta_dev;
  decode_ws(plan, float_ws, &mp.ws_o, &mp.ws_lse);
  mp.out = out; mp.o_s0 = out_strides[0]; mp.o_s1 = out_strides[1];
  mp.lse = lse;
  mp.num_kv_heads = plan->num_kv_heads;
  mp.group = plan->num_qo_heads / plan->num_kv_heads;
  mp.num_qo_heads = plan->num_qo_heads;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool bf = plan->dtype == BSKV_BF16;
  if (plan->head_dim == 128)
    return bf ? launch_merge_t<__nv_bfloat16, 128>(plan, mp, st) : launch_merge_t<__half, 128>(plan, mp, st);
  return bf ? launch_merge_t<__nv_bfloat16, 64>(plan, mp, st) : launch_merge_t<__half, 64>(plan, mp, st);
}

extern "C" bskv_status bskv_run_decode(const bskv_plan* plan, const void* q,
                                       const int64_t* q_strides, const void* kv_cache,
                                       const int64_t* kv_strides, void* out,
                                       const int64_t* out_strides, float* lse, float sm_scale,
                                       void* float_ws, size_t float_ws_bytes, void* stream) {
  if (bskv_status s = bskv_run_decode_partial(plan, q, q_strides, kv_cache, kv_strides, out,
                                              out_strides, lse, sm_scale, float_ws,
                                              float_ws_bytes, stream))
    return s;
  return bskv_decode_merge(plan, out, out_strides, lse, float_ws, float_ws_bytes, stream);
}

extern "C" bskv_status bskv_merge_states(const float* v, const float* s, int64_t seq_len,
                                         int32_t num_states, int32_t num_heads,
                                         int32_t head_dim, void* v_out, int32_t out_dtype,
                                         float* s_out, void* stream) {
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
  if (!plan || plan->kind != KIND_DECODE) { set_error("run_decode_noalloc: not a decode plan"); return BSKV_ERR_INVALID_ARG; }
  const size_t meta_words = plan->meta.size();
  if (meta_words > kNoAllocMetaWords || plan->float_ws_bytes > kNoAllocScratchBytes) {
    set_error("run_decode_noalloc: plan needs %zu metadata bytes and %zu scratch bytes; the "
              "static arrays hold %zu and %zu (use bskv_run_decode with caller workspaces)",
              meta_words * 4, plan->float_ws_bytes, kNoAllocMetaWords * 4, kNoAllocScratchBytes);
    return BSKV_ERR_UNSUPPORTED;
  }
  if (!q_strides || !kv_strides || !out_strides) { set_error("run_decode_noalloc: NULL strides"); return BSKV_ERR_INVALID_ARG; }
  const int ps = plan->page_size;
  if (!(ps == 8 || ps % 16 == 0)) {
    set_error("run_decode_noalloc: page_size %d unsupported (8 or a multiple of 16)", ps);
    return BSKV_ERR_UNSUPPORTED;
  }
  const int esz = 2;
  const int Hkv = plan->num_kv_heads, D = plan->head_dim;
  for (int i = 0; i < 4; ++i) {
    if (kv_strides[i] <= 0 || (kv_strides[i] * esz) % 16 != 0) {
      set_error("run_decode_noalloc: kv stride %d must be positive and 16-byte aligned", i);
      return BSKV_ERR_INVALID_ARG;
    }
  }
  if ((q_strides[0] * esz) % 4 || (q_strides[1] * esz) % 4 || (out_strides[0] * esz) % 4 ||
      (out_strides[1] * esz) % 4) {
    set_error("run_decode_noalloc: q/out strides must be multiples of 2 elements");
    return BSKV_ERR_INVALID_ARG;
  }
  if (plan->batch == 0) return BSKV_OK;
  if (!q || !kv_cache || !out) { set_error("run_decode_noalloc: NULL tensor"); return BSKV_ERR_INVALID_ARG; }
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out)) { set_error("run_decode_noalloc: tensors must be 16-byte aligned"); return BSKV_ERR_INVALID_ARG; }
  NoAllocPtrs st_ptrs;
  if (bskv_status s = noalloc_ptrs(&st_ptrs)) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The metadata is copied into the static array on the caller's stream; nothing in the
  // scratch array has to start at zero (every partial state is written before it is read).
  if (bskv_status s = cuda_check(cudaMemcpyAsync(st_ptrs.meta, plan->meta.data(), meta_words * 4,
                                                 cudaMemcpyHostToDevice, st),
                                 "run_decode_noalloc: metadata copy"))
    return s;
  DecodeParams dp{};
  dp.meta = st_ptrs.meta;
  dp.q = q; dp.q_s0 = q_strides[0]; dp.q_s1 = q_strides[1];
  dp.out = out; dp.o_s0 = out_strides[0]; dp.o_s1 = out_strides[1];
  dp.lse = lse;
  const int g = plan->num_qo_heads / Hkv;
  decode_ws(plan, st_ptrs.scratch, &dp.ws_o, &dp.ws_lse);
  dp.num_kv_heads = Hkv; dp.group = g; dp.page_size = ps; dp.num_qo_heads = plan->num_qo_heads;
  dp.scale_log2 = sm_scale * 1.4426950408889634f;
  if (bskv_status s = status_args(&dp.st)) return s;
  CUtensorMap map;
  const uint64_t dims[5] = {uint64_t(D), uint64_t(ps), uint64_t(Hkv), 2, uint64_t(plan->num_pages)};
  const uint64_t strides[4] = {uint64_t(kv_strides[3]) * esz, uint64_t(kv_strides[2]) * esz,
                               uint64_t(kv_strides[1]) * esz, uint64_t(kv_strides[0]) * esz};
  const uint32_t box[5] = {64, uint32_t(ps < kTile ? ps : kTile), 1, 1, 1};
  const CUtensorMapDataType dt =
      plan->dtype == BSKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  if (bskv_status s = encode_tiled(&map, dt, 5, kv_cache, dims, strides, box,
                                   CU_TENSOR_MAP_SWIZZLE_128B))
    return s;
  MergeParams mp{};
  mp.meta = st_ptrs.meta;
  mp.ws_o = dp.ws_o; mp.ws_lse = dp.ws_lse;
  mp.out = out; mp.o_s0 = out_strides[0]; mp.o_s1 = out_strides[1];
  mp.lse = lse;
  mp.num_kv_heads = Hkv; mp.group = g; mp.num_qo_heads = plan->num_qo_heads;
  const bool bf = plan->dtype == BSKV_BF16;
  bskv_status s = BSKV_OK;
  if (D == 128) {
    s = bf ? launch_decode_t<__nv_bfloat16, 128>(plan, map, dp, st) : launch_decode_t<__half, 128>(plan, map, dp, st);
    if (s == BSKV_OK)
      s = bf ? launch_merge_t<__nv_bfloat16, 128>(plan, mp, st) : launch_merge_t<__half, 128>(plan, mp, st);
  } else {
    s = bf ? launch_decode_t<__nv_bfloat16, 64>(plan, map, dp, st) : launch_decode_t<__half, 64>(plan, map, dp, st);
    if (s == BSKV_OK)
      s = bf ? launch_merge_t<__nv_bfloat16, 64>(plan, mp, st) : launch_merge_t<__half, 64>(plan, mp, st);
  }
  return s;
}
