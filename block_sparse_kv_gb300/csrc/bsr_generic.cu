// BSR block-sparse attention, general shapes (any R, C; head_dim 64 or 128).
//
// Method: "flashinfer.sparse - FlashInfer 0.7.4 documentation", BlockSparseAttentionWrapper:
// the mask is a bsr_matrix with indptr (MB+1), indices (< NB = N/C), block size R x C, any
// (R, C); num_qo_heads a multiple of num_kv_heads (GQA); causal is a token-level mask;
// run() returns out [M, Hq, D] and optionally lse [M, Hq].
//
// Design: persistent CTAs of 4 warps; each unit is (row block i, kv head h, 64-row tile),
// its 64 rows being the (token, query head) pairs of row block i that share kv head h, so
// every K/V tile loaded serves all grouped heads. K/V tiles of 32 tokens (16 for blocks of at
// most 16 columns) are staged with cp.async into a double-buffered, XOR-swizzled
// shared-memory tile and consumed by mma.sync m16n8k16 (fp32 accumulate) with an online
// softmax, FlashAttention-2 style.
// The tensor-core (tcgen05) kernel covers the large R = C = 64 shapes; this one covers
// everything else.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "launch.h"

namespace bskv {
namespace {

using namespace dev;

struct BsrParams {
  const int32_t* meta;
  const void* q;
  int64_t q_s0, q_s1;
  const void* k;
  int64_t k_s0, k_s1;
  const void* v;
  int64_t v_s0, v_s1;
  // paged KV cache (paged prefill): element (page, K/V, kv head, slot) at these strides
  const void* kv;
  int64_t kv_s0, kv_s1, kv_s2, kv_s3;
  void* out;
  int64_t o_s0, o_s1;
  float* lse;
  int64_t lse_st, lse_sh;  // lse element strides of a token and of a head
  int M, N, R, C, Hq, Hkv, group, causal;
  // per-block token mask, bits packed little-endian within bytes over (nnz, R, C); NULL =
  // every listed block is full
  const uint8_t* mask;
  float scale_log2;
  StatusArgs st;
};

// Key tokens per tile (KT): 32, two 16-key sub-blocks per online-softmax update, or 16 for
// blocks of at most 16 columns (a 32-key tile would be half empty there).
static_assert(kBsrVarTile == 32, "variable-block plans list 32-key tiles");

// kMode 0: block-sparse (row block, listed column blocks); 1: variable blocks and 2: paged
// prefill, whose unit rows and key tiles come from the metadata lists (paged tiles also
// name their page and first slot, and causal is aligned per request).
template <typename T, int D, int kMode, int kKT>
__global__ void __launch_bounds__(128) bsr_generic_kernel(const BsrParams p) {
  constexpr int kSub = kKT / 16;
  constexpr bool kList = kMode != 0;
  constexpr int kDesc = kMode == 2 ? 5 : 4;   // words per unit descriptor
  constexpr int kTileW = kMode == 2 ? 4 : 2;  // words per key tile
  constexpr int kRowBytes = D * 2;
  constexpr int kChunks = kRowBytes / 16;
  constexpr int kTileBytes = kKT * kRowBytes;
  __shared__ __align__(128) uint8_t sm[2][2][kTileBytes];  // [buffer][K/V]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* hdr = p.meta;
  const int32_t* wptr = hdr + hdr[H_OFF_WORKERS];
  const int4* units = reinterpret_cast<const int4*>(hdr + hdr[H_OFF_CHUNKS]);
  const int32_t* indptr = hdr + hdr[H_OFF_AUX0];
  const int32_t* indices = hdr + hdr[H_OFF_AUX1];
  const int g = p.group;
  const int subtiles = (p.C + kKT - 1) / kKT;
  using Mma = MmaOp<T>;

  for (int ui = wptr[blockIdx.x]; ui < wptr[blockIdx.x + 1]; ++ui) {
    const int4 un = units[ui];
    const int i = un.y, h = un.z, rt = un.w;
    // The unit's query rows and key tiles: row block i of R rows and its listed column
    // blocks, or (variable blocks) the lists of descriptor un.x.
    int row0 = i * p.R, nrows = p.R, tb = 0, te = 0, shift = p.N - p.M;
    if constexpr (kList) {
      const int32_t* dsc = indptr + kDesc * int64_t(un.x);
      row0 = dsc[0];
      nrows = dsc[1];
      tb = dsc[2];
      te = dsc[3];
      if constexpr (kMode == 2) shift = dsc[4];
    }
    // This thread's two packed rows (mma rows r0 and r0 + 8 of the warp's 16).
    const int pr0 = rt * kBsrGenericRows + warp * 16 + (lane >> 2);
    const int pr1 = pr0 + 8;
    const int tok0 = row0 + pr0 / g, tok1 = row0 + pr1 / g;
    const int hd0 = h * g + pr0 % g, hd1 = h * g + pr1 % g;
    const bool v0 = pr0 < nrows * g && tok0 < p.M;
    const bool v1 = pr1 < nrows * g && tok1 < p.M;
    const T* qb = static_cast<const T*>(p.q);
    const int cq = lane & 3;
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int d0 = kk * 16 + 2 * cq;
      const T* q0 = qb + int64_t(tok0) * p.q_s0 + int64_t(hd0) * p.q_s1;
      const T* q1 = qb + int64_t(tok1) * p.q_s0 + int64_t(hd1) * p.q_s1;
      qa[kk][0] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + d0) : 0u;
      qa[kk][1] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + d0) : 0u;
      qa[kk][2] = v0 ? *reinterpret_cast<const uint32_t*>(q0 + d0 + 8) : 0u;
      qa[kk][3] = v1 ? *reinterpret_cast<const uint32_t*>(q1 + d0 + 8) : 0u;
    }
    float o[D / 8][4];
#pragma unroll
    for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    const int e0 = kList ? 0 : indptr[i], e1 = kList ? 0 : indptr[i + 1];
    const int ntiles = kList ? te - tb : (e1 - e0) * subtiles;
    // Stage tile n (block e0 + n / subtiles, sub-tile n % subtiles) into buffer `buf`.
    auto load = [&](int n, int buf) {
      int kt0, lim = p.N;
      int64_t base = 0;  // paged: element offset of the tile's first K row
      if constexpr (kMode == 2) {
        const int32_t* tl = indices + kTileW * int64_t(tb + n);
        kt0 = tl[0];
        lim = tl[1];
        base = int64_t(tl[2]) * p.kv_s0 + int64_t(h) * p.kv_s2 + int64_t(tl[3]) * p.kv_s3;
      } else if constexpr (kMode == 1) {
        kt0 = indices[kTileW * (tb + n)];
      } else {
        const int j = indices[e0 + n / subtiles];  // block-sparse mode only: subtiles >= 1
        kt0 = j * p.C + (n % subtiles) * kKT;
      }
      for (int c = threadIdx.x; c < kKT * kChunks; c += 128) {
        const int row = c / kChunks, ch = c % kChunks;
        const int tok = kt0 + row;
        const uint32_t off = swz(row, ch, kRowBytes);
        if (tok < lim) {
          const T* ks;
          const T* vs;
          if constexpr (kMode == 2) {
            ks = static_cast<const T*>(p.kv) + base + int64_t(row) * p.kv_s3;
            vs = ks + p.kv_s1;
          } else {
            ks = static_cast<const T*>(p.k) + int64_t(tok) * p.k_s0 + int64_t(h) * p.k_s1;
            vs = static_cast<const T*>(p.v) + int64_t(tok) * p.v_s0 + int64_t(h) * p.v_s1;
          }
          cp_async_16(&sm[buf][0][off], ks + ch * 8);
          cp_async_16(&sm[buf][1][off], vs + ch * 8);
        } else {
          *reinterpret_cast<uint4*>(&sm[buf][0][off]) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(&sm[buf][1][off]) = make_uint4(0, 0, 0, 0);
        }
      }
      cp_async_commit();
    };
    if (ntiles > 0) load(0, 0);
    for (int n = 0; n < ntiles; ++n) {
      if (n + 1 < ntiles) {
        load(n + 1, (n + 1) & 1);
        cp_async_wait<1>();
      } else {
        cp_async_wait<0>();
      }
      __syncthreads();
      const int buf = n & 1;
      const int eb = kList ? 0 : e0 + n / subtiles;  // the block's position in indices
      const int j = kList ? 0 : indices[eb];
      // first key of the tile and end of its column block (of its key range, of its tile)
      const int kt0 = kList ? indices[kTileW * (tb + n)] : j * p.C + (n % subtiles) * kKT;
      const int kend = kList ? indices[kTileW * (tb + n) + 1] : j * p.C + p.C;
      float s[2 * kSub][4];
#pragma unroll
      for (int nt = 0; nt < 2 * kSub; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
      {
        const int mi = lane >> 3;
#pragma unroll
        for (int sb = 0; sb < kSub; ++sb) {
          const int trow = sb * 16 + (mi >> 1) * 8 + (lane & 7);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const int ch = kk * 2 + (mi & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(smem_u32(&sm[buf][0][0]) + swz(trow, ch, kRowBytes), b0, b1, b2, b3);
            Mma::run(s[2 * sb], qa[kk], b0, b1);
            Mma::run(s[2 * sb + 1], qa[kk], b2, b3);
          }
        }
      }
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2 * kSub; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kt = kt0 + nt * 8 + 2 * cq + (e & 1);
          const int qt = (e < 2) ? tok0 : tok1;
          bool vis = kt < kend;
          if (kMode == 0 && p.mask) {
            // bit (eb * R + row in block) * C + column in block; rows past M are never stored
            const int64_t bit = (int64_t(eb) * p.R + (qt - i * p.R)) * p.C + (kt - j * p.C);
            vis = vis && qt < p.M && ((__ldg(p.mask + (bit >> 3)) >> (bit & 7)) & 1);
          } else if (p.causal) {
            // bottom-right aligned: query qt - row0 of its request (or row qt of the whole
            // sequence) sees keys up to itself plus the shift
            vis = vis && (kt <= (kMode == 2 ? qt - row0 : qt) + shift);
          }
          s[nt][e] = vis ? s[nt][e] * p.scale_log2 : -INFINITY;
        }
        mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      // A row that has seen no visible key yet keeps reference 0 so that nothing is NaN.
      const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
      const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
      const float a0 = fast_exp2(m0 - ref0), a1 = fast_exp2(m1 - ref1);
      m0 = mn0;
      m1 = mn1;
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2 * kSub; ++nt) {
        s[nt][0] = fast_exp2(s[nt][0] - ref0);
        s[nt][1] = fast_exp2(s[nt][1] - ref0);
        s[nt][2] = fast_exp2(s[nt][2] - ref1);
        s[nt][3] = fast_exp2(s[nt][3] - ref1);
        ps0 += s[nt][0] + s[nt][1];
        ps1 += s[nt][2] + s[nt][3];
      }
      l0 = l0 * a0 + ps0;
      l1 = l1 * a1 + ps1;
#pragma unroll
      for (int nn = 0; nn < D / 8; ++nn) {
        o[nn][0] *= a0;
        o[nn][1] *= a0;
        o[nn][2] *= a1;
        o[nn][3] *= a1;
      }
#pragma unroll
      for (int sb = 0; sb < kSub; ++sb) {
        uint32_t pa[4] = {Mma::pack(s[2 * sb][0], s[2 * sb][1]),
                          Mma::pack(s[2 * sb][2], s[2 * sb][3]),
                          Mma::pack(s[2 * sb + 1][0], s[2 * sb + 1][1]),
                          Mma::pack(s[2 * sb + 1][2], s[2 * sb + 1][3])};
        const int mi = lane >> 3;
        const int trow = sb * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
        for (int dd = 0; dd < D / 16; ++dd) {
          const int ch = dd * 2 + (mi >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_u32(&sm[buf][1][0]) + swz(trow, ch, kRowBytes), b0, b1, b2, b3);
          Mma::run(o[2 * dd], pa, b0, b1);
          Mma::run(o[2 * dd + 1], pa, b2, b3);
        }
      }
      __syncthreads();
    }
    float lt0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
    lt0 += __shfl_xor_sync(0xffffffffu, lt0, 2);
    float lt1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
    lt1 += __shfl_xor_sync(0xffffffffu, lt1, 2);
    const float inv0 = lt0 > 0.f ? 1.f / lt0 : 0.f, inv1 = lt1 > 0.f ? 1.f / lt1 : 0.f;
    T* ob = static_cast<T*>(p.out);
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      const int d = n * 8 + 2 * cq;
      if (v0)
        *reinterpret_cast<uint32_t*>(ob + int64_t(tok0) * p.o_s0 + int64_t(hd0) * p.o_s1 + d) =
            Mma::pack(o[n][0] * inv0, o[n][1] * inv0);
      if (v1)
        *reinterpret_cast<uint32_t*>(ob + int64_t(tok1) * p.o_s0 + int64_t(hd1) * p.o_s1 + d) =
            Mma::pack(o[n][2] * inv1, o[n][3] * inv1);
    }
    if (p.lse && cq == 0) {
      if (v0) p.lse[int64_t(tok0) * p.lse_st + int64_t(hd0) * p.lse_sh] = lt0 > 0.f ? (m0 + __log2f(lt0)) * kLn2 : -INFINITY;
      if (v1) p.lse[int64_t(tok1) * p.lse_st + int64_t(hd1) * p.lse_sh] = lt1 > 0.f ? (m1 + __log2f(lt1)) * kLn2 : -INFINITY;
    }
  }
}

}  // namespace

bskv_status launch_bsr_tcgen05(const bskv_plan* plan, const void* q, const int64_t* qs,
                               const void* k, const int64_t* ks, const void* v,
                               const int64_t* vs, void* out, const int64_t* os, float* lse,
                               float sm_scale, const uint8_t* mask, cudaStream_t st);
bskv_status launch_prefill_tcgen05(const bskv_plan* plan, const void* q, const int64_t* qs,
                                   const void* kv, const int64_t* kvs, void* out,
                                   const int64_t* os, float* lse, float sm_scale,
                                   cudaStream_t st);

}  // namespace bskv

using namespace bskv;

namespace {

template <int kMode, int kKT>
void launch_generic(const bskv_plan* plan, const BsrParams& p, int grid, cudaStream_t st) {
  const bool bf = plan->dtype == BSKV_BF16;
  if (plan->head_dim == 128) {
    if (bf) bsr_generic_kernel<__nv_bfloat16, 128, kMode, kKT><<<grid, 128, 0, st>>>(p);
    else bsr_generic_kernel<__half, 128, kMode, kKT><<<grid, 128, 0, st>>>(p);
  } else {
    if (bf) bsr_generic_kernel<__nv_bfloat16, 64, kMode, kKT><<<grid, 128, 0, st>>>(p);
    else bsr_generic_kernel<__half, 64, kMode, kKT><<<grid, 128, 0, st>>>(p);
  }
}

bskv_status run_bsr(const bskv_plan* plan, const void* q, const int64_t* q_strides,
                    const void* k, const int64_t* k_strides, const void* v,
                    const int64_t* v_strides, void* out, const int64_t* out_strides, float* lse,
                    float sm_scale, const uint8_t* mask, void* stream) {
  const int variant = plan && plan->kind == KIND_BSR ? meta_word(plan, H_VARIANT) : -1;
  const bool var = variant == BSR_VARIABLE;
  if (variant == BSR_PAGED_PREFILL || variant == BSR_PAGED_PREFILL_TC) {
    set_error("run_bsr: a paged prefill plan runs through bskv_run_prefill_paged");
    return BSKV_ERR_INVALID_ARG;
  }
  if (!plan || plan->kind != KIND_BSR) { set_error("run_bsr: not a BSR plan"); return BSKV_ERR_INVALID_ARG; }
  if (!plan->meta_dev) { set_error("run_bsr: plan not uploaded (bskv_plan_upload)"); return BSKV_ERR_INVALID_ARG; }
  if (!q_strides || !k_strides || !v_strides || !out_strides) { set_error("run_bsr: NULL strides"); return BSKV_ERR_INVALID_ARG; }
  if (plan->M == 0) return BSKV_OK;
  if (!q || !k || !v || !out) { set_error("run_bsr: NULL tensor"); return BSKV_ERR_INVALID_ARG; }
  const int64_t* all[4] = {q_strides, k_strides, v_strides, out_strides};
  for (auto s : all)
    if (s[0] <= 0 || s[1] <= 0 || (s[0] * 2) % 16 || (s[1] * 2) % 16) {
      set_error("run_bsr: strides must be positive multiples of 8 elements"); return BSKV_ERR_INVALID_ARG;
    }
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) { set_error("run_bsr: tensors must be 16-byte aligned"); return BSKV_ERR_INVALID_ARG; }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (variant == BSR_TCGEN05 || variant == BSR_VARIABLE_TC)
    return launch_bsr_tcgen05(plan, q, q_strides, k, k_strides, v, v_strides, out, out_strides,
                              lse, sm_scale, mask, st);
  BsrParams p{};
  p.meta = plan->meta_dev;
  p.q = q; p.q_s0 = q_strides[0]; p.q_s1 = q_strides[1];
  p.k = k; p.k_s0 = k_strides[0]; p.k_s1 = k_strides[1];
  p.v = v; p.v_s0 = v_strides[0]; p.v_s1 = v_strides[1];
  p.out = out; p.o_s0 = out_strides[0]; p.o_s1 = out_strides[1];
  p.lse = lse;
  // lse [M, Hq] for block-sparse plans, [Hq, M] (head-major) for variable-block plans
  p.lse_st = var ? 1 : plan->num_qo_heads;
  p.lse_sh = var ? plan->M : 1;
  p.M = plan->M; p.N = plan->N; p.R = plan->R; p.C = plan->C;
  p.Hq = plan->num_qo_heads; p.Hkv = plan->num_kv_heads; p.group = p.Hq / p.Hkv;
  p.causal = plan->causal;
  p.mask = mask;
  p.scale_log2 = sm_scale_log2(sm_scale, plan->head_dim);
  if (bskv_status s = status_args(&p.st)) return s;
  const int grid = meta_word(plan, H_GRID);
  if (grid == 0) return BSKV_OK;
  const bool narrow = !var && plan->C <= 16;  // 16-key tiles
  if (var) launch_generic<1, 32>(plan, p, grid, st);
  else if (narrow) launch_generic<0, 16>(plan, p, grid, st);
  else launch_generic<0, 32>(plan, p, grid, st);
  return cuda_check(cudaGetLastError(), "bsr kernel launch");
}

}  // namespace

extern "C" bskv_status bskv_run_bsr(const bskv_plan* plan, const void* q, const int64_t* q_strides,
                                    const void* k, const int64_t* k_strides, const void* v,
                                    const int64_t* v_strides, void* out,
                                    const int64_t* out_strides, float* lse, float sm_scale,
                                    void* float_ws, size_t float_ws_bytes, void* stream) {
  BSKV_NVTX_RANGE("bskv_run_bsr");
  (void)float_ws;
  (void)float_ws_bytes;
  if (plan && plan->masked) { set_error("run_bsr: the plan expects a token mask (bskv_run_bsr_masked)"); return BSKV_ERR_INVALID_ARG; }
  if (plan && plan->kind == KIND_BSR &&
      (meta_word(plan, H_VARIANT) == BSR_VARIABLE || meta_word(plan, H_VARIANT) == BSR_VARIABLE_TC)) {
    set_error("run_bsr: a variable-block plan runs through bskv_run_bsr_variable");
    return BSKV_ERR_INVALID_ARG;
  }
  return run_bsr(plan, q, q_strides, k, k_strides, v, v_strides, out, out_strides, lse, sm_scale,
                 nullptr, stream);
}

extern "C" bskv_status bskv_run_bsr_masked(const bskv_plan* plan, const void* q,
                                           const int64_t* q_strides, const void* k,
                                           const int64_t* k_strides, const void* v,
                                           const int64_t* v_strides, const void* packed_mask,
                                           size_t packed_mask_bytes, void* out,
                                           const int64_t* out_strides, float* lse,
                                           float sm_scale, void* stream) {
  BSKV_NVTX_RANGE("bskv_run_bsr_masked");
  if (!plan || plan->kind != KIND_BSR || !plan->masked) { set_error("run_bsr_masked: not a masked BSR plan (bskv_plan_bsr_masked)"); return BSKV_ERR_INVALID_ARG; }
  const int32_t MB = (plan->M + plan->R - 1) / plan->R;
  const int32_t* meta = plan->meta.data();
  const int64_t nnz = plan->M > 0 ? meta[meta[H_OFF_AUX0] + MB] : 0;
  const size_t need = size_t((nnz * plan->R * plan->C + 7) / 8);
  if (need > 0 && (!packed_mask || packed_mask_bytes < need)) {
    set_error("run_bsr_masked: packed mask of %zu bytes, %zu needed", packed_mask_bytes, need);
    return BSKV_ERR_INVALID_ARG;
  }
  if (reinterpret_cast<uintptr_t>(packed_mask) & 15) { set_error("run_bsr_masked: packed mask must be 16-byte aligned"); return BSKV_ERR_INVALID_ARG; }
  return run_bsr(plan, q, q_strides, k, k_strides, v, v_strides, out, out_strides, lse, sm_scale,
                 static_cast<const uint8_t*>(packed_mask), stream);
}

extern "C" bskv_status bskv_run_bsr_variable(const bskv_plan* plan, const void* q,
                                             const int64_t* q_strides, const void* k,
                                             const int64_t* k_strides, const void* v,
                                             const int64_t* v_strides, void* out,
                                             const int64_t* out_strides, float* lse,
                                             float sm_scale, void* stream) {
  BSKV_NVTX_RANGE("bskv_run_bsr_variable");
  if (!plan || plan->kind != KIND_BSR || !plan->meta.size() ||
      (plan->meta[H_VARIANT] != BSR_VARIABLE && plan->meta[H_VARIANT] != BSR_VARIABLE_TC)) {
    set_error("run_bsr_variable: not a variable-block plan (bskv_plan_bsr_variable)");
    return BSKV_ERR_INVALID_ARG;
  }
  return run_bsr(plan, q, q_strides, k, k_strides, v, v_strides, out, out_strides, lse, sm_scale,
                 nullptr, stream);
}

extern "C" bskv_status bskv_run_prefill_paged(const bskv_plan* plan, const void* q,
                                              const int64_t* q_strides, const void* kv_cache,
                                              const int64_t* kv_strides, void* out,
                                              const int64_t* out_strides, float* lse,
                                              float sm_scale, void* stream) {
  BSKV_NVTX_RANGE("bskv_run_prefill_paged");
  if (!plan || plan->kind != KIND_BSR || plan->meta.empty() ||
      (plan->meta[H_VARIANT] != BSR_PAGED_PREFILL && plan->meta[H_VARIANT] != BSR_PAGED_PREFILL_TC)) {
    set_error("run_prefill_paged: not a paged prefill plan (bskv_plan_prefill_paged)");
    return BSKV_ERR_INVALID_ARG;
  }
  if (!plan->meta_dev) { set_error("run_prefill_paged: plan not uploaded (bskv_plan_upload)"); return BSKV_ERR_INVALID_ARG; }
  if (!q_strides || !kv_strides || !out_strides) { set_error("run_prefill_paged: NULL strides"); return BSKV_ERR_INVALID_ARG; }
  if (plan->M == 0) return BSKV_OK;
  if (!q || !kv_cache || !out) { set_error("run_prefill_paged: NULL tensor"); return BSKV_ERR_INVALID_ARG; }
  const int64_t* qo[2] = {q_strides, out_strides};
  for (auto st2 : qo)
    if (st2[0] <= 0 || st2[1] <= 0 || (st2[0] * 2) % 16 || (st2[1] * 2) % 16) {
      set_error("run_prefill_paged: q/out strides must be positive multiples of 8 elements"); return BSKV_ERR_INVALID_ARG;
    }
  for (int i = 0; i < 4; ++i)
    if (kv_strides[i] < 0 || (kv_strides[i] * 2) % 16) {
      set_error("run_prefill_paged: kv strides must be non-negative multiples of 8 elements"); return BSKV_ERR_INVALID_ARG;
    }
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out)) { set_error("run_prefill_paged: tensors must be 16-byte aligned"); return BSKV_ERR_INVALID_ARG; }
  if (plan->meta[H_VARIANT] == BSR_PAGED_PREFILL_TC)
    return launch_prefill_tcgen05(plan, q, q_strides, kv_cache, kv_strides, out, out_strides, lse,
                                  sm_scale, static_cast<cudaStream_t>(stream));
  BsrParams p{};
  p.meta = plan->meta_dev;
  p.q = q; p.q_s0 = q_strides[0]; p.q_s1 = q_strides[1];
  p.kv = kv_cache;
  p.kv_s0 = kv_strides[0]; p.kv_s1 = kv_strides[1]; p.kv_s2 = kv_strides[2]; p.kv_s3 = kv_strides[3];
  p.out = out; p.o_s0 = out_strides[0]; p.o_s1 = out_strides[1];
  p.lse = lse;
  p.lse_st = plan->num_qo_heads;
  p.lse_sh = 1;
  p.M = plan->M; p.N = 0; p.R = 0; p.C = 0;
  p.Hq = plan->num_qo_heads; p.Hkv = plan->num_kv_heads; p.group = p.Hq / p.Hkv;
  p.causal = plan->causal;
  p.mask = nullptr;
  p.scale_log2 = sm_scale_log2(sm_scale, plan->head_dim);
  if (bskv_status s = status_args(&p.st)) return s;
  const int grid = meta_word(plan, H_GRID);
  if (grid == 0) return BSKV_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  launch_generic<2, 32>(plan, p, grid, st);
  return cuda_check(cudaGetLastError(), "prefill kernel launch");
}
