// BSR block-sparse attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// Method: "flashinfer.sparse - FlashInfer 0.7.4 documentation", BlockSparseAttentionWrapper
// (bsr_matrix block mask; num_qo_heads a multiple of num_kv_heads; causal token mask; run()
// returns out [M, Hq, D] and lse [M, Hq]).
//
// Shape served: R = C = 64, head_dim 128, g = Hq/Hkv in {2, 4}, fp16 or bf16. One unit is
// (row block i, kv head h): the 64 query tokens of row block i times the g query heads that
// share kv head h, i.e. one or two M=128 tiles (two heads per tile, head-major), so every
// K/V block that is loaded feeds all grouped heads.
//
// GB300 design (persistent, one CTA per SM, 12 warps):
//   warp 0   TMA producer: Q tiles (3-D tensor map, 128B swizzle) once per unit, K and V
//            blocks of the unit's column list into a 3-stage ring;
//   warp 1   allocates 512 TMEM columns; lane 0 issues every tcgen05.mma:
//            S_m = Q_m K^T (M=128, N=64, K=128, K-major operands) into a double-buffered
//            S region of TMEM, then O_m += P_m V (M=128, N=128, K=64; V MN-major);
//            completion is signalled with tcgen05.commit on mbarriers;
//   warps 4-7 / 8-11  one warpgroup per M tile: thread = row = TMEM lane. Each reads its S
//            row (tcgen05.ld), applies scale and the causal mask, keeps a running max with
//            lazy rescaling (O is rescaled in TMEM only when the max grows by more than 2^8),
//            writes P (fp16/bf16) into a 128B-swizzled K-major tile for the PV MMA, and in
//            the epilogue normalises O from TMEM and stores out and lse.
// The MMA pipe runs QK of block j+1 while the warpgroups do the softmax of block j.
// Every wait is bounded; on a timeout the CTA drains its copies and MMAs, frees TMEM and
// returns after recording BSKV_ERR_TIMEOUT.
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "launch.h"

namespace bskv {
namespace {

using namespace dev;

constexpr int kBlk = 64;          // R = C = 64
constexpr int kD = 128;
constexpr int kStagesKV = 3;
constexpr int kThreads = 384;
constexpr uint32_t kKPanel = 64 * 128;      // [64 rows x 64 elements] of 16 bits
constexpr uint32_t kQTile = 2 * 128 * 128;  // [128 rows x 128 elements]: 2 panels of 16 KB
constexpr uint32_t kKVStage = 4 * kKPanel;  // K (2 panels) then V (2 panels)
constexpr uint32_t kPTile = 128 * 128;      // [128 rows x 64 elements]
constexpr uint32_t kTmemCols = 512;

struct TcParams {
  const int32_t* meta;
  void* out;
  int64_t o_s0, o_s1;
  float* lse;
  int M, N, Hq, Hkv, group, causal;
  float scale_log2;
  StatusArgs st;
};

template <int NM>
struct Smem {
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kP = kQ + NM * kQTile;
  static constexpr uint32_t kKV = kP + NM * 2 * kPTile;
  static constexpr uint32_t kBar = kKV + kStagesKV * kKVStage;
  static constexpr uint32_t kBytes = kBar + 512;
};

struct Bars {
  uint64_t q_full, q_empty, drain;
  uint64_t kv_full[kStagesKV], kv_empty[kStagesKV];
  uint64_t s_full[2][2];  // [m][buffer]
  uint64_t p_full[2][2];
  uint64_t o_done[2], o_free[2];
  uint32_t tmem_base;
  int abort;
};

template <typename T>
struct Fmt;
template <>
struct Fmt<__half> {
  static constexpr uint32_t v = 0;
};
template <>
struct Fmt<__nv_bfloat16> {
  static constexpr uint32_t v = 1;
};

__device__ __forceinline__ uint32_t pack2(__half, float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack2(__nv_bfloat16, float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <typename T, int NM>
__global__ void __launch_bounds__(kThreads, 1)
    bsr_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, const TcParams p) {
  using L = Smem<NM>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  Bars& B = *reinterpret_cast<Bars*>(sm + L::kBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* hdr = p.meta;
  const int32_t* wptr = hdr + hdr[H_OFF_WORKERS];
  const int4* units = reinterpret_cast<const int4*>(hdr + hdr[H_OFF_CHUNKS]);
  const int32_t* indptr = hdr + hdr[H_OFF_AUX0];
  const int32_t* indices = hdr + hdr[H_OFF_AUX1];
  const int u0 = wptr[blockIdx.x], u1 = wptr[blockIdx.x + 1];
  const bool forced = forced_timeout(p.st);

  if (threadIdx.x == 0) {
    mbar_init(&B.q_full, 1);
    mbar_init(&B.q_empty, 1);
    mbar_init(&B.drain, 1);
    for (int s = 0; s < kStagesKV; ++s) {
      mbar_init(&B.kv_full[s], 1);
      mbar_init(&B.kv_empty[s], 1);
    }
    for (int m = 0; m < 2; ++m) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(&B.s_full[m][b], 1);
        mbar_init(&B.p_full[m][b], 128);
      }
      mbar_init(&B.o_done[m], 1);
      mbar_init(&B.o_free[m], 128);
    }
    B.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&B.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B.tmem_base;
  volatile int* abort_flag = &B.abort;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&qmap);
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      uint32_t qc = 0, kvc = 0;
      bool ok = true;
      for (int ui = u0; ui < u1 && ok; ++ui) {
        const int4 un = units[ui];
        const int i = un.y, h = un.z;
        const int e0 = indptr[i], e1 = indptr[i + 1];
        if (e1 == e0) continue;
        if (*abort_flag || !mbar_wait(&B.q_empty, (qc & 1u) ^ 1u, p.st, forced)) { ok = false; break; }
        mbar_arrive_expect_tx(&B.q_full, NM * kQTile);
        for (int m = 0; m < NM; ++m)
          for (int hl = 0; hl < 2; ++hl)
            for (int pn = 0; pn < 2; ++pn)
              tma_load_3d(sm + L::kQ + m * kQTile + pn * (kQTile / 2) + hl * kKPanel, &qmap,
                          pn * 64, h * p.group + m * 2 + hl, i * kBlk, &B.q_full);
        ++qc;
        for (int e = e0; e < e1; ++e, ++kvc) {
          const int s = kvc % kStagesKV;
          if (*abort_flag || !mbar_wait(&B.kv_empty[s], ((kvc / kStagesKV) & 1u) ^ 1u, p.st, forced)) {
            ok = false;
            break;
          }
          const int j = indices[e];
          uint8_t* dst = sm + L::kKV + s * kKVStage;
          mbar_arrive_expect_tx(&B.kv_full[s], kKVStage);
          tma_load_3d(dst, &kmap, 0, h, j * kBlk, &B.kv_full[s]);
          tma_load_3d(dst + kKPanel, &kmap, 64, h, j * kBlk, &B.kv_full[s]);
          tma_load_3d(dst + 2 * kKPanel, &vmap, 0, h, j * kBlk, &B.kv_full[s]);
          tma_load_3d(dst + 3 * kKPanel, &vmap, 64, h, j * kBlk, &B.kv_full[s]);
        }
      }
      if (!ok) {
        *abort_flag = 1;
        // Wait (bounded, not forcible) for every copy this thread issued to land.
        if (qc > 0) mbar_wait(&B.q_full, (qc - 1) & 1u, p.st, false);
        for (int s = 0; s < kStagesKV; ++s) {
          // the last use of stage s that was issued: kvc' < kvc with kvc' % stages == s
          if (kvc > uint32_t(s)) {
            const uint32_t last = ((kvc - 1 - s) / kStagesKV) * kStagesKV + s;
            mbar_wait(&B.kv_full[s], (last / kStagesKV) & 1u, p.st, false);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t fmt = Fmt<T>::v;
      constexpr uint32_t idesc_qk = umma_idesc(128, 64, fmt, fmt, 0, 0);
      constexpr uint32_t idesc_pv = umma_idesc(128, 128, fmt, fmt, 0, 1);
      const uint32_t sbase = smem_u32(sm);
      uint32_t qc = 0, kvc = 0, G = 0, uc = 0;
      bool ok = true;
      auto pv = [&](uint32_t g_step, uint32_t kv_use, bool first) -> bool {
        const int s = kv_use % kStagesKV;
        const uint32_t vaddr = sbase + L::kKV + s * kKVStage + 2 * kKPanel;
        for (int m = 0; m < NM; ++m) {
          const uint32_t b = g_step & 1u;
          if (*abort_flag || !mbar_wait(&B.p_full[m][b], (g_step >> 1) & 1u, p.st, forced)) return false;
          if (first && (*abort_flag || !mbar_wait(&B.o_free[m], (uc & 1u) ^ 1u, p.st, forced))) return false;
          tc_fence_after();
          const uint32_t paddr = sbase + L::kP + (m * 2 + b) * kPTile;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = umma_desc(paddr + kk * 32, 16, 1024, kSwz128);
            const uint64_t bd = umma_desc(vaddr + kk * 2048, kKPanel, 1024, kSwz128);
            umma_f16(tmem + m * 128, a, bd, idesc_pv, (first && kk == 0) ? 0u : 1u);
          }
          umma_commit(&B.o_done[m]);
        }
        umma_commit(&B.kv_empty[s]);
        return true;
      };
      for (int ui = u0; ui < u1 && ok; ++ui) {
        const int4 un = units[ui];
        const int i = un.y;
        const int e0 = indptr[i], e1 = indptr[i + 1];
        const int n = e1 - e0;
        if (n == 0) continue;
        if (*abort_flag || !mbar_wait(&B.q_full, qc & 1u, p.st, forced)) { ok = false; break; }
        ++qc;
        tc_fence_after();
        const uint32_t kv_first = kvc;
        for (int j = 0; j < n; ++j, ++kvc) {
          const int s = kvc % kStagesKV;
          if (*abort_flag || !mbar_wait(&B.kv_full[s], (kvc / kStagesKV) & 1u, p.st, forced)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kaddr = sbase + L::kKV + s * kKVStage;
          const uint32_t gj = G + j;
          for (int m = 0; m < NM; ++m) {
            const uint32_t qaddr = sbase + L::kQ + m * kQTile;
            const uint32_t sd = tmem + 256 + (m * 2 + (gj & 1u)) * 64;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t a = umma_desc(qaddr + (kk / 4) * (kQTile / 2) + (kk % 4) * 32, 16, 1024, kSwz128);
              const uint64_t bd = umma_desc(kaddr + (kk / 4) * kKPanel + (kk % 4) * 32, 16, 1024, kSwz128);
              umma_f16(sd, a, bd, idesc_qk, kk > 0 ? 1u : 0u);
            }
            umma_commit(&B.s_full[m][gj & 1u]);
          }
          if (j >= 1 && !pv(gj - 1, kv_first + j - 1, j == 1)) { ok = false; break; }
        }
        if (!ok) break;
        if (!pv(G + n - 1, kv_first + n - 1, n == 1)) { ok = false; break; }
        umma_commit(&B.q_empty);
        G += n;
        ++uc;
      }
      if (!ok) *abort_flag = 1;
      // All MMAs issued by this thread complete before TMEM is released.
      umma_commit(&B.drain);
      mbar_wait(&B.drain, 0, p.st, false);
    }
  } else if (warp >= 4 && warp < 4 + 4 * NM) {
    // ------------------------------------------------------------------ softmax warpgroups
    const int m = (warp - 4) >> 2;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;                    // row of the M tile = TMEM lane
    const uint32_t lane_base = uint32_t(q4 * 32) << 16;
    const int hl = m * 2 + r / kBlk;                 // head within the group
    uint8_t* const prow = sm + L::kP + m * 2 * kPTile + r * 128;
    uint32_t G = 0, od = 0;
    bool ok = true;
    for (int ui = u0; ui < u1 && ok; ++ui) {
      const int4 un = units[ui];
      const int i = un.y, h = un.z;
      const int e0 = indptr[i], e1 = indptr[i + 1];
      const int n = e1 - e0;
      const int tok = i * kBlk + (r % kBlk);
      const int head = h * p.group + hl;
      T* orow = static_cast<T*>(p.out) + int64_t(tok) * p.o_s0 + int64_t(head) * p.o_s1;
      if (n == 0) {
        if (tok < p.M) {
          for (int c = 0; c < kD; c += 8) *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
          if (p.lse) p.lse[int64_t(tok) * p.Hq + head] = -INFINITY;
        }
        continue;
      }
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < n; ++j, ++G) {
        const uint32_t b = G & 1u;
        if (!warp_wait(&B.s_full[m][b], (G >> 1) & 1u, p.st, forced, abort_flag)) { ok = false; break; }
        tc_fence_after();
        uint32_t sr[64];
        const uint32_t scol = tmem + lane_base + 256 + (m * 2 + b) * 64;
        tmem_ld32(scol, sr);
        tmem_ld32(scol + 32, sr + 32);
        tmem_ld_wait();
        float s[64];
        const int jb = indices[e0 + j];
        const int lim = tok + (p.N - p.M);
        const bool mask = p.causal && (jb * kBlk + kBlk - 1 > lim);
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          float x = __uint_as_float(sr[c]) * p.scale_log2;
          if (mask && jb * kBlk + c > lim) x = -INFINITY;
          s[c] = x;
          mx = fmaxf(mx, x);
        }
        // Lazy rescaling: keep the reference max unless the row max grew by more than 8
        // (a factor 2^8), so O in TMEM is rarely touched and P stays below 256.
        float m_use = m_run, alpha = 1.f;
        bool rescale = false;
        if (m_run == -INFINITY) {
          m_use = mx;
        } else if (mx > m_run + 8.f) {
          m_use = mx;
          alpha = fast_exp2(m_run - mx);
          rescale = true;
        }
        const float ref = m_use == -INFINITY ? 0.f : m_use;
        float sum = 0.f;
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float a0 = fast_exp2(s[c] - ref), a1 = fast_exp2(s[c + 1] - ref);
          sum += a0 + a1;
          pk[c / 2] = pack2(T(), a0, a1);
        }
        l_run = l_run * alpha + sum;
        m_run = m_use;
        // The O rescale (tcgen05.ld/st, warp-collective) runs for the whole warp when any
        // of its rows needs it; the other rows multiply by 1.
        rescale = __any_sync(0xffffffffu, rescale);
        // P buffer b was last read by PV of step G-2; observe completions up to PV(G-1)
        // (also required before touching O).
        while (od < G) {
          if (!warp_wait(&B.o_done[m], od & 1u, p.st, forced, abort_flag)) { ok = false; break; }
          ++od;
        }
        if (!ok) break;
        uint8_t* pr = prow + b * kPTile;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(pr + ((c ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        if (rescale && j > 0) {
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < kD; cc += 32) {
            uint32_t ov[32];
            tmem_ld32(tmem + lane_base + m * 128 + cc, ov);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
            tmem_st32(tmem + lane_base + m * 128 + cc, ov);
          }
          tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&B.p_full[m][b]);
      }
      if (!ok) break;
      // Epilogue: wait for the unit's last PV, normalise and store.
      while (od < G) {
        if (!warp_wait(&B.o_done[m], od & 1u, p.st, forced, abort_flag)) { ok = false; break; }
        ++od;
      }
      if (!ok) break;
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
      for (int cc = 0; cc < kD; cc += 32) {
        uint32_t ov[32];
        tmem_ld32(tmem + lane_base + m * 128 + cc, ov);
        tmem_ld_wait();
        if (tok < p.M) {
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint4 w;
            w.x = pack2(T(), __uint_as_float(ov[c]) * inv, __uint_as_float(ov[c + 1]) * inv);
            w.y = pack2(T(), __uint_as_float(ov[c + 2]) * inv, __uint_as_float(ov[c + 3]) * inv);
            w.z = pack2(T(), __uint_as_float(ov[c + 4]) * inv, __uint_as_float(ov[c + 5]) * inv);
            w.w = pack2(T(), __uint_as_float(ov[c + 6]) * inv, __uint_as_float(ov[c + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + cc + c) = w;
          }
        }
      }
      if (tok < p.M && p.lse)
        p.lse[int64_t(tok) * p.Hq + head] =
            l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
      tc_fence_before();
      mbar_arrive(&B.o_free[m]);
    }
    if (!ok) *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <typename T, int NM>
bskv_status launch_t(const bskv_plan* plan, const CUtensorMap& qm, const CUtensorMap& km,
                     const CUtensorMap& vm, const TcParams& tp, cudaStream_t st) {
  const int grid = meta_word(plan, H_GRID);
  if (grid == 0) return BSKV_OK;
  const size_t smem = Smem<NM>::kBytes + 1024;
  auto kern = bsr_tc_kernel<T, NM>;
  if (bskv_status s = cuda_check(
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)),
          "bsr_tc: cudaFuncSetAttribute"))
    return s;
  kern<<<grid, kThreads, smem, st>>>(qm, km, vm, tp);
  return cuda_check(cudaGetLastError(), "bsr_tc launch");
}

}  // namespace

bskv_status launch_bsr_tcgen05(const bskv_plan* plan, const void* q, const int64_t* qs,
                               const void* k, const int64_t* ks, const void* v,
                               const int64_t* vs, void* out, const int64_t* os, float* lse,
                               float sm_scale, cudaStream_t st) {
  const int g = plan->num_qo_heads / plan->num_kv_heads;
  if (!(plan->R == kBlk && plan->C == kBlk && plan->head_dim == kD && (g == 2 || g == 4))) {
    set_error("run_bsr: tensor-core kernel needs R = C = 64, head_dim 128, group 2 or 4");
    return BSKV_ERR_UNSUPPORTED;
  }
  TcParams tp{};
  tp.meta = plan->meta_dev;
  tp.out = out; tp.o_s0 = os[0]; tp.o_s1 = os[1];
  tp.lse = lse;
  tp.M = plan->M; tp.N = plan->N; tp.Hq = plan->num_qo_heads; tp.Hkv = plan->num_kv_heads;
  tp.group = g; tp.causal = plan->causal;
  tp.scale_log2 = sm_scale * 1.4426950408889634f;
  if (bskv_status s = status_args(&tp.st)) return s;
  const CUtensorMapDataType dt =
      plan->dtype == BSKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap qm, km, vm;
  const uint32_t box[3] = {64, 1, 64};
  {
    const uint64_t dims[3] = {uint64_t(kD), uint64_t(plan->num_qo_heads), uint64_t(plan->M)};
    const uint64_t str[2] = {uint64_t(qs[1]) * 2, uint64_t(qs[0]) * 2};
    if (bskv_status s = encode_tiled(&qm, dt, 3, q, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return s;
  }
  {
    const uint64_t dims[3] = {uint64_t(kD), uint64_t(plan->num_kv_heads), uint64_t(plan->N)};
    const uint64_t sk[2] = {uint64_t(ks[1]) * 2, uint64_t(ks[0]) * 2};
    const uint64_t sv[2] = {uint64_t(vs[1]) * 2, uint64_t(vs[0]) * 2};
    if (bskv_status s = encode_tiled(&km, dt, 3, k, dims, sk, box, CU_TENSOR_MAP_SWIZZLE_128B)) return s;
    if (bskv_status s = encode_tiled(&vm, dt, 3, v, dims, sv, box, CU_TENSOR_MAP_SWIZZLE_128B)) return s;
  }
  const bool bf = plan->dtype == BSKV_BF16;
  if (g == 4)
    return bf ? launch_t<__nv_bfloat16, 2>(plan, qm, km, vm, tp, st) : launch_t<__half, 2>(plan, qm, km, vm, tp, st);
  return bf ? launch_t<__nv_bfloat16, 1>(plan, qm, km, vm, tp, st) : launch_t<__half, 1>(plan, qm, km, vm, tp, st);
}

}  // namespace bskv
