// Sparse MLA FP8 decode on the 5th-generation tensor cores (tcgen05 kind::f8f6f4 + TMEM).
//
// Method: "Sparse MLA" (MATE 0.2.6), sparse_mla_fp8_decode: E4M3 query [batch, q_len,
// heads, 576], E4M3 cache rows of 576 values (512 latent + 64 rotated), int32 physical-token
// indices [batch, q_len, top_k] shared by all heads, seq_lens[b] valid entries, bmm1_scale
// on the QK product and bmm2_scale on the output, BF16 output of 512 values and FP32 LSE;
// "FlashInfer Compatibility Wrapper", scale folding. V is the first 512 values of a row.
//
// GB300 design (persistent, one CTA per SM, 12 warps). The work unit is (query token,
// latent half): all 128 heads form the M=128 rows of every MMA and the CTA accumulates
// O for one 256-value half of the output in TMEM (256 columns), so S and O fit side by side
// (the full 128 x 512 fp32 accumulator alone would fill TMEM). S is computed by both halves.
//   warps 0-5  two gather groups of 96 threads taking alternate tiles: a group stages the
//              tile's 64 row ids in shared memory, copies the rows with 16-byte cp.async
//              (consecutive threads, consecutive chunks of a row) into the swizzled panels
//              (row r, chunk c -> chunk c ^ (r mod 8)) and publishes the tile as soon as its
//              own copies have landed. Thread 0 also TMA-loads the query tile (four
//              128B-swizzled panels of 128 B plus one 64B-swizzled panel for the rotated
//              tail). On this part many-row gathers are faster through the load/store pipes
//              than through TMA tile::gather4, which moves 128-byte pieces one at a time;
//   warp 6     allocates TMEM; lane 0 issues S = Q K^T (M=128, N=64, K=576: 18 MMAs of K=32)
//              and O += P V_half (M=128, N=256, K=64; the gathered panels serve as the
//              MN-major V operand), advancing prebuilt descriptors by address only;
//   warps 8-15 two softmax warpgroups; thread = head = TMEM lane, each group owns 32 of a
//              tile's 64 columns and 128 of the 256 output values. The row max and, at the end,
//              the row sum are combined through shared memory; lazy max rescaling (threshold
//              2^8); exponentials as packed f16x2 (ex2.approx.f16x2) converted straight to
//              E4M3 for the PV MMA; the epilogue writes bf16 out or the split-KV partial state.
#include <cuda_fp8.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "launch.h"

namespace bskv {
namespace {

using namespace dev;

constexpr int kRows = 64;                     // gathered rows per tile
constexpr int kStages = 3;
constexpr int kThreads = 512;
constexpr uint32_t kNopePanelQ = 128 * 128;   // [128 heads x 128 B]
constexpr uint32_t kRopePanelQ = 128 * 64;    // [128 heads x 64 B]
constexpr uint32_t kQBytes = 4 * kNopePanelQ + kRopePanelQ;  // 72 KB
constexpr uint32_t kNopePanelK = kRows * 128;  // 8 KB
constexpr uint32_t kRopePanelK = kRows * 64;   // 4 KB
constexpr uint32_t kStageBytes = 4 * kNopePanelK + kRopePanelK;  // 36 KB
constexpr uint32_t kPBytes = 128 * 64;         // [128 heads x 64 tokens] E4M3
constexpr uint32_t kSmemQ = 0;
constexpr uint32_t kSmemKV = kSmemQ + kQBytes;
constexpr uint32_t kSmemP = kSmemKV + kStages * kStageBytes;
constexpr uint32_t kSmemBar = kSmemP + 2 * kPBytes;
constexpr uint32_t kSmemIdx = kSmemBar + 512;  // [stages][64] sanitised row ids
// [3][2 groups][128]: row maxima by tile parity (slots 0, 1) and row sums (slot 2)
constexpr uint32_t kSmemRed = kSmemIdx + kStages * kRows * 4;
constexpr uint32_t kSmemBytes = kSmemRed + 3 * 2 * 128 * 4;
constexpr int kGatherThreads = 96;  // per group
constexpr uint32_t kTmemCols = 512;
constexpr int kVD = kMlaVDim;  // 256

struct MlaParams {
  const int32_t* meta;
  const uint8_t* kv;
  int64_t num_rows;
  const int32_t* indices;
  int top_k, heads;
  float scale_log2;  // bmm1_scale * log2(e)
  float bmm2;
  __nv_bfloat16* out;
  float* lse;
  float* ws_o;
  float* ws_lse;
  StatusArgs st;
};

struct Bars {
  uint64_t q_full, q_empty, drain;
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done, o_free;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ __half2 h2exp2_approx(__half2 x) {
  uint32_t in = *reinterpret_cast<uint32_t*>(&x), out;
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(out) : "r"(in));
  return *reinterpret_cast<__half2*>(&out);
}

// Two f16 values (low, high) to E4M3 (low byte, high byte), round to nearest even, saturating.
__device__ __forceinline__ uint32_t half2_to_e4m3x2(__half2 x) {
  const uint32_t in = *reinterpret_cast<uint32_t*>(&x);
  uint16_t out;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(out) : "r"(in));
  return out;
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_kernel(const __grid_constant__ CUtensorMap qmap_nope,
               const __grid_constant__ CUtensorMap qmap_rope,
               const __grid_constant__ CUtensorMap kvmap_nope,
               const __grid_constant__ CUtensorMap kvmap_rope, const MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  Bars& B = *reinterpret_cast<Bars*>(sm + kSmemBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* hdr = p.meta;
  const int32_t* wptr = hdr + hdr[H_OFF_WORKERS];
  const int4* chunks = reinterpret_cast<const int4*>(hdr + hdr[H_OFF_CHUNKS]);
  const int c0 = wptr[blockIdx.x], c1 = wptr[blockIdx.x + 1];
  const bool forced = forced_timeout(p.st);

  if (threadIdx.x == 0) {
    mbar_init(&B.q_full, 1);
    mbar_init(&B.q_empty, 1);
    mbar_init(&B.drain, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&B.kv_full[s], kGatherThreads);
      mbar_init(&B.kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&B.s_full[b], 1);
      mbar_init(&B.p_full[b], 256);
    }
    mbar_init(&B.o_done, 1);
    mbar_init(&B.o_free, 256);
    B.abort = 0;
    fence_mbar_init();
  }
  if (warp == 6) {
    tmem_alloc(&B.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = B.tmem_base;
  volatile int* abort_flag = &B.abort;

  if (warp < 6) {
    // -------------------------------------------------------------- gather groups
    // Group grp (0/1) owns the tiles with kvc % 2 == grp. A tile is published (kv_full, 128
    // arrivals) once the group's own copies of it are complete, so no tile waits for the
    // issue of another; with three stages, gathering tile t only needs the stage released by
    // PV(t-3), which the MMA issues after QK(t-2): no cycle. Decisions of a group go through
    // bar_and on its own named barrier (1 + grp, 96 threads).
    const int grp = threadIdx.x / kGatherThreads;
    const int pt = threadIdx.x % kGatherThreads;
    const uint32_t bar_id = 1 + grp;
    int32_t* idx_smem = reinterpret_cast<int32_t*>(sm + kSmemIdx);
    // This thread's 24 chunks of a tile: chunk id pt + 96 k -> (row, 16-byte column).
    constexpr int kPer = (kRows * 36) / kGatherThreads;
    uint32_t off[kPer];
    uint16_t col[kPer];
    uint8_t rowk[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int cid = pt + kGatherThreads * k;
      const int r = cid / 36, q = cid % 36;
      off[k] = q < 32 ? (q >> 3) * kNopePanelK + r * 128 + (((q & 7) ^ (r & 7)) << 4)
                      : 4 * kNopePanelK + r * 64 + ((((q - 32) & 3) ^ ((r >> 1) & 3)) << 4);
      col[k] = uint16_t(q * 16);
      rowk[k] = uint8_t(r);
    }
    uint32_t qc = 0, kvc = 0;
    bool ok = true;
    for (int ci = c0; ci < c1 && ok; ++ci) {
      const int4 ch = chunks[ci];
      const int n = ch.x / kMlaVSplit;
      const int32_t* idx_row = p.indices + int64_t(n) * p.top_k;
      bool good = true;
      if (grp == 0 && pt == 0) {
        good = !*abort_flag && mbar_wait(&B.q_empty, (qc & 1u) ^ 1u, p.st, forced);
        if (good) {
          mbar_arrive_expect_tx(&B.q_full, kQBytes);
          for (int pn = 0; pn < 4; ++pn)
            tma_load_2d(sm + kSmemQ + pn * kNopePanelQ, &qmap_nope, pn * 128, n * p.heads, &B.q_full);
          tma_load_2d(sm + kSmemQ + 4 * kNopePanelQ, &qmap_rope, 512, n * p.heads, &B.q_full);
        }
      }
      if (grp == 0) ++qc;
      ok = bar_and(bar_id, kGatherThreads, good);
      if (!ok) break;
      for (int t0 = ch.y; t0 < ch.z; t0 += kRows, ++kvc) {
        if ((kvc & 1u) != uint32_t(grp)) continue;
        const int s = kvc % kStages;
        int32_t my_id = 0;
        if (pt < kRows && t0 + pt < ch.z) {
          my_id = __ldg(idx_row + t0 + pt);
          if (my_id < 0 || my_id >= p.num_rows) {
            record_error(p.st, BSKV_ERR_DEVICE_INDEX);
            my_id = 0;
          }
        }
        good = !*abort_flag && mbar_wait(&B.kv_empty[s], ((kvc / kStages) & 1u) ^ 1u, p.st, forced);
        int32_t* ib = idx_smem + s * kRows;
        if (pt < kRows) ib[pt] = my_id;
        ok = bar_and(bar_id, kGatherThreads, good);
        if (!ok) break;
        uint8_t* stage = sm + kSmemKV + s * kStageBytes;
        const int valid = ch.z - t0;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          if (rowk[k] < valid)
            cp_async_16(stage + off[k], p.kv + int64_t(ib[rowk[k]]) * 576 + col[k]);
          else
            *reinterpret_cast<uint4*>(stage + off[k]) = make_uint4(0, 0, 0, 0);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async_smem();
        mbar_arrive(&B.kv_full[s]);
      }
    }
    if (!ok) *abort_flag = 1;
    if (grp == 0 && pt == 0 && qc > 0 && !ok) mbar_wait(&B.q_full, (qc - 1) & 1u, p.st, false);
  } else if (warp == 6) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = umma_idesc(128, 64, 0, 0, 0, 0);
      constexpr uint32_t idesc_pv = umma_idesc(128, kVD, 0, 0, 0, 1);
      const uint32_t sbase = smem_u32(sm);
      uint32_t qc = 0, kvc = 0, G = 0, cc = 0;
      bool ok = true;
      const uint64_t dp = umma_desc(sbase + kSmemP, 16, 512, kSwz64);
      const uint64_t dv = umma_desc(sbase + kSmemKV, kNopePanelK, 1024, kSwz128);
      auto pv = [&](uint32_t g, uint32_t kv_use, bool first, int vh) -> bool {
        const int s = kv_use % kStages;
        const uint32_t b = g & 1u;
        if (*abort_flag || !mbar_wait(&B.p_full[b], (g >> 1) & 1u, p.st, forced)) return false;
        if (first && (*abort_flag || !mbar_wait(&B.o_free, (cc & 1u) ^ 1u, p.st, forced))) return false;
        tc_fence_after();
        const uint64_t a0 = dp + ((b * kPBytes) >> 4);
        const uint64_t b0 = dv + ((s * kStageBytes + (2 * vh) * kNopePanelK) >> 4);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
          umma_f8(tmem, a0 + kk * 2, b0 + kk * 256, idesc_pv, (first && kk == 0) ? 0u : 1u);
        umma_commit(&B.o_done);
        umma_commit(&B.kv_empty[s]);
        return true;
      };
      // Descriptors are built once; a k-step only advances the start-address field
      // (bits 0-13, in 16-byte units), which cannot carry out for shared addresses.
      const uint64_t dq_n = umma_desc(sbase + kSmemQ, 16, 1024, kSwz128);
      const uint64_t dq_r = umma_desc(sbase + kSmemQ + 4 * kNopePanelQ, 16, 512, kSwz64);
      const uint64_t dk_n = umma_desc(sbase + kSmemKV, 16, 1024, kSwz128);
      const uint64_t dk_r = umma_desc(sbase + kSmemKV + 4 * kNopePanelK, 16, 512, kSwz64);
      for (int ci = c0; ci < c1 && ok; ++ci) {
        const int4 ch = chunks[ci];
        const int vh = ch.x % kMlaVSplit;
        const int nt = (ch.z - ch.y + kRows - 1) / kRows;
        if (*abort_flag || !mbar_wait(&B.q_full, qc & 1u, p.st, forced)) { ok = false; break; }
        ++qc;
        tc_fence_after();
        const uint32_t kv_first = kvc;
        for (int t = 0; t < nt; ++t, ++kvc) {
          const int s = kvc % kStages;
          if (*abort_flag || !mbar_wait(&B.kv_full[s], (kvc / kStages) & 1u, p.st, forced)) { ok = false; break; }
          tc_fence_after();
          const uint32_t so = (s * kStageBytes) >> 4;
          const uint32_t sd = tmem + 256 + ((G + t) & 1u) * 64;
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {
            const uint32_t qo = ((kk >> 2) * kNopePanelQ + (kk & 3) * 32) >> 4;
            const uint32_t ko = ((kk >> 2) * kNopePanelK + (kk & 3) * 32) >> 4;
            umma_f8(sd, dq_n + qo, dk_n + so + ko, idesc_qk, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            umma_f8(sd, dq_r + kk * 2, dk_r + so + kk * 2, idesc_qk, 1u);
          umma_commit(&B.s_full[(G + t) & 1u]);
          if (t >= 1 && !pv(G + t - 1, kv_first + t - 1, t == 1, vh)) { ok = false; break; }
        }
        if (!ok) break;
        if (!pv(G + nt - 1, kv_first + nt - 1, nt == 1, vh)) { ok = false; break; }
        umma_commit(&B.q_empty);
        G += nt;
        ++cc;
      }
      if (!ok) *abort_flag = 1;
      umma_commit(&B.drain);
      mbar_wait(&B.drain, 0, p.st, false);
    }
  } else if (warp >= 8) {
    // -------------------------------------------------------------- softmax warpgroups
    const int wg = (warp - 8) >> 2;          // 0: columns 0-31 / O 0-127; 1: 32-63 / 128-255
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;            // head
    const uint32_t lane_base = uint32_t(q4 * 32) << 16;
    float* red = reinterpret_cast<float*>(sm + kSmemRed);  // [parity][group][row]
    uint32_t G = 0, od = 0;
    bool ok = true;
    for (int ci = c0; ci < c1 && ok; ++ci) {
      const int4 ch = chunks[ci];
      const int n = ch.x / kMlaVSplit, vh = ch.x % kMlaVSplit;
      const int nt = (ch.z - ch.y + kRows - 1) / kRows;
      float m_run = -INFINITY, l_run = 0.f;
      for (int t = 0; t < nt; ++t, ++G) {
        const uint32_t b = G & 1u;
        bool good = warp_wait(&B.s_full[b], (G >> 1) & 1u, p.st, forced, abort_flag);
        uint32_t sr[32];
        if (good) {
          tc_fence_after();
          tmem_ld32(tmem + lane_base + 256 + b * 64 + wg * 32, sr);
          tmem_ld_wait();
        }
        const int valid = min(kRows, ch.z - (ch.y + t * kRows)) - wg * 32;
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float x = c < valid ? __uint_as_float(sr[c]) * p.scale_log2 : -INFINITY;
          sr[c] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
        red[(b * 2 + wg) * 128 + r] = mx;
        // both groups meet here once per tile (named barrier 3, 256 threads)
        ok = bar_and(3, 256, good);
        if (!ok) break;
        mx = fmaxf(mx, red[(b * 2 + (wg ^ 1)) * 128 + r]);
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
        // p = 2^(x - ref) in f16x2 pairs, straight to E4M3 pairs; partial row sum in f16x2.
        uint32_t pk[8];
        __half2 hsum = __float2half2_rn(0.f);
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const __half2 h0 = __floats2half2_rn(__uint_as_float(sr[c]) - ref, __uint_as_float(sr[c + 1]) - ref);
          const __half2 h1 = __floats2half2_rn(__uint_as_float(sr[c + 2]) - ref, __uint_as_float(sr[c + 3]) - ref);
          const __half2 e0 = h2exp2_approx(h0), e1 = h2exp2_approx(h1);
          hsum = __hadd2(hsum, __hadd2(e0, e1));
          pk[c / 4] = half2_to_e4m3x2(e0) | (half2_to_e4m3x2(e1) << 16);
        }
        const float2 fs = __half22float2(hsum);
        l_run = l_run * alpha + (fs.x + fs.y);
        m_run = m_use;
        rescale = __any_sync(0xffffffffu, rescale);
        while (od < G) {
          if (!warp_wait(&B.o_done, od & 1u, p.st, forced, abort_flag)) { ok = false; break; }
          ++od;
        }
        if (!ok) break;
        // this group's two 16-byte chunks (2 wg, 2 wg + 1) of the 64-byte P row, SW64 layout
        uint8_t* prow = sm + kSmemP + b * kPBytes + r * 64;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int cc = 2 * wg + c;
          *reinterpret_cast<uint4*>(prow + ((cc ^ ((r >> 1) & 3)) << 4)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        if (rescale && t > 0) {
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < kVD / 2; cc += 32) {
            uint32_t ov[32];
            const uint32_t ta = tmem + lane_base + wg * (kVD / 2) + cc;
            tmem_ld32(ta, ov);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
            tmem_st32(ta, ov);
          }
          tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&B.p_full[b]);
      }
      if (!ok) break;
      // Epilogue: combine the two partial row sums, then each group stores its 128 values.
      red[(4 + wg) * 128 + r] = l_run;
      ok = bar_and(3, 256, true);
      if (!ok) break;
      const float l_tot = red[4 * 128 + r] + red[5 * 128 + r];
      while (od < G) {
        if (!warp_wait(&B.o_done, od & 1u, p.st, forced, abort_flag)) { ok = false; break; }
        ++od;
      }
      if (!ok) break;
      tc_fence_after();
      const float scale = l_tot > 0.f ? p.bmm2 / l_tot : 0.f;
      const float lse = l_tot > 0.f ? (m_run + __log2f(l_tot)) * kLn2 : -INFINITY;
      const bool row_ok = r < p.heads;
      const int slot = ch.w;
#pragma unroll 1
      for (int cc = 0; cc < kVD / 2; cc += 32) {
        uint32_t ov[32];
        tmem_ld32(tmem + lane_base + wg * (kVD / 2) + cc, ov);
        tmem_ld_wait();
        if (!row_ok) continue;
        const int col = wg * (kVD / 2) + cc;
        if (slot < 0) {
          __nv_bfloat16* dst = p.out + (int64_t(n) * p.heads + r) * 512 + vh * kVD + col;
#pragma unroll
          for (int c = 0; c < 32; c += 8) {
            uint4 w;
            __nv_bfloat162 h0 = __floats2bfloat162_rn(__uint_as_float(ov[c]) * scale, __uint_as_float(ov[c + 1]) * scale);
            __nv_bfloat162 h1 = __floats2bfloat162_rn(__uint_as_float(ov[c + 2]) * scale, __uint_as_float(ov[c + 3]) * scale);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(ov[c + 4]) * scale, __uint_as_float(ov[c + 5]) * scale);
            __nv_bfloat162 h3 = __floats2bfloat162_rn(__uint_as_float(ov[c + 6]) * scale, __uint_as_float(ov[c + 7]) * scale);
            w.x = *reinterpret_cast<uint32_t*>(&h0);
            w.y = *reinterpret_cast<uint32_t*>(&h1);
            w.z = *reinterpret_cast<uint32_t*>(&h2);
            w.w = *reinterpret_cast<uint32_t*>(&h3);
            *reinterpret_cast<uint4*>(dst + c) = w;
          }
        } else {
          float* dst = p.ws_o + (int64_t(slot) * 128 + r) * kVD + col;
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            *reinterpret_cast<float4*>(dst + c) =
                make_float4(__uint_as_float(ov[c]) * scale, __uint_as_float(ov[c + 1]) * scale,
                            __uint_as_float(ov[c + 2]) * scale, __uint_as_float(ov[c + 3]) * scale);
        }
      }
      if (row_ok && wg == 0) {
        if (slot < 0) {
          if (p.lse && vh == 0) p.lse[int64_t(n) * p.heads + r] = lse;
        } else {
          p.ws_lse[int64_t(slot) * 128 + r] = lse;
        }
      }
      tc_fence_before();
      mbar_arrive(&B.o_free);
    }
    if (!ok) *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 6) tmem_dealloc(tmem, kTmemCols);
}

// Merge split-KV pieces of (query token, latent half) units; zero-fill empty ones.
__global__ void __launch_bounds__(128)
    mla_merge_kernel(const int32_t* __restrict__ meta, const float* __restrict__ ws_o,
                     const float* __restrict__ ws_lse, int heads, __nv_bfloat16* __restrict__ out,
                     float* __restrict__ lse) {
  const int NM = meta[H_MERGES];
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= NM * heads) return;
  const int item = gw / heads, h = gw % heads;
  const int32_t* mi = meta + meta[H_OFF_MERGES] + 3 * item;
  const int unit = mi[0], first = mi[1], count = mi[2];
  const int n = unit / kMlaVSplit, vh = unit % kMlaVSplit;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float lse_out = -INFINITY;
  if (count > 0) {
    float mx = -INFINITY;
    for (int c = lane; c < count; c += 32) mx = fmaxf(mx, ws_lse[int64_t(first + c) * 128 + h]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    float tot = 0.f;
    if (mx > -INFINITY) {
      for (int c = 0; c < count; ++c) {
        const float wgt = expf(ws_lse[int64_t(first + c) * 128 + h] - mx);
        tot += wgt;
        const float4* src = reinterpret_cast<const float4*>(ws_o + (int64_t(first + c) * 128 + h) * kVD + lane * 8);
        const float4 x0 = src[0], x1 = src[1];
        acc[0] += wgt * x0.x; acc[1] += wgt * x0.y; acc[2] += wgt * x0.z; acc[3] += wgt * x0.w;
        acc[4] += wgt * x1.x; acc[5] += wgt * x1.y; acc[6] += wgt * x1.z; acc[7] += wgt * x1.w;
      }
      const float inv = 1.f / tot;
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] *= inv;
      lse_out = mx + logf(tot);
    }
  }
  __nv_bfloat16* dst = out + (int64_t(n) * heads + h) * 512 + vh * kVD + lane * 8;
  uint4 w;
  __nv_bfloat162 h0 = __floats2bfloat162_rn(acc[0], acc[1]);
  __nv_bfloat162 h1 = __floats2bfloat162_rn(acc[2], acc[3]);
  __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[4], acc[5]);
  __nv_bfloat162 h3 = __floats2bfloat162_rn(acc[6], acc[7]);
  w.x = *reinterpret_cast<uint32_t*>(&h0);
  w.y = *reinterpret_cast<uint32_t*>(&h1);
  w.z = *reinterpret_cast<uint32_t*>(&h2);
  w.w = *reinterpret_cast<uint32_t*>(&h3);
  *reinterpret_cast<uint4*>(dst) = w;
  if (lse && vh == 0 && lane == 0) lse[int64_t(n) * heads + h] = lse_out;
}

}  // namespace
}  // namespace bskv

using namespace bskv;

extern "C" bskv_status bskv_run_mla_sparse(const bskv_plan* plan, const void* query,
                                           const void* kv_rows, int64_t num_rows,
                                           const int32_t* indices, float bmm1_scale,
                                           float bmm2_scale, void* out, float* lse,
                                           void* float_ws, size_t float_ws_bytes, void* stream) {
  if (!plan || plan->kind != KIND_MLA) { set_error("run_mla_sparse: not an MLA plan"); return BSKV_ERR_INVALID_ARG; }
  if (!plan->meta_dev) { set_error("run_mla_sparse: plan not uploaded (bskv_plan_upload)"); return BSKV_ERR_INVALID_ARG; }
  if (plan->batch == 0) return BSKV_OK;
  if (!query || !kv_rows || !indices || !out) { set_error("run_mla_sparse: NULL tensor"); return BSKV_ERR_INVALID_ARG; }
  if (!aligned16(query) || !aligned16(kv_rows) || !aligned16(out) || (reinterpret_cast<uintptr_t>(indices) & 3)) {
    set_error("run_mla_sparse: tensors must be 16-byte aligned (indices 4-byte)");
    return BSKV_ERR_INVALID_ARG;
  }
  if (num_rows < 1) { set_error("run_mla_sparse: num_rows must be positive"); return BSKV_ERR_INVALID_ARG; }
  if (float_ws_bytes < plan->float_ws_bytes || (plan->float_ws_bytes && !float_ws)) {
    set_error("run_mla_sparse: float workspace of %zu bytes, %zu needed", float_ws_bytes, plan->float_ws_bytes);
    return BSKV_ERR_WORKSPACE_TOO_SMALL;
  }
  if (float_ws && !aligned16(float_ws)) { set_error("run_mla_sparse: float workspace must be 16-byte aligned"); return BSKV_ERR_INVALID_ARG; }
  const int64_t nq = int64_t(plan->batch) * plan->q_len;
  MlaParams mp{};
  mp.meta = plan->meta_dev;
  mp.kv = static_cast<const uint8_t*>(kv_rows);
  mp.num_rows = num_rows;
  mp.indices = indices;
  mp.top_k = plan->top_k;
  mp.heads = plan->num_qo_heads;
  mp.scale_log2 = bmm1_scale * 1.4426950408889634f;
  mp.bmm2 = bmm2_scale;
  mp.out = static_cast<__nv_bfloat16*>(out);
  mp.lse = lse;
  const int slots = meta_word(plan, H_SLOTS);
  mp.ws_o = static_cast<float*>(float_ws);
  mp.ws_lse = slots ? reinterpret_cast<float*>(static_cast<uint8_t*>(float_ws) +
                                               ((size_t(slots) * 128 * kVD * 4 + 255) & ~size_t(255)))
                    : nullptr;
  if (bskv_status s = status_args(&mp.st)) return s;
  CUtensorMap qn, qr;
  const uint64_t dims[2] = {576, uint64_t(nq * plan->num_qo_heads)};
  const uint64_t str[1] = {576};
  const uint32_t box_n[2] = {128, 128}, box_r[2] = {64, 128};
  if (bskv_status s = encode_tiled(&qn, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, query, dims, str, box_n,
                                   CU_TENSOR_MAP_SWIZZLE_128B))
    return s;
  if (bskv_status s = encode_tiled(&qr, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, query, dims, str, box_r,
                                   CU_TENSOR_MAP_SWIZZLE_64B))
    return s;
  CUtensorMap kn, kr;
  {
    const uint64_t kd[2] = {576, uint64_t(num_rows)};
    const uint32_t gb_n[2] = {128, 1}, gb_r[2] = {64, 1};
    if (bskv_status s = encode_tiled(&kn, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, kv_rows, kd, str, gb_n,
                                     CU_TENSOR_MAP_SWIZZLE_128B))
      return s;
    if (bskv_status s = encode_tiled(&kr, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, kv_rows, kd, str, gb_r,
                                     CU_TENSOR_MAP_SWIZZLE_64B))
      return s;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int grid = meta_word(plan, H_GRID);
  if (grid > 0) {
    const size_t smem = kSmemBytes + 1024;
    if (bskv_status s = cuda_check(cudaFuncSetAttribute(mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)),
                                   "mla: cudaFuncSetAttribute"))
      return s;
    mla_kernel<<<grid, kThreads, smem, st>>>(qn, qr, kn, kr, mp);
    if (bskv_status s = cuda_check(cudaGetLastError(), "mla kernel launch")) return s;
  }
  const int nm = meta_word(plan, H_MERGES);
  if (nm > 0) {
    const int warps = nm * plan->num_qo_heads;
    mla_merge_kernel<<<(warps + 3) / 4, 128, 0, st>>>(plan->meta_dev, mp.ws_o, mp.ws_lse,
                                                      plan->num_qo_heads, mp.out, lse);
    if (bskv_status s = cuda_check(cudaGetLastError(), "mla merge launch")) return s;
  }
  return BSKV_OK;
}
