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
// GB300 design (persistent, one CTA per SM, 12 warps). A tcgen05.mma costs about the same
// time for N = 64 and N = 128 and reaches the dense peak only at N = 256, so the column
// blocks of a row are taken in pairs: one step is S = Q K^T over 128 keys (N = 128) and
// O += P V over the same 128 keys (K = 128, N = head_dim = 128).
//   warp 0   TMA producer: Q tiles (3-D tensor map, 128B swizzle) once per unit; K and V of
//            a block pair into one stage ([128 keys x 128 B] panels), 2 stages (3 for g = 2);
//   warp 1   allocates 512 TMEM columns and issues the MMAs (the warp stays converged, one
//            elected lane executes them). With two M tiles the jobs alternate tile 0 /
//            tile 1 (ping-pong): while one warpgroup turns S into P, the tensor core runs
//            the other tile's PV and next QK. With one M tile, S is double
//            buffered instead. P is written back into TMEM over S (16-bit, two per column)
//            and feeds the PV MMA as its A operand; V is an MN-major shared-memory operand;
//   warps 4-7 / 8-11  one warpgroup per M tile: thread = row = TMEM lane. It reads its
//            S row once into registers (four loads, one wait), applies scale and the causal
//            mask, keeps a running max with lazy rescaling (O in TMEM is rescaled only when
//            the max grows by more than 2^8), forms P = 2^x (packed f16x2 for fp16 inputs)
//            and stores it over the S columns with tcgen05.st; the epilogue normalises O and
//            stores out and lse. With two M tiles each warp stages its 32 rows of a 64-value
//            panel (128B-swizzled, 4 KB) in shared memory and writes them with one tensor
//            store, so the output leaves in whole lines instead of one row per thread.
// The same engine serves the list-driven rows ("flashinfer.sparse",
// VariableBlockSparseAttentionWrapper; batch prefill over a paged KV cache): a unit is then a
// 64-token tile of a variable row block or of a request's queries, its keys a list of steps
// of up to 128 contiguous keys (paged: whole pages, one TMA box per page through a 5-D map of
// the cache). Columns past a step's last key, or past the causal limit of a row, are masked;
// V rows past the last key of a partial step (garbage slots of a page, rows the step did not
// load) are zeroed before PV so that 0 * NaN cannot reach O; rows past the tile's last token
// are computed but not stored.
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
constexpr int kThreads = 384;
constexpr uint32_t kKPanel = 64 * 128;          // [64 rows x 64 elements] of 16 bits
constexpr uint32_t kPairPanel = 128 * 128;      // [128 rows x 64 elements]
constexpr uint32_t kQTile = 2 * 128 * 128;      // [128 rows x 128 elements]: 2 panels
constexpr uint32_t kStageBytes = 4 * kPairPanel;  // K pair (2 panels) then V pair (2 panels)
constexpr uint32_t kTmemCols = 512;
// TMEM columns: O of M tile m at 256 m; S (and P over it) of slot z at 128 + 256 z.

struct TcParams {
  const int32_t* meta;
  void* out;
  int64_t o_s0, o_s1;
  float* lse;
  int64_t lse_st, lse_sh;  // lse element strides of a token and of a head
  int M, N, Hq, Hkv, group, causal;
  int step_words, page_size;  // list plans: words per key step; paged: tokens per page
  // per-block token mask (bits little-endian over (nnz, 64, 64): one 64-bit word per row of
  // a block, bit c = key c), or NULL
  const unsigned long long* mask;
  float scale_log2;
  StatusArgs st;
};

template <int NM>
struct Cfg {
  static constexpr int kStages = NM == 2 ? 2 : 3;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kKV = kQ + NM * kQTile;
  // epilogue staging with two M tiles: one 4 KB box ([32 rows x 128 B]) per softmax warp
  static constexpr uint32_t kOut = kKV + kStages * kStageBytes;
  static constexpr uint32_t kOutBytes = NM == 2 ? 8 * 4096 : 0;
  static constexpr uint32_t kBar = kOut + kOutBytes;
  static constexpr uint32_t kBytes = kBar + 512;
};

struct Bars {
  uint64_t q_full[2], q_empty[2], drain;  // Q per M tile
  uint64_t kv_full[3], kv_empty[3];
  uint64_t s_full[2], p_half[2], p_full[2];  // per S slot: P of the first 64 keys / of all
  uint64_t o_done[2], o_free[2];  // per M tile
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

// P for two logits (log2 domain, reference subtracted): returns them packed in T and their
// values as float. fp16 uses the packed f16x2 exponential (P is fp16 anyway); bf16 keeps
// the fp32 exponential, since a bf16 argument would lose too much precision.
// Row-sum accumulator of P: for fp16, eight packed f16x2 partial sums (each takes at most
// 16 pairs of values <= 2^8 per 128-key step, well inside f16 range), turned into one float
// per step; for bf16, eight float partial sums.
template <typename T>
struct PSum;
template <>
struct PSum<__half> {
  __half2 h[8];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int q = 0; q < 8; ++q) h[q] = __float2half2_rn(0.f);
  }
  __device__ __forceinline__ float total() const {
    float2 a = __half22float2(__hadd2(__hadd2(h[0], h[1]), __hadd2(h[2], h[3])));
    float2 b = __half22float2(__hadd2(__hadd2(h[4], h[5]), __hadd2(h[6], h[7])));
    return (a.x + a.y) + (b.x + b.y);
  }
};
template <>
struct PSum<__nv_bfloat16> {
  float f[8];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int q = 0; q < 8; ++q) f[q] = 0.f;
  }
  __device__ __forceinline__ float total() const {
    return ((f[0] + f[1]) + (f[2] + f[3])) + ((f[4] + f[5]) + (f[6] + f[7]));
  }
};
template <typename T>
__device__ __forceinline__ uint32_t exp2_pack(float x0, float x1, PSum<T>& acc, int q);
template <>
__device__ __forceinline__ uint32_t exp2_pack<__half>(float x0, float x1, PSum<__half>& acc, int q) {
  const __half2 in = __floats2half2_rn(x0, x1);
  uint32_t out;
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(out) : "r"(*reinterpret_cast<const uint32_t*>(&in)));
  acc.h[q] = __hadd2(acc.h[q], *reinterpret_cast<const __half2*>(&out));
  return out;
}
template <>
__device__ __forceinline__ uint32_t exp2_pack<__nv_bfloat16>(float x0, float x1,
                                                              PSum<__nv_bfloat16>& acc, int q) {
  const float v0 = fast_exp2(x0), v1 = fast_exp2(x1);
  acc.f[q] += v0 + v1;
  return pack2(__nv_bfloat16(), v0, v1);
}

// A unit as every role sees it: tokens [tok0, tok0 + ntok) of the tile (ntok <= 64), kv
// head h, its blocks (BSR: indices[e0, e0 + n)) or its key steps (lists: steps e0 .. e0 +
// n - 1), and the causal key limit of its first token (row t sees keys <= lim + t).
struct Unit {
  int tok0, ntok, h, e0, n, lim;
};

// kMode 0: block-sparse; 1: block-sparse with a per-block token mask (a separate
// instantiation, so that the unmasked softmax carries none of its code); 2: variable
// blocks; 3: paged prefill (2 and 3 read their units and key steps from the plan's lists).
template <typename T, int NM, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    bsr_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
                  const TcParams p) {
  using L = Cfg<NM>;
  constexpr int S = L::kStages;
  constexpr bool kMask = kMode == 1;
  constexpr bool kList = kMode >= 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  Bars& B = *reinterpret_cast<Bars*>(sm + L::kBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* hdr = p.meta;
  const int32_t* wptr = hdr + hdr[H_OFF_WORKERS];
  const int4* units = reinterpret_cast<const int4*>(hdr + hdr[H_OFF_CHUNKS]);
  const int32_t* indptr = hdr + hdr[H_OFF_AUX0];   // lists: unit descriptors
  const int32_t* indices = hdr + hdr[H_OFF_AUX1];  // lists: key steps
  const int u0 = wptr[blockIdx.x], u1 = wptr[blockIdx.x + 1];
  const bool forced = forced_timeout(p.st);
  auto unit_of = [&](int ui) -> Unit {
    const int4 un = units[ui];
    Unit u;
    u.h = un.z;
    if constexpr (kList) {
      const int32_t* d = indptr + kBsrTcUnitWords * int64_t(un.x);
      u.tok0 = d[0];
      u.ntok = d[1];
      u.e0 = d[2];
      u.n = d[3] - d[2];
      u.lim = d[4];
    } else {
      const int i = un.y;
      u.tok0 = i * kBlk;
      u.ntok = min(kBlk, p.M - u.tok0);
      u.e0 = indptr[i];
      u.n = indptr[i + 1] - u.e0;
      u.lim = u.tok0 + (p.N - p.M);
    }
    return u;
  };
  // steps of a unit (a BSR step is a pair of blocks) and 64-key halves of step j
  auto nsteps = [&](const Unit& u) -> int { return kList ? u.n : (u.n + 1) >> 1; };
  auto step_halves = [&](const Unit& u, int j) -> int {
    if constexpr (kList) {
      const int32_t* st = indices + int64_t(p.step_words) * (u.e0 + j);
      return st[1] - st[0] > kBlk ? 2 : 1;
    } else {
      return min(2, u.n - 2 * j);
    }
  };

  if (threadIdx.x == 0) {
    for (int m = 0; m < 2; ++m) {
      mbar_init(&B.q_full[m], 1);
      mbar_init(&B.q_empty[m], 1);
    }
    mbar_init(&B.drain, 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(&B.kv_full[s], 1);
      mbar_init(&B.kv_empty[s], 1);
    }
    for (int z = 0; z < 2; ++z) {
      mbar_init(&B.s_full[z], 1);
      mbar_init(&B.p_half[z], 128);
      mbar_init(&B.p_full[z], 128);
      mbar_init(&B.o_done[z], 1);
      mbar_init(&B.o_free[z], 128);
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
    // Converged like the MMA issuer; the elected lane issues the copies.
    {
      const uint32_t leader = elect_leader();
      if (leader) {
        prefetch_tensormap(&qmap);
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
      }
      __syncwarp();
      uint32_t qc = 0, kvc = 0;
      uint32_t qi[2] = {0u, 0u};  // Q tiles issued
      // Q is read once (evict first); a K/V block serves every row block that lists it
      // (evict last), so it stays in L2 while the Q and output streams pass through.
      const uint64_t pol_q = l2_evict_first_policy(), pol_kv = l2_evict_last_policy();
      bool ok = true;
      // Q of M tile m for the unit (64 tokens from tok0, kv head h), once the previous unit's
      // last QK on that tile has completed.
      auto load_q = [&](int m, const Unit& u) -> bool {
        if (!issuer_wait(&B.q_empty[m], (qc & 1u) ^ 1u, p.st, forced, abort_flag)) return false;
        mbar_arrive_expect_tx_w(leader, &B.q_full[m], kQTile);
        for (int hl = 0; hl < 2; ++hl)
          for (int pn = 0; pn < 2; ++pn)
            tma_load_3d_hint_w(leader, sm + L::kQ + m * kQTile + pn * (kQTile / 2) + hl * kKPanel, &qmap,
                             pn * 64, u.h * p.group + m * 2 + hl, u.tok0, &B.q_full[m], pol_q);
        ++qi[m];
        return true;
      };
      // K and V of step j of the unit into the next stage: BSR, column blocks e0 + 2j and
      // e0 + 2j + 1; variable blocks, the keys from the step's start in 64-key boxes; paged
      // prefill, the step's pages, one box of page_size slots each.
      auto load_kv = [&](const Unit& u, int j) -> bool {
        const int s = kvc % S;
        if (!issuer_wait(&B.kv_empty[s], ((kvc / S) & 1u) ^ 1u, p.st, forced, abort_flag)) return false;
        uint8_t* dst = sm + L::kKV + s * kStageBytes;
        if constexpr (kMode == 3) {
          const int32_t* st = indices + int64_t(p.step_words) * (u.e0 + j);
          const int ps = p.page_size;
          const int npg = (st[1] - st[0] + ps - 1) / ps;
          mbar_arrive_expect_tx_w(leader, &B.kv_full[s], uint32_t(npg * ps * 128 * 4));
          for (int k = 0; k < npg; ++k) {
            const int page = st[2 + k];
            for (int pn = 0; pn < 2; ++pn) {
              tma_load_5d_hint_w(leader, dst + pn * kPairPanel + k * ps * 128, &kmap, pn * 64, 0, u.h, 0,
                                 page, &B.kv_full[s], pol_kv);
              tma_load_5d_hint_w(leader, dst + 2 * kPairPanel + pn * kPairPanel + k * ps * 128, &kmap,
                                 pn * 64, 0, u.h, 1, page, &B.kv_full[s], pol_kv);
            }
          }
        } else {
          const int nb = step_halves(u, j);
          mbar_arrive_expect_tx_w(leader, &B.kv_full[s], nb * 4 * kKPanel);
          const int k0 = kList ? indices[int64_t(p.step_words) * (u.e0 + j)] : 0;
          for (int b = 0; b < nb; ++b) {
            const int key = kList ? k0 + b * kBlk : indices[u.e0 + 2 * j + b] * kBlk;
            for (int pn = 0; pn < 2; ++pn) {
              tma_load_3d_hint_w(leader, dst + pn * kPairPanel + b * kKPanel, &kmap, pn * 64, u.h, key,
                               &B.kv_full[s], pol_kv);
              tma_load_3d_hint_w(leader, dst + 2 * kPairPanel + pn * kPairPanel + b * kKPanel, &vmap,
                               pn * 64, u.h, key, &B.kv_full[s], pol_kv);
            }
          }
        }
        ++kvc;
        return true;
      };
      for (int ui = u0; ui < u1 && ok; ++ui) {
        const Unit u = unit_of(ui);
        const int ns = nsteps(u);
        if (ns == 0) continue;
        // Order: Q of tile 0 (free one job before tile 1's), the first K/V step (its stage
        // is freed before tile 1's last QK completes), then Q of tile 1 and the other steps.
        ok = load_q(0, u) && load_kv(u, 0) && (NM == 1 || load_q(1, u));
        for (int j = 1; j < ns && ok; ++j) ok = load_kv(u, j);
        ++qc;
      }
      if (!ok) {
        *abort_flag = 1;
        for (int m = 0; m < 2; ++m)
          if (qi[m] > 0) mbar_wait(&B.q_full[m], (qi[m] - 1) & 1u, p.st, false);
        for (int s = 0; s < S; ++s) {
          if (kvc > uint32_t(s)) {
            const uint32_t last = ((kvc - 1 - s) / S) * S + s;
            mbar_wait(&B.kv_full[s], (last / S) & 1u, p.st, false);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // The warp stays converged through the loop; one elected lane executes the tcgen05
    // instructions (a lone lane in a divergent branch issues MMAs less than half as fast
    // while the softmax warps of its SM sub-partition are busy).
    {
      const uint32_t leader = elect_leader();
      constexpr uint32_t fmt = Fmt<T>::v;
      constexpr uint32_t idesc_qk128 = umma_idesc(128, 128, fmt, fmt, 0, 0);
      constexpr uint32_t idesc_qk64 = umma_idesc(128, 64, fmt, fmt, 0, 0);
      constexpr uint32_t idesc_pv = umma_idesc(128, 128, fmt, fmt, 0, 1);
      const uint32_t sbase = smem_u32(sm);
      // Descriptors are built once; steps advance the start-address field (16-byte units).
      const uint64_t dq = umma_desc(sbase + L::kQ, 16, 1024, kSwz128);
      const uint64_t dk = umma_desc(sbase + L::kKV, 16, 1024, kSwz128);
      const uint64_t dv = umma_desc(sbase + L::kKV + 2 * kPairPanel, kPairPanel, 1024, kSwz128);
      uint32_t qc = 0, kvc = 0, J = 0, uc = 0;
      bool ok = true;
      for (int ui = u0; ui < u1 && ok; ++ui) {
        const Unit u = unit_of(ui);
        const int steps = nsteps(u);
        if (steps == 0) continue;
        const int NJ = steps * NM;
        const uint32_t kv_first = kvc;
        // QK of local job jl into S slot (J + jl) & 1.
        auto qk = [&](int jl) -> bool {
          const int j = NM == 2 ? (jl >> 1) : jl;
          const int m = NM == 2 ? (jl & 1) : 0;
          const uint32_t step = kv_first + j;
          const int s = step % S;
          if (m == 0 && !issuer_wait(&B.kv_full[s], (step / S) & 1u, p.st, forced, abort_flag)) return false;
          if (jl < NM && !issuer_wait(&B.q_full[m], qc & 1u, p.st, forced, abort_flag)) return false;
          tc_fence_after();
          const int nb = step_halves(u, j);
          const uint32_t z = (J + jl) & 1u;
          const uint32_t sd = tmem + 128 + 256 * z;
          const uint32_t qo = (m * kQTile) >> 4, ko = (s * kStageBytes) >> 4;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t pq = ((kk >> 2) * (kQTile / 2) + (kk & 3) * 32) >> 4;
            const uint32_t pk = ((kk >> 2) * kPairPanel + (kk & 3) * 32) >> 4;
            umma_f16_w(leader, sd, dq + qo + pq, dk + ko + pk, nb == 2 ? idesc_qk128 : idesc_qk64,
                     kk > 0 ? 1u : 0u);
          }
          umma_commit_w(leader, &B.s_full[z]);
          // Q of tile m is not read after the unit's last QK on it: release it so the next
          // unit's Q loads while this unit's last jobs and epilogue run.
          if (jl == NJ - NM + m) umma_commit_w(leader, &B.q_empty[m]);
          return true;
        };
        if (!qk(0) || (NJ > 1 && !qk(1))) { ok = false; break; }
        for (int jl = 0; jl < NJ; ++jl) {
          const uint32_t Jg = J + jl, z = Jg & 1u;
          const int j = NM == 2 ? (jl >> 1) : jl;
          const int m = NM == 2 ? (jl & 1) : 0;
          if (!issuer_wait(kList ? &B.p_full[z] : &B.p_half[z], (Jg >> 1) & 1u, p.st, forced,
                           abort_flag)) { ok = false; break; }
          if (j == 0 && !issuer_wait(&B.o_free[m], (uc & 1u) ^ 1u, p.st, forced, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const int nb = step_halves(u, j);
          const int s = (kv_first + j) % S;
          const uint32_t vo = (s * kStageBytes) >> 4;
          const uint32_t pa = tmem + 128 + 256 * z;
          // a block pair is 8 MMAs (K = 16 keys each), a lone last block 4; a list step only
          // the 16-key slices that hold its keys (the V rows past them are zero, see softmax)
          if constexpr (kList) {
            const int32_t* st = indices + int64_t(p.step_words) * (u.e0 + j);
            const int nk = (st[1] - st[0] + 15) >> 4;
#pragma unroll 1
            for (int kk = 0; kk < nk; ++kk)
              umma_f16_ts_w(leader, tmem + 256 * m, pa + kk * 8, dv + vo + kk * (2048 >> 4), idesc_pv,
                            (j == 0 && kk == 0) ? 0u : 1u);
          } else if (nb == 2) {
            // a block pair: the first block's slices once its P is in TMEM, then the second's
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_f16_ts_w(leader, tmem + 256 * m, pa + kk * 8, dv + vo + kk * (2048 >> 4), idesc_pv,
                            (j == 0 && kk == 0) ? 0u : 1u);
            if (!issuer_wait(&B.p_full[z], (Jg >> 1) & 1u, p.st, forced, abort_flag)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int kk = 4; kk < 8; ++kk)
              umma_f16_ts_w(leader, tmem + 256 * m, pa + kk * 8, dv + vo + kk * (2048 >> 4), idesc_pv, 1u);
          } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_f16_ts_w(leader, tmem + 256 * m, pa + kk * 8, dv + vo + kk * (2048 >> 4), idesc_pv,
                            (j == 0 && kk == 0) ? 0u : 1u);
          }
          umma_commit_w(leader, &B.o_done[m]);
          if (m == NM - 1) umma_commit_w(leader, &B.kv_empty[s]);
          if (jl + 2 < NJ && !qk(jl + 2)) { ok = false; break; }
        }
        if (!ok) break;
        kvc = kv_first + steps;
        J += NJ;
        ++uc;
        ++qc;
      }
      if (!ok) *abort_flag = 1;
      umma_commit_w(leader, &B.drain);
      mbar_wait(&B.drain, 0, p.st, false);
    }
  } else if (warp >= 4 && warp < 4 + 4 * NM) {
    // ------------------------------------------------------------------ softmax warpgroups
    const int m = (warp - 4) >> 2;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;                    // row of the M tile = TMEM lane
    const uint32_t lane_base = uint32_t(q4 * 32) << 16;
    const int hl = m * 2 + r / kBlk;                 // head within the group
    uint32_t J = 0, cnt = 0, od = 0;
    uint32_t kvs = 0;  // K/V steps of the previous units (the stage of step j is (kvs + j) % S)
    bool ok = true;
    for (int ui = u0; ui < u1 && ok; ++ui) {
      const Unit u = unit_of(ui);
      const int t64 = r % kBlk;  // token of this row within the unit's 64
      const bool row_ok = t64 < u.ntok;
      const int tok = u.tok0 + t64;
      const int head = u.h * p.group + hl;
      // this row's output and lse (formed where they are written, not held across the steps)
      auto out_row = [&]() {
        return static_cast<T*>(p.out) + int64_t(tok) * p.o_s0 + int64_t(head) * p.o_s1;
      };
      auto lse_at = [&]() -> float& { return p.lse[int64_t(tok) * p.lse_st + int64_t(head) * p.lse_sh]; };
      const int steps = nsteps(u);
      if (steps == 0) {
        if (row_ok) {
          T* orow = out_row();
          for (int c = 0; c < kD; c += 8) *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
          if (p.lse) lse_at() = -INFINITY;
        }
        continue;
      }
      const int lim = u.lim + t64;  // causal: the last key this row sees
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < steps; ++j) {
        const uint32_t Jg = J + (NM == 2 ? 2 * j + m : j), z = Jg & 1u;
        // the step's column blocks (lists: key range) are read before waiting for S (off the
        // critical path)
        const int nb = step_halves(u, j);
        int jb0 = 0, jb1 = 0, kvalid = 2 * kBlk, cmax = 2 * kBlk;
        if constexpr (kList) {
          const int32_t* st = indices + int64_t(p.step_words) * (u.e0 + j);
          kvalid = st[1] - st[0];
          // columns at or past cmax are masked: past the step's keys, or past the causal limit
          cmax = p.causal ? min(kvalid, lim - st[0] + 1) : kvalid;
        } else {
          jb0 = indices[u.e0 + 2 * j];
          jb1 = nb == 2 ? indices[u.e0 + 2 * j + 1] : jb0;
        }
        // this row's token-mask words of the step's blocks, read before the wait as well
        unsigned long long mw0 = ~0ull, mw1 = ~0ull;
        if (kMask) {
          mw0 = __ldg(p.mask + (int64_t(u.e0 + 2 * j) * kBlk + (r & (kBlk - 1))));
          if (nb == 2) mw1 = __ldg(p.mask + (int64_t(u.e0 + 2 * j + 1) * kBlk + (r & (kBlk - 1))));
        }
        if (!warp_wait(&B.s_full[z], (Jg >> 1) & 1u, p.st, forced, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t scol = tmem + lane_base + 128 + 256 * z;
        // The whole S row goes to registers in one read; P may then overwrite it in TMEM.
        uint32_t sr[128];
        tmem_ld32(scol, sr);
        tmem_ld32(scol + 32, sr + 32);
        if (nb == 2) {
          tmem_ld32(scol + 64, sr + 64);
          tmem_ld32(scol + 96, sr + 96);
        }
        tmem_ld_wait();
        // row max as 8 independent partial maxima (short dependency chains)
        float mxp[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) mxp[q] = -INFINITY;
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          if (bb < nb) {
            if constexpr (kList) {
              if (cmax < 64 * (bb + 1)) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                  if (64 * bb + c >= cmax) sr[64 * bb + c] = __float_as_uint(-INFINITY);
              }
            } else {
              const int k0 = (bb ? jb1 : jb0) * kBlk;
              const unsigned long long mw = bb ? mw1 : mw0;
              if (kMask && mw != ~0ull) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                  if (!((mw >> c) & 1ull)) sr[64 * bb + c] = __float_as_uint(-INFINITY);
              }
              if (p.causal && (k0 + kBlk - 1 > lim)) {
#pragma unroll
                for (int c = 0; c < 64; ++c)
                  if (k0 + c > lim) sr[64 * bb + c] = __float_as_uint(-INFINITY);
              }
            }
#pragma unroll
            for (int c = 0; c < 64; c += 2)
              mxp[(c >> 1) & 7] = fmax3(mxp[(c >> 1) & 7], __uint_as_float(sr[64 * bb + c]),
                                        __uint_as_float(sr[64 * bb + c + 1]));
          }
        }
        float mx = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                         fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
        mx *= p.scale_log2;
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
        rescale = __any_sync(0xffffffffu, rescale);
        // All earlier PVs into this tile's O must be complete before a rescale. With two M
        // tiles that is already implied: this tile's previous PV was issued before the QK
        // whose completion produced S, so exactly cnt PVs have completed (od = cnt keeps the
        // phase count exact for the epilogue's wait). With one tile, wait for it.
        if (NM == 2) {
          od = cnt;
        } else {
          while (od < cnt) {
            if (!warp_wait(&B.o_done[m], od & 1u, p.st, forced, abort_flag)) { ok = false; break; }
            ++od;
          }
          if (!ok) break;
        }
        // P = 2^(s * scale - ref), 32 keys at a time into packed columns [16 ck, 16 ck + 16).
        // Block-sparse steps hand the first block's P to the issuer before forming the
        // second's (its PV slices start meanwhile); O is rescaled in between, when the S row's
        // first half no longer holds registers.
        PSum<T> sp;
        sp.zero();
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nr2 = make_float2(-ref, -ref);
#pragma unroll
        for (int ck = 0; ck < 2; ++ck) {
          {  // keys 32 ck .. 32 ck + 31 of the first block
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              const float2 x = ffma2(make_float2(__uint_as_float(sr[32 * ck + c]),
                                                 __uint_as_float(sr[32 * ck + c + 1])),
                                     sc2, nr2);
              pk[c / 2] = exp2_pack<T>(x.x, x.y, sp, (c >> 1) & 7);
            }
            tmem_st16(scol + 16 * ck, pk);
          }
        }
        if (rescale && j > 0) {
#pragma unroll 1
          for (int cc = 0; cc < kD; cc += 32) {
            uint32_t ov[32];
            tmem_ld32(tmem + lane_base + 256 * m + cc, ov);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
            tmem_st32(tmem + lane_base + 256 * m + cc, ov);
          }
        }
        if constexpr (kList) {
          // V rows of a partial step past its last key up to the next multiple of 16 (a page's
          // unused slots, rows no box of this step wrote), which the step's last PV slice
          // reads, are zeroed before PV: their P is 0, but 0 * NaN is not. The first M tile's
          // PV is issued before the second's, so its warpgroup does it.
          if (m == 0 && r >= kvalid && r < ((kvalid + 15) & ~15)) {
            uint8_t* vrow = sm + L::kKV + ((kvs + j) % S) * kStageBytes + 2 * kPairPanel + r * 128;
#pragma unroll
            for (int pn = 0; pn < 2; ++pn)
#pragma unroll
              for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4*>(vrow + pn * kPairPanel + c * 16) = make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
          }
        }
        if constexpr (!kList) {
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&B.p_half[z]);
        }
#pragma unroll
        for (int ck = 2; ck < 4; ++ck) {
          if (ck < 2 * nb) {
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 32; c += 2) {
              const float2 x = ffma2(make_float2(__uint_as_float(sr[32 * ck + c]),
                                                 __uint_as_float(sr[32 * ck + c + 1])),
                                     sc2, nr2);
              pk[c / 2] = exp2_pack<T>(x.x, x.y, sp, (c >> 1) & 7);
            }
            tmem_st16(scol + 16 * ck, pk);
          }
        }
        const float sum = sp.total();
        l_run = l_run * alpha + sum;
        m_run = m_use;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&B.p_full[z]);
        ++cnt;
      }
      if (!ok) break;
      J += steps * NM;
      kvs += steps;
      // Epilogue: wait for the unit's last PV into this tile, normalise and store.
      while (od < cnt) {
        if (!warp_wait(&B.o_done[m], od & 1u, p.st, forced, abort_flag)) { ok = false; break; }
        ++od;
      }
      if (!ok) break;
      tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      if constexpr (NM == 2) {
        // Rows q4*32 .. q4*32+31 of the tile are 32 consecutive tokens of one head: per
        // 64-value panel, lane = token row of a [32 x 128 B] box (16-byte chunk c at
        // c ^ (row & 7)), then lane 0 stores the box. Tokens past M are clipped by the store.
        uint8_t* stg = sm + L::kOut + (m * 4 + q4) * 4096;
        const uint64_t pol_out = l2_evict_first_policy();  // written once
        const uint32_t row_addr = smem_u32(stg) + lane * 128;
        // a warp whose 32 tokens are not all in the unit (the last tile of a row range) stores
        // its valid rows one by one instead: a box would reach into the next unit's rows
        const bool full_box = (q4 & 1) * 32 + 32 <= u.ntok;
        T* orow = out_row();
#pragma unroll 1
        for (int pn = 0; pn < 2 && !full_box; ++pn) {
#pragma unroll 1
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t ov[32];
            tmem_ld32(tmem + lane_base + 256 * m + pn * 64 + hf * 32, ov);
            tmem_ld_wait();
            if (row_ok) {
#pragma unroll
              for (int c = 0; c < 32; c += 8) {
                uint4 w;
                w.x = pack2(T(), __uint_as_float(ov[c]) * inv, __uint_as_float(ov[c + 1]) * inv);
                w.y = pack2(T(), __uint_as_float(ov[c + 2]) * inv, __uint_as_float(ov[c + 3]) * inv);
                w.z = pack2(T(), __uint_as_float(ov[c + 4]) * inv, __uint_as_float(ov[c + 5]) * inv);
                w.w = pack2(T(), __uint_as_float(ov[c + 6]) * inv, __uint_as_float(ov[c + 7]) * inv);
                *reinterpret_cast<uint4*>(orow + pn * 64 + hf * 32 + c) = w;
              }
            }
          }
        }
#pragma unroll 1
        for (int pn = 0; pn < 2 && full_box; ++pn) {
          // the box's previous store has finished reading it
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
#pragma unroll 1
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t ov[32];
            tmem_ld32(tmem + lane_base + 256 * m + pn * 64 + hf * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              const int c = c4 * 8, c8 = hf * 4 + c4;
              uint4 w;
              w.x = pack2(T(), __uint_as_float(ov[c]) * inv, __uint_as_float(ov[c + 1]) * inv);
              w.y = pack2(T(), __uint_as_float(ov[c + 2]) * inv, __uint_as_float(ov[c + 3]) * inv);
              w.z = pack2(T(), __uint_as_float(ov[c + 4]) * inv, __uint_as_float(ov[c + 5]) * inv);
              w.w = pack2(T(), __uint_as_float(ov[c + 6]) * inv, __uint_as_float(ov[c + 7]) * inv);
              sts128(row_addr + ((c8 ^ (lane & 7)) << 4), w);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d_hint(&omap, stg, pn * 64, head, u.tok0 + (q4 & 1) * 32, pol_out);
            bulk_commit();
          }
        }
      } else {
        T* orow = out_row();
#pragma unroll
        for (int cc = 0; cc < kD; cc += 32) {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_base + 256 * m + cc, ov);
          tmem_ld_wait();
          if (row_ok) {
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
      }
      if (row_ok && p.lse) lse_at() = l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
      tc_fence_before();
      mbar_arrive(&B.o_free[m]);
    }
    if (!ok) *abort_flag = 1;
    // the output stores must be complete before the CTA exits
    if (NM == 2 && lane == 0) bulk_wait_all0();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <typename T, int NM, int kMode>
bskv_status launch_t(const bskv_plan* plan, const CUtensorMap& qm, const CUtensorMap& km,
                     const CUtensorMap& vm, const CUtensorMap& om, const TcParams& tp,
                     cudaStream_t st) {
  const int grid = meta_word(plan, H_GRID);
  if (grid == 0) return BSKV_OK;
  const size_t smem = Cfg<NM>::kBytes + 1024;
  auto kern = bsr_tc_kernel<T, NM, kMode>;
  if (bskv_status s = cuda_check(
          cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)),
          "bsr_tc: cudaFuncSetAttribute"))
    return s;
  kern<<<grid, kThreads, smem, st>>>(qm, km, vm, om, tp);
  return cuda_check(cudaGetLastError(), "bsr_tc launch");
}

template <int kMode>
bskv_status launch_mode(const bskv_plan* plan, const CUtensorMap& qm, const CUtensorMap& km,
                        const CUtensorMap& vm, const CUtensorMap& om, const TcParams& tp,
                        cudaStream_t st) {
  const bool bf = plan->dtype == BSKV_BF16;
  if (tp.group == 4)
    return bf ? launch_t<__nv_bfloat16, 2, kMode>(plan, qm, km, vm, om, tp, st)
              : launch_t<__half, 2, kMode>(plan, qm, km, vm, om, tp, st);
  return bf ? launch_t<__nv_bfloat16, 1, kMode>(plan, qm, km, vm, om, tp, st)
            : launch_t<__half, 1, kMode>(plan, qm, km, vm, om, tp, st);
}

// Parameters and the Q / output tensor maps shared by every mode: q and out as (head_dim,
// head, token) with the caller's strides, boxes of 64 values x 1 head x 64 (Q) or 32 (out)
// tokens.
bskv_status tc_common(const bskv_plan* plan, const void* q, const int64_t* qs, void* out,
                      const int64_t* os, float* lse, float sm_scale, TcParams* tp,
                      CUtensorMap* qm, CUtensorMap* om) {
  const int g = plan->num_qo_heads / plan->num_kv_heads;
  if (!(plan->head_dim == kD && (g == 2 || g == 4))) {
    set_error("bsr_tc: the tensor-core kernel needs head_dim 128 and group 2 or 4");
    return BSKV_ERR_UNSUPPORTED;
  }
  *tp = TcParams{};
  tp->meta = plan->meta_dev;
  tp->out = out; tp->o_s0 = os[0]; tp->o_s1 = os[1];
  tp->lse = lse;
  tp->lse_st = plan->num_qo_heads;
  tp->lse_sh = 1;
  tp->M = plan->M; tp->N = plan->N; tp->Hq = plan->num_qo_heads; tp->Hkv = plan->num_kv_heads;
  tp->group = g; tp->causal = plan->causal;
  tp->scale_log2 = sm_scale_log2(sm_scale, plan->head_dim);
  if (bskv_status s = status_args(&tp->st)) return s;
  const CUtensorMapDataType dt =
      plan->dtype == BSKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint32_t box[3] = {64, 1, 64};
  const uint64_t dims[3] = {uint64_t(kD), uint64_t(plan->num_qo_heads), uint64_t(plan->M)};
  {
    const uint64_t str[2] = {uint64_t(qs[1]) * 2, uint64_t(qs[0]) * 2};
    if (bskv_status s = encode_tiled(qm, dt, 3, q, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return s;
  }
  if (g == 4) {
    // output boxes of 32 tokens x 1 head x 64 values (the epilogue's per-warp stores)
    const uint32_t obox[3] = {64, 1, 32};
    const uint64_t str[2] = {uint64_t(os[1]) * 2, uint64_t(os[0]) * 2};
    if (bskv_status s = encode_tiled(om, dt, 3, out, dims, str, obox, CU_TENSOR_MAP_SWIZZLE_128B)) return s;
  } else {
    *om = *qm;  // unused with one M tile
  }
  return BSKV_OK;
}

}  // namespace

bskv_status launch_bsr_tcgen05(const bskv_plan* plan, const void* q, const int64_t* qs,
                               const void* k, const int64_t* ks, const void* v,
                               const int64_t* vs, void* out, const int64_t* os, float* lse,
                               float sm_scale, const uint8_t* mask, cudaStream_t st) {
  const int variant = meta_word(plan, H_VARIANT);
  if (!(variant == BSR_TCGEN05 || variant == BSR_VARIABLE_TC) ||
      (variant == BSR_TCGEN05 && !(plan->R == kBlk && plan->C == kBlk))) {
    set_error("run_bsr: not a tensor-core block-sparse plan");
    return BSKV_ERR_INVALID_ARG;
  }
  TcParams tp;
  CUtensorMap qm, km, vm, om;
  if (bskv_status s = tc_common(plan, q, qs, out, os, lse, sm_scale, &tp, &qm, &om)) return s;
  tp.mask = reinterpret_cast<const unsigned long long*>(mask);
  if (variant == BSR_VARIABLE_TC) {
    // head-major lse [num_qo_heads, qo_len]
    tp.lse_st = 1;
    tp.lse_sh = plan->M;
    tp.step_words = 2;
  }
  const CUtensorMapDataType dt =
      plan->dtype == BSKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  {
    const uint32_t box[3] = {64, 1, 64};
    const uint64_t dims[3] = {uint64_t(kD), uint64_t(plan->num_kv_heads), uint64_t(plan->N)};
    const uint64_t sk[2] = {uint64_t(ks[1]) * 2, uint64_t(ks[0]) * 2};
    const uint64_t sv[2] = {uint64_t(vs[1]) * 2, uint64_t(vs[0]) * 2};
    if (bskv_status s = encode_tiled(&km, dt, 3, k, dims, sk, box, CU_TENSOR_MAP_SWIZZLE_128B)) return s;
    if (bskv_status s = encode_tiled(&vm, dt, 3, v, dims, sv, box, CU_TENSOR_MAP_SWIZZLE_128B)) return s;
  }
  if (variant == BSR_VARIABLE_TC) return launch_mode<2>(plan, qm, km, vm, om, tp, st);
  if (mask) return launch_mode<1>(plan, qm, km, vm, om, tp, st);
  return launch_mode<0>(plan, qm, km, vm, om, tp, st);
}

bskv_status launch_prefill_tcgen05(const bskv_plan* plan, const void* q, const int64_t* qs,
                                   const void* kv, const int64_t* kvs, void* out,
                                   const int64_t* os, float* lse, float sm_scale,
                                   cudaStream_t st) {
  if (meta_word(plan, H_VARIANT) != BSR_PAGED_PREFILL_TC || !bsr_tc_page_size(plan->page_size)) {
    set_error("run_prefill_paged: not a tensor-core paged prefill plan");
    return BSKV_ERR_INVALID_ARG;
  }
  for (int i = 0; i < 4; ++i)
    if (kvs[i] <= 0) {
      set_error("run_prefill_paged: kv strides must be positive for the tensor-core kernel");
      return BSKV_ERR_INVALID_ARG;
    }
  TcParams tp;
  CUtensorMap qm, km, om;
  if (bskv_status s = tc_common(plan, q, qs, out, os, lse, sm_scale, &tp, &qm, &om)) return s;
  tp.page_size = plan->page_size;
  tp.step_words = 2 + kBsrTcStep / plan->page_size;
  // the cache as (head_dim, slot, kv head, K/V, page), one page of one head per box
  const CUtensorMapDataType dt =
      plan->dtype == BSKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint64_t dims[5] = {uint64_t(kD), uint64_t(plan->page_size), uint64_t(plan->num_kv_heads), 2,
                            uint64_t(plan->num_pages)};
  const uint64_t strides[4] = {uint64_t(kvs[3]) * 2, uint64_t(kvs[2]) * 2, uint64_t(kvs[1]) * 2,
                               uint64_t(kvs[0]) * 2};
  const uint32_t box[5] = {64, uint32_t(plan->page_size), 1, 1, 1};
  if (bskv_status s = encode_tiled(&km, dt, 5, kv, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return s;
  return launch_mode<3>(plan, qm, km, km, om, tp, st);
}

}  // namespace bskv
