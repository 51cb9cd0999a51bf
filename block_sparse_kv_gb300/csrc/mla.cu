// Sparse MLA FP8 decode on the 5th-generation tensor cores (tcgen05 kind::f8f6f4 + TMEM).
//
// Method: "Sparse MLA" (MATE 0.2.6), sparse_mla_fp8_decode: E4M3 query [batch, q_len,
// heads, 576], E4M3 cache rows of 576 values (512 latent + 64 rotated), int32 physical-token
// indices [batch, q_len, top_k] shared by all heads, seq_lens[b] valid entries, bmm1_scale
// on the QK product and bmm2_scale on the output, BF16 output of 512 values and FP32 LSE;
// "FlashInfer Compatibility Wrapper", scale folding. V is the first 512 values of a row.
//
// GB300 design (persistent, clusters of two CTAs, one CTA per SM, 16 warps). A work unit is
// one query token; the two CTAs of a cluster take the same units, CTA rank v accumulating
// the 256 output values of latent half v in TMEM. Both compute the same S = Q K^T (128 heads
// = the M=128 rows, 128 gathered rows = N, K = 576), so each gathered row is needed by both:
// each CTA gathers half of a tile's rows and pushes them into its partner's shared memory.
// TMEM (512 columns): O (256), the query's 512 latent bytes as the E4M3 A operand of QK
// (128, four values per column), S (128). Shared memory: the query's 64-byte rotated tail,
// P (the hi and lo E4M3 terms of one tile), and the gathered tiles split by lifetime: a K part (the other
// latent half and the tail, freed once QK has read it; two slots) and a V part (the unit's
// latent half, freed after PV; three slots).
//   warps 0-5  gather: 192 threads copy this CTA's 64 rows of a tile (16-byte cp.async into
//              128B-swizzled panels), then the leader arms kv_full for the partner's half and
//              pushes this half to the partner with five shared-to-shared bulk copies. Row ids
//              are fetched one tile ahead. On a paged cache (the kPaged instantiation) a whole
//              tile is instead loaded by each CTA with TMA boxes of page slots, issued by one
//              thread: no cp.async and no push;
//   warp 6     allocates TMEM; one elected lane of the converged warp issues QK (16 MMAs
//              with A in TMEM, 2 with the tail in shared memory, N = 128) and PV (A = P in
//              shared memory, B = the V part read MN-major, N = 256; once for the hi and once
//              for the lo terms of P, into the same accumulator); slot releases are
//              committed to both CTAs' barriers;
//   warp 7     TMA-loads the query tail once per token;
//   warps 8-15 two softmax warpgroups; thread = head = TMEM lane, each group owns 64 of a
//              tile's columns and 128 of the 256 output values: it reads S (and releases it
//              for the next QK at once), combines the row max with the other group, applies
//              lazy rescaling (threshold 2^4), forms 16 P with packed f16x2 exponentials and
//              splits it into two E4M3 terms (hi = e4m3(16 P), lo = e4m3(16 P - hi)), and writes
//              O (bf16) or the split-KV partial state in the epilogue
//              (per warp, 128B-swizzled boxes in the idle P buffers and tensor stores); at a
//              token's last tile it also writes the next token's query into TMEM.
#include <cuda_fp8.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "launch.h"

namespace bskv {
namespace {

using namespace dev;

constexpr int kRows = 128;                    // gathered rows per tile
constexpr int kKSlots = 2;                    // K parts in flight (freed after QK)
constexpr int kVSlots = 3;                    // V parts in flight (freed after PV)
constexpr int kThreads = 512;
constexpr int kGatherThreads = 192;           // warps 0-5
constexpr int kHalfRows = kRows / 2;          // rows each CTA of the pair gathers per tile
constexpr uint32_t kPanel = kRows * 128;      // [128 rows x 128 B]: 16 KB
constexpr uint32_t kRopePanel = kRows * 64;   // [128 rows x 64 B]: 8 KB
constexpr uint32_t kKPart = 2 * kPanel + kRopePanel;  // other latent half + rotated tail
constexpr uint32_t kVPart = 2 * kPanel;               // the unit's latent half
// bytes of one CTA's half tile: 64 rows of the four 128-byte panels and of the 64-byte tail
constexpr uint32_t kHalfTileBytes = 4 * (kHalfRows * 128) + kHalfRows * 64;
constexpr uint32_t kPBytes = 128 * 128;               // [128 heads x 128 keys] E4M3
constexpr uint32_t kSmemQR = 0;                                  // query tail, 8 KB
constexpr uint32_t kSmemP = kSmemQR + kRopePanel;                // 2 x 16 KB
constexpr uint32_t kSmemK = kSmemP + 2 * kPBytes;                // 2 x 40 KB
constexpr uint32_t kSmemV = kSmemK + kKSlots * kKPart;           // 3 x 32 KB
constexpr uint32_t kSmemBar = kSmemV + kVSlots * kVPart;
constexpr uint32_t kSmemIdx = kSmemBar + 256;                    // [3][128] row ids
// [3][2 groups][128]: row maxima by tile parity (slots 0, 1) and row sums (slot 2)
constexpr uint32_t kSmemRed = kSmemIdx + kVSlots * kRows * 4;
constexpr uint32_t kSmemBytes = kSmemRed + 3 * 2 * 128 * 4;
constexpr uint32_t kTmemCols = 512;
constexpr int kVD = kMlaVDim;  // 256
// TMEM columns: O (the unit's 256 output values) at 0, the query's 512 latent bytes at 256
// (E4M3, four per column: the A operand of QK), S at 384.
constexpr uint32_t kTmemQ = 256, kTmemS = 384;

struct MlaParams {
  const int32_t* meta;
  const uint8_t* q;
  const uint8_t* kv;
  int64_t num_rows;
  const int32_t* indices;
  // paged decode (indices NULL): request n's token t is cache row
  // pg_indices[pg_indptr[n] + t / page_size] * page_size + t % page_size
  const int32_t* pg_indptr;
  const int32_t* pg_indices;
  int page_size;
  // paged decode: rows per TMA box of the cache maps (whole tiles are then loaded by TMA,
  // page by page, into both CTAs), or 0 (every tile gathered row by row)
  int tma_box;
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
  uint64_t q_full, qr_full, q_empty, drain;
  uint64_t kv_full[kVSlots], v_empty[kVSlots], k_empty[kKSlots];
  uint64_t s_full, s_empty, p_full, o_done;
  uint64_t o_free;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");
static_assert(kSmemBytes + 1024 <= 232448, "shared memory");

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

// Two E4M3 values (low byte, high byte) to f16 (low, high); exact.
__device__ __forceinline__ __half2 e4m3x2_to_half2(uint32_t x) {
  const uint16_t in = uint16_t(x);
  uint32_t out;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(in));
  return *reinterpret_cast<__half2*>(&out);
}

// Query token of a chunk (a unit is one query token; the CTA pair splits its latent halves).
__device__ __forceinline__ int chunk_token(const int4& ch) { return ch.x; }

// The softmax weights enter PV as two E4M3 terms: 16 p ~ hi + lo with hi = e4m3(16 p) and
// lo = e4m3(16 p - hi), both multiplied with the same V into the same accumulator, so a weight
// carries about 2^-8 relative rounding instead of the 2^-4 of a single E4M3 code (which, with
// the weights split between two groups of rows of different values, can move an output by
// twice the FP8 tolerance at any list length). The two P buffers hold hi and lo of one tile,
// a tile's PV is 8 MMAs, and the lazy-rescale threshold is 2^4 so that 16 p stays below 448.
template <bool kPaged>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_kernel(const __grid_constant__ CUtensorMap qmap_rope, const __grid_constant__ CUtensorMap omap,
               const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap kvmap,
               const __grid_constant__ CUtensorMap kvmap_tail, const MlaParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  Bars& B = *reinterpret_cast<Bars*>(sm + kSmemBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* hdr = p.meta;
  const int32_t* wptr = hdr + hdr[H_OFF_WORKERS];
  const int4* chunks = reinterpret_cast<const int4*>(hdr + hdr[H_OFF_CHUNKS]);
  // The two CTAs of a cluster take the same chunks: CTA rank v computes latent half v.
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int vh = int(rank);
  const int c0 = wptr[blockIdx.x >> 1], c1 = wptr[(blockIdx.x >> 1) + 1];
  const bool forced = forced_timeout(p.st);

  if (threadIdx.x == 0) {
    mbar_init(&B.q_full, 256);
    mbar_init(&B.qr_full, 1);
    mbar_init(&B.q_empty, 1);
    mbar_init(&B.drain, 1);
    // kv_full: this CTA's gather leader (after its half landed) + the peer's half as tx bytes;
    // v_empty / k_empty: both CTAs' MMA issuers (a slot is refilled in both at once).
    for (int s = 0; s < kVSlots; ++s) {
      mbar_init(&B.kv_full[s], 1);
      mbar_init(&B.v_empty[s], 2);
    }
    for (int s = 0; s < kKSlots; ++s) mbar_init(&B.k_empty[s], 2);
    mbar_init(&B.s_full, 1);
    mbar_init(&B.s_empty, 256);
    mbar_init(&B.p_full, 256);
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
  cluster_sync();  // both CTAs' barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = B.tmem_base;
  volatile int* abort_flag = &B.abort;
  const uint32_t peer_abort = mapa_shared(smem_u32(&B.abort), peer);
  auto raise_abort = [&]() {
    *abort_flag = 1;
    st_cluster_u32(peer_abort, 1u);
  };

  if (warp < 6) {
    // -------------------------------------------------------------- gather group
    // A tile is 128 rows x 576 bytes; CTA rank c copies rows 64 c .. 64 c + 63 with 16-byte
    // cp.async (192 threads, 12 chunks each) and its leader then pushes them into the peer's
    // shared memory with five bulk copies, so each row is read from L2 once per pair. Panels
    // are 128B-swizzled (row r, 16-byte chunk c -> chunk c ^ (r mod 8)); the 64-byte tail
    // uses the 64-byte pattern. The unit's latent half goes to a V part, the other half and
    // the tail to a K part; the peer, computing the other half, files the same panels the
    // other way round. Decisions go through bar_and on named barrier 1 (192 threads).
    // A whole tile of the paged cache (its 128 tokens in whole boxes of page slots) is
    // instead loaded by each CTA itself with TMA: five boxes per box of rows (four 128-byte
    // latent panels, 128B-swizzled, and the tail, 64B-swizzled, the same layouts), issued by
    // one thread, with no cp.async and no push; the partial last tile of a request is
    // gathered as above, which zero-fills the rows past its last token.
    const int pt = threadIdx.x;
    int32_t* idx_smem = reinterpret_cast<int32_t*>(sm + kSmemIdx);
    constexpr int kPer = (kHalfRows * 36) / kGatherThreads;  // 12 chunks per thread
    uint32_t off[kPer];  // bit 31: V part
    uint16_t col[kPer];
    uint8_t rowk[kPer];  // tile row
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int cid = pt + kGatherThreads * j;
      const int r = int(rank) * kHalfRows + cid / 36, q = cid % 36;
      if (q < 32) {
        const int pn = q >> 3;
        off[j] = ((pn >> 1) == vh ? 0x80000000u : 0u) |
                 uint32_t((pn & 1) * kPanel + r * 128 + (((q & 7) ^ (r & 7)) << 4));
      } else {
        off[j] = uint32_t(2 * kPanel + r * 64 + ((((q - 32) & 3) ^ ((r >> 1) & 3)) << 4));
      }
      col[j] = uint16_t(q * 16);
      rowk[j] = uint8_t(r);
    }
    // The peer's copy of this CTA's rows: nope panel pn is in the peer's V part when its half
    // is the peer's (pn / 2 != vh), else in its K part; the tail always in the K part.
    const uint32_t sbase = smem_u32(sm);
    const uint32_t peer_base = mapa_shared(sbase, peer);
    uint32_t kvc = 0, armed = 0;
    bool ok = true;
    // tile row whose id this thread loads: a paged cache needs every row's (the whole tile
    // may be loaded by TMA), a sparse list only this CTA's half
    constexpr bool all_ids = kPaged;
    const int tr = all_ids ? pt : int(rank) * kHalfRows + pt;
    const int nids = all_ids ? kRows : kHalfRows;
    // Row id of tile row tr of the tile of chunk cn that starts at row u0, loaded one tile
    // ahead. The chunk descriptors are held in registers (the next one read at the start of
    // a chunk), so the id is one independent load that nothing waits for until the next
    // tile: a load chained behind the descriptor's would stall the id threads, and with
    // them the whole gather group, for two L2 round trips per tile.
    // Paged decode: the row of token t of the chunk's request comes from the page table,
    // page_ptr = kv_indptr of the request (read once per chunk, when its first row ids are).
    auto load_id = [&](const int4& cn, int page_ptr, int u0) -> int32_t {
      if (pt >= nids || u0 + tr >= cn.z) return 0;
      const int t = u0 + tr;
      if constexpr (kPaged) {
        const int pg = __ldg(p.pg_indices + page_ptr + t / p.page_size);
        return pg * p.page_size + t % p.page_size;
      }
      return __ldg(p.indices + int64_t(cn.x) * p.top_k + t);
    };
    auto page_ptr_of = [&](const int4& cn) -> int {
      return kPaged && pt < nids ? __ldg(p.pg_indptr + cn.x) : 0;
    };
    int4 ch = c0 < c1 ? chunks[c0] : make_int4(0, 0, 0, 0);
    int cptr = c0 < c1 ? page_ptr_of(ch) : 0;
    int32_t next_id = c0 < c1 ? load_id(ch, cptr, ch.y) : 0;
    for (int ci = c0; ci < c1 && ok; ++ci) {
      const int4 nch = ci + 1 < c1 ? chunks[ci + 1] : make_int4(0, 0, 0, 0);
      int nptr = 0;
      for (int t0 = ch.y; t0 < ch.z; t0 += kRows, ++kvc) {
        const int v = kvc % kVSlots, k = kvc % kKSlots;
        int32_t my_id = next_id;
        if (t0 + kRows < ch.z) {
          next_id = load_id(ch, cptr, t0 + kRows);
        } else if (ci + 1 < c1) {
          nptr = page_ptr_of(nch);
          next_id = load_id(nch, nptr, nch.y);
        } else {
          next_id = 0;
        }
        if (my_id < 0 || my_id >= p.num_rows) {
          record_error(p.st, BSKV_ERR_DEVICE_INDEX);
          my_id = 0;
        }
        bool good = !*abort_flag &&
                    mbar_wait(&B.v_empty[v], ((kvc / kVSlots) & 1u) ^ 1u, p.st, forced) &&
                    mbar_wait(&B.k_empty[k], ((kvc / kKSlots) & 1u) ^ 1u, p.st, forced);
        // the push of tile kvc - 2 (same K slot) must have read its source before it is
        // overwritten; the push of kvc - 1 may still be running
        if (pt == 0) bulk_wait_read1();
        int32_t* ib = idx_smem + v * kRows;
        if (pt < nids) ib[tr] = my_id;
        ok = bar_and(1, kGatherThreads, good);
        if (!ok) break;
        uint8_t* vbase = sm + kSmemV + v * kVPart;
        uint8_t* kbase = sm + kSmemK + k * kKPart;
        const int valid = ch.z - t0;
        if (kPaged && p.tma_box > 0 && valid >= kRows) {
          if (pt == 0) {
            mbar_arrive_expect_tx(&B.kv_full[v], kRows * 576);
            ++armed;
            for (int r0 = 0; r0 < kRows; r0 += p.tma_box) {
              const int id = ib[r0];  // row id of the box's first token: page * page_size + slot
              const int page = id / p.page_size, slot = id % p.page_size;
#pragma unroll
              for (int pn = 0; pn < 4; ++pn)
                tma_load_3d(((pn >> 1) == vh ? vbase : kbase) + (pn & 1) * kPanel + r0 * 128,
                            &kvmap, pn * 128, slot, page, &B.kv_full[v]);
              tma_load_3d(kbase + 2 * kPanel + r0 * 64, &kvmap_tail, 512, slot, page,
                          &B.kv_full[v]);
            }
          }
          continue;
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
          uint8_t* dst = ((off[j] >> 31) ? vbase : kbase) + (off[j] & 0x7fffffffu);
          if (rowk[j] < valid)
            cp_async_16(dst, p.kv + int64_t(ib[rowk[j]]) * 576 + col[j]);
          else
            *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        }
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async_smem();
        ok = bar_and(1, kGatherThreads, !*abort_flag);
        if (!ok) break;
        if (pt == 0) {
          // this half is in place: arm kv_full for the peer's half and push ours to the peer
          mbar_arrive_expect_tx(&B.kv_full[v], kHalfTileBytes);
          ++armed;
          const uint32_t vo = kSmemV + v * kVPart, ko = kSmemK + k * kKPart;
          const uint32_t rows_off = rank * kHalfRows;
          const uint32_t mbar = mapa_shared(smem_u32(&B.kv_full[v]), peer);
#pragma unroll
          for (int pn = 0; pn < 4; ++pn) {
            const uint32_t in_panel = (pn & 1) * kPanel + rows_off * 128;
            const uint32_t src = ((pn >> 1) == vh ? vo : ko) + in_panel;
            const uint32_t dst = ((pn >> 1) != vh ? vo : ko) + in_panel;
            bulk_s2s_cluster(peer_base + dst, sm + src, kHalfRows * 128, mbar);
          }
          bulk_s2s_cluster(peer_base + ko + 2 * kPanel + rows_off * 64,
                           sm + ko + 2 * kPanel + rows_off * 64, kHalfRows * 64, mbar);
          bulk_commit();
        }
      }
      ch = nch;
      cptr = nptr;
    }
    if (pt == 0) bulk_wait_read0();
    if (!ok) raise_abort();
    if (pt == 0 && !ok) {
      // tiles this CTA armed may still receive the peer's half: let it land (bounded)
      const uint32_t from = armed > uint32_t(kVSlots) ? armed - kVSlots : 0u;
      for (uint32_t a = from; a < armed; ++a)
        mbar_wait(&B.kv_full[a % kVSlots], (a / kVSlots) & 1u, p.st, false);
    }
  } else if (warp == 7) {
    // -------------------------------------------------------------- query tail loader
    // The rotated 64-byte tail of the query tile (128 heads, 64B swizzle) is TMA-loaded once
    // per token; the two latent halves of a token reuse it.
    if (lane == 0) {
      uint32_t qc = 0;
      bool ok = true;
      int cur = -1;
      for (int ci = c0; ci < c1; ++ci) {
        const int n = chunk_token(chunks[ci]);
        if (n == cur) continue;
        cur = n;
        if (*abort_flag || !mbar_wait(&B.q_empty, (qc & 1u) ^ 1u, p.st, forced)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&B.qr_full, kRopePanel);
        tma_load_2d(sm + kSmemQR, &qmap_rope, 512, n * p.heads, &B.qr_full);
        ++qc;
      }
      if (!ok) raise_abort();
      // the last load issued must land before the CTA may exit (bounded, not forcible)
      if (qc > 0) mbar_wait(&B.qr_full, (qc - 1) & 1u, p.st, false);
    }
  } else if (warp == 6) {
    // -------------------------------------------------------------- MMA issuer
    // The warp stays converged; one elected lane executes the tcgen05 instructions.
    {
      const uint32_t leader = elect_leader();
      constexpr uint32_t idesc_qk = umma_idesc(128, kRows, 0, 0, 0, 0);
      constexpr uint32_t idesc_pv = umma_idesc(128, kVD, 0, 0, 0, 1);
      const uint32_t sbase = smem_u32(sm);
      uint32_t qc = 0, kvc = 0, cc = 0;
      bool ok = true;
      // P: K-major, 128B swizzle. V part: MN-major, 128-byte atoms along the output values
      // (LBO = panel stride), 8-row groups along the rows (SBO = 1024).
      const uint64_t dp = umma_desc(sbase + kSmemP, 16, 1024, kSwz128);
      const uint64_t dv = umma_desc(sbase + kSmemV, kPanel, 1024, kSwz128);
      const uint64_t dqr = umma_desc(sbase + kSmemQR, 16, 512, kSwz64);
      const uint64_t dkn = umma_desc(sbase + kSmemK, 16, 1024, kSwz128);
      const uint64_t dvn = umma_desc(sbase + kSmemV, 16, 1024, kSwz128);
      const uint64_t dkr = umma_desc(sbase + kSmemK + 2 * kPanel, 16, 512, kSwz64);
      // PV of tile g: P buffer 0 holds the hi terms, buffer 1 the lo terms (one p_full and
      // one o_done phase per tile)
      auto pv = [&](uint32_t g, bool first) -> bool {
        const uint32_t v = g % kVSlots;
        if (!issuer_wait(&B.p_full, g & 1u, p.st, forced, abort_flag)) return false;
        if (first && !issuer_wait(&B.o_free, (cc & 1u) ^ 1u, p.st, forced, abort_flag)) return false;
        tc_fence_after();
        const uint64_t b0 = dv + ((v * kVPart) >> 4);
#pragma unroll
        for (int kk = 0; kk < kRows / 32; ++kk)
          umma_f8_w(leader, tmem, dp + kk * 2, b0 + kk * 256, idesc_pv, (first && kk == 0) ? 0u : 1u);
#pragma unroll
        for (int kk = 0; kk < kRows / 32; ++kk)
          umma_f8_w(leader, tmem, dp + (kPBytes >> 4) + kk * 2, b0 + kk * 256, idesc_pv, 1u);
        umma_commit_w(leader, &B.o_done);
        umma_commit_mc_w(leader, &B.v_empty[v], 0x3);  // both CTAs' V part free
        return true;
      };
      int cur = -1;
      for (int ci = c0; ci < c1 && ok; ++ci) {
        const int4 ch = chunks[ci];
        const int n = chunk_token(ch);
        const int nt = (ch.z - ch.y + kRows - 1) / kRows;
        const bool last_use = ci + 1 == c1 || chunk_token(chunks[ci + 1]) != n;
        if (n != cur) {
          if (!issuer_wait(&B.q_full, qc & 1u, p.st, forced, abort_flag) ||
              !issuer_wait(&B.qr_full, qc & 1u, p.st, forced, abort_flag)) { ok = false; break; }
          ++qc;
          cur = n;
        }
        const uint32_t g0 = kvc;
        for (int t = 0; t < nt; ++t, ++kvc) {
          const uint32_t v = kvc % kVSlots, k = kvc % kKSlots;
          if (!issuer_wait(&B.kv_full[v], (kvc / kVSlots) & 1u, p.st, forced, abort_flag)) { ok = false; break; }
          // S is single-buffered: the softmax must have read the previous tile's S.
          if (kvc > 0 && !issuer_wait(&B.s_empty, (kvc - 1) & 1u, p.st, forced, abort_flag)) { ok = false; break; }
          tc_fence_after();
          // S = Q K^T over the 512 latent values (A from TMEM) and the 64-value tail.
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {
            const int pn = kk >> 2;
            const uint64_t bd = ((pn >> 1) == vh ? dvn + ((v * kVPart) >> 4) : dkn + ((k * kKPart) >> 4)) +
                                (((pn & 1) * kPanel + (kk & 3) * 32) >> 4);
            umma_f8_ts_w(leader, tmem + kTmemS, tmem + kTmemQ + kk * 8, bd, idesc_qk, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            umma_f8_w(leader, tmem + kTmemS, dqr + kk * 2, dkr + ((k * kKPart) >> 4) + kk * 2, idesc_qk, 1u);
          umma_commit_w(leader, &B.s_full);
          umma_commit_mc_w(leader, &B.k_empty[k], 0x3);  // both CTAs' K part free
          if (t + 1 == nt && last_use) umma_commit_w(leader, &B.q_empty);
          if (t >= 1 && !pv(kvc - 1, t == 1)) { ok = false; break; }
        }
        if (!ok) break;
        if (!pv(g0 + nt - 1, nt == 1)) { ok = false; break; }
        ++cc;
      }
      if (!ok) raise_abort();
      umma_commit_w(leader, &B.drain);
      mbar_wait(&B.drain, 0, p.st, false);
    }
  } else {
    // -------------------------------------------------------------- softmax warpgroups
    // Group wg owns tile columns 64 wg .. 64 wg + 63, output values 128 wg .. 128 wg + 127
    // and query bytes 256 wg .. 256 wg + 255; thread = head = TMEM lane.
    const int wg = (warp - 8) >> 2;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;            // head
    const uint32_t lane_base = uint32_t(q4 * 32) << 16;
    float* red = reinterpret_cast<float*>(sm + kSmemRed);  // [slot][group][row]
    uint32_t G = 0, qc = 0;
    uint32_t od_next = 0;  // next tile whose PV is not yet waited for
    bool ok = true;
    // Wait for the PVs of all tiles up to `upto` (o_done completes one phase per tile).
    auto consume = [&](int64_t upto) -> bool {
      while (int64_t(od_next) <= upto) {
        if (!warp_wait(&B.o_done, od_next & 1u, p.st, forced, abort_flag)) return false;
        ++od_next;
      }
      return true;
    };
    // Query latent bytes of head r for token n into TMEM, once the previous token's last QK
    // has completed (q_empty); then q_full.
    auto load_q = [&](int n) -> bool {
      if (!warp_wait(&B.q_empty, (qc & 1u) ^ 1u, p.st, forced, abort_flag)) return false;
      ++qc;
      tc_fence_after();
#pragma unroll 1
      for (int hlf = 0; hlf < 2; ++hlf) {
        uint32_t qv[32];
        if (r < p.heads) {
          const uint4* src = reinterpret_cast<const uint4*>(
              p.q + (int64_t(n) * p.heads + r) * 576 + wg * 256 + hlf * 128);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 x4 = __ldg(src + i);
            qv[4 * i] = x4.x; qv[4 * i + 1] = x4.y; qv[4 * i + 2] = x4.z; qv[4 * i + 3] = x4.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) qv[i] = 0u;
        }
        tmem_st32(tmem + lane_base + kTmemQ + wg * 64 + hlf * 32, qv);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&B.q_full);
      return true;
    };
    int cur = -1;
    for (int ci = c0; ci < c1 && ok; ++ci) {
      const int4 ch = chunks[ci];
      const int n = chunk_token(ch);
      const int nt = (ch.z - ch.y + kRows - 1) / kRows;
      if (n != cur) {
        // first chunk of this CTA (later tokens are loaded during the previous chunk)
        cur = n;
        ok = load_q(n);
        if (!ok) break;
      }
      // token of the next chunk, if it needs a new query
      const int n_next = ci + 1 < c1 && chunk_token(chunks[ci + 1]) != n ? chunk_token(chunks[ci + 1]) : -1;
      float m_run = -INFINITY, l_run = 0.f;
      for (int t = 0; t < nt; ++t, ++G) {
        const uint32_t b = G & 1u;  // tile parity: slot of the row-max exchange
        bool good = warp_wait(&B.s_full, G & 1u, p.st, forced, abort_flag);
        uint32_t sr[64];
        if (good) {
          tc_fence_after();
          const uint32_t sa = tmem + lane_base + kTmemS + wg * 64;
          tmem_ld32(sa, sr);
          tmem_ld32(sa + 32, sr + 32);
          tmem_ld_wait();
          tc_fence_before();
        }
        mbar_arrive(&B.s_empty);  // S may be overwritten by the next QK
        if (t + 1 == nt && n_next >= 0) {
          // The last QK of this token has completed (its S is loaded): bring the next
          // token's query in now, so the next chunk's QK overlaps this tile and the epilogue.
          good = good && load_q(n_next);
          cur = n_next;
        }
        const int valid = min(kRows, ch.z - (ch.y + t * kRows)) - wg * 64;
        // scaled logits, kept in place as float bits
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), z2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float2 y = ffma2(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sc2, z2);
          sr[c] = __float_as_uint(y.x);
          sr[c + 1] = __float_as_uint(y.y);
        }
        if (valid < 64) {
#pragma unroll
          for (int c = 0; c < 64; ++c) sr[c] = c < valid ? sr[c] : __float_as_uint(-INFINITY);
        }
        auto x = [&](int c) { return __uint_as_float(sr[c]); };
        float m8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          m8[j] = fmax3(fmax3(x(j), x(j + 8), x(j + 16)), fmax3(x(j + 24), x(j + 32), x(j + 40)),
                        fmaxf(x(j + 48), x(j + 56)));
        float mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
        red[(b * 2 + wg) * 128 + r] = mx;
        // both groups meet here once per tile (named barrier 3, 256 threads)
        ok = bar_and(3, 256, good);
        if (!ok) break;
        mx = fmaxf(mx, red[(b * 2 + (wg ^ 1)) * 128 + r]);
        float m_use = m_run, alpha = 1.f;
        bool rescale = false;
        if (m_run == -INFINITY) {
          m_use = mx;
        } else if (mx > m_run + 4.f) {
          m_use = mx;
          alpha = fast_exp2(m_run - mx);
          rescale = true;
        }
        const float ref = m_use == -INFINITY ? 0.f : m_use;
        rescale = __any_sync(0xffffffffu, rescale);
        // The P buffers were last read by the PV of tile G - 1.
        if (!consume(int64_t(G) - 1)) { ok = false; break; }
        // 16 p = 2^(x - ref + 4) in f16x2 pairs, straight to E4M3 pairs (hi and lo terms),
        // 16 keys (one 16-byte chunk of the 128B-swizzled P row) at a time; row sum of 16 p in
        // f16x2 (the LSE takes the 2^4 out again).
        uint8_t* prow = sm + kSmemP + r * 128;
        const float2 one2 = make_float2(1.f, 1.f), nr2 = make_float2(4.f - ref, 4.f - ref);
        __half2 hs[4];
#pragma unroll
        for (int c16 = 0; c16 < 4; ++c16) {
          uint32_t pk[4], lk[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c = c16 * 16 + j * 4;
            const float2 d0 = ffma2(make_float2(x(c), x(c + 1)), one2, nr2);
            const float2 d1 = ffma2(make_float2(x(c + 2), x(c + 3)), one2, nr2);
            const __half2 e0 = h2exp2_approx(__floats2half2_rn(d0.x, d0.y));
            const __half2 e1 = h2exp2_approx(__floats2half2_rn(d1.x, d1.y));
            const __half2 s2 = __hadd2(e0, e1);
            hs[j] = c16 == 0 ? s2 : __hadd2(hs[j], s2);
            const uint32_t h0 = half2_to_e4m3x2(e0), h1 = half2_to_e4m3x2(e1);
            pk[j] = h0 | (h1 << 16);
            // the remainder after the first code is exact in f16; its own code is the lo term
            const __half2 r0 = __hsub2(e0, e4m3x2_to_half2(h0));
            const __half2 r1 = __hsub2(e1, e4m3x2_to_half2(h1));
            lk[j] = half2_to_e4m3x2(r0) | (half2_to_e4m3x2(r1) << 16);
          }
          const int cc = 4 * wg + c16;
          *reinterpret_cast<uint4*>(prow + ((cc ^ (r & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4*>(prow + kPBytes + ((cc ^ (r & 7)) << 4)) =
              make_uint4(lk[0], lk[1], lk[2], lk[3]);
        }
        const float2 fs = __half22float2(__hadd2(__hadd2(hs[0], hs[1]), __hadd2(hs[2], hs[3])));
        l_run = l_run * alpha + (fs.x + fs.y);
        m_run = m_use;
        if (rescale && t > 0) {
          if (!consume(int64_t(G) - 1)) { ok = false; break; }
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
        mbar_arrive(&B.p_full);
      }
      if (!ok) break;
      // Epilogue: combine the two partial row sums, then each group stores its 128 values.
      red[(4 + wg) * 128 + r] = l_run;
      ok = bar_and(3, 256, true);
      if (!ok) break;
      const float l_tot = red[4 * 128 + r] + red[5 * 128 + r];
      if (!consume(int64_t(G) - 1)) { ok = false; break; }
      tc_fence_after();
      const float scale = l_tot > 0.f ? p.bmm2 / l_tot : 0.f;
      // (l_tot sums 16 p: the LSE takes the 2^4 out)
      const float lse = l_tot > 0.f ? (m_run + __log2f(l_tot) - 4.f) * kLn2 : -INFINITY;
      const bool row_ok = r < p.heads;
      const int slot = ch.w;
      // Each warp stages its 32 heads x 128 bytes of a box (128B-swizzled) in its own 4 KB of
      // the P buffers, whose PVs have all completed, and lane 0 writes the box with a tensor
      // store: the output or the split partial leaves in whole lines. A box holds 64 bf16 or
      // 32 float values per head.
      uint8_t* stg = sm + kSmemP + (warp - 8) * 4096;
      const uint32_t row_addr = smem_u32(stg) + lane * 128;
      const int nbox = slot < 0 ? 2 : 4;
#pragma unroll 1
      for (int bx = 0; bx < nbox; ++bx) {
        if (lane == 0) bulk_wait_read0();  // the previous box has been read
        __syncwarp();
        if (slot < 0) {
#pragma unroll 1
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t ov[32];
            tmem_ld32(tmem + lane_base + wg * (kVD / 2) + bx * 64 + hf * 32, ov);
            tmem_ld_wait();
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
              const int c = c4 * 8;
              __nv_bfloat162 h0 = __floats2bfloat162_rn(__uint_as_float(ov[c]) * scale, __uint_as_float(ov[c + 1]) * scale);
              __nv_bfloat162 h1 = __floats2bfloat162_rn(__uint_as_float(ov[c + 2]) * scale, __uint_as_float(ov[c + 3]) * scale);
              __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(ov[c + 4]) * scale, __uint_as_float(ov[c + 5]) * scale);
              __nv_bfloat162 h3 = __floats2bfloat162_rn(__uint_as_float(ov[c + 6]) * scale, __uint_as_float(ov[c + 7]) * scale);
              sts128(row_addr + (((hf * 4 + c4) ^ (lane & 7)) << 4),
                     make_uint4(*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1),
                                *reinterpret_cast<uint32_t*>(&h2), *reinterpret_cast<uint32_t*>(&h3)));
            }
          }
        } else {
          uint32_t ov[32];
          tmem_ld32(tmem + lane_base + wg * (kVD / 2) + bx * 32, ov);
          tmem_ld_wait();
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            const int c = c8 * 4;
            sts128(row_addr + ((c8 ^ (lane & 7)) << 4),
                   make_uint4(__float_as_uint(__uint_as_float(ov[c]) * scale),
                              __float_as_uint(__uint_as_float(ov[c + 1]) * scale),
                              __float_as_uint(__uint_as_float(ov[c + 2]) * scale),
                              __float_as_uint(__uint_as_float(ov[c + 3]) * scale)));
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (slot < 0) {
            if (q4 * 32 < p.heads)  // rows past the last head are clipped by the store
              tma_store_3d(&omap, stg, vh * kVD + wg * (kVD / 2) + bx * 64, q4 * 32, n);
          } else
            tma_store_2d(&wmap, stg, wg * (kVD / 2) + bx * 32, (slot * 2 + vh) * 128 + q4 * 32);
          bulk_commit();
        }
      }
      // The next chunk writes P only after every warp has passed its first tile's group
      // barrier; this warp gets there after its stores have read the staging.
      if (lane == 0) bulk_wait_read0();
      __syncwarp();
      if (row_ok && wg == 0) {
        if (slot < 0) {
          if (p.lse && vh == 0) p.lse[int64_t(n) * p.heads + r] = lse;
        } else {
          p.ws_lse[int64_t(slot * 2 + vh) * 128 + r] = lse;
        }
      }
      tc_fence_before();
      mbar_arrive(&B.o_free);
    }
    if (lane == 0) bulk_wait_all0();  // output stores complete before the CTA exits
    if (!ok) raise_abort();
  }
  tc_fence_before();
  // Neither CTA leaves while the other may still copy into its shared memory.
  cluster_sync();
  tc_fence_after();
  if (warp == 6) tmem_dealloc(tmem, kTmemCols);
}

// Merge split-KV pieces of query-token units (each piece holds both latent halves, slots
// 2 s and 2 s + 1); zero-fill empty ones. One warp per (unit, half, head); a lane owns 8 of
// the 256 values. Pieces are combined in slot order with the log-sum-exp merge (running
// max m, scale exp(m - m'), weight exp(lse_c - m')), the loads of four pieces in flight
// together.
__global__ void __launch_bounds__(128)
    mla_merge_kernel(const int32_t* __restrict__ meta, const float* __restrict__ ws_o,
                     const float* __restrict__ ws_lse, int heads, __nv_bfloat16* __restrict__ out,
                     float* __restrict__ lse) {
  const int NM = meta[H_MERGES];
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= NM * kMlaVSplit * heads) return;
  const int item = gw / (kMlaVSplit * heads), vh = (gw / heads) % kMlaVSplit, h = gw % heads;
  const int32_t* mi = meta + meta[H_OFF_MERGES] + 3 * item;
  const int n = mi[0], first = mi[1], count = mi[2];
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  float m = -INFINITY, l = 0.f;
  for (int c0 = 0; c0 < count; c0 += 4) {
    float bl[4];
    float4 bx[4][2];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (c0 + j < count) {
        const int64_t sh = (int64_t(first + c0 + j) * kMlaVSplit + vh) * 128 + h;
        bl[j] = __ldg(ws_lse + sh);
        const float4* src = reinterpret_cast<const float4*>(ws_o + sh * kVD + lane * 8);
        bx[j][0] = __ldg(src);
        bx[j][1] = __ldg(src + 1);
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (c0 + j >= count) continue;
      const float mn = fmaxf(m, bl[j]);
      const float sc = m == -INFINITY ? 0.f : expf(m - mn);
      const float w = expf(bl[j] - mn);
      l = l * sc + w;
      const float x[8] = {bx[j][0].x, bx[j][0].y, bx[j][0].z, bx[j][0].w,
                          bx[j][1].x, bx[j][1].y, bx[j][1].z, bx[j][1].w};
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = acc[i] * sc + w * x[i];
      m = mn;
    }
  }
  const float inv = count > 0 ? 1.f / l : 0.f;
  __nv_bfloat16* dst = out + (int64_t(n) * heads + h) * 512 + vh * kVD + lane * 8;
  uint4 w4;
  __nv_bfloat162 h0 = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
  __nv_bfloat162 h1 = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
  __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[4] * inv, acc[5] * inv);
  __nv_bfloat162 h3 = __floats2bfloat162_rn(acc[6] * inv, acc[7] * inv);
  w4.x = *reinterpret_cast<uint32_t*>(&h0);
  w4.y = *reinterpret_cast<uint32_t*>(&h1);
  w4.z = *reinterpret_cast<uint32_t*>(&h2);
  w4.w = *reinterpret_cast<uint32_t*>(&h3);
  *reinterpret_cast<uint4*>(dst) = w4;
  if (lse && vh == 0 && lane == 0) lse[int64_t(n) * heads + h] = count > 0 ? m + logf(l) : -INFINITY;
}

// The decode over validated arguments: `indices` holds plan->top_k row ids per query token
// (NULL for a paged plan, whose rows come from its page table); the float workspace holds
// the split-KV partials.
bskv_status run_mla(const bskv_plan* plan, const void* query, const void* kv_rows,
                    int64_t num_rows, const int32_t* indices, float bmm1_scale, float bmm2_scale,
                    void* out, float* lse, void* float_ws, cudaStream_t st) {
  const bool paged = plan->mla_variant == MLA_PAGED;
  const int64_t nq = int64_t(plan->batch) * plan->q_len;
  MlaParams mp{};
  mp.meta = plan->meta_dev;
  mp.kv = static_cast<const uint8_t*>(kv_rows);
  mp.num_rows = num_rows;
  mp.indices = indices;
  if (paged) {  // the page table rides in the uploaded metadata (aux0 = kv_indptr, aux1 = kv_indices)
    mp.pg_indptr = plan->meta_dev + meta_word(plan, H_OFF_AUX0);
    mp.pg_indices = plan->meta_dev + meta_word(plan, H_OFF_AUX1);
    mp.page_size = plan->page_size;
  }
  mp.top_k = plan->top_k;
  mp.heads = plan->num_qo_heads;
  mp.scale_log2 = bmm1_scale * 1.4426950408889634f;
  mp.bmm2 = bmm2_scale;
  mp.out = static_cast<__nv_bfloat16*>(out);
  mp.lse = lse;
  const int slots = meta_word(plan, H_SLOTS);
  mp.ws_o = static_cast<float*>(float_ws);
  mp.ws_lse = slots ? reinterpret_cast<float*>(static_cast<uint8_t*>(float_ws) +
                                               ((size_t(slots) * kMlaVSplit * 128 * kVD * 4 + 255) &
                                                ~size_t(255)))
                    : nullptr;
  if (bskv_status s = status_args(&mp.st)) return s;
  mp.q = static_cast<const uint8_t*>(query);
  CUtensorMap qr;
  const uint64_t dims[2] = {576, uint64_t(nq * plan->num_qo_heads)};
  const uint64_t str[1] = {576};
  const uint32_t box_r[2] = {64, 128};
  if (bskv_status s = encode_tiled(&qr, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, query, dims, str, box_r,
                                   CU_TENSOR_MAP_SWIZZLE_64B))
    return s;
  // epilogue stores: out as [token][head][512] bf16 in boxes of 32 heads x 64 values; the
  // split partials as [(slot, half, head)][256] float in boxes of 32 rows x 32 values
  CUtensorMap om, wm;
  {
    const uint64_t od[3] = {512, uint64_t(plan->num_qo_heads), uint64_t(nq)};
    const uint64_t os[2] = {512 * 2, uint64_t(plan->num_qo_heads) * 512 * 2};
    const uint32_t ob[3] = {64, uint32_t(std::min(32, plan->num_qo_heads)), 1};
    if (bskv_status s = encode_tiled(&om, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out, od, os, ob,
                                     CU_TENSOR_MAP_SWIZZLE_128B))
      return s;
  }
  if (slots > 0) {
    const uint64_t wd[2] = {uint64_t(kVD), uint64_t(slots) * kMlaVSplit * 128};
    const uint64_t ws[1] = {uint64_t(kVD) * 4};
    const uint32_t wb[2] = {32, 32};
    if (bskv_status s = encode_tiled(&wm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, float_ws, wd, ws, wb,
                                     CU_TENSOR_MAP_SWIZZLE_128B))
      return s;
  } else {
    wm = om;  // no split partials
  }
  // paged cache as [page][slot][576] bytes: whole tiles load by boxes of min(page_size, 128)
  // slots (a page size that is a multiple of 8 and divides 128 or is a multiple of it, so
  // that every box lands on a swizzle-atom boundary of the panels)
  CUtensorMap kvm = qr, kvt = qr;
  const int ps = plan->page_size;
  if (paged && ps >= 8 && ps % 8 == 0 && (kRows % ps == 0 || ps % kRows == 0)) {
    const int box = std::min(ps, kRows);
    const uint64_t kd[3] = {576, uint64_t(ps), uint64_t(plan->num_pages)};
    const uint64_t ks[2] = {576, uint64_t(576) * uint64_t(ps)};
    const uint32_t kb[3] = {128, uint32_t(box), 1}, kbt[3] = {64, uint32_t(box), 1};
    if (bskv_status s = encode_tiled(&kvm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, kv_rows, kd, ks, kb,
                                     CU_TENSOR_MAP_SWIZZLE_128B))
      return s;
    if (bskv_status s = encode_tiled(&kvt, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, kv_rows, kd, ks, kbt,
                                     CU_TENSOR_MAP_SWIZZLE_64B))
      return s;
    mp.tma_box = box;
  }
  const int grid = meta_word(plan, H_GRID);
  if (grid > 0) {
    const size_t smem = kSmemBytes + 1024;
    auto kern = paged ? mla_kernel<true> : mla_kernel<false>;
    if (bskv_status s = cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)),
                                   "mla: cudaFuncSetAttribute"))
      return s;
    kern<<<grid, kThreads, smem, st>>>(qr, om, wm, kvm, kvt, mp);
    if (bskv_status s = cuda_check(cudaGetLastError(), "mla kernel launch")) return s;
  }
  const int nm = meta_word(plan, H_MERGES);
  if (nm > 0) {
    const int warps = nm * kMlaVSplit * plan->num_qo_heads;
    mla_merge_kernel<<<(warps + 3) / 4, 128, 0, st>>>(plan->meta_dev, mp.ws_o, mp.ws_lse,
                                                      plan->num_qo_heads, mp.out, lse);
    if (bskv_status s = cuda_check(cudaGetLastError(), "mla merge launch")) return s;
  }
  return BSKV_OK;
}

}  // namespace
}  // namespace bskv

using namespace bskv;

extern "C" bskv_status bskv_run_mla_sparse(const bskv_plan* plan, const void* query,
                                           const void* kv_rows, int64_t num_rows,
                                           const int32_t* indices, float bmm1_scale,
                                           float bmm2_scale, void* out, float* lse,
                                           void* float_ws, size_t float_ws_bytes, void* stream) {
  BSKV_NVTX_RANGE("bskv_run_mla_sparse");
  if (!plan || plan->kind != KIND_MLA || plan->mla_variant != MLA_SPARSE) { set_error("run_mla_sparse: not a sparse MLA plan"); return BSKV_ERR_INVALID_ARG; }
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
  return run_mla(plan, query, kv_rows, num_rows, indices, bmm1_scale, bmm2_scale, out, lse,
                 float_ws, static_cast<cudaStream_t>(stream));
}

extern "C" bskv_status bskv_run_mla_paged(const bskv_plan* plan, const void* query,
                                          const void* kv_pages, float bmm1_scale,
                                          float bmm2_scale, void* out, float* lse,
                                          void* float_ws, size_t float_ws_bytes, void* stream) {
  BSKV_NVTX_RANGE("bskv_run_mla_paged");
  if (!plan || plan->kind != KIND_MLA || plan->mla_variant != MLA_PAGED) { set_error("run_mla_paged: not a paged MLA plan"); return BSKV_ERR_INVALID_ARG; }
  if (!plan->meta_dev) { set_error("run_mla_paged: plan not uploaded (bskv_plan_upload)"); return BSKV_ERR_INVALID_ARG; }
  if (plan->batch == 0) return BSKV_OK;
  if (!query || !kv_pages || !out) { set_error("run_mla_paged: NULL tensor"); return BSKV_ERR_INVALID_ARG; }
  if (!aligned16(query) || !aligned16(kv_pages) || !aligned16(out)) {
    set_error("run_mla_paged: tensors must be 16-byte aligned");
    return BSKV_ERR_INVALID_ARG;
  }
  if (float_ws_bytes < plan->float_ws_bytes || (plan->float_ws_bytes && !float_ws)) {
    set_error("run_mla_paged: float workspace of %zu bytes, %zu needed", float_ws_bytes, plan->float_ws_bytes);
    return BSKV_ERR_WORKSPACE_TOO_SMALL;
  }
  if (float_ws && !aligned16(float_ws)) { set_error("run_mla_paged: float workspace must be 16-byte aligned"); return BSKV_ERR_INVALID_ARG; }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return run_mla(plan, query, kv_pages, int64_t(plan->num_pages) * plan->page_size, nullptr,
                 bmm1_scale, bmm2_scale, out, lse, float_ws, st);
}
