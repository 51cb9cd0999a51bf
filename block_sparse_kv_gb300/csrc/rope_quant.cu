// Fused RoPE + FP8 E4M3 quantisation of MLA query and key rows (512 NoPE + 64 RoPE values).
//
// Method: "Sparse MLA" (MATE 0.2.6), mla_rope_quantize_fp8 (rotary arithmetic in float32
// on the 64-value tail; cos/sin cache columns [:32] cos and [32:] sin; is_neox selects
// contiguous halves or adjacent even/odd pairs; Q_fp8 = cast(Q * quant_scale_q),
// K_fp8 = cast(K * quant_scale_kv); outputs may be strided slices of 576-byte rows).
//
// GB300 design: a pure HBM stream (2.0 bytes in per byte out, plus the cache row). A warp
// takes its rows 32 at a time: each lane first resolves one row's index chain (its rotary
// position; for a paged append also its request, position and page, three dependent loads),
// so the chain costs one latency per 32 rows; then the warp handles two rows per iteration,
// taking their positions and destinations from the owning lanes by shuffle, and issues every
// load of both rows (row data, then the cos/sin values the positions select) before it
// converts anything. Each lane loads 32 bytes of NoPE (two
// 16-byte loads) and writes 16 bytes of E4M3, and 4 bytes of the RoPE tail, exchanging
// rotation partners with one shuffle (neox) or none (even/odd).
// cvt.rn.satfinite.e4m3x2.f32 does the cast (RNE, saturating to +-448).
#include <cuda_fp8.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"
#include "launch.h"

namespace bskv {
namespace {

using namespace dev;

struct RopeParams {
  // query group
  const __nv_bfloat16* q_rope;
  int64_t qr_s0, qr_s1;
  const __nv_bfloat16* q_nope;
  int64_t qn_s0, qn_s1;
  const void* pos_q;
  int64_t nnz_q;
  int heads;
  uint8_t* q_rope_out;
  int64_t qro_s0, qro_s1;
  uint8_t* q_nope_out;
  int64_t qno_s0, qno_s1;
  // key group
  const __nv_bfloat16* k_rope;
  int64_t kr_s;
  const __nv_bfloat16* k_nope;
  int64_t kn_s;
  const void* pos_k;
  int64_t nnz_k;
  uint8_t* k_rope_out;
  int64_t kro_s;
  uint8_t* k_nope_out;
  int64_t kno_s;
  // paged append (app_indptr non-NULL): key row t goes to cache row page * page_size + slot
  // of the page table entry of (app_batch[t], app_pos[t]); k_*_out then address the cache
  const int32_t* app_batch;
  const int32_t* app_pos;
  const int32_t* app_indptr;
  const int32_t* app_indices;
  int32_t app_requests, app_page_size;
  int64_t app_num_pages;
  // shared
  const void* cos_sin;
  int64_t max_seq_len;
  float scale_q, scale_kv;
  StatusArgs st;
};

__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  return static_cast<uint16_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// Streaming loads: each input byte is read once, so keep it out of L1.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_stream4(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// One row's inputs, loaded before any of them is used so that a warp keeps the loads of
// two rows in flight at once (the row data does not wait for the position, and only the
// cos/sin values depend on it).
struct RowIn {
  uint4 x0, x1;      // this lane's 16 NoPE values
  uint32_t rw;       // this lane's 2 RoPE values
  float c0, c1, s0, s1;
  bool valid;        // position inside [0, max_seq_len)
};

// Cache row of an appended key row of request b at position q, or -1 when its request,
// position or page is out of range (two dependent loads; the row's data loads do not wait
// for them).
__device__ __forceinline__ int64_t append_row(const RopeParams& p, int32_t b, int32_t q) {
  if (b < 0 || b >= p.app_requests || q < 0) return -1;
  const int64_t slot = int64_t(__ldg(p.app_indptr + b)) + q / p.app_page_size;
  if (slot >= __ldg(p.app_indptr + b + 1)) return -1;
  const int32_t page = __ldg(p.app_indices + slot);
  if (page < 0 || page >= p.app_num_pages) return -1;
  return int64_t(page) * p.app_page_size + q % p.app_page_size;
}

__device__ __forceinline__ void row_ptrs(const RopeParams& p, int64_t r, int64_t q_rows,
                                         const __nv_bfloat16*& rope, const __nv_bfloat16*& nope,
                                         uint8_t*& rope_out, uint8_t*& nope_out, float& scale,
                                         bool& dst_ok) {
  dst_ok = true;
  if (r < q_rows) {
    const int64_t t = r / p.heads;
    const int h = int(r % p.heads);
    rope = p.q_rope + t * p.qr_s0 + h * p.qr_s1;
    nope = p.q_nope + t * p.qn_s0 + h * p.qn_s1;
    rope_out = p.q_rope_out + t * p.qro_s0 + h * p.qro_s1;
    nope_out = p.q_nope_out + t * p.qno_s0 + h * p.qno_s1;
    scale = p.scale_q;
  } else {
    const int64_t t = r - q_rows;
    rope = p.k_rope + t * p.kr_s;
    nope = p.k_nope + t * p.kn_s;
    // a paged append resolves the destination later (resolve_dst), after the row's data
    // loads are in flight
    rope_out = p.k_rope_out + t * p.kro_s;
    nope_out = p.k_nope_out + t * p.kno_s;
    scale = p.scale_kv;
  }
}

// Index chain of row r, resolved by one lane for the warp: its rotary position and, for an
// appended key row, its cache row (-1 when the destination is out of range).
template <typename PosT, bool kAppend>
__device__ __forceinline__ void row_chain(const RopeParams& p, int64_t r, int64_t q_rows,
                                          int64_t& pos, int64_t& dst) {
  dst = 0;
  if (r < q_rows) {
    pos = int64_t(__ldg(static_cast<const PosT*>(p.pos_q) + r / p.heads));
  } else {
    const int64_t t = r - q_rows;
    pos = int64_t(__ldg(static_cast<const PosT*>(p.pos_k) + t));
    if (kAppend) dst = append_row(p, __ldg(p.app_batch + t), __ldg(p.app_pos + t));
  }
}

// Destination of an appended key row r (rows past the query rows only) from its cache row.
__device__ __forceinline__ void resolve_dst(const RopeParams& p, int64_t r, int64_t q_rows,
                                            int64_t d, uint8_t*& rope_out, uint8_t*& nope_out,
                                            bool& dst_ok) {
  if (r < q_rows) return;
  dst_ok = d >= 0;
  if (!dst_ok) d = 0;
  rope_out = p.k_rope_out + d * p.kro_s;
  nope_out = p.k_nope_out + d * p.kno_s;
}

template <bool kNeox, typename CacheT>
__device__ __forceinline__ void load_row(const __nv_bfloat16* rope, const __nv_bfloat16* nope,
                                         int64_t pos, int64_t max_seq_len, const CacheT* cache,
                                         int lane, RowIn& in) {
  const uint4* src = reinterpret_cast<const uint4*>(nope) + 2 * lane;
  in.x0 = ld_stream16(src);
  in.x1 = ld_stream16(src + 1);
  in.rw = ld_stream4(reinterpret_cast<const unsigned int*>(rope) + lane);
  in.valid = pos >= 0 && pos < max_seq_len;
  const int64_t pc = in.valid ? pos : 0;  // loads stay in bounds; the row is skipped later
  const int i0 = kNeox ? ((2 * lane) & 31) : lane;  // frequency index of the first element
  auto cs = [&](int i) -> float {
    if constexpr (sizeof(CacheT) == 4) {
      return __ldg(reinterpret_cast<const float*>(cache) + pc * 64 + i);
    } else {
      const uint16_t b = __ldg(reinterpret_cast<const unsigned short*>(cache) + pc * 64 + i);
      return __uint_as_float(uint32_t(b) << 16);
    }
  };
  in.c0 = cs(i0);
  in.s0 = cs(32 + i0);
  if (kNeox) {
    in.c1 = cs(i0 + 1);
    in.s1 = cs(32 + i0 + 1);
  }
}

template <bool kNeox>
__device__ __forceinline__ void store_row(const RowIn& in, uint8_t* rope_out, uint8_t* nope_out,
                                          float scale, int lane, const StatusArgs& st,
                                          bool dst_ok) {
  // The neox partner exchange is a warp shuffle, so it runs before the validity test.
  const float e0 = bf16_lo(in.rw), e1 = bf16_hi(in.rw);
  float r0, r1;
  if (kNeox) {
    // Pair i = (i, i + 32): lanes 0-15 hold the first halves, lanes 16-31 the partners.
    const float p0 = __shfl_xor_sync(0xffffffffu, e0, 16);
    const float p1 = __shfl_xor_sync(0xffffffffu, e1, 16);
    if (lane < 16) {
      r0 = __fsub_rn(__fmul_rn(e0, in.c0), __fmul_rn(p0, in.s0));
      r1 = __fsub_rn(__fmul_rn(e1, in.c1), __fmul_rn(p1, in.s1));
    } else {
      r0 = __fadd_rn(__fmul_rn(e0, in.c0), __fmul_rn(p0, in.s0));
      r1 = __fadd_rn(__fmul_rn(e1, in.c1), __fmul_rn(p1, in.s1));
    }
  } else {
    r0 = __fsub_rn(__fmul_rn(e0, in.c0), __fmul_rn(e1, in.s0));
    r1 = __fadd_rn(__fmul_rn(e1, in.c0), __fmul_rn(e0, in.s0));
  }
  if (!in.valid || !dst_ok) {
    if (lane == 0) record_error(st, BSKV_ERR_DEVICE_INDEX);
    return;
  }
  const uint32_t w[8] = {in.x0.x, in.x0.y, in.x0.z, in.x0.w, in.x1.x, in.x1.y, in.x1.z, in.x1.w};
  uint32_t packed[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint16_t a = cvt_e4m3x2(bf16_lo(w[2 * i]) * scale, bf16_hi(w[2 * i]) * scale);
    const uint16_t b = cvt_e4m3x2(bf16_lo(w[2 * i + 1]) * scale, bf16_hi(w[2 * i + 1]) * scale);
    packed[i] = uint32_t(a) | (uint32_t(b) << 16);
  }
  *reinterpret_cast<uint4*>(nope_out + 16 * lane) =
      make_uint4(packed[0], packed[1], packed[2], packed[3]);
  *reinterpret_cast<uint16_t*>(rope_out + 2 * lane) =
      cvt_e4m3x2(__fmul_rn(r0, scale), __fmul_rn(r1, scale));
}

// kAppend: key rows go to the paged cache through the page table.
template <bool kNeox, typename PosT, typename CacheT, bool kAppend>
__global__ void __launch_bounds__(256) rope_quant_kernel(const RopeParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t W = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int64_t q_rows = p.q_rope ? p.nnz_q * p.heads : 0;
  const int64_t total = q_rows + (p.k_rope ? p.nnz_k : 0);
  const CacheT* cache = static_cast<const CacheT*>(p.cos_sin);
  // Rows base + i W (i < 32) of this warp: lane i resolves row i's chain, then the warp takes
  // the rows two at a time (rows 2k and 2k + 1 of the 32), every load of both issued before
  // use.
  for (int64_t base = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; base < total;
       base += 32 * W) {
    const int64_t my_r = base + int64_t(lane) * W;
    int64_t my_pos = 0, my_dst = 0;
    if (my_r < total) row_chain<PosT, kAppend>(p, my_r, q_rows, my_pos, my_dst);
#pragma unroll 1
    for (int k = 0; k < 16; ++k) {
      const int64_t ra = base + int64_t(2 * k) * W;
      if (ra >= total) break;  // warp-uniform
      const int64_t rb = ra + W;
      const bool has_b = rb < total;
      const int64_t pos_a = __shfl_sync(0xffffffffu, my_pos, 2 * k);
      const int64_t pos_b = __shfl_sync(0xffffffffu, my_pos, 2 * k + 1);
      const __nv_bfloat16 *rope_a, *nope_a, *rope_b, *nope_b;
      uint8_t *ro_a, *no_a, *ro_b, *no_b;
      float sc_a, sc_b;
      bool ok_a, ok_b;
      row_ptrs(p, ra, q_rows, rope_a, nope_a, ro_a, no_a, sc_a, ok_a);
      row_ptrs(p, has_b ? rb : ra, q_rows, rope_b, nope_b, ro_b, no_b, sc_b, ok_b);
      RowIn a, b;
      load_row<kNeox, CacheT>(rope_a, nope_a, pos_a, p.max_seq_len, cache, lane, a);
      load_row<kNeox, CacheT>(rope_b, nope_b, has_b ? pos_b : pos_a, p.max_seq_len, cache, lane, b);
      if (kAppend) {
        const int64_t dst_a = __shfl_sync(0xffffffffu, my_dst, 2 * k);
        const int64_t dst_b = __shfl_sync(0xffffffffu, my_dst, 2 * k + 1);
        resolve_dst(p, ra, q_rows, dst_a, ro_a, no_a, ok_a);
        if (has_b) resolve_dst(p, rb, q_rows, dst_b, ro_b, no_b, ok_b);
      }
      store_row<kNeox>(a, ro_a, no_a, sc_a, lane, p.st, ok_a);
      if (has_b) store_row<kNeox>(b, ro_b, no_b, sc_b, lane, p.st, ok_b);
    }
  }
}

// Blocks of this kernel resident on one SM times the SM count, cached per device.
template <typename Kernel>
bskv_status resident_grid(Kernel kernel, int threads, int* out) {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (bskv_status s = cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) return s;
  const int slot = dev < 64 ? dev : 63;
  int v = dev < 64 ? cache[slot].load(std::memory_order_relaxed) : 0;
  if (v == 0) {
    int sms = 0, occ = 0;
    if (bskv_status s = cuda_check(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute"))
      return s;
    if (bskv_status s = cuda_check(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, 0), "cudaOccupancyMaxActiveBlocksPerMultiprocessor"))
      return s;
    v = sms * (occ > 0 ? occ : 1);
    if (dev < 64) cache[slot].store(v, std::memory_order_relaxed);
  }
  *out = v;
  return BSKV_OK;
}

template <bool kNeox, typename PosT, typename CacheT>
bskv_status launch_rope_t(const RopeParams& p, int64_t rows, cudaStream_t st) {
  auto kernel = p.app_indptr ? rope_quant_kernel<kNeox, PosT, CacheT, true>
                             : rope_quant_kernel<kNeox, PosT, CacheT, false>;
  int resident = 0;
  if (bskv_status s = resident_grid(kernel, 256, &resident)) return s;
  // One wave of resident blocks; fewer when there are fewer than one row per warp.
  const int64_t want = (rows + 7) / 8;
  const int blocks = int(want < resident ? want : resident);
  kernel<<<blocks, 256, 0, st>>>(p);
  return cuda_check(cudaGetLastError(), "rope_quantize_fp8 launch");
}

template <bool kNeox>
bskv_status launch_rope(const RopeParams& p, int pos_dtype, int cache_dtype, cudaStream_t st) {
  const int64_t rows = (p.q_rope ? p.nnz_q * p.heads : 0) + (p.k_rope ? p.nnz_k : 0);
  if (rows == 0) return BSKV_OK;
  if (pos_dtype == BSKV_INT32)
    return cache_dtype == BSKV_FP32 ? launch_rope_t<kNeox, int32_t, float>(p, rows, st)
                                    : launch_rope_t<kNeox, int32_t, __nv_bfloat16>(p, rows, st);
  return cache_dtype == BSKV_FP32 ? launch_rope_t<kNeox, int64_t, float>(p, rows, st)
                                  : launch_rope_t<kNeox, int64_t, __nv_bfloat16>(p, rows, st);
}

}  // namespace
}  // namespace bskv

using namespace bskv;

namespace bskv {
namespace {

// The checks and launch shared by both entry points; `app` (nullable) fills the paged
// append fields of the parameters.
bskv_status rope_entry(
    const void* q_rope, const int64_t* q_rope_strides, const void* q_nope,
    const int64_t* q_nope_strides, const void* pos_q, int64_t nnz_q, int32_t num_heads,
    void* q_rope_out, const int64_t* q_rope_out_strides, void* q_nope_out,
    const int64_t* q_nope_out_strides, const void* k_rope, int64_t k_rope_stride,
    const void* k_nope, int64_t k_nope_stride, const void* pos_k, int64_t nnz_k,
    void* k_rope_out, int64_t k_rope_out_stride, void* k_nope_out, int64_t k_nope_out_stride,
    int32_t pos_dtype, const void* cos_sin, int32_t cos_sin_dtype, int64_t max_seq_len,
    int32_t is_neox, float quant_scale_q, float quant_scale_kv, void* stream,
    const RopeParams* app) {
  RopeParams p{};
  if (app) {
    p.app_batch = app->app_batch; p.app_pos = app->app_pos;
    p.app_indptr = app->app_indptr; p.app_indices = app->app_indices;
    p.app_requests = app->app_requests; p.app_page_size = app->app_page_size;
    p.app_num_pages = app->app_num_pages;
  }
  const bool has_q = q_rope || q_nope || q_rope_out || q_nope_out || pos_q;
  const bool has_k = k_rope || k_nope || k_rope_out || k_nope_out || pos_k;
  if (pos_dtype != BSKV_INT32 && pos_dtype != BSKV_INT64) { set_error("rope_quantize_fp8: pos dtype %s unsupported", dtype_name(pos_dtype)); return BSKV_ERR_UNSUPPORTED; }
  if (cos_sin_dtype != BSKV_FP32 && cos_sin_dtype != BSKV_BF16) { set_error("rope_quantize_fp8: cos_sin dtype %s unsupported", dtype_name(cos_sin_dtype)); return BSKV_ERR_UNSUPPORTED; }
  if (!cos_sin || max_seq_len < 1) { set_error("rope_quantize_fp8: cos_sin cache missing"); return BSKV_ERR_INVALID_ARG; }
  if (has_q) {
    if (!q_rope || !q_nope || !q_rope_out || !q_nope_out || !pos_q || !q_rope_strides ||
        !q_nope_strides || !q_rope_out_strides || !q_nope_out_strides) {
      set_error("rope_quantize_fp8: the query group needs all of q_rope, q_nope, pos_q and both outputs");
      return BSKV_ERR_INVALID_ARG;
    }
    if (nnz_q < 0 || num_heads < 1) { set_error("rope_quantize_fp8: nnz_q=%lld num_heads=%d", (long long)nnz_q, num_heads); return BSKV_ERR_INVALID_ARG; }
    const int64_t in_s[4] = {q_rope_strides[0], q_rope_strides[1], q_nope_strides[0], q_nope_strides[1]};
    for (int i = 0; i < 4; ++i)
      if ((in_s[i] * 2) % 16) { set_error("rope_quantize_fp8: query input strides must be multiples of 8 elements"); return BSKV_ERR_INVALID_ARG; }
    if (q_nope_out_strides[0] % 16 || q_nope_out_strides[1] % 16 || q_rope_out_strides[0] % 2 || q_rope_out_strides[1] % 2) {
      set_error("rope_quantize_fp8: q_nope_out strides must be multiples of 16 bytes, q_rope_out of 2");
      return BSKV_ERR_INVALID_ARG;
    }
    if (!aligned16(q_rope) || !aligned16(q_nope) || !aligned16(q_nope_out) || (reinterpret_cast<uintptr_t>(q_rope_out) & 1)) {
      set_error("rope_quantize_fp8: misaligned query tensor"); return BSKV_ERR_INVALID_ARG;
    }
    p.q_rope = static_cast<const __nv_bfloat16*>(q_rope); p.qr_s0 = q_rope_strides[0]; p.qr_s1 = q_rope_strides[1];
    p.q_nope = static_cast<const __nv_bfloat16*>(q_nope); p.qn_s0 = q_nope_strides[0]; p.qn_s1 = q_nope_strides[1];
    p.pos_q = pos_q; p.nnz_q = nnz_q; p.heads = num_heads;
    p.q_rope_out = static_cast<uint8_t*>(q_rope_out); p.qro_s0 = q_rope_out_strides[0]; p.qro_s1 = q_rope_out_strides[1];
    p.q_nope_out = static_cast<uint8_t*>(q_nope_out); p.qno_s0 = q_nope_out_strides[0]; p.qno_s1 = q_nope_out_strides[1];
  }
  if (has_k) {
    if (!k_rope || !k_nope || !k_rope_out || !k_nope_out || !pos_k) {
      set_error("rope_quantize_fp8: the key group needs all of k_rope, k_nope, pos_k and both outputs");
      return BSKV_ERR_INVALID_ARG;
    }
    if (nnz_k < 0) { set_error("rope_quantize_fp8: nnz_k=%lld", (long long)nnz_k); return BSKV_ERR_INVALID_ARG; }
    if ((k_rope_stride * 2) % 16 || (k_nope_stride * 2) % 16 || k_nope_out_stride % 16 || k_rope_out_stride % 2) {
      set_error("rope_quantize_fp8: key strides misaligned"); return BSKV_ERR_INVALID_ARG;
    }
    if (!aligned16(k_rope) || !aligned16(k_nope) || !aligned16(k_nope_out) || (reinterpret_cast<uintptr_t>(k_rope_out) & 1)) {
      set_error("rope_quantize_fp8: misaligned key tensor"); return BSKV_ERR_INVALID_ARG;
    }
    p.k_rope = static_cast<const __nv_bfloat16*>(k_rope); p.kr_s = k_rope_stride;
    p.k_nope = static_cast<const __nv_bfloat16*>(k_nope); p.kn_s = k_nope_stride;
    p.pos_k = pos_k; p.nnz_k = nnz_k;
    p.k_rope_out = static_cast<uint8_t*>(k_rope_out); p.kro_s = k_rope_out_stride;
    p.k_nope_out = static_cast<uint8_t*>(k_nope_out); p.kno_s = k_nope_out_stride;
  }
  p.cos_sin = cos_sin; p.max_seq_len = max_seq_len;
  p.scale_q = quant_scale_q; p.scale_kv = quant_scale_kv;
  if (bskv_status s = status_args(&p.st)) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return is_neox ? launch_rope<true>(p, pos_dtype, cos_sin_dtype, st)
                 : launch_rope<false>(p, pos_dtype, cos_sin_dtype, st);
}

}  // namespace
}  // namespace bskv

extern "C" bskv_status bskv_rope_quantize_fp8(
    const void* q_rope, const int64_t* q_rope_strides, const void* q_nope,
    const int64_t* q_nope_strides, const void* pos_q, int64_t nnz_q, int32_t num_heads,
    void* q_rope_out, const int64_t* q_rope_out_strides, void* q_nope_out,
    const int64_t* q_nope_out_strides, const void* k_rope, int64_t k_rope_stride,
    const void* k_nope, int64_t k_nope_stride, const void* pos_k, int64_t nnz_k,
    void* k_rope_out, int64_t k_rope_out_stride, void* k_nope_out, int64_t k_nope_out_stride,
    int32_t pos_dtype, const void* cos_sin, int32_t cos_sin_dtype, int64_t max_seq_len,
    int32_t is_neox, float quant_scale_q, float quant_scale_kv, void* stream) {
  BSKV_NVTX_RANGE("bskv_rope_quantize_fp8");
  return rope_entry(q_rope, q_rope_strides, q_nope, q_nope_strides, pos_q, nnz_q, num_heads,
                    q_rope_out, q_rope_out_strides, q_nope_out, q_nope_out_strides, k_rope,
                    k_rope_stride, k_nope, k_nope_stride, pos_k, nnz_k, k_rope_out,
                    k_rope_out_stride, k_nope_out, k_nope_out_stride, pos_dtype, cos_sin,
                    cos_sin_dtype, max_seq_len, is_neox, quant_scale_q, quant_scale_kv, stream,
                    nullptr);
}

extern "C" bskv_status bskv_rope_quantize_fp8_append_paged(
    const void* q_rope, const int64_t* q_rope_strides, const void* q_nope,
    const int64_t* q_nope_strides, const void* pos_q, int64_t nnz_q, int32_t num_heads,
    void* q_rope_out, const int64_t* q_rope_out_strides, void* q_nope_out,
    const int64_t* q_nope_out_strides, const void* k_rope, int64_t k_rope_stride,
    const void* k_nope, int64_t k_nope_stride, const void* pos_k, int64_t nnz_k,
    const int32_t* batch_indices, const int32_t* positions, const int32_t* kv_indptr,
    const int32_t* kv_indices, int32_t batch, int32_t page_size, int64_t num_pages,
    void* kv_pages, int32_t pos_dtype, const void* cos_sin, int32_t cos_sin_dtype,
    int64_t max_seq_len, int32_t is_neox, float quant_scale_q, float quant_scale_kv,
    void* stream) {
  BSKV_NVTX_RANGE("bskv_rope_quantize_fp8_append_paged");
  if (!k_rope || !k_nope || !pos_k || !batch_indices || !positions || !kv_indptr ||
      !kv_indices || !kv_pages) {
    set_error("rope_quantize_fp8_append_paged: the key rows, their positions, batch_indices, "
              "positions, the page table and kv_pages are all required");
    return BSKV_ERR_INVALID_ARG;
  }
  if (batch < 1 || page_size < 1 || num_pages < 1 || nnz_k < 0) {
    set_error("rope_quantize_fp8_append_paged: batch=%d page_size=%d num_pages=%lld nnz_k=%lld",
              batch, page_size, (long long)num_pages, (long long)nnz_k);
    return BSKV_ERR_INVALID_ARG;
  }
  if ((reinterpret_cast<uintptr_t>(batch_indices) | reinterpret_cast<uintptr_t>(positions) |
       reinterpret_cast<uintptr_t>(kv_indptr) | reinterpret_cast<uintptr_t>(kv_indices)) & 3) {
    set_error("rope_quantize_fp8_append_paged: index arrays must be 4-byte aligned");
    return BSKV_ERR_INVALID_ARG;
  }
  RopeParams app{};
  app.app_batch = batch_indices; app.app_pos = positions;
  app.app_indptr = kv_indptr; app.app_indices = kv_indices;
  app.app_requests = batch; app.app_page_size = page_size; app.app_num_pages = num_pages;
  uint8_t* cache = static_cast<uint8_t*>(kv_pages);
  return rope_entry(q_rope, q_rope_strides, q_nope, q_nope_strides, pos_q, nnz_q, num_heads,
                    q_rope_out, q_rope_out_strides, q_nope_out, q_nope_out_strides, k_rope,
                    k_rope_stride, k_nope, k_nope_stride, pos_k, nnz_k, cache + 512, 576, cache,
                    576, pos_dtype, cos_sin, cos_sin_dtype, max_seq_len, is_neox, quant_scale_q,
                    quant_scale_kv, stream, &app);
}
