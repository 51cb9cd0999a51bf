"""RoPE on the 64-value tail and FP8 quantisation of MLA query/key rows, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows "Sparse MLA" (MATE 0.2.6 API docs), section "RoPE and FP8 quantization"
(mla_rope_quantize_fp8 parameters), and "FlashInfer Compatibility Wrapper", section
"RoPE and FP8 quantization":
  * the rotary cache is [max_seq_len, 64], the cosines in its first 32 columns and the
    sines in the last 32; every position must lie in [0, max_seq_len);
  * is_neox=True pairs tail value i with value i + 32 (the first half against the
    second), is_neox=False pairs values 2i and 2i + 1;
  * the quant scales multiply the values before the FP8 cast:
    Q_fp8 = cast(Q * quant_scale_q), KV_fp8 = cast(KV * quant_scale_kv),
    for both the 512-value NoPE part and the rotated 64-value tail.
Reading taken where the pages are silent: pair i (i < 32) uses cos = cache[pos, i]
and sin = cache[pos, 32 + i] in both layouts, and rotates (x, y) to
(x*cos - y*sin, y*cos + x*sin). The arithmetic is exact float64 on the stored cache
values; the single rounding is the E4M3 cast.

The paged append (FlashInfer cheat page, benchmark README:
rope_quantize_fp8_append_paged_kv_cache, which rotates, quantises and writes the key rows
into a paged cache in one call; page table of the "FlashInfer" agent-skill summary, KV-Cache Formats) writes the
same key rows into a paged latent cache. Reading: key row i belongs to request
batch_indices[i] at token position positions[i]; it lands in page
kv_indices[kv_indptr[b] + positions[i] // page_size], slot positions[i] % page_size, as
512 NoPE codes followed by the 64 rotated codes.
"""

import numpy as np

from .numerics import bf16_bits_to_f64, e4m3_encode

ROPE_DIM = 64
NOPE_DIM = 512


def rotate(x, cos, sin, is_neox):
    """Rotate rows of x [..., 64] by per-row cos/sin [..., 32] (float64)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    if is_neox:
        a, b = x[..., :32], x[..., 32:]
        out[..., :32] = a * cos - b * sin
        out[..., 32:] = b * cos + a * sin
    else:
        a, b = x[..., 0::2], x[..., 1::2]
        out[..., 0::2] = a * cos - b * sin
        out[..., 1::2] = b * cos + a * sin
    return out


def cache_rows(cos_sin, pos, cache_dtype="f32"):
    """Gather (cos, sin) [n, 32] in float64 for positions ``pos`` from the stored cache."""
    pos = np.asarray(pos, dtype=np.int64)
    cs = np.asarray(cos_sin)
    if np.any(pos < 0) or np.any(pos >= cs.shape[0]):
        raise ValueError("position outside [0, max_seq_len)")
    if cache_dtype == "f32":
        rows = cs[pos].astype(np.float64)
    elif cache_dtype == "bf16":
        rows = bf16_bits_to_f64(cs[pos])
    else:
        raise ValueError(cache_dtype)
    return rows[:, :32], rows[:, 32:]


def mla_rope_quantize_fp8(q_rope_bits, k_rope_bits, q_nope_bits, k_nope_bits, cos_sin,
                          pos_q, pos_k, is_neox=True, quant_scale_q=1.0, quant_scale_kv=1.0,
                          cache_dtype="f32"):
    """Return (q_rope_out, k_rope_out, q_nope_out, k_nope_out) as E4M3 codes.

    q_rope [nq, H, 64], q_nope [nq, H, 512], k_rope [nk, 64], k_nope [nk, 512] are
    bfloat16 bit patterns; pos_q [nq] and pos_k [nk] are positions. Any group may be
    None (its outputs are then None). The pages' single-nnz form is pos_q == pos_k.
    """
    outs = [None, None, None, None]
    if q_rope_bits is not None:
        c, s = cache_rows(cos_sin, pos_q, cache_dtype)
        qr = bf16_bits_to_f64(q_rope_bits)
        rq = rotate(qr, c[:, None, :], s[:, None, :], is_neox)
        outs[0] = e4m3_encode(rq * quant_scale_q)
        outs[2] = e4m3_encode(bf16_bits_to_f64(q_nope_bits) * quant_scale_q)
    if k_rope_bits is not None:
        c, s = cache_rows(cos_sin, pos_k, cache_dtype)
        kr = bf16_bits_to_f64(k_rope_bits)
        rk = rotate(kr, c, s, is_neox)
        outs[1] = e4m3_encode(rk * quant_scale_kv)
        outs[3] = e4m3_encode(bf16_bits_to_f64(k_nope_bits) * quant_scale_kv)
    return tuple(outs)


def rope_quantize_fp8_append_paged(k_rope_bits, k_nope_bits, cos_sin, pos_k, batch_indices,
                                   positions, kv_indptr, kv_indices, kv_pages, page_size,
                                   is_neox=True, quant_scale_kv=1.0, cache_dtype="f32"):
    """The key rows of mla_rope_quantize_fp8, appended: returns a copy of the paged cache
    kv_pages [num_pages, page_size, 576] (E4M3 codes) with each row written to its slot."""
    _, kr, _, kn = mla_rope_quantize_fp8(None, k_rope_bits, None, k_nope_bits, cos_sin, None,
                                         pos_k, is_neox, 1.0, quant_scale_kv, cache_dtype)
    out = np.array(kv_pages, dtype=np.uint8, copy=True)
    for i in range(len(kn)):
        b, q = int(batch_indices[i]), int(positions[i])
        slot = int(kv_indptr[b]) + q // page_size
        if slot >= int(kv_indptr[b + 1]):
            raise ValueError("position past the request's pages")
        page = int(kv_indices[slot])
        out[page, q % page_size, :NOPE_DIM] = kn[i]
        out[page, q % page_size, NOPE_DIM:] = kr[i]
    return out
