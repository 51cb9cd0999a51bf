"""Attention restricted to a CSR-indexed key set, as plain dense masked softmax (float64).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Every index form is expanded into the plain definition: for query row i and query
head h (key/value head h // (Hq/Hkv)),
    logits_j = sm_scale * <q_i, k_j>       for the keys j visible to row i
    out_i    = sum_j softmax(logits)_j v_j
    lse_i    = log sum_j exp(logits_j)     (natural log, of the scaled logits)
A row that sees no key gets out = 0 and lse = -inf.

Sources:
  * BSR mask and GQA: "flashinfer.sparse - FlashInfer 0.7.4 documentation",
    BlockSparseAttentionWrapper: the mask is a SciPy bsr_matrix (indptr of length
    MB+1, MB = ceil_div(M, R); indices < NB = N // C); the 3x3 worked example checks
    the result against dense attention with the same boolean mask; plan(mask=(nnz, R, C))
    selects the visible pairs inside each listed block and then causal does not apply
    (packed_mask: the same entries packed as bits; reading: little-endian bit order within
    a byte, as numpy.packbits(bitorder="little")); num_qo_heads must
    be a multiple of num_kv_heads (grouped-query attention); sm_scale defaults to
    1/sqrt(head_dim); run() returns out [M, Hq, D] and lse [M, Hq].
  * causal: plan() parameter "causal"; for M != N the mask is aligned bottom-right,
    key j visible to query i iff j <= i + (N - M) (FlashInfer cheat page, benchmark
    README flag --causal: multi-query decode uses bottom-right causal masking).
  * Variable blocks: "flashinfer.sparse", VariableBlockSparseAttentionWrapper: plan(
    block_mask_map (num_kv_heads, MB, NB), block_row_sz (num_kv_heads, MB), block_col_sz
    (num_kv_heads, NB)); each kv head its own pattern, shared by its query heads; run(q
    (num_qo_heads, qo_len, head_dim), k/v (num_kv_heads, kv_len, head_dim)) returns out of
    q's shape and lse (num_qo_heads, qo_len). Reading: blocks are consecutive in the order
    given, and causal keeps key j for query i iff j <= i + (kv_len - qo_len).
  * Paged KV: "FlashInfer" agent-skill summary, KV-Cache Formats / Paged KV-Cache:
    kv_cache (num_pages, 2, num_kv_heads, page_size, head_dim), kv_indptr (batch+1,),
    kv_indices, kv_last_page_len (batch,). Reading: request b owns pages
    kv_indices[kv_indptr[b]:kv_indptr[b+1]] in order, and its length is
    (n_pages - 1) * page_size + kv_last_page_len[b].
  * Paged prefill: FlashInfer cheat page, benchmark README (BatchPrefillWithPagedKVCacheWrapper,
    the paged-cache prefill wrapper); "FlashInfer" agent-skill summary, Batch prefill
    and Append (causal prefill of new tokens against the cache). Reading: request b's queries
    are the last qo_len_b tokens of its sequence, so causal is aligned bottom-right.
  * Sparse MLA: "Sparse MLA" (MATE 0.2.6), sparse_mla_fp8_decode: FP8 query
    [batch, q_len, heads, 576], FP8 cache rows of 576 values, int32 physical-token
    indices [batch, q_len, top_k] shared by all heads, seq_lens[b] valid entries,
    bmm1_scale on the QK product, bmm2_scale on the output, BF16 output of 512 values
    (kv_lora_rank) and FP32 LSE. Reading: V is the first 512 values of each row.
  * Dense paged MLA: "FlashInfer" agent-skill summary, Multi-Head Latent Attention (MLA)
    (BatchMLAPagedAttentionWrapper; trtllm_batch_decode_with_kv_cache_mla over the latent
    cache) and FlashInfer cheat page, benchmark README (BatchMLAPagedAttentionWrapper: MLA
    attention of the DeepSeek models). Reading: the sparse MLA contraction over all tokens
    of the request, whose 576-value latent rows are paged with the page table of Paged KV.
  * merge: FlashInfer cheat page, docs/api/cascade.rst (merge_state, merge_states);
    "FlashInfer" agent-skill summary, Cascade Inference (merge attention states).
"""

import numpy as np

from .numerics import bits_to_f64, e4m3_decode


def masked_attention(q, k, v, sm_scale, mask=None):
    """Dense masked softmax attention.

    q [Mq, Hq, D], k [Nk, Hkv, D], v [Nk, Hkv, Dv] float64; mask [Mq, Nk] bool (True =
    visible) shared by all heads, or None for all visible.
    Returns out [Mq, Hq, Dv] and lse [Mq, Hq] (float64).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    Mq, Hq, _ = q.shape
    Nk, Hkv, Dv = v.shape
    if Hq % Hkv != 0:
        raise ValueError("num_kv_heads must divide num_qo_heads")
    g = Hq // Hkv
    out = np.zeros((Mq, Hq, Dv))
    lse = np.full((Mq, Hq), -np.inf)
    if Nk == 0 or Mq == 0:
        return out, lse
    for h in range(Hq):
        kh = h // g
        logits = sm_scale * (q[:, h, :] @ k[:, kh, :].T)
        if mask is not None:
            logits = np.where(mask, logits, -np.inf)
        m = logits.max(axis=1)
        live = np.isfinite(m)
        ms = np.where(live, m, 0.0)
        p = np.exp(logits - ms[:, None])
        p = np.where(np.isfinite(logits), p, 0.0)
        l = p.sum(axis=1)
        o = (p @ v[:, kh, :]) / np.where(live, l, 1.0)[:, None]
        out[:, h, :] = np.where(live[:, None], o, 0.0)
        lse[:, h] = np.where(live, ms + np.log(np.where(live, l, 1.0)), -np.inf)
    return out, lse


# ---------------------------------------------------------------------------------------
# BSR block-sparse mask
# ---------------------------------------------------------------------------------------

def bsr_mask(indptr, indices, M, N, R, C, causal=False, rows=None, block_mask=None):
    """Dense boolean mask [len(rows), N] of a BSR block mask (rows default to all M).

    ``block_mask`` (nnz, R, C) optionally selects the visible pairs inside each listed block
    (entry [e, i % R, j % C] for the block at position e of ``indices``); causal is then not
    applied (it only acts when no mask is given)."""
    indptr = np.asarray(indptr, dtype=np.int64)
    indices = np.asarray(indices, dtype=np.int64)
    MB = (M + R - 1) // R
    NB = N // C
    if N % C != 0:
        raise ValueError("N must be divisible by C")
    if indptr.shape != (MB + 1,):
        raise ValueError("indptr must have MB + 1 entries")
    rows = np.arange(M) if rows is None else np.asarray(rows, dtype=np.int64)
    mask = np.zeros((len(rows), N), dtype=bool)
    for r, i in enumerate(rows):
        bi = i // R
        for e in range(indptr[bi], indptr[bi + 1]):
            j = indices[e]
            if not (0 <= j < NB):
                raise ValueError("column block index out of range")
            if block_mask is None:
                mask[r, j * C:(j + 1) * C] = True
            else:
                mask[r, j * C:(j + 1) * C] = block_mask[e, i % R]
    if causal and block_mask is None:
        cols = np.arange(N)
        mask &= cols[None, :] <= (rows[:, None] + (N - M))
    return mask


def bsr_attention(q_bits, k_bits, v_bits, dtype, indptr, indices, M, N, R, C,
                  sm_scale=None, causal=False, rows=None, block_mask=None):
    """BSR block-sparse attention from stored 16-bit inputs.

    q [M, Hq, D], k/v [N, Hkv, D] as uint16 bit patterns of ``dtype`` ('fp16'/'bf16').
    ``rows`` restricts the computation to some query rows (returned in that order).
    """
    q = bits_to_f64(q_bits, dtype)
    D = q.shape[-1]
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    rows_idx = np.arange(M) if rows is None else np.asarray(rows, dtype=np.int64)
    mask = bsr_mask(indptr, indices, M, N, R, C, causal, rows_idx, block_mask)
    k = bits_to_f64(k_bits, dtype)
    v = bits_to_f64(v_bits, dtype)
    return masked_attention(q[rows_idx], k, v, sm_scale, mask)


# ---------------------------------------------------------------------------------------
# Variable-block sparse attention
# ---------------------------------------------------------------------------------------

def variable_block_mask(block_mask_map, block_row_sz, block_col_sz, causal=False, rows=None):
    """Dense boolean masks [Hkv, qo_len, kv_len]: kv head h cuts the query tokens into
    consecutive row blocks of block_row_sz[h] tokens and the keys into consecutive column
    blocks of block_col_sz[h]; block (a, c) is visible iff block_mask_map[h, a, c].
    ``rows`` optionally lists the query tokens to build (then [Hkv, len(rows), kv_len])."""
    bm = np.asarray(block_mask_map, dtype=bool)
    rs = np.asarray(block_row_sz, dtype=np.int64)
    cs = np.asarray(block_col_sz, dtype=np.int64)
    H, MB, NB = bm.shape
    qo, kv = int(rs[0].sum()), int(cs[0].sum())
    sel = np.arange(qo) if rows is None else np.asarray(rows, dtype=np.int64)
    out = np.zeros((H, len(sel), kv), dtype=bool)
    for h in range(H):
        if rs[h].sum() != qo or cs[h].sum() != kv:
            raise ValueError("every kv head must cover the same lengths")
        r0 = np.concatenate([[0], np.cumsum(rs[h])])
        c0 = np.concatenate([[0], np.cumsum(cs[h])])
        for a in range(MB):
            inside = (sel >= r0[a]) & (sel < r0[a + 1])   # the selected tokens of row block a
            for c in range(NB):
                if bm[h, a, c]:
                    out[h, inside, c0[c]:c0[c + 1]] = True
    if causal:
        i = sel[:, None]
        j = np.arange(kv)[None, :]
        out &= (j <= i + (kv - qo))[None]
    return out


def variable_block_attention(q_bits, k_bits, v_bits, dtype, block_mask_map, block_row_sz,
                             block_col_sz, sm_scale=None, causal=False, rows=None):
    """Variable-block sparse attention from stored 16-bit inputs, head-major as on the page:
    q [Hq, qo_len, D], k/v [Hkv, kv_len, D]. Returns out [Hq, qo_len, D] and lse [Hq, qo_len];
    query head hq uses kv head hq // (Hq / Hkv) and that head's mask. ``rows`` optionally lists
    the query tokens to compute (then out [Hq, len(rows), D], lse [Hq, len(rows)])."""
    if rows is not None:
        q_bits = np.asarray(q_bits)[:, np.asarray(rows, dtype=np.int64)]
    q = bits_to_f64(q_bits, dtype)
    k = bits_to_f64(k_bits, dtype)
    v = bits_to_f64(v_bits, dtype)
    Hq, L, D = q.shape
    Hkv = k.shape[0]
    g = Hq // Hkv
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    masks = variable_block_mask(block_mask_map, block_row_sz, block_col_sz, causal, rows)
    out = np.zeros((Hq, L, v.shape[-1]))
    lse = np.zeros((Hq, L))
    for h in range(Hkv):
        qg = q[h * g:(h + 1) * g].transpose(1, 0, 2)           # [L, g, D]
        o, l = masked_attention(qg, k[h][:, None, :], v[h][:, None, :], sm_scale, masks[h])
        out[h * g:(h + 1) * g] = o.transpose(1, 0, 2)
        lse[h * g:(h + 1) * g] = l.T
    return out, lse


# ---------------------------------------------------------------------------------------
# Paged KV decode
# ---------------------------------------------------------------------------------------

def paged_kv_len(kv_indptr, kv_last_page_len, page_size, b):
    n = int(kv_indptr[b + 1]) - int(kv_indptr[b])
    if n == 0:
        return 0
    return (n - 1) * page_size + int(kv_last_page_len[b])


def paged_kv(kv_bits, dtype, kv_indptr, kv_indices, kv_last_page_len, page_size, b):
    """Logical K, V [L_b, Hkv, D] (float64) of request b, from its page list."""
    pages = np.asarray(kv_indices[int(kv_indptr[b]):int(kv_indptr[b + 1])], dtype=np.int64)
    L = paged_kv_len(kv_indptr, kv_last_page_len, page_size, b)
    Hkv, D = kv_bits.shape[2], kv_bits.shape[4]
    if L == 0:
        return np.zeros((0, Hkv, D)), np.zeros((0, Hkv, D))
    blk = kv_bits[pages]                       # [n, 2, Hkv, ps, D]
    kb = blk[:, 0].transpose(0, 2, 1, 3).reshape(-1, Hkv, D)[:L]
    vb = blk[:, 1].transpose(0, 2, 1, 3).reshape(-1, Hkv, D)[:L]
    return bits_to_f64(kb, dtype), bits_to_f64(vb, dtype)


def paged_decode(q_bits, kv_bits, dtype, kv_indptr, kv_indices, kv_last_page_len, page_size,
                 sm_scale=None, requests=None):
    """Batch decode over a paged KV cache: one query token per request.

    q [B, Hq, D] and kv_cache [pages, 2, Hkv, page_size, D] as 16-bit bit patterns.
    Returns out [len(requests), Hq, D], lse [len(requests), Hq].
    """
    B, Hq, D = q_bits.shape
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    reqs = range(B) if requests is None else requests
    outs, lses = [], []
    for b in reqs:
        k, v = paged_kv(kv_bits, dtype, kv_indptr, kv_indices, kv_last_page_len, page_size, b)
        q = bits_to_f64(q_bits[b:b + 1], dtype)
        o, l = masked_attention(q, k, v, sm_scale)
        outs.append(o[0])
        lses.append(l[0])
    return np.stack(outs), np.stack(lses)


def paged_prefill(q_bits, kv_bits, dtype, qo_indptr, kv_indptr, kv_indices, kv_last_page_len,
                  page_size, sm_scale=None, causal=True, requests=None):
    """Batch prefill over a paged KV cache: request b's query tokens
    q[qo_indptr[b]:qo_indptr[b+1]] (the last qo_len_b tokens of its sequence) attend to the
    L_b keys of its pages; causal keeps key j for local query t iff j <= t + L_b - qo_len_b.
    q [total_qo, Hq, D] and the cache as 16-bit patterns. Returns the rows of the requested
    requests (all by default) in order: out [n, Hq, D], lse [n, Hq]."""
    D = q_bits.shape[-1]
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    reqs = range(len(qo_indptr) - 1) if requests is None else requests
    outs, lses = [], []
    for b in reqs:
        q = bits_to_f64(q_bits[int(qo_indptr[b]):int(qo_indptr[b + 1])], dtype)
        k, v = paged_kv(kv_bits, dtype, kv_indptr, kv_indices, kv_last_page_len, page_size, b)
        nq, L = q.shape[0], k.shape[0]
        mask = None
        if causal:
            mask = np.arange(L)[None, :] <= (np.arange(nq)[:, None] + (L - nq))
        o, l = masked_attention(q, k, v, sm_scale, mask)
        outs.append(o)
        lses.append(l)
    return np.concatenate(outs), np.concatenate(lses)


# ---------------------------------------------------------------------------------------
# Sparse MLA FP8 decode
# ---------------------------------------------------------------------------------------

KV_LORA_RANK = 512
QK_DIM = 576


def mla_sparse_decode(query_codes, kv_codes, indices, seq_lens, bmm1_scale, bmm2_scale,
                      queries=None):
    """Sparse MLA decode from E4M3 codes.

    query [B, T, H, 576] and kv rows [rows, 576] as uint8 E4M3 codes; indices
    [B, T, top_k] int32 row ids; seq_lens [B]. ``queries`` optionally lists (b, t)
    pairs to compute. Returns out [n, H, 512] and lse [n, H] (float64), with
    out = bmm2_scale * softmax(bmm1_scale * q k^T) v and lse of the bmm1-scaled logits.
    """
    B, T, H, Dq = query_codes.shape
    if Dq != QK_DIM or kv_codes.shape[-1] != QK_DIM:
        raise ValueError("MLA rows must hold 576 values")
    qs = [(b, t) for b in range(B) for t in range(T)] if queries is None else queries
    outs, lses = [], []
    for b, t in qs:
        n = int(seq_lens[b])
        idx = np.asarray(indices[b, t, :n], dtype=np.int64)
        if np.any(idx < 0) or np.any(idx >= kv_codes.shape[0]):
            raise ValueError("sparse index out of range")
        kv = e4m3_decode(kv_codes[idx])                  # [n, 576]
        q = e4m3_decode(query_codes[b, t])               # [H, 576]
        o, l = masked_attention(q[None], kv[:, None, :], kv[:, None, :KV_LORA_RANK],
                                bmm1_scale)
        outs.append(bmm2_scale * o[0])
        lses.append(l[0])
    return np.stack(outs), np.stack(lses)


def mla_paged_decode(query_codes, kv_page_codes, kv_indptr, kv_indices, kv_last_page_len,
                     page_size, bmm1_scale, bmm2_scale, requests=None):
    """Dense paged MLA decode from E4M3 codes: one query token per request attends to every
    token of its request.

    query [B, H, 576] and the latent cache [pages, page_size, 576] as uint8 E4M3 codes; the
    page table as for paged_decode (request b owns pages kv_indices[kv_indptr[b]:
    kv_indptr[b+1]] in order, length (n_b - 1) * page_size + kv_last_page_len[b]). The
    request's logical rows are its pages' rows concatenated and cut to that length; then
    the sparse MLA definition applies to them (same scales, V = the first 512 values).
    Returns out [n, H, 512] and lse [n, H] (float64).
    """
    B, H, Dq = query_codes.shape
    if Dq != QK_DIM or kv_page_codes.shape[-1] != QK_DIM:
        raise ValueError("MLA rows must hold 576 values")
    reqs = range(B) if requests is None else requests
    outs, lses = [], []
    for b in reqs:
        L = paged_kv_len(kv_indptr, kv_last_page_len, page_size, b)
        pages = np.asarray(kv_indices[int(kv_indptr[b]):int(kv_indptr[b + 1])], dtype=np.int64)
        rows = kv_page_codes[pages].reshape(-1, QK_DIM)[:L]       # [L, 576] codes, in order
        kv = e4m3_decode(rows)
        q = e4m3_decode(query_codes[b])                            # [H, 576]
        o, l = masked_attention(q[None], kv[:, None, :], kv[:, None, :KV_LORA_RANK], bmm1_scale)
        outs.append(bmm2_scale * o[0])
        lses.append(l[0])
    return np.stack(outs), np.stack(lses)


# ---------------------------------------------------------------------------------------
# Merge of attention states
# ---------------------------------------------------------------------------------------

def merge_states(v, s, axis=1):
    """Merge attention states along ``axis``.

    v [..., S, ..., D] partial outputs, each normalised over its own key set; s the
    matching natural-log LSE (v without its last dim). The merged state is
        lse = log sum_c exp(s_c),   out = sum_c exp(s_c - lse) v_c,
    which equals attention over the union of the key sets. States with lse = -inf
    (no key) carry no weight; if all are empty, out = 0 and lse = -inf.
    """
    v = np.asarray(v, dtype=np.float64)
    s = np.asarray(s, dtype=np.float64)
    m = np.max(s, axis=axis, keepdims=True)
    live = np.isfinite(m)
    ms = np.where(live, m, 0.0)
    w = np.exp(s - ms)
    w = np.where(np.isfinite(s), w, 0.0)
    tot = np.sum(w, axis=axis, keepdims=True)
    lse = np.where(live, ms + np.log(np.where(live, tot, 1.0)), -np.inf)
    wn = w / np.where(live, tot, 1.0)
    out = np.sum(wn[..., None] * v, axis=axis)
    return out, np.squeeze(lse, axis=axis)
