"""Seeded generators for the workloads of CSR-indexed sparse/paged attention.

Every generator takes a seed and the sizes of its workload and returns a dict of
torch tensors plus the integer parameters. Index structures are always drawn on the
CPU from ``torch.Generator().manual_seed(seed)``. Bulk N(0,1) tensors are drawn in
float32 on ``device`` (a generator seeded with ``seed + 1``) and cast to the
workload dtype by torch (round to nearest even). Whoever checks a result reads the
very same stored bytes as whoever computes it.
"""

import math

import torch

_SLAB = 1 << 26  # elements per float32 draw, to bound temporary memory


def _cpu_gen(seed):
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def _dev_gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed + 1)
    return g


def _randn(shape, dtype, gen, device, scale=1.0):
    """N(0,1) float32 draws cast to ``dtype``, drawn in slabs along dim 0."""
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, _SLAB):
        e = min(n, s + _SLAB)
        x = torch.randn(e - s, generator=gen, dtype=torch.float32, device=device)
        if scale != 1.0:
            x.mul_(scale)
        flat[s:e].copy_(x.to(dtype))
    return out


def _uniform_int(g, lo, hi, n):
    """n integers uniform in [lo, hi] inclusive."""
    return torch.randint(lo, hi + 1, (n,), generator=g, dtype=torch.int64)


# --------------------------------------------------------------------------------------
# BSR block-sparse attention
# --------------------------------------------------------------------------------------

def bsr_inputs(seed, M, N, R, C, num_qo_heads, num_kv_heads, head_dim, dtype=torch.float16,
               pattern="random", density=0.5, p_off=0.1, causal=False, q_scale=1.0,
               device="cpu", tensors=True):
    """Block-sparse attention inputs.

    pattern "random": each of the MB x NB blocks is kept with probability ``density``;
    a row block left empty gets one uniformly chosen column block.
    pattern "diag_lower": every diagonal block, plus each strictly-lower block kept
    independently with probability ``p_off``.
    pattern "full": every block.
    Column indices of a row are sorted ascending (CSR form).
    """
    g = _cpu_gen(seed)
    MB = (M + R - 1) // R
    NB = N // C
    rows = []
    if pattern == "random":
        keep = torch.rand((MB, NB), generator=g) < density
        for i in range(MB):
            if not bool(keep[i].any()):
                j = int(torch.randint(0, NB, (1,), generator=g))
                keep[i, j] = True
            rows.append(torch.nonzero(keep[i]).flatten())
    elif pattern == "diag_lower":
        assert MB <= NB
        keep = torch.rand((MB, NB), generator=g) < p_off
        keep = torch.tril(keep, diagonal=-1)
        keep[torch.arange(MB), torch.arange(MB)] = True
        for i in range(MB):
            rows.append(torch.nonzero(keep[i]).flatten())
    elif pattern == "full":
        for i in range(MB):
            rows.append(torch.arange(NB))
    else:
        raise ValueError(pattern)
    counts = torch.tensor([len(r) for r in rows], dtype=torch.int64)
    indptr = torch.zeros(MB + 1, dtype=torch.int32)
    indptr[1:] = torch.cumsum(counts, 0).to(torch.int32)
    indices = (torch.cat(rows) if rows else torch.zeros(0, dtype=torch.int64)).to(torch.int32)

    q = k = v = None
    if tensors:
        dg = _dev_gen(seed, device)
        q = _randn((M, num_qo_heads, head_dim), dtype, dg, device, q_scale)
        k = _randn((N, num_kv_heads, head_dim), dtype, dg, device)
        v = _randn((N, num_kv_heads, head_dim), dtype, dg, device)
    return dict(q=q, k=k, v=v, indptr=indptr, indices=indices, M=M, N=N, R=R, C=C,
                num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                causal=causal, sm_scale=1.0 / math.sqrt(head_dim), seed=seed)


# --------------------------------------------------------------------------------------
# Paged-KV decode
# --------------------------------------------------------------------------------------

def paged_decode_inputs(seed, batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                        len_lo, len_hi, dtype=torch.bfloat16, canary_frac=0.1,
                        lengths=None, q_scale=1.0, device="cpu", tensors=True):
    """One query token per request over a paged KV cache (HND pages).

    kv lengths L_b are uniform integers in [len_lo, len_hi] (or ``lengths``). Request b
    owns ceil(L_b / page_size) pages; all pages are a random permutation of a shared
    pool holding ``canary_frac`` extra pages. Unreferenced pool pages and the slots past
    each last page's valid length hold NaN, so a read of anything outside the page
    table poisons the output.

    kv_cache layout: [num_pages, 2, num_kv_heads, page_size, head_dim] (index 0 = K).
    """
    g = _cpu_gen(seed)
    if lengths is None:
        lengths = _uniform_int(g, len_lo, len_hi, batch)
    else:
        lengths = torch.as_tensor(lengths, dtype=torch.int64)
    npages = (lengths + page_size - 1) // page_size
    total = int(npages.sum())
    pool = total + int(math.ceil(canary_frac * total))
    pool = max(pool, 1)
    perm = torch.randperm(pool, generator=g)
    kv_indices = perm[:total].to(torch.int32)
    kv_indptr = torch.zeros(batch + 1, dtype=torch.int32)
    kv_indptr[1:] = torch.cumsum(npages, 0).to(torch.int32)
    last = lengths - (npages - 1) * page_size
    last = torch.where(npages == 0, torch.zeros_like(last), last).to(torch.int32)

    kv_cache = q = None
    if tensors:
        dg = _dev_gen(seed, device)
        kv_cache = _randn((pool, 2, num_kv_heads, page_size, head_dim), dtype, dg, device)
        unused = perm[total:].to(device)
        if unused.numel():
            kv_cache[unused] = float("nan")
        for b in range(batch):
            n = int(npages[b])
            if n == 0:
                continue
            lp = int(kv_indices[int(kv_indptr[b]) + n - 1])
            lb = int(last[b])
            if lb < page_size:
                kv_cache[lp, :, :, lb:, :] = float("nan")
        q = _randn((batch, num_qo_heads, head_dim), dtype, dg, device, q_scale)
    return dict(q=q, kv_cache=kv_cache, kv_indptr=kv_indptr, kv_indices=kv_indices,
                kv_last_page_len=last, kv_lens=lengths.to(torch.int32), batch=batch,
                num_qo_heads=num_qo_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                page_size=page_size, num_pages=pool, sm_scale=1.0 / math.sqrt(head_dim),
                seed=seed)


def paged_prefill_inputs(seed, batch, num_qo_heads, num_kv_heads, head_dim, page_size, len_lo,
                         len_hi, qo_lo, qo_hi, dtype=torch.bfloat16, lengths=None,
                         qo_lens=None, device="cpu"):
    """Batch prefill over a paged KV cache: the cache of paged_decode_inputs (lengths L_b,
    permuted pages, NaN canaries) plus qo_len_b = min(U[qo_lo, qo_hi], L_b) query tokens per
    request (or ``qo_lens``), ragged in q [total_qo, Hq, D] with qo_indptr."""
    d = paged_decode_inputs(seed, batch, num_qo_heads, num_kv_heads, head_dim, page_size,
                            len_lo, len_hi, dtype=dtype, lengths=lengths, device=device)
    g = _cpu_gen(seed + 3)
    if qo_lens is None:
        qo_lens = [min(int(x), int(L)) for x, L in zip(_uniform_int(g, qo_lo, qo_hi, batch),
                                                         d["kv_lens"])]
    qo_indptr = torch.zeros(batch + 1, dtype=torch.int32)
    qo_indptr[1:] = torch.cumsum(torch.tensor(qo_lens, dtype=torch.int64), 0).to(torch.int32)
    dg = _dev_gen(seed + 5, device)
    q = _randn((int(qo_indptr[-1]), num_qo_heads, head_dim), dtype, dg, device)
    d.update(q=q, qo_indptr=qo_indptr, qo_lens=torch.tensor(qo_lens, dtype=torch.int32),
             dtype=dtype)
    return d


# --------------------------------------------------------------------------------------
# MLA sparse FP8 decode and its RoPE + FP8 prologue
# --------------------------------------------------------------------------------------

def rope_cos_sin_cache(max_seq_len, rotary_dim=64, theta=1e4, dtype=torch.float32):
    """cos/sin cache [max_seq_len, rotary_dim]: columns [:half] cos, [half:] sin.

    Column i < half holds cos(p * theta^(-2i/rotary_dim)) and column half + i the
    matching sine, computed in float64 and stored in ``dtype``.
    """
    half = rotary_dim // 2
    p = torch.arange(max_seq_len, dtype=torch.float64)[:, None]
    inv = theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / rotary_dim)
    ang = p * inv[None, :]
    return torch.cat([torch.cos(ang), torch.sin(ang)], dim=1).to(dtype).contiguous()


def mla_inputs(seed, batch, heads, top_k, pool_rows, ctx_lo, ctx_hi, q_len=1,
               max_seq_len=65536, theta=1e4, seq_lens=None, q_scale=1.0,
               cache_dtype=torch.float32, device="cpu"):
    """Inputs of the RoPE+FP8 prologue and of the sparse MLA decode.

    * q_nope [batch*q_len, heads, 512], q_rope [batch*q_len, heads, 64] bf16 ~ N(0,1)
    * k_nope [pool_rows, 512], k_rope [pool_rows, 64] bf16 ~ N(0,1); pool row r sits at
      rotary position r (pos_k = arange)
    * cos_sin [max_seq_len, 64] (float64 formula stored in ``cache_dtype``)
    * per query token (b, t): a context of length L ~ U[ctx_lo, ctx_hi] at pool rows
      [off, off + L) with off ~ U[0, pool_rows - L]; ``top_k`` distinct indices drawn
      uniformly from it; the query's own position is off + L - 1.
    * seq_lens [batch] valid sparse lengths (default: top_k for every request)
    """
    assert pool_rows <= max_seq_len
    g = _cpu_gen(seed)
    nq = batch * q_len
    indices = torch.empty((batch, q_len, top_k), dtype=torch.int32)
    pos_q = torch.empty(nq, dtype=torch.int32)
    for n in range(nq):
        L = int(_uniform_int(g, ctx_lo, ctx_hi, 1))
        L = min(L, pool_rows)
        assert L >= top_k
        off = int(_uniform_int(g, 0, pool_rows - L, 1))
        sel = torch.randperm(L, generator=g)[:top_k] + off
        indices[n // q_len, n % q_len] = sel.to(torch.int32)
        pos_q[n] = off + L - 1
    if seq_lens is None:
        seq_lens = torch.full((batch,), top_k, dtype=torch.int32)
    else:
        seq_lens = torch.as_tensor(seq_lens, dtype=torch.int32)

    dg = _dev_gen(seed, device)
    q_nope = _randn((nq, heads, 512), torch.bfloat16, dg, device, q_scale)
    q_rope = _randn((nq, heads, 64), torch.bfloat16, dg, device, q_scale)
    k_nope = _randn((pool_rows, 512), torch.bfloat16, dg, device)
    k_rope = _randn((pool_rows, 64), torch.bfloat16, dg, device)
    cos_sin = rope_cos_sin_cache(max_seq_len, 64, theta, cache_dtype).to(device)
    pos_k = torch.arange(pool_rows, dtype=torch.int32)
    return dict(q_nope=q_nope, q_rope=q_rope, k_nope=k_nope, k_rope=k_rope, cos_sin=cos_sin,
                pos_q=pos_q, pos_k=pos_k, indices=indices, seq_lens=seq_lens, batch=batch,
                q_len=q_len, heads=heads, top_k=top_k, pool_rows=pool_rows,
                max_seq_len=max_seq_len, seed=seed)


def variable_block_inputs(seed, num_qo_heads, num_kv_heads, head_dim, MB, NB, qo_len, kv_len,
                          density=0.5, dtype=torch.float16, causal=False, empty_row_block=None,
                          device="cpu"):
    """Variable-block sparse attention inputs (head-major tensors, as on the page).

    Every kv head cuts qo_len query tokens into MB and kv_len keys into NB consecutive blocks
    of random positive sizes (a fresh cut per head) and keeps each block with probability
    ``density`` (``empty_row_block``: that row block of every head keeps none).
    q [Hq, qo_len, D], k/v [Hkv, kv_len, D] ~ N(0,1) cast to ``dtype``.
    """
    g = _cpu_gen(seed)
    H = num_kv_heads

    def parts(total, n):
        out = []
        for _ in range(H):
            cuts = sorted((torch.randperm(total - 1, generator=g)[:n - 1] + 1).tolist())
            out.append([b - a for a, b in zip([0] + cuts, cuts + [total])])
        return torch.tensor(out, dtype=torch.int32)

    row_sz = parts(qo_len, MB)
    col_sz = parts(kv_len, NB)
    bm = torch.rand((H, MB, NB), generator=g) < density
    if empty_row_block is not None:
        bm[:, empty_row_block, :] = False
    dg = _dev_gen(seed, device)
    q = _randn((num_qo_heads, qo_len, head_dim), dtype, dg, device)
    k = _randn((H, kv_len, head_dim), dtype, dg, device)
    v = _randn((H, kv_len, head_dim), dtype, dg, device)
    return dict(q=q, k=k, v=v, block_mask_map=bm, block_row_sz=row_sz, block_col_sz=col_sz,
                num_qo_heads=num_qo_heads, num_kv_heads=H, head_dim=head_dim, MB=MB, NB=NB,
                qo_len=qo_len, kv_len=kv_len, causal=causal, dtype=dtype, seed=seed)


E4M3_NAN = 0x7F  # canary code for cache slots no request may read


def _e4m3_codes(shape, gen, device, scale=1.0):
    """uint8 E4M3 codes of N(0,1) float32 draws (torch cast, round to nearest even)."""
    out = torch.empty(shape, dtype=torch.uint8, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, _SLAB):
        e = min(n, s + _SLAB)
        x = torch.randn(e - s, generator=gen, dtype=torch.float32, device=device)
        if scale != 1.0:
            x.mul_(scale)
        flat[s:e].copy_(x.to(torch.float8_e4m3fn).view(torch.uint8))
    return out


def mla_paged_inputs(seed, batch, heads, page_size, len_lo, len_hi, spare=0.1, lens=None,
                     q_scale=1.0, device="cpu"):
    """Inputs of the dense paged MLA decode.

    * request b has L_b ~ U[len_lo, len_hi] tokens (or ``lens``) in n_b = ceil(L_b / page_size)
      pages; the pages of all requests are a random permutation of the pool pages
      [0, P), P = sum n_b + ceil(spare * sum n_b) (the spare pages are canaries);
    * kv_indptr [batch+1], kv_indices, kv_last_page_len [batch] int32 (the page table);
    * query [batch, heads, 576] and kv_pages [P, page_size, 576]: uint8 E4M3 codes of
      N(0,1) draws; every slot past a request's last token and every spare page holds the
      E4M3 NaN code, so a read outside the request shows up.
    """
    g = _cpu_gen(seed)
    if lens is None:
        lens = [int(x) for x in _uniform_int(g, len_lo, len_hi, batch)]
    lens = [int(x) for x in lens]
    npg = [(L + page_size - 1) // page_size for L in lens]
    used = sum(npg)
    P = max(1, used + int(math.ceil(spare * used)))
    perm = torch.randperm(P, generator=g).to(torch.int32)
    kv_indptr = torch.zeros(batch + 1, dtype=torch.int32)
    kv_indptr[1:] = torch.cumsum(torch.tensor(npg, dtype=torch.int64), 0).to(torch.int32)
    kv_indices = perm[:used].clone()
    kv_last_page_len = torch.tensor([L - (n - 1) * page_size if n > 0 else 0
                                     for L, n in zip(lens, npg)], dtype=torch.int32)
    dg = _dev_gen(seed, device)
    query = _e4m3_codes((batch, heads, 576), dg, device, q_scale)
    kv_pages = _e4m3_codes((P, page_size, 576), dg, device)
    kv_pages[perm[used:].to(torch.int64).to(device)] = E4M3_NAN
    for b in range(batch):
        n = npg[b]
        lp = int(kv_last_page_len[b])
        if n > 0 and lp < page_size:
            kv_pages[int(kv_indices[int(kv_indptr[b]) + n - 1]), lp:] = E4M3_NAN
    return dict(query=query, kv_pages=kv_pages, kv_indptr=kv_indptr, kv_indices=kv_indices,
                kv_last_page_len=kv_last_page_len, lens=torch.tensor(lens, dtype=torch.int32),
                batch=batch, heads=heads, page_size=page_size, num_pages=P, seed=seed)


def mla_append_inputs(seed, batch, page_size, len_lo, len_hi, new_tokens, lens=None,
                      max_seq_len=65536, theta=1e4, device="cpu"):
    """Inputs of the RoPE + FP8 append into a paged latent cache.

    Request b holds L_b ~ U[len_lo, len_hi] tokens (or ``lens``) plus ``new_tokens`` more,
    in the pages of mla_paged_inputs (canary-filled cache, permuted pages). The appended
    rows are the last ``new_tokens`` positions of every request: batch_indices,
    positions (also their rotary positions pos_k), k_rope [nnz, 64] and k_nope [nnz, 512]
    bf16 ~ N(0,1), and the cos/sin cache.
    """
    g = _cpu_gen(seed + 7)
    if lens is None:
        lens = [int(x) for x in _uniform_int(g, len_lo, len_hi, batch)]
    total = [int(L) + new_tokens for L in lens]
    d = mla_paged_inputs(seed, batch=batch, heads=1, page_size=page_size, len_lo=0, len_hi=0,
                         lens=total, device=device)
    bi, pos = [], []
    for b, L in enumerate(lens):
        bi += [b] * new_tokens
        pos += list(range(int(L), int(L) + new_tokens))
    assert max(pos, default=0) < max_seq_len
    nnz = len(pos)
    dg = _dev_gen(seed + 11, device)
    k_rope = _randn((nnz, 64), torch.bfloat16, dg, device)
    k_nope = _randn((nnz, 512), torch.bfloat16, dg, device)
    cos_sin = rope_cos_sin_cache(max_seq_len, 64, theta, torch.float32).to(device)
    positions = torch.tensor(pos, dtype=torch.int32)
    return dict(kv_pages=d["kv_pages"], kv_indptr=d["kv_indptr"], kv_indices=d["kv_indices"],
                kv_last_page_len=d["kv_last_page_len"], num_pages=d["num_pages"],
                page_size=page_size, batch=batch, batch_indices=torch.tensor(bi, dtype=torch.int32),
                positions=positions, pos_k=positions.clone(), k_rope=k_rope, k_nope=k_nope,
                cos_sin=cos_sin, max_seq_len=max_seq_len, seed=seed)


# --------------------------------------------------------------------------------------
# The five workloads at full size (seeds 1000 + index)
# --------------------------------------------------------------------------------------

CONFIGS = {
    "bsr_tiny": dict(kind="bsr", seed=1000, M=64, N=64, R=16, C=16, num_qo_heads=4,
                     num_kv_heads=2, head_dim=64, dtype=torch.float16, pattern="random",
                     density=0.5, causal=False),
    "paged_decode": dict(kind="decode", seed=1001, batch=64, num_qo_heads=32, num_kv_heads=8,
                         head_dim=128, page_size=16, len_lo=512, len_hi=4096,
                         dtype=torch.bfloat16),
    "bsr_prefill": dict(kind="bsr", seed=1002, M=16384, N=16384, R=64, C=64, num_qo_heads=32,
                        num_kv_heads=8, head_dim=128, dtype=torch.float16,
                        pattern="diag_lower", p_off=0.1, causal=True),
    "mla_decode": dict(kind="mla", seed=1003, batch=128, heads=128, top_k=2048,
                       pool_rows=65536, ctx_lo=8192, ctx_hi=32768, max_seq_len=65536),
    "split_decode": dict(kind="decode", seed=1004, batch=8, num_qo_heads=64, num_kv_heads=8,
                         head_dim=128, page_size=64, len_lo=131072, len_hi=131072,
                         dtype=torch.bfloat16),
    "mla_paged": dict(kind="mla_paged", seed=1005, batch=128, heads=128, page_size=64,
                      len_lo=2048, len_hi=8192),
    "bsr_variable": dict(kind="bsr_variable", seed=1007, num_qo_heads=32, num_kv_heads=8,
                         head_dim=128, MB=128, NB=128, qo_len=16384, kv_len=16384,
                         density=0.1, dtype=torch.float16, causal=True),
    "prefill_paged": dict(kind="prefill_paged", seed=1008, batch=16, num_qo_heads=32,
                          num_kv_heads=8, head_dim=128, page_size=16, len_lo=2048,
                          len_hi=8192, qo_lo=1024, qo_hi=1024, dtype=torch.bfloat16),
    "mla_append": dict(kind="mla_append", seed=1006, batch=128, page_size=64, len_lo=2048,
                       len_hi=8192, new_tokens=512),
}


def make(name, device="cpu", **overrides):
    """Build a named workload (optionally with some sizes overridden)."""
    cfg = dict(CONFIGS[name])
    cfg.update(overrides)
    kind = cfg.pop("kind")
    if kind == "bsr":
        return bsr_inputs(device=device, **cfg)
    if kind == "decode":
        return paged_decode_inputs(device=device, **cfg)
    if kind == "mla":
        return mla_inputs(device=device, **cfg)
    if kind == "mla_paged":
        return mla_paged_inputs(device=device, **cfg)
    if kind == "bsr_variable":
        return variable_block_inputs(device=device, **cfg)
    if kind == "prefill_paged":
        return paged_prefill_inputs(device=device, **cfg)
    if kind == "mla_append":
        return mla_append_inputs(device=device, **cfg)
    raise ValueError(kind)
