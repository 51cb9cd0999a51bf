"""Pins of the oracle's attention, index expansions and merge (CPU only).

Pins, none of which re-types the oracle's own formula:
  * the BSR worked example of the FlashInfer sparse page (3x3 mask, R = C = 1): the BSR
    expansion reproduces the printed boolean mask, and BSR attention equals dense
    attention under that mask (library routine: torch SDPA with attn_mask, float64);
  * all blocks present equals unmasked SDPA; causal equals SDPA is_causal; GQA equals
    SDPA on kv heads repeated with repeat_interleave (head h uses kv head h // g);
  * brute force: pure-Python triple loop on tiny inputs;
  * special cases: one visible key gives out = v and lse = logit; identical keys give
    the mean of v; a row that sees nothing gives 0 and -inf;
  * paged decode is invariant to page size and page permutation, and one page holding
    the whole sequence equals dense attention;
  * merging states of any split equals the unsplit result; merging one state is the
    identity;
  * sparse MLA over indices covering a whole small context equals dense attention on
    the decoded rows; permuting the indices changes nothing; the scale folding rule of
    the MATE wrapper page holds;
  * dense paged MLA with page_size 1 equals sparse MLA over the page list; it is
    invariant to page size and to where the pages sit in the pool; canary slots (NaN
    codes) past a request's end and in spare pages are never read; a request without
    pages gives 0 and -inf.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synth
from oracle import attention as att
from oracle import numerics as nx
from oracle import rope

HERE = os.path.dirname(os.path.abspath(__file__))


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _sdpa(q, k, v, scale, mask=None, causal=False):
    """Library reference: torch SDPA in float64 with kv heads repeated (h -> h // g)."""
    Hq, Hkv = q.shape[1], k.shape[1]
    g = Hq // Hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k).repeat_interleave(g, dim=1).permute(1, 0, 2)
    vt = torch.from_numpy(v).repeat_interleave(g, dim=1).permute(1, 0, 2)
    m = None if mask is None else torch.from_numpy(mask)
    o = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, is_causal=causal, scale=scale)
    return o.permute(1, 0, 2).numpy()


def test_worked_example_mask_and_result():
    ex = json.load(open(os.path.join(HERE, "golden", "bsr_worked_example.json")))
    mask = att.bsr_mask(ex["indptr"], ex["indices"], ex["M"], ex["N"], ex["R"], ex["C"])
    np.testing.assert_array_equal(mask, np.array(ex["mask"], dtype=bool))
    d = synth.bsr_inputs(7, ex["M"], ex["N"], ex["R"], ex["C"], ex["num_qo_heads"],
                         ex["num_kv_heads"], ex["head_dim"], pattern="full")
    out, lse = att.bsr_attention(_bits(d["q"]), _bits(d["k"]), _bits(d["v"]), "fp16",
                                 ex["indptr"], ex["indices"], ex["M"], ex["N"], ex["R"], ex["C"])
    q = d["q"].double().numpy(); k = d["k"].double().numpy(); v = d["v"].double().numpy()
    ref = _sdpa(q, k, v, 1 / math.sqrt(ex["head_dim"]), mask=np.array(ex["mask"], dtype=bool))
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_all_blocks_equals_dense(causal):
    d = synth.bsr_inputs(11, 48, 48, 16, 8, 4, 2, 32, pattern="full", causal=causal)
    out, lse = att.bsr_attention(_bits(d["q"]), _bits(d["k"]), _bits(d["v"]), "fp16",
                                 d["indptr"].numpy(), d["indices"].numpy(), 48, 48, 16, 8,
                                 causal=causal)
    q = d["q"].double().numpy(); k = d["k"].double().numpy(); v = d["v"].double().numpy()
    ref = _sdpa(q, k, v, d["sm_scale"], causal=causal)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    # lse against a direct logsumexp (library routine)
    g = 2
    logits = np.einsum("mhd,nhd->mhn", q, np.repeat(k, g, axis=1)) * d["sm_scale"]
    if causal:
        logits = np.where(np.tril(np.ones((48, 48), bool))[:, None, :], logits, -np.inf)
    np.testing.assert_allclose(lse, torch.logsumexp(torch.from_numpy(logits), -1).numpy(),
                               rtol=1e-12)


def test_bottom_right_causal_when_m_less_than_n():
    d = synth.bsr_inputs(12, 8, 24, 4, 8, 2, 1, 16, pattern="full", causal=True)
    mask = att.bsr_mask(d["indptr"].numpy(), d["indices"].numpy(), 8, 24, 4, 8, causal=True)
    # query i (of 8) sees keys j <= i + 16: the last query row sees all 24 keys
    assert mask[-1].all() and mask[0].sum() == 17


def test_brute_force_tiny():
    rng = np.random.default_rng(2)
    M, N, Hq, Hkv, D = 5, 7, 4, 2, 3
    q, k, v = rng.standard_normal((M, Hq, D)), rng.standard_normal((N, Hkv, D)), rng.standard_normal((N, Hkv, D))
    mask = rng.random((M, N)) < 0.6
    mask[:, 0] = True
    out, lse = att.masked_attention(q, k, v, 0.7, mask)
    for i in range(M):
        for h in range(Hq):
            kh = h // (Hq // Hkv)
            logits = [sum(q[i, h, t] * k[j, kh, t] for t in range(D)) * 0.7 if mask[i, j] else None
                      for j in range(N)]
            mx = max(x for x in logits if x is not None)
            w = [math.exp(x - mx) if x is not None else 0.0 for x in logits]
            tot = sum(w)
            for t in range(D):
                ref = sum(w[j] * v[j, kh, t] for j in range(N)) / tot
                assert abs(out[i, h, t] - ref) < 1e-12
            assert abs(lse[i, h] - (mx + math.log(tot))) < 1e-12


def test_special_cases():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((2, 2, 8)); k = rng.standard_normal((5, 1, 8)); v = rng.standard_normal((5, 1, 8))
    mask = np.zeros((2, 5), bool)
    mask[0, 3] = True  # one visible key; row 1 sees nothing
    out, lse = att.masked_attention(q, k, v, 0.3, mask)
    np.testing.assert_allclose(out[0, 0], v[3, 0], rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0], 0.3 * q[0, 0] @ k[3, 0], rtol=1e-14)
    assert (out[1] == 0).all() and np.isneginf(lse[1]).all()
    kk = np.repeat(k[:1], 5, axis=0)
    out, _ = att.masked_attention(q, kk, v, 0.3)
    np.testing.assert_allclose(out[:, 0], np.repeat(v[:, 0].mean(0, keepdims=True), 2, 0), rtol=1e-13)


def _paged(seed, page_size, lengths, Hq=4, Hkv=2, D=16):
    return synth.paged_decode_inputs(seed, len(lengths), Hq, Hkv, D, page_size, 0, 0,
                                     lengths=lengths)


def test_paged_invariance_to_page_size_and_permutation():
    lengths = [1, 17, 40, 64, 5]
    base = _paged(21, 64, lengths)
    B, Hq, D = base["q"].shape
    # Rebuild the same logical K/V with other page sizes and a fresh page permutation.
    ks, vs = [], []
    for b in range(B):
        k, v = att.paged_kv(_bits(base["kv_cache"]), "bf16", base["kv_indptr"].numpy(),
                            base["kv_indices"].numpy(), base["kv_last_page_len"].numpy(), 64, b)
        ks.append(k); vs.append(v)
    ref, ref_lse = att.paged_decode(_bits(base["q"]), _bits(base["kv_cache"]), "bf16",
                                    base["kv_indptr"].numpy(), base["kv_indices"].numpy(),
                                    base["kv_last_page_len"].numpy(), 64)
    for ps, seed in [(1, 1), (16, 2), (7, 3)]:
        other = _paged(100 + seed, ps, lengths)
        cache = other["kv_cache"].clone()
        for b in range(B):
            pages = other["kv_indices"][other["kv_indptr"][b]:other["kv_indptr"][b + 1]]
            kb = torch.from_numpy(ks[b]).to(torch.bfloat16)
            vb = torch.from_numpy(vs[b]).to(torch.bfloat16)
            for n, p in enumerate(pages.tolist()):
                seg = slice(n * ps, min((n + 1) * ps, lengths[b]))
                cnt = seg.stop - seg.start
                cache[p, 0, :, :cnt] = kb[seg].transpose(0, 1)
                cache[p, 1, :, :cnt] = vb[seg].transpose(0, 1)
        out, lse = att.paged_decode(_bits(base["q"]), _bits(cache), "bf16",
                                    other["kv_indptr"].numpy(), other["kv_indices"].numpy(),
                                    other["kv_last_page_len"].numpy(), ps)
        np.testing.assert_array_equal(out, ref)
        np.testing.assert_array_equal(lse, ref_lse)


def test_single_page_equals_dense():
    d = _paged(31, 64, [64, 64])
    out, lse = att.paged_decode(_bits(d["q"]), _bits(d["kv_cache"]), "bf16", d["kv_indptr"].numpy(),
                                d["kv_indices"].numpy(), d["kv_last_page_len"].numpy(), 64)
    for b in range(2):
        page = int(d["kv_indices"][b])
        k = d["kv_cache"][page, 0].transpose(0, 1).double().numpy()
        v = d["kv_cache"][page, 1].transpose(0, 1).double().numpy()
        q = d["q"][b:b + 1].double().numpy()
        np.testing.assert_allclose(out[b], _sdpa(q, k, v, d["sm_scale"])[0], rtol=1e-12, atol=1e-14)


def test_merge_of_any_split_equals_unsplit():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((3, 4, 8)); k = rng.standard_normal((50, 4, 8)); v = rng.standard_normal((50, 4, 8))
    full, full_lse = att.masked_attention(q, k, v, 0.4)
    cuts = [0, 7, 8, 30, 50]
    parts = [att.masked_attention(q, k[a:b], v[a:b], 0.4) for a, b in zip(cuts[:-1], cuts[1:])]
    vv = np.stack([p[0] for p in parts], axis=1)  # [M, S, H, D]
    ss = np.stack([p[1] for p in parts], axis=1)
    out, lse = att.merge_states(vv, ss, axis=1)
    np.testing.assert_allclose(out, full, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, full_lse, rtol=1e-13)
    one, one_lse = att.merge_states(vv[:, :1], ss[:, :1], axis=1)
    np.testing.assert_allclose(one, vv[:, 0], rtol=1e-15)
    np.testing.assert_array_equal(one_lse, ss[:, 0])
    empty = att.merge_states(np.zeros((1, 2, 1, 4)), np.full((1, 2, 1), -np.inf), axis=1)
    assert (empty[0] == 0).all() and np.isneginf(empty[1]).all()


def _mla_small(seed=41, H=8, pool=256, top_k=128):
    d = synth.mla_inputs(seed, batch=2, heads=H, top_k=top_k, pool_rows=pool, ctx_lo=top_k,
                         ctx_hi=top_k, max_seq_len=pool)
    qr, kr, qn, kn = rope.mla_rope_quantize_fp8(
        _bits(d["q_rope"]), _bits(d["k_rope"]), _bits(d["q_nope"]), _bits(d["k_nope"]),
        d["cos_sin"].numpy(), d["pos_q"].numpy(), d["pos_k"].numpy(), True)
    query = np.concatenate([qn, qr], axis=-1).reshape(2, 1, H, 576)
    kv = np.concatenate([kn, kr], axis=-1)
    return d, query, kv


def test_mla_full_context_equals_dense_and_is_permutation_invariant():
    d, query, kv = _mla_small()
    idx = d["indices"].numpy()
    scale = 1 / math.sqrt(576)
    out, lse = att.mla_sparse_decode(query, kv, idx, d["seq_lens"].numpy(), scale, 1.0)
    for b in range(2):
        rows = np.sort(idx[b, 0])  # the whole context (top_k == context length)
        assert len(np.unique(rows)) == len(rows) == 128
        K = nx.e4m3_decode(kv[rows])
        Q = nx.e4m3_decode(query[b, 0])
        ref = _sdpa(Q[None], K[:, None, :], K[:, None, :512], scale)[0]
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-14)
    perm = idx[:, :, ::-1].copy()
    out2, lse2 = att.mla_sparse_decode(query, kv, perm, d["seq_lens"].numpy(), scale, 1.0)
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13)


def test_mla_duplicate_indices_count_as_list_entries():
    """Index lists are lists, not sets (the reading for duplicates): listing every row twice
    doubles every softmax weight, so the output is unchanged and the LSE grows by ln 2."""
    d, query, kv = _mla_small(seed=44)
    idx, sl = d["indices"].numpy(), d["seq_lens"].numpy()
    scale = 1 / math.sqrt(576)
    out, lse = att.mla_sparse_decode(query, kv, idx, sl, scale, 1.0)
    twice = np.concatenate([idx, idx], axis=-1)
    out2, lse2 = att.mla_sparse_decode(query, kv, twice, 2 * sl, scale, 1.0)
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(lse2, lse + math.log(2.0), rtol=1e-13)


def test_mla_scale_folding():
    """Quantising with scales (sq, skv) and decoding with bmm1 = a/(sq*skv), bmm2 = 1/skv
    equals decoding unit-scale rows with bmm1 = a when the scaled values stay exact."""
    d, query, kv = _mla_small(seed=43)
    idx, sl = d["indices"].numpy(), d["seq_lens"].numpy()
    a = 1 / math.sqrt(576)
    sq, skv = 2.0, 0.5
    qv, kvv = nx.e4m3_decode(query), nx.e4m3_decode(kv)
    ok_q = np.abs(qv) >= 2.0 ** -5
    ok_k = np.abs(kvv) >= 2.0 ** -5
    q1 = nx.e4m3_encode(np.where(ok_q, qv, 0.0)); k1 = nx.e4m3_encode(np.where(ok_k, kvv, 0.0))
    q2 = nx.e4m3_encode(nx.e4m3_decode(q1) * sq); k2 = nx.e4m3_encode(nx.e4m3_decode(k1) * skv)
    o1, l1 = att.mla_sparse_decode(q1, k1, idx, sl, a, 1.0)
    o2, l2 = att.mla_sparse_decode(q2, k2, idx, sl, a / (sq * skv), 1.0 / skv)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l2, l1, rtol=1e-12)


def test_mla_seq_lens_limit_the_rows():
    d, query, kv = _mla_small(seed=44)
    idx = d["indices"].numpy()
    sl = np.array([64, 0], np.int32)
    out, lse = att.mla_sparse_decode(query, kv, idx, sl, 0.05, 1.0)
    ref, ref_lse = att.mla_sparse_decode(query, kv, idx[:, :, :64], np.array([64, 0]), 0.05, 1.0)
    np.testing.assert_array_equal(out, ref)
    assert (out[1] == 0).all() and np.isneginf(lse[1]).all()


# ---------------------------------------------------------------------------------------
# dense paged MLA
# ---------------------------------------------------------------------------------------

def _relayout(d, page_size, seed):
    """The same logical rows of every request in a new cache with another page size and
    the pages at other (random) pool positions; canaries elsewhere."""
    g = torch.Generator().manual_seed(seed)
    lens = d["lens"].tolist()
    old = d["kv_pages"].numpy()
    logical = []
    for b, L in enumerate(lens):
        pg = d["kv_indices"][int(d["kv_indptr"][b]):int(d["kv_indptr"][b + 1])].numpy()
        logical.append(old[pg].reshape(-1, 576)[:L])
    npg = [(L + page_size - 1) // page_size for L in lens]
    P = sum(npg) + 3
    perm = torch.randperm(P, generator=g).numpy()
    cache = np.full((P, page_size, 576), synth.E4M3_NAN, np.uint8)
    indptr = np.concatenate([[0], np.cumsum(npg)]).astype(np.int32)
    indices = perm[:sum(npg)].astype(np.int32)
    last = np.zeros(len(lens), np.int32)
    for b, L in enumerate(lens):
        for t in range(L):
            cache[indices[indptr[b] + t // page_size], t % page_size] = logical[b][t]
        if npg[b]:
            last[b] = L - (npg[b] - 1) * page_size
    return cache, indptr, indices, last


def test_mla_paged_page_size_one_equals_sparse():
    d = synth.mla_paged_inputs(51, batch=3, heads=8, page_size=1, len_lo=0, len_hi=0,
                               lens=[37, 1, 90])
    q, cache = d["query"].numpy(), d["kv_pages"].numpy()
    ip, ix, lp = d["kv_indptr"].numpy(), d["kv_indices"].numpy(), d["kv_last_page_len"].numpy()
    out, lse = att.mla_paged_decode(q, cache, ip, ix, lp, 1, 0.05, 1.5)
    top = 128
    idx = np.zeros((3, 1, top), np.int32)
    for b in range(3):
        n = ip[b + 1] - ip[b]
        idx[b, 0, :n] = ix[ip[b]:ip[b + 1]]
    ref, ref_lse = att.mla_sparse_decode(q[:, None], cache.reshape(-1, 576), idx,
                                         d["lens"].numpy(), 0.05, 1.5)
    np.testing.assert_array_equal(out, ref)
    np.testing.assert_array_equal(lse, ref_lse)


@pytest.mark.parametrize("ps_from,ps_to", [(16, 64), (64, 1), (7, 16)])
def test_mla_paged_invariant_to_page_size_and_placement(ps_from, ps_to):
    d = synth.mla_paged_inputs(52, batch=4, heads=8, page_size=ps_from, len_lo=0, len_hi=0,
                               lens=[200, 64, 1, 129])
    q = d["query"].numpy()
    out, lse = att.mla_paged_decode(q, d["kv_pages"].numpy(), d["kv_indptr"].numpy(),
                                    d["kv_indices"].numpy(), d["kv_last_page_len"].numpy(),
                                    ps_from, 1 / math.sqrt(576), 1.0)
    assert np.isfinite(out).all() and np.isfinite(lse).all()  # no canary slot was read
    cache, ip, ix, lp = _relayout(d, ps_to, seed=5)
    out2, lse2 = att.mla_paged_decode(q, cache, ip, ix, lp, ps_to, 1 / math.sqrt(576), 1.0)
    np.testing.assert_array_equal(out2, out)
    np.testing.assert_array_equal(lse2, lse)


def test_mla_paged_full_request_equals_dense_and_empty_request():
    d = synth.mla_paged_inputs(53, batch=2, heads=4, page_size=16, len_lo=0, len_hi=0,
                               lens=[40, 0])
    q, cache = d["query"].numpy(), d["kv_pages"].numpy()
    out, lse = att.mla_paged_decode(q, cache, d["kv_indptr"].numpy(), d["kv_indices"].numpy(),
                                    d["kv_last_page_len"].numpy(), 16, 0.07, 1.0)
    pages = d["kv_indices"].numpy()[:3]
    K = nx.e4m3_decode(cache[pages].reshape(-1, 576)[:40])
    Q = nx.e4m3_decode(q[0])
    ref = _sdpa(Q[None], K[:, None, :], K[:, None, :512], 0.07)[0]
    np.testing.assert_allclose(out[0], ref, rtol=1e-12, atol=1e-14)
    assert (out[1] == 0).all() and np.isneginf(lse[1]).all()


# ---------------------------------------------------------------------------------------
# BSR with a per-block token mask
# ---------------------------------------------------------------------------------------

def _bsr_small(seed, M, N, R, C, Hq=4, Hkv=2, D=16, density=0.6):
    d = synth.bsr_inputs(seed, M, N, R, C, Hq, Hkv, D, pattern="random", density=density)
    return d, _bits(d["q"]), _bits(d["k"]), _bits(d["v"])


def test_bsr_all_true_token_mask_equals_unmasked():
    d, q, k, v = _bsr_small(61, 20, 24, 4, 8)
    nnz = int(d["indptr"][-1])
    full = np.ones((nnz, 4, 8), bool)
    a = att.bsr_attention(q, k, v, "fp16", d["indptr"], d["indices"], 20, 24, 4, 8)
    b = att.bsr_attention(q, k, v, "fp16", d["indptr"], d["indices"], 20, 24, 4, 8, block_mask=full)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_bsr_token_mask_of_the_causal_pattern_equals_causal():
    """All blocks listed; each block's mask is the causal pattern restricted to it."""
    M = N = 16
    R = C = 4
    MB = NB = 4
    indptr = np.arange(0, MB * NB + 1, NB)
    indices = np.tile(np.arange(NB), MB)
    bm = np.zeros((MB * NB, R, C), bool)
    for a in range(MB):
        for c in range(NB):
            for r in range(R):
                for cc in range(C):
                    bm[a * NB + c, r, cc] = c * C + cc <= a * R + r
    d, q, k, v = _bsr_small(62, M, N, R, C)
    ref = att.bsr_attention(q, k, v, "fp16", indptr, indices, M, N, R, C, causal=True)
    got = att.bsr_attention(q, k, v, "fp16", indptr, indices, M, N, R, C, block_mask=bm,
                            causal=True)
    np.testing.assert_array_equal(got[0], ref[0])
    np.testing.assert_array_equal(got[1], ref[1])


def test_bsr_token_mask_brute_force_and_empty_rows():
    """Pure-Python loops over the pairs the mask keeps; a row whose pairs are all masked
    gives 0 and -inf."""
    M, N, R, C = 6, 8, 3, 4
    d, qb, kb, vb = _bsr_small(63, M, N, R, C, Hq=2, Hkv=1, D=4, density=1.0)
    nnz = int(d["indptr"][-1])
    bm = np.asarray(torch.rand((nnz, R, C), generator=torch.Generator().manual_seed(5)) < 0.5)
    bm[:, 1, :] = False  # rows 1 and 4 see nothing
    out, lse = att.bsr_attention(qb, kb, vb, "fp16", d["indptr"], d["indices"], M, N, R, C,
                                 sm_scale=0.5, block_mask=bm)
    q = nx.bits_to_f64(qb, "fp16"); k = nx.bits_to_f64(kb, "fp16"); v = nx.bits_to_f64(vb, "fp16")
    ip, ix = d["indptr"], d["indices"]
    for i in range(M):
        for h in range(2):
            keys = []
            for e in range(int(ip[i // R]), int(ip[i // R + 1])):
                for cc in range(C):
                    if bm[e, i % R, cc]:
                        keys.append(int(ix[e]) * C + cc)
            if not keys:
                assert (out[i, h] == 0).all() and math.isinf(lse[i, h]) and lse[i, h] < 0
                continue
            logits = [0.5 * sum(q[i, h, t] * k[j, 0, t] for t in range(4)) for j in keys]
            mx = max(logits)
            w = [math.exp(x - mx) for x in logits]
            den = sum(w)
            for t in range(4):
                ref = sum(wi * v[j, 0, t] for wi, j in zip(w, keys)) / den
                assert abs(out[i, h, t] - ref) <= 1e-12
            assert abs(lse[i, h] - (mx + math.log(den))) <= 1e-12


def test_packed_mask_bit_order_reading():
    """The reading of packed_mask: entry t of the flattened (nnz, R, C) mask is bit t % 8 of
    byte t // 8, which is numpy.packbits with bitorder='little'."""
    g = np.random.default_rng(7)
    m = g.random(77) < 0.5
    packed = np.packbits(m, bitorder="little")
    for t in range(77):
        assert bool((packed[t // 8] >> (t % 8)) & 1) == m[t]


# ---------------------------------------------------------------------------------------
# variable-block sparse attention
# ---------------------------------------------------------------------------------------

def test_variable_block_page_example_mask_and_result():
    ex = json.load(open(os.path.join(HERE, "golden", "variable_block_example.json")))
    m = att.variable_block_mask(ex["block_mask_map"], ex["block_row_sz"], ex["block_col_sz"])
    np.testing.assert_array_equal(m[0], np.array(ex["dense_mask"], bool))
    g = torch.Generator().manual_seed(9)
    L, D = ex["seq_len"], 16
    q = torch.randn((1, L, D), generator=g).to(torch.float16)
    k = torch.randn((1, L, D), generator=g).to(torch.float16)
    v = torch.randn((1, L, D), generator=g).to(torch.float16)
    out, lse = att.variable_block_attention(_bits(q), _bits(k), _bits(v), "fp16",
                                            ex["block_mask_map"], ex["block_row_sz"],
                                            ex["block_col_sz"])
    qd = nx.bits_to_f64(_bits(q), "fp16")[0][:, None, :]
    kd = nx.bits_to_f64(_bits(k), "fp16")[0][:, None, :]
    vd = nx.bits_to_f64(_bits(v), "fp16")[0][:, None, :]
    ref = _sdpa(qd, kd, vd, 1 / math.sqrt(D), mask=np.array(ex["dense_mask"], bool))
    np.testing.assert_allclose(out[0], ref[:, 0, :], rtol=1e-12, atol=1e-14)


def test_variable_blocks_of_equal_size_are_bsr():
    """Uniform sizes R x C with the same map for every kv head give BSR attention."""
    M, N, R, C, Hq, Hkv, D = 24, 32, 4, 8, 4, 2, 16
    d = synth.bsr_inputs(71, M, N, R, C, Hq, Hkv, D, pattern="random", density=0.5)
    MB, NB = M // R, N // C
    bm = np.zeros((MB, NB), bool)
    ip, ix = d["indptr"].numpy(), d["indices"].numpy()
    for a in range(MB):
        bm[a, ix[ip[a]:ip[a + 1]]] = True
    qh = d["q"].permute(1, 0, 2).contiguous()
    kh = d["k"].permute(1, 0, 2).contiguous()
    vh = d["v"].permute(1, 0, 2).contiguous()
    for causal in (False, True):
        out, lse = att.variable_block_attention(
            _bits(qh), _bits(kh), _bits(vh), "fp16", np.stack([bm] * Hkv), [[R] * MB] * Hkv,
            [[C] * NB] * Hkv, causal=causal)
        ref, ref_lse = att.bsr_attention(_bits(d["q"]), _bits(d["k"]), _bits(d["v"]), "fp16", ip,
                                         ix, M, N, R, C, causal=causal)
        np.testing.assert_allclose(out.transpose(1, 0, 2), ref, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse.T, ref_lse, rtol=1e-12)


def test_variable_block_heads_follow_their_kv_head():
    """Query heads 0-1 use kv head 0's map and sizes, heads 2-3 kv head 1's: each pair equals
    a one-kv-head computation with that head's pattern alone."""
    g = torch.Generator().manual_seed(11)
    L, Lk, D = 10, 12, 8
    q = torch.randn((4, L, D), generator=g).to(torch.float16)
    k = torch.randn((2, Lk, D), generator=g).to(torch.float16)
    v = torch.randn((2, Lk, D), generator=g).to(torch.float16)
    bmap = [[[1, 0, 1], [0, 1, 0]], [[0, 1, 1], [1, 1, 0]]]
    rsz = [[4, 6], [7, 3]]
    csz = [[5, 4, 3], [2, 2, 8]]
    out, lse = att.variable_block_attention(_bits(q), _bits(k), _bits(v), "fp16", bmap, rsz, csz)
    for h in range(2):
        o1, l1 = att.variable_block_attention(_bits(q[2 * h:2 * h + 2]), _bits(k[h:h + 1]),
                                              _bits(v[h:h + 1]), "fp16", [bmap[h]], [rsz[h]],
                                              [csz[h]])
        np.testing.assert_array_equal(out[2 * h:2 * h + 2], o1)
        np.testing.assert_array_equal(lse[2 * h:2 * h + 2], l1)
    m = att.variable_block_mask(bmap, rsz, csz)
    assert m[1, 0, :].tolist() == [False] * 2 + [True] * 10   # row block 0 of head 1: cols 1, 2


@pytest.mark.parametrize("causal", [False, True])
def test_variable_block_selected_rows_are_the_full_rows(causal):
    """The rows= selection computes exactly the selected rows of the full result (mask and
    attention), bit for bit, in the order given."""
    d = synth.variable_block_inputs(30, 4, 2, 16, 3, 4, 40, 50, density=0.6, causal=causal)
    args = (_bits(d["q"]), _bits(d["k"]), _bits(d["v"]), "fp16", d["block_mask_map"].numpy(),
            d["block_row_sz"].numpy(), d["block_col_sz"].numpy())
    out, lse = att.variable_block_attention(*args, causal=causal)
    rows = [39, 0, 17, 18, 5]
    o2, l2 = att.variable_block_attention(*args, causal=causal, rows=rows)
    np.testing.assert_array_equal(o2, out[:, rows])
    np.testing.assert_array_equal(l2, lse[:, rows])
    m = att.variable_block_mask(*args[4:], causal=causal)
    np.testing.assert_array_equal(att.variable_block_mask(*args[4:], causal=causal, rows=rows),
                                  m[:, rows])


# ---------------------------------------------------------------------------------------
# batch prefill over a paged KV cache
# ---------------------------------------------------------------------------------------

def test_paged_prefill_one_query_is_decode():
    """qo_len 1 with causal: the last token sees its whole request, i.e. paged decode."""
    d = synth.paged_prefill_inputs(81, 4, 8, 2, 16, 16, 1, 90, 1, 1, lengths=[1, 17, 40, 90])
    ip, ix, lp = d["kv_indptr"].numpy(), d["kv_indices"].numpy(), d["kv_last_page_len"].numpy()
    out, lse = att.paged_prefill(_bits(d["q"]), _bits(d["kv_cache"]), "bf16",
                                 d["qo_indptr"].numpy(), ip, ix, lp, 16)
    ref, ref_lse = att.paged_decode(_bits(d["q"]), _bits(d["kv_cache"]), "bf16", ip, ix, lp, 16)
    np.testing.assert_array_equal(out, ref)
    np.testing.assert_array_equal(lse, ref_lse)


def test_paged_prefill_whole_sequence_is_sdpa_causal():
    """One request whose queries are its whole sequence: standard causal attention."""
    d = synth.paged_prefill_inputs(82, 1, 4, 2, 16, 8, 0, 0, 0, 0, lengths=[37], qo_lens=[37])
    k, v = att.paged_kv(_bits(d["kv_cache"]), "bf16", d["kv_indptr"].numpy(),
                        d["kv_indices"].numpy(), d["kv_last_page_len"].numpy(), 8, 0)
    out, _ = att.paged_prefill(_bits(d["q"]), _bits(d["kv_cache"]), "bf16",
                               d["qo_indptr"].numpy(), d["kv_indptr"].numpy(),
                               d["kv_indices"].numpy(), d["kv_last_page_len"].numpy(), 8)
    q = nx.bits_to_f64(_bits(d["q"]), "bf16")
    ref = _sdpa(q, k, v, 1 / math.sqrt(16), causal=True)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)


def test_paged_prefill_bottom_right_and_page_size_invariance():
    """The first of qo_len queries sees L - qo_len + 1 keys; relayout with another page size
    changes nothing."""
    lengths, qo = [30, 64], [5, 64]
    d = synth.paged_prefill_inputs(83, 2, 4, 4, 16, 16, 0, 0, 0, 0, lengths=lengths, qo_lens=qo)
    args = (d["qo_indptr"].numpy(), d["kv_indptr"].numpy(), d["kv_indices"].numpy(),
            d["kv_last_page_len"].numpy(), 16)
    out, lse = att.paged_prefill(_bits(d["q"]), _bits(d["kv_cache"]), "bf16", *args)
    k, v = att.paged_kv(_bits(d["kv_cache"]), "bf16", *args[1:], 0)
    q0 = nx.bits_to_f64(_bits(d["q"][:1]), "bf16")
    one, _ = att.masked_attention(q0, k[:26], v[:26], 1 / math.sqrt(16))
    np.testing.assert_allclose(out[0], one[0], rtol=1e-12, atol=1e-14)
    other = synth.paged_prefill_inputs(84, 2, 4, 4, 16, 7, 0, 0, 0, 0, lengths=lengths, qo_lens=qo)
    cache = other["kv_cache"].clone()
    for b in range(2):
        kb, vb = att.paged_kv(_bits(d["kv_cache"]), "bf16", *args[1:], b)
        pages = other["kv_indices"][other["kv_indptr"][b]:other["kv_indptr"][b + 1]]
        for n, p in enumerate(pages.tolist()):
            seg = slice(n * 7, min((n + 1) * 7, lengths[b]))
            cnt = seg.stop - seg.start
            cache[p, 0, :, :cnt] = torch.from_numpy(kb[seg]).to(torch.bfloat16).transpose(0, 1)
            cache[p, 1, :, :cnt] = torch.from_numpy(vb[seg]).to(torch.bfloat16).transpose(0, 1)
    out2, lse2 = att.paged_prefill(_bits(d["q"]), _bits(cache), "bf16", d["qo_indptr"].numpy(),
                                   other["kv_indptr"].numpy(), other["kv_indices"].numpy(),
                                   other["kv_last_page_len"].numpy(), 7)
    np.testing.assert_array_equal(out2, out)
    np.testing.assert_array_equal(lse2, lse)
