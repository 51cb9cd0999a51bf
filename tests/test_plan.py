"""Plans: bit-exact metadata against the oracle's restatement, invariants, and host-side
fault injection (every malformed input is rejected before anything is launched)."""

import os
import re
import subprocess
import sys

import numpy as np
import pytest
import torch

import block_sparse_kv_gb300 as bskv
import synth
from oracle import attention as att
from oracle import plan_ref

SMS = 152


def _decode_plan(d, num_sms=SMS, max_workers=0):
    return bskv.bskv_plan_decode(d["kv_indptr"], d["kv_indices"], d["kv_last_page_len"],
                                 d["num_pages"], d["page_size"], d["num_qo_heads"],
                                 d["num_kv_heads"], d["head_dim"], torch.bfloat16,
                                 num_sms=num_sms, max_workers=max_workers)


def _check_linear(meta, unit_len, tile):
    s = plan_ref.sections(meta)
    seen = {u: [] for u in range(len(unit_len))}
    for c in s["chunks"]:
        seen[c[0]].append((c[1], c[2], c[3]))
    for u, L in enumerate(unit_len):
        segs = sorted(seen[u])
        pos = 0
        for a, b, slot in segs:
            assert a == pos and b > a and a % tile == 0
            pos = b
        assert pos == L  # every token of every unit exactly once
        if len(segs) == 1:
            assert segs[0][2] == -1
        else:
            assert all(sl >= 0 for _, _, sl in segs)
    # balance: tiles per worker differ by at most one
    per = []
    for w in range(s["workers"]):
        cs = s["chunks"][s["worker_ptr"][w]:s["worker_ptr"][w + 1]]
        per.append(sum((c[2] - c[1] + tile - 1) // tile for c in cs))
    if per:
        assert max(per) - min(per) <= 1 + len(unit_len)  # a worker can be cut at unit ends
        assert sum(per) == sum((L + tile - 1) // tile for L in unit_len)
    assert s["slots"] == sum(1 for c in s["chunks"] if c[3] >= 0)


@pytest.mark.parametrize("name,over", [
    ("paged_decode", dict(tensors=False)),
    ("paged_decode", dict(batch=5, len_lo=1, len_hi=100)),
    ("paged_decode", dict(batch=3, page_size=64, len_lo=64, len_hi=64)),
    ("split_decode", dict(len_lo=4096, len_hi=4096, batch=2)),
])
def test_decode_plan_bit_exact(lib, name, over):
    d = synth.make(name, **over)
    p = _decode_plan(d)
    meta = p.metadata()
    ref = plan_ref.decode_meta(d["kv_indptr"].tolist(), d["kv_indices"].tolist(),
                               d["kv_last_page_len"].tolist(), d["batch"], d["page_size"],
                               d["num_qo_heads"], d["num_kv_heads"], SMS)
    assert meta == ref
    lens = plan_ref.decode_units(d["kv_indptr"].tolist(), d["kv_last_page_len"].tolist(),
                                 d["batch"], d["page_size"], d["num_kv_heads"])
    _check_linear(meta, lens, 16)
    # pages of at most 16 tokens take the page-major variant: one unit per request here
    group = d["page_size"] <= 16
    assert plan_ref.sections(meta)["variant"] == (1 if group else 0)
    assert len(lens) == d["batch"] * (1 if group else d["num_kv_heads"])


def test_decode_plan_full_long_context(lib):
    d = synth.make("split_decode", tensors=False)
    p = _decode_plan(d)
    meta = p.metadata()
    assert meta == plan_ref.decode_meta(d["kv_indptr"].tolist(), d["kv_indices"].tolist(),
                                        d["kv_last_page_len"].tolist(), 8, 64, 64, 8, SMS)
    _check_linear(meta, [131072] * 64, 16)
    s = plan_ref.sections(meta)
    assert s["workers"] == SMS * 8 and s["grid"] == SMS


def test_decode_plan_zero_length_and_max_workers(lib):
    indptr = [0, 0, 3, 3, 4]
    idx = [5, 1, 2, 0]
    last = [0, 7, 0, 16]
    p = bskv.bskv_plan_decode(indptr, idx, last, 6, 16, 4, 2, 64, torch.bfloat16, num_sms=1,
                              max_workers=3)
    meta = p.metadata()
    assert meta == plan_ref.decode_meta(indptr, idx, last, 4, 16, 4, 2, 1, 3)
    s = plan_ref.sections(meta)
    zero_units = {m[0] for m in s["merges"] if m[2] == 0}
    assert s["variant"] == 1 and zero_units == {0, 2}  # requests 0 and 2 (both kv heads)
    # the same requests with 32-token pages take the per-kv-head variant
    p = bskv.bskv_plan_decode(indptr, idx, [0, 7, 0, 32], 6, 32, 4, 2, 64, torch.bfloat16,
                              num_sms=1, max_workers=3)
    meta = p.metadata()
    assert meta == plan_ref.decode_meta(indptr, idx, [0, 7, 0, 32], 4, 32, 4, 2, 1, 3)
    s = plan_ref.sections(meta)
    zero_units = {m[0] for m in s["merges"] if m[2] == 0}
    assert s["variant"] == 0 and zero_units == {0, 1, 4, 5}  # requests 0 and 2, both kv heads


@pytest.mark.parametrize("name,over", [
    ("bsr_tiny", {}),
    ("bsr_prefill", {}),
    ("bsr_prefill", dict(M=2048, N=2048, num_qo_heads=8)),
    ("bsr_prefill", dict(M=1000, N=1024, R=32, C=16, pattern="random")),
])
def test_bsr_plan_bit_exact(lib, name, over):
    d = synth.make(name, tensors=False, **over)
    args = (d["indptr"], d["indices"], d["M"], d["N"], d["R"], d["C"], d["num_qo_heads"],
            d["num_kv_heads"], d["head_dim"])
    p = bskv.bskv_plan_bsr(*args, causal=d["causal"], dtype=torch.float16, num_sms=SMS)
    meta = p.metadata()
    assert meta == plan_ref.bsr_meta(d["indptr"].tolist(), d["indices"].tolist(), *args[2:], SMS)
    s = plan_ref.sections(meta)
    units = sorted(c[0] for c in s["chunks"])
    assert units == list(range(s["units"]))  # each unit exactly once
    # LPT bound: no CTA exceeds the mean load by more than the largest unit
    MB = (d["M"] + d["R"] - 1) // d["R"]
    rows = np.diff(d["indptr"].numpy())
    per_unit = s["units"] // (MB * d["num_kv_heads"])
    loads = []
    for c in range(s["grid"]):
        us = s["chunks"][s["worker_ptr"][c]:s["worker_ptr"][c + 1]]
        loads.append(sum(1 + rows[u[1]] for u in us))
    assert max(loads) <= sum(loads) / len(loads) + 1 + rows.max()
    g = d["num_qo_heads"] // d["num_kv_heads"]
    if d["R"] == 64 and d["C"] == 64 and d["head_dim"] == 128 and 64 * g in (128, 256):
        assert s["variant"] == 1 and per_unit == 1
    else:
        assert s["variant"] == 0


@pytest.mark.parametrize("batch,q_len,seq", [(128, 1, None), (3, 2, [64, 0, 130]), (1, 1, [2048])])
def test_mla_plan_bit_exact(lib, batch, q_len, seq):
    top_k = 2048 if seq is None else 192 if batch == 3 else 2048
    seq_lens = [top_k] * batch if seq is None else seq
    p = bskv.bskv_plan_mla_sparse(seq_lens, batch, q_len, 128, top_k, num_sms=SMS)
    meta = p.metadata()
    assert meta == plan_ref.mla_meta(seq_lens, batch, q_len, SMS)
    lens = [s for s in seq_lens for _ in range(q_len)]
    _check_linear(meta, lens, 128)
    assert plan_ref.sections(meta)["grid"] == 2 * plan_ref.sections(meta)["workers"]


def test_mla_plan_splits_only_when_it_pays(lib):
    """128 queries of 16 tiles on 76 cluster workers: whole queries (busiest worker 32 tiles,
    split partition 27: within the 7-tile penalty), so no partial states and no merge; three
    queries of 16 tiles: the split partition (1 tile per worker against 16 whole)."""
    p = bskv.bskv_plan_mla_sparse([2048] * 128, 128, 1, 128, 2048, num_sms=SMS)
    s = plan_ref.sections(p.metadata())
    assert s["slots"] == 0 and s["merges_n"] == 0 and s["workers"] == 76
    assert all(c[1] == 0 and c[2] == 2048 and c[3] == -1 for c in s["chunks"])
    assert p.workspace_sizes()[1] == 0
    p = bskv.bskv_plan_mla_sparse([2048] * 3, 3, 1, 128, 2048, num_sms=SMS)
    s = plan_ref.sections(p.metadata())
    assert s["slots"] > 0 and s["merges_n"] == 3


@pytest.mark.parametrize("lens,ps", [([5, 0, 130], 16), ([2048] * 7, 64), ([1, 64, 65, 300], 1)])
def test_mla_paged_plan_bit_exact(lib, lens, ps):
    d = synth.mla_paged_inputs(61, batch=len(lens), heads=16, page_size=ps, len_lo=0, len_hi=0,
                               lens=lens)
    ip, ix, lp = d["kv_indptr"], d["kv_indices"], d["kv_last_page_len"]
    p = bskv.bskv_plan_mla_paged(ip, ix, lp, len(lens), d["num_pages"], ps, 128, num_sms=SMS)
    meta = p.metadata()
    assert meta == plan_ref.mla_paged_meta(ip.tolist(), ix.tolist(), lp.tolist(), len(lens), ps, SMS)
    _check_linear(meta, lens, 128)
    # the float workspace holds only split-KV partial states (both latent halves)
    _, fb = p.workspace_sizes()
    slots = plan_ref.sections(meta)["slots"]
    assert (fb == 0) == (slots == 0) and fb >= slots * 2 * 128 * 257 * 4


# ---------------------------------------------------------------------------------------
# fault injection on the host: each malformed input returns an error and plans nothing
# ---------------------------------------------------------------------------------------

def _expect(status, fn, *a, **k):
    with pytest.raises(bskv.BskvError) as e:
        fn(*a, **k)
    assert e.value.status == status, str(e.value)


def test_decode_plan_rejects_bad_inputs(lib):
    f = bskv.bskv_plan_decode
    ok = dict(num_pages=4, page_size=16, num_qo_heads=8, num_kv_heads=2, head_dim=128, num_sms=4)
    f([0, 2], [0, 1], [5], **ok)  # sanity: valid
    _expect("ERR_INVALID_ARG", f, [1, 2], [0, 1], [5], **ok)           # indptr[0] != 0
    _expect("ERR_INVALID_ARG", f, [0, 2, 1], [0, 1], [5, 1], **ok)     # decreasing indptr
    _expect("ERR_INVALID_ARG", f, [0, 2], [0, 4], [5], **ok)           # page id out of range
    _expect("ERR_INVALID_ARG", f, [0, 2], [0, -1], [5], **ok)
    _expect("ERR_INVALID_ARG", f, [0, 2], [0, 1], [0], **ok)           # last page len 0
    _expect("ERR_INVALID_ARG", f, [0, 2], [0, 1], [17], **ok)          # > page_size
    _expect("ERR_INVALID_ARG", f, [0, 2], [0, 1], [5], **{**ok, "num_kv_heads": 3})
    _expect("ERR_UNSUPPORTED", f, [0, 2], [0, 1], [5], **{**ok, "head_dim": 96})
    _expect("ERR_UNSUPPORTED", f, [0, 2], [0, 1], [5], **{**ok, "num_qo_heads": 64, "num_kv_heads": 2})
    _expect("ERR_INVALID_ARG", f, [0, 2], [0, 1], [5], **{**ok, "page_size": 0})


def test_bsr_plan_rejects_bad_inputs(lib):
    f = bskv.bskv_plan_bsr
    f([0, 1, 2], [0, 1], 4, 4, 2, 2, 2, 1, 64, num_sms=2)  # valid
    _expect("ERR_INVALID_ARG", f, [0, 1, 2], [0, 1], 4, 5, 2, 2, 2, 1, 64, num_sms=2)   # N % C
    _expect("ERR_INVALID_ARG", f, [0, 1, 2], [0, 2], 4, 4, 2, 2, 2, 1, 64, num_sms=2)   # index >= NB
    _expect("ERR_INVALID_ARG", f, [0, 2, 2], [1, 1], 4, 4, 2, 2, 2, 1, 64, num_sms=2)   # duplicate
    _expect("ERR_INVALID_ARG", f, [0, 2, 1], [0, 1], 4, 4, 2, 2, 2, 1, 64, num_sms=2)   # decreasing
    _expect("ERR_INVALID_ARG", f, [1, 1, 2], [0, 1], 4, 4, 2, 2, 2, 1, 64, num_sms=2)   # indptr[0]
    _expect("ERR_INVALID_ARG", f, [0, 1, 2], [0, 1], 4, 4, 2, 2, 3, 2, 64, num_sms=2)   # heads
    _expect("ERR_UNSUPPORTED", f, [0, 1, 2], [0, 1], 4, 4, 2, 2, 2, 1, 80, num_sms=2)   # head_dim


def test_mla_plan_rejects_bad_inputs(lib):
    f = bskv.bskv_plan_mla_sparse
    f([64], 1, 1, 128, 64, num_sms=2)
    _expect("ERR_INVALID_ARG", f, [64], 1, 1, 128, 96, num_sms=2)    # top_k % 64
    _expect("ERR_INVALID_ARG", f, [65], 1, 1, 128, 64, num_sms=2)    # seq_len > top_k
    _expect("ERR_INVALID_ARG", f, [-1], 1, 1, 128, 64, num_sms=2)
    _expect("ERR_UNSUPPORTED", f, [64], 1, 1, 256, 64, num_sms=2)    # heads > 128


@pytest.mark.parametrize("M,N,R,C,Hq,Hkv,D", [(200, 256, 64, 64, 32, 8, 128), (64, 64, 16, 16, 4, 2, 64)])
def test_bsr_masked_plan_bit_exact(lib, M, N, R, C, Hq, Hkv, D):
    d = synth.bsr_inputs(95, M, N, R, C, Hq, Hkv, D, pattern="random", density=0.5,
                         tensors=False)
    p = bskv.bskv_plan_bsr_masked(d["indptr"], d["indices"], M, N, R, C, Hq, Hkv, D, num_sms=SMS)
    meta = p.metadata()
    assert meta == plan_ref.bsr_meta(d["indptr"].tolist(), d["indices"].tolist(), M, N, R, C,
                                     Hq, Hkv, D, SMS)
    assert plan_ref.sections(meta)["variant"] == (1 if R == 64 else 0)


def test_mla_paged_plan_rejects_bad_inputs(lib):
    f = bskv.bskv_plan_mla_paged
    ok = dict(num_pages=4, page_size=16, num_heads=128, num_sms=4)
    f([0, 2], [0, 1], [5], 1, **ok)  # valid
    _expect("ERR_INVALID_ARG", f, [1, 2], [0, 1], [5], 1, **ok)          # indptr[0] != 0
    _expect("ERR_INVALID_ARG", f, [0, 2, 1], [0, 1], [5, 1], 2, **ok)    # decreasing
    _expect("ERR_INVALID_ARG", f, [0, 2], [0, 4], [5], 1, **ok)          # page id >= num_pages
    _expect("ERR_INVALID_ARG", f, [0, 2], [0, -1], [5], 1, **ok)
    _expect("ERR_INVALID_ARG", f, [0, 2], [0, 1], [0], 1, **ok)          # last page len 0
    _expect("ERR_INVALID_ARG", f, [0, 2], [0, 1], [17], 1, **ok)         # > page_size
    _expect("ERR_INVALID_ARG", f, [0, 2], [0, 1], [5], 1, **{**ok, "page_size": 0})
    _expect("ERR_UNSUPPORTED", f, [0, 2], [0, 1], [5], 1, **{**ok, "num_heads": 129})
    _expect("ERR_UNSUPPORTED", f, [0, 2], [0, 1], [5], 1, **{**ok, "num_pages": 1 << 30, "page_size": 4})


def test_run_without_upload_is_rejected(lib):
    p = bskv.bskv_plan_bsr([0, 1], [0], 2, 2, 2, 2, 2, 1, 64, num_sms=2)
    lib_ = bskv.load_library()
    s = (bskv.ctypes.c_int64 * 2)(64, 64)
    code = lib_.bskv_run_bsr(p.handle, 16, s, 16, s, 16, s, 16, s, None, 1.0, None, 0, None)
    assert bskv.STATUS[code] == "ERR_INVALID_ARG"
    assert "not uploaded" in bskv.bskv_last_error_message()


@pytest.mark.parametrize("D,causal", [(64, False), (128, False), (128, True)])
@pytest.mark.parametrize("seed,H,MB,NB", [(1, 2, 3, 4), (2, 8, 16, 16), (3, 1, 1, 1)])
def test_bsr_variable_plan_bit_exact(lib, seed, H, MB, NB, D, causal):
    """head_dim 64: the general kernel's plan (variant 2); 128 with 2 query heads per kv head:
    the tensor-core plan (variant 4), with and without causal trimming of the steps."""
    g = torch.Generator().manual_seed(seed)
    bm = (torch.rand((H, MB, NB), generator=g) < 0.5).to(torch.uint8)

    def parts(total, n):  # n positive sizes summing to total, a fresh cut per kv head
        out = []
        for _ in range(H):
            cuts = sorted((torch.randperm(total - 1, generator=g)[:n - 1] + 1).tolist())
            out.append([b - a for a, b in zip([0] + cuts, cuts + [total])])
        return torch.tensor(out, dtype=torch.int32)

    rs = parts(50 * MB, MB)
    cs = parts(40 * NB, NB)
    p = bskv.bskv_plan_bsr_variable(bm, rs, cs, 2 * H, H, D, causal=causal, num_sms=SMS)
    meta = p.metadata()
    assert meta == plan_ref.bsr_variable_meta(bm.tolist(), rs.tolist(), cs.tolist(), 2 * H, H, SMS,
                                              head_dim=D, causal=causal)
    s = plan_ref.sections(meta)
    assert s["variant"] == (4 if D == 128 else 2)


def test_bsr_variable_plan_rejects_bad_inputs(lib):
    f = bskv.bskv_plan_bsr_variable
    bm = torch.ones((2, 2, 2), dtype=torch.uint8)
    f(bm, [[1, 2], [2, 1]], [[3, 1], [2, 2]], 2, 2, 64, num_sms=2)  # valid
    _expect("ERR_INVALID_ARG", f, bm, [[1, 2], [2, 2]], [[3, 1], [2, 2]], 2, 2, 64, num_sms=2)  # qo lengths differ
    _expect("ERR_INVALID_ARG", f, bm, [[1, 2], [2, 1]], [[3, 1], [2, 3]], 2, 2, 64, num_sms=2)  # kv lengths differ
    _expect("ERR_INVALID_ARG", f, bm, [[0, 3], [2, 1]], [[3, 1], [2, 2]], 2, 2, 64, num_sms=2)  # empty block
    _expect("ERR_INVALID_ARG", f, bm, [[1, 2], [2, 1]], [[3, 1], [2, 2]], 3, 2, 64, num_sms=2)  # heads
    _expect("ERR_UNSUPPORTED", f, bm, [[1, 2], [2, 1]], [[3, 1], [2, 2]], 2, 2, 96, num_sms=2)  # head_dim


@pytest.mark.parametrize("D,causal", [(64, True), (128, True), (128, False)])
@pytest.mark.parametrize("lengths,qo,ps", [([1, 17, 40, 90], [1, 17, 3, 64], 16),
                                           ([2048, 300], [1024, 300], 64), ([5], [5], 1),
                                           ([700, 0, 129], [300, 0, 129], 8),
                                           ([1000, 77], [1, 77], 128)])
def test_prefill_paged_plan_bit_exact(lib, lengths, qo, ps, D, causal):
    """head_dim 64 (or page_size 1): the general kernel's plan (variant 3); head_dim 128 with
    page_size 8 .. 128: the tensor-core plan (variant 5)."""
    d = synth.paged_prefill_inputs(85, len(lengths), 32, 8, 128, ps, 0, 0, 0, 0,
                                   lengths=lengths, qo_lens=qo)
    args = [d["qo_indptr"].tolist(), d["kv_indptr"].tolist(), d["kv_indices"].tolist(),
            d["kv_last_page_len"].tolist()]
    p = bskv.bskv_plan_prefill_paged(*args, d["num_pages"], ps, 32, 8, D, causal=causal,
                                     num_sms=SMS)
    meta = p.metadata()
    assert meta == plan_ref.prefill_paged_meta(*args, ps, 32, 8, SMS, head_dim=D, causal=causal)
    assert plan_ref.sections(meta)["variant"] == (5 if D == 128 and ps != 1 else 3)


# ---------------------------------------------------------------------------------------
# invariants of the list-driven plans, checked against the oracle's definitions (not
# against the restated rule)
# ---------------------------------------------------------------------------------------

def _aux(meta):
    return meta[meta[11]:meta[12]], meta[meta[12]:meta[14]]


@pytest.mark.parametrize("seed", [3, 4])
def test_variable_plan_tiles_cover_exactly_the_visible_keys(lib, seed):
    d = synth.variable_block_inputs(seed, 8, 4, 64, 7, 9, 500, 700, density=0.45)
    bm, rs, cs = d["block_mask_map"], d["block_row_sz"], d["block_col_sz"]
    p = bskv.bskv_plan_bsr_variable(bm, rs, cs, 8, 4, 64, num_sms=SMS)
    meta = p.metadata()
    desc, tiles = _aux(meta)
    mask = att.variable_block_mask(bm.numpy(), rs.numpy(), cs.numpy())   # [H, qo, kv]
    H, MB = 4, 7
    g = 2
    seen_rows = np.zeros((H, 500 * g), int)
    for c in plan_ref.sections(meta)["chunks"]:
        x, a, h, rt = c
        r0, nr, tb, te = desc[4 * x:4 * x + 4]
        assert x == h * MB + a
        keys = np.zeros(700, bool)
        for t in range(tb, te):
            k0, ke = tiles[2 * t], tiles[2 * t + 1]
            assert 0 <= k0 < ke <= 700
            keys[k0:min(ke, k0 + 32)] = True
        for row in range(r0, r0 + nr):
            np.testing.assert_array_equal(keys, mask[h, row])
        lo, hi = rt * 64, min((rt + 1) * 64, nr * g)
        seen_rows[h, r0 * g + lo:r0 * g + hi] += 1
    assert (seen_rows == 1).all()  # every (token, query head) row in exactly one unit


def test_prefill_plan_tiles_address_every_key_once(lib):
    lengths, qo, ps = [1, 17, 40, 90, 0], [1, 17, 3, 64, 0], 16
    d = synth.paged_prefill_inputs(86, 5, 8, 2, 64, ps, 0, 0, 0, 0, lengths=lengths,
                                   qo_lens=qo, device="cpu")
    p = bskv.bskv_plan_prefill_paged(d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                                     d["kv_last_page_len"], d["num_pages"], ps, 8, 2, 64,
                                     num_sms=SMS)
    meta = p.metadata()
    desc, tiles = _aux(meta)
    ip, ix = d["kv_indptr"].numpy(), d["kv_indices"].numpy()
    for b in range(5):
        r0, nq, tb, te, shift = desc[5 * b:5 * b + 5]
        assert r0 == int(d["qo_indptr"][b]) and nq == qo[b] and shift == lengths[b] - qo[b]
        covered = []
        for t in range(tb, te):
            k0, ke, page, slot = tiles[4 * t:4 * t + 4]
            assert ke - k0 <= 32 and slot + (ke - k0) <= ps      # never crosses its page
            for k in range(k0, ke):
                assert page == ix[ip[b] + k // ps] and slot + (k - k0) == k % ps
                covered.append(k)
        assert covered == list(range(lengths[b]))


def test_plan_log_lines():
    """BSKV_LOGLEVEL=2 makes a plan print its decisions (kernel, units, workers, workspace
    bytes) and the per-worker spread to stderr; unset, a plan prints nothing."""
    code = ("import torch, block_sparse_kv_gb300 as b, synth\n"
            "d = synth.make('paged_decode')\n"
            "b.bskv_plan_decode(d['kv_indptr'], d['kv_indices'], d['kv_last_page_len'],"
            " d['num_pages'], 16, 32, 8, 128, torch.bfloat16, num_sms=152)\n"
            "t = synth.make('bsr_tiny')\n"
            "b.bskv_plan_bsr(t['indptr'], t['indices'], 64, 64, 16, 16, 4, 2, 64, num_sms=152)\n")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, BSKV_LOGLEVEL="2", PYTHONPATH=root)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       cwd=root, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stderr.splitlines() if ln.startswith("[bskv]")]
    assert any(re.search(r"bskv_plan_decode: kernel decode_group_kernel.*workers (\d+)", ln)
               and int(re.search(r"workers (\d+)", ln).group(1)) <= 152 for ln in lines), lines
    assert any("bskv_plan_bsr: kernel bsr_generic_kernel" in ln for ln in lines), lines
    assert any("work items per worker" in ln for ln in lines), lines
    env["BSKV_LOGLEVEL"] = "0"
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       cwd=root, timeout=300)
    assert r.returncode == 0 and "[bskv]" not in r.stderr


@pytest.mark.parametrize("causal", [False, True])
def test_variable_tc_plan_steps_cover_exactly_the_visible_keys(lib, causal):
    """Tensor-core variable-block plan: for every row of every unit, the keys of its steps
    (cut at the row's causal limit) are exactly the row of the oracle's dense mask, steps
    hold at most 128 keys, and every (token, kv head) sits in exactly one unit."""
    H, MB, NB, L, Lk = 4, 7, 9, 500, 700
    d = synth.variable_block_inputs(21, 8, H, 128, MB, NB, L, Lk, density=0.45, causal=causal)
    bm, rs, cs = d["block_mask_map"], d["block_row_sz"], d["block_col_sz"]
    p = bskv.bskv_plan_bsr_variable(bm, rs, cs, 8, H, 128, causal=causal, num_sms=SMS)
    meta = p.metadata()
    assert plan_ref.sections(meta)["variant"] == 4
    desc, steps = _aux(meta)
    mask = att.variable_block_mask(bm.numpy(), rs.numpy(), cs.numpy(), causal=causal)
    seen = np.zeros((H, L), int)
    for c in plan_ref.sections(meta)["chunks"]:
        x, _, h, _ = c
        tok0, valid, tb, te, lim = desc[5 * x:5 * x + 5]
        assert 1 <= valid <= 64
        keys = np.zeros(Lk, bool)
        for t in range(tb, te):
            k0, ke = steps[2 * t], steps[2 * t + 1]
            assert 0 <= k0 < ke <= Lk and ke - k0 <= 128
            keys[k0:ke] = True
        for r in range(valid):
            row = keys.copy()
            if causal:
                row[lim + r + 1:] = False
            np.testing.assert_array_equal(row, mask[h, tok0 + r])
        seen[h, tok0:tok0 + valid] += 1
    assert (seen == 1).all()


@pytest.mark.parametrize("ps,causal", [(16, True), (8, True), (128, False), (64, True)])
def test_prefill_tc_plan_steps_address_every_visible_key_once(lib, ps, causal):
    """Tensor-core paged-prefill plan: per row, the keys of the unit's steps (cut at the
    row's causal limit) are exactly the keys the row sees; a step's listed pages are the
    request's pages for its keys (-1 past them); every (query token, kv head) is in one unit."""
    lengths, qo = [1, 17, 300, 90, 0, 257], [1, 17, 130, 64, 0, 200]
    Hkv = 2
    d = synth.paged_prefill_inputs(87, len(lengths), 8, Hkv, 128, ps, 0, 0, 0, 0,
                                   lengths=lengths, qo_lens=qo, device="cpu")
    p = bskv.bskv_plan_prefill_paged(d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                                     d["kv_last_page_len"], d["num_pages"], ps, 8, Hkv, 128,
                                     causal=causal, num_sms=SMS)
    meta = p.metadata()
    assert plan_ref.sections(meta)["variant"] == 5
    desc, steps = _aux(meta)
    words = 2 + 128 // ps
    qi, ip, ix = d["qo_indptr"].numpy(), d["kv_indptr"].numpy(), d["kv_indices"].numpy()
    seen = np.zeros((int(qi[-1]), Hkv), int)
    for c in plan_ref.sections(meta)["chunks"]:
        x, _, h, _ = c
        tok0, valid, tb, te, lim = desc[5 * x:5 * x + 5]
        b = int(np.searchsorted(qi, tok0, side="right") - 1)
        L, nq = lengths[b], qo[b]
        keys = np.zeros(L, bool)
        for t in range(tb, te):
            st = steps[words * t:words * (t + 1)]
            k0, ke = st[0], st[1]
            assert k0 % 128 == 0 and 0 <= k0 < ke <= L and ke - k0 <= 128
            keys[k0:ke] = True
            for k in range(128 // ps):
                kk = k0 + k * ps
                want = int(ix[ip[b] + kk // ps]) if kk < ke else -1
                assert st[2 + k] == want
        for r in range(valid):
            t_local = tok0 - int(qi[b]) + r
            want = np.arange(L) <= t_local + L - nq if causal else np.ones(L, bool)
            row = keys.copy()
            if causal:
                row[lim + r + 1:] = False
            np.testing.assert_array_equal(row, want)
        seen[tok0:tok0 + valid, h] += 1
    assert (seen == 1).all()
