"""GPU parity of the dense paged MLA FP8 decode.

Gate: |gpu - oracle| <= 3e-2 + 3e-2 |oracle| on the bf16 output and the LSE (the sparse MLA
gate). The GPU rounds each softmax weight p_j to E4M3 before the PV product (relative error
at most 2^-4) and the oracle does not; over thousands of keys those errors average out far
below the gate, but a request with a handful of keys can carry the whole worst case, so for
a request shorter than 64 tokens the output gate adds bmm2 * 2^-4 * sum_j p_j |v_j| / sum_j p_j
(per head and value, from the decoded rows). Inputs carry NaN canary codes in every cache
slot no request may read (past a request's last token and in the spare pages), so a read
outside the page table poisons the output.
"""

import math

import numpy as np
import pytest
import torch

import block_sparse_kv_gb300 as bskv
import synth
from oracle import attention as att
from oracle import numerics as nx
from gpu_util import assert_close, to64, u8

pytestmark = pytest.mark.gpu
TOL = 3e-2
SCALE = 1.0 / math.sqrt(576)


def _run(cuda, d, bmm1=SCALE, bmm2=1.0, repeat=False):
    p = bskv.bskv_plan_mla_paged(d["kv_indptr"], d["kv_indices"], d["kv_last_page_len"],
                                 d["batch"], d["num_pages"], d["page_size"], d["heads"])
    q = d["query"].to(cuda)
    kv = d["kv_pages"].to(cuda)
    out, lse = bskv.bskv_run_mla_paged(p, q, kv, bmm1, bmm2, return_lse=True)
    if repeat:
        out2 = bskv.bskv_run_mla_paged(p, q, kv, bmm1, bmm2)
        torch.cuda.synchronize()
        assert torch.equal(out, out2)
    torch.cuda.synchronize()
    return out, lse


def _oracle(d, bmm1=SCALE, bmm2=1.0, requests=None):
    return att.mla_paged_decode(u8(d["query"]), u8(d["kv_pages"]), d["kv_indptr"].numpy(),
                                d["kv_indices"].numpy(), d["kv_last_page_len"].numpy(),
                                d["page_size"], bmm1, bmm2, requests=requests)


def _p_rounding_bound(d, reqs, bmm1, bmm2):
    """bmm2 * 2^-4 * sum_j p_j |v_j| / sum_j p_j for the requests shorter than 64 tokens
    (0 elsewhere): the most one E4M3 rounding of every softmax weight can move the output."""
    q_all = nx.e4m3_decode(u8(d["query"]))
    cache = u8(d["kv_pages"])
    ip, ix = d["kv_indptr"].numpy(), d["kv_indices"].numpy()
    lens = d["lens"].numpy()
    ps = d["page_size"]
    out = np.zeros((len(reqs), q_all.shape[1], 512))
    for i, b in enumerate(reqs):
        L = int(lens[b])
        if L == 0 or L >= 64:
            continue
        rows = np.array([ix[ip[b] + t // ps] * ps + t % ps for t in range(L)])
        kv = nx.e4m3_decode(cache.reshape(-1, 576)[rows])
        s = bmm1 * (q_all[b] @ kv.T)                       # [H, L]
        p = np.exp(s - s.max(axis=1, keepdims=True))
        out[i] = bmm2 * 2.0 ** -4 * (p @ np.abs(kv[:, :512])) / p.sum(axis=1, keepdims=True)
    return out


def _check(out, lse, ref, ref_lse, reqs=None, slack=None):
    o = to64(out)
    l = lse.cpu().numpy().astype(np.float64)
    if reqs is not None:
        o, l = o[reqs], l[reqs]
    if slack is not None:
        # the E4M3 rounding of P, added to the gate of the short requests only
        with np.errstate(invalid="ignore"):
            err = np.abs(o - ref)
        inside = err <= TOL + TOL * np.abs(ref) + slack
        assert inside.all(), ("out", int((~inside).sum()), float(np.nanmax(err - slack)))
        assert np.isfinite(o).all()
    else:
        assert_close(o, ref, TOL, TOL, "out")
    fin = np.isfinite(ref_lse)
    assert (np.isneginf(l) == ~fin).all()
    assert_close(l[fin], ref_lse[fin], TOL, TOL, "lse")


@pytest.mark.parametrize("lens,ps,heads", [
    ([5, 0, 130, 64, 1], 16, 128),     # empty request, one token, tile and page edges
    ([300, 2048, 17], 64, 128),        # a long request split across workers (merge path)
    ([1, 2, 129, 1000], 1, 16),        # page_size 1, fewer heads
    ([257, 256, 255, 3], 7, 64),       # a page size that is not a power of two
])
def test_mla_paged_small(cuda, lens, ps, heads):
    d = synth.mla_paged_inputs(71, batch=len(lens), heads=heads, page_size=ps, len_lo=0,
                               len_hi=0, lens=lens)
    bskv.bskv_get_device_status(reset=True)
    out, lse = _run(cuda, d, repeat=True)
    ref, ref_lse = _oracle(d)
    _check(out, lse, ref, ref_lse, slack=_p_rounding_bound(d, list(range(len(lens))), SCALE, 1.0))
    assert bskv.bskv_get_device_status() == 0


def test_mla_paged_scales(cuda):
    d = synth.mla_paged_inputs(72, batch=3, heads=128, page_size=64, len_lo=0, len_hi=0,
                               lens=[700, 64, 129])
    out, lse = _run(cuda, d, bmm1=0.11, bmm2=0.5)
    ref, ref_lse = _oracle(d, 0.11, 0.5)
    _check(out, lse, ref, ref_lse)


def test_mla_paged_full_workload_sampled(cuda):
    """The benchmark's workload (128 requests of 2048-8192 tokens, page_size 64), in the
    launch configuration the benchmark times, checked on sampled requests."""
    d = synth.make("mla_paged", device="cuda")
    bskv.bskv_get_device_status(reset=True)
    out, lse = _run(cuda, d)
    reqs = [0, 1, 37, 64, 101, 127]
    ref, ref_lse = _oracle(d, requests=reqs)
    _check(out, lse, ref, ref_lse, reqs)
    assert torch.isfinite(out.float()).all()  # no canary was read anywhere
    assert bskv.bskv_get_device_status() == 0


def test_mla_paged_rejects_a_sparse_plan_and_small_workspace(cuda):
    d = synth.mla_paged_inputs(73, batch=2, heads=128, page_size=16, len_lo=0, len_hi=0,
                               lens=[40, 3])
    sp = bskv.bskv_plan_mla_sparse([64, 64], 2, 1, 128, 64)
    q = d["query"].to(cuda)
    kv = d["kv_pages"].to(cuda)
    with pytest.raises(bskv.BskvError) as e:
        bskv.bskv_run_mla_paged(sp, q, kv, SCALE)
    assert e.value.status == "ERR_INVALID_ARG"
    p = bskv.bskv_plan_mla_paged(d["kv_indptr"], d["kv_indices"], d["kv_last_page_len"], 2,
                                 d["num_pages"], 16, 128)
    p.upload(cuda, float_ws=torch.empty(16, dtype=torch.uint8, device=cuda))
    with pytest.raises(bskv.BskvError) as e:
        bskv.bskv_run_mla_paged(p, q, kv, SCALE)
    assert e.value.status == "ERR_WORKSPACE_TOO_SMALL"
