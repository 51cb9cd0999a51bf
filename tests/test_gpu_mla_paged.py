"""GPU parity of the dense paged MLA FP8 decode.

Gate: |gpu - oracle| <= 3e-2 + 3e-2 |oracle| on the bf16 output and the LSE (the sparse MLA
gate), for every request length from 1 token up. Inputs carry NaN canary codes in every cache
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


def _check(out, lse, ref, ref_lse, reqs=None):
    o = to64(out)
    l = lse.cpu().numpy().astype(np.float64)
    if reqs is not None:
        o, l = o[reqs], l[reqs]
    assert np.isfinite(o).all()
    assert_close(o, ref, TOL, TOL, "out")
    fin = np.isfinite(ref_lse)
    assert (np.isneginf(l) == ~fin).all()
    assert_close(l[fin], ref_lse[fin], TOL, TOL, "lse")


@pytest.mark.parametrize("lens,ps,heads", [
    ([5, 0, 130, 64, 1], 16, 128),     # empty request, one token, tile and page edges
    ([300, 2048, 17], 64, 128),        # a long request split across workers (merge path)
    ([1, 2, 129, 1000], 1, 16),        # page_size 1, fewer heads
    ([257, 256, 255, 3], 7, 64),       # a page size that is not a power of two
    # whole tiles by TMA boxes of page slots: 16 boxes of 8, one box of 128, boxes of 128
    # at slot 0 and 128 of a 256-slot page; the partial last tiles gathered row by row
    ([777, 40, 128], 8, 128),
    ([300, 128, 513], 128, 64),
    ([1000, 256, 129], 256, 128),
])
def test_mla_paged_small(cuda, lens, ps, heads):
    d = synth.mla_paged_inputs(71, batch=len(lens), heads=heads, page_size=ps, len_lo=0,
                               len_hi=0, lens=lens)
    bskv.bskv_get_device_status(reset=True)
    out, lse = _run(cuda, d, repeat=True)
    ref, ref_lse = _oracle(d)
    _check(out, lse, ref, ref_lse)
    assert bskv.bskv_get_device_status() == 0


def test_mla_paged_scales(cuda):
    d = synth.mla_paged_inputs(72, batch=3, heads=128, page_size=64, len_lo=0, len_hi=0,
                               lens=[700, 64, 129])
    out, lse = _run(cuda, d, bmm1=0.11, bmm2=0.5)
    ref, ref_lse = _oracle(d, 0.11, 0.5)
    _check(out, lse, ref, ref_lse)


def test_mla_paged_full_workload(cuda):
    """The benchmark's workload (128 requests of 2048-8192 tokens, page_size 64), in the
    launch configuration the benchmark times, every request checked."""
    d = synth.make("mla_paged", device="cuda")
    bskv.bskv_get_device_status(reset=True)
    out, lse = _run(cuda, d)
    reqs = list(range(d["batch"]))
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
    # one long request: split across workers, so its partial states need float workspace
    e2 = synth.mla_paged_inputs(74, batch=1, heads=128, page_size=16, len_lo=0, len_hi=0,
                                lens=[2048])
    p = bskv.bskv_plan_mla_paged(e2["kv_indptr"], e2["kv_indices"], e2["kv_last_page_len"], 1,
                                 e2["num_pages"], 16, 128)
    assert p.workspace_sizes()[1] > 16
    p.upload(cuda, float_ws=torch.empty(16, dtype=torch.uint8, device=cuda))
    with pytest.raises(bskv.BskvError) as e:
        bskv.bskv_run_mla_paged(p, e2["query"].to(cuda), e2["kv_pages"].to(cuda), SCALE)
    assert e.value.status == "ERR_WORKSPACE_TOO_SMALL"
