"""GPU parity of merge_states and of the general BSR kernel against the oracle."""

import json
import math
import os

import numpy as np
import pytest
import torch

import block_sparse_kv_gb300 as bskv
import synth
from oracle import attention as att
from gpu_util import assert_close, bits, to64

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_merge_states(cuda, out_dtype):
    g = torch.Generator().manual_seed(400)
    seq, S, H, D = 37, 5, 6, 128
    v = torch.randn((seq, S, H, D), generator=g)
    s = torch.randn((seq, S, H), generator=g) * 4
    s[3, :, 2] = -float("inf")  # a row with no key in any state
    s[4, 1:, 0] = -float("inf")  # only one live state
    vo, so = bskv.bskv_merge_states(v.to(cuda), s.to(cuda), out_dtype=out_dtype)
    torch.cuda.synchronize()
    ref, ref_s = att.merge_states(v.double().numpy(), s.double().numpy(), axis=1)
    tol = 1e-5 if out_dtype == torch.float32 else TOL
    assert_close(to64(vo), ref, tol, tol, "v")
    assert_close(so.cpu().numpy(), ref_s, 1e-5, 1e-5, "s")


def _bsr_case(cuda, d, dtype):
    dt = "bf16" if dtype == torch.bfloat16 else "fp16"
    p = bskv.bskv_plan_bsr(d["indptr"], d["indices"], d["M"], d["N"], d["R"], d["C"],
                           d["num_qo_heads"], d["num_kv_heads"], d["head_dim"],
                           causal=d["causal"], dtype=dtype)
    out, lse = bskv.bskv_run_bsr(p, d["q"].to(cuda), d["k"].to(cuda), d["v"].to(cuda),
                                 return_lse=True)
    torch.cuda.synchronize()
    assert bskv.bskv_get_device_status() == 0
    ref, ref_lse = att.bsr_attention(bits(d["q"]), bits(d["k"]), bits(d["v"]), dt,
                                     d["indptr"].numpy(), d["indices"].numpy(), d["M"], d["N"],
                                     d["R"], d["C"], d["sm_scale"], d["causal"])
    st = assert_close(to64(out), ref, TOL, TOL, "out")
    assert_close(lse.cpu().numpy(), ref_lse, TOL, TOL, "lse")
    return st, p


def test_bsr_worked_example(cuda):
    """The page's own example: M = N = 3, R = C = 1, 32 query / 8 kv heads, head_dim 128,
    fp16, the 3 x 3 block mask from tests/golden (its dense mask as printed). The GPU result
    equals the oracle's dense attention under that mask, and the default scale (0 = the
    library's 1/sqrt(head_dim)) gives the same bits as passing 1/sqrt(128)."""
    here = os.path.dirname(os.path.abspath(__file__))
    ex = json.load(open(os.path.join(here, "golden", "bsr_worked_example.json")))
    M, N, R, C = ex["M"], ex["N"], ex["R"], ex["C"]
    Hq, Hkv, D = ex["num_qo_heads"], ex["num_kv_heads"], ex["head_dim"]
    d = synth.bsr_inputs(7, M, N, R, C, Hq, Hkv, D, pattern="full")
    indptr = torch.tensor(ex["indptr"], dtype=torch.int32)
    indices = torch.tensor(ex["indices"], dtype=torch.int32)
    p = bskv.bskv_plan_bsr(indptr, indices, M, N, R, C, Hq, Hkv, D, dtype=torch.float16)
    q, k, v = d["q"].to(cuda), d["k"].to(cuda), d["v"].to(cuda)
    out, lse = bskv.bskv_run_bsr(p, q, k, v, return_lse=True)
    out2 = bskv.bskv_run_bsr(p, q, k, v, sm_scale=1.0 / math.sqrt(D))
    torch.cuda.synchronize()
    assert bskv.bskv_get_device_status() == 0
    assert torch.equal(out, out2)
    mask = att.bsr_mask(ex["indptr"], ex["indices"], M, N, R, C)
    np.testing.assert_array_equal(mask, np.array(ex["mask"], dtype=bool))
    ref, ref_lse = att.bsr_attention(bits(d["q"]), bits(d["k"]), bits(d["v"]), "fp16",
                                     ex["indptr"], ex["indices"], M, N, R, C)
    assert_close(to64(out), ref, TOL, TOL, "out")
    assert_close(lse.cpu().numpy(), ref_lse, TOL, TOL, "lse")


def test_bsr_tiny_workload(cuda):
    """M = N = 64, R = C = 16, 4/2 heads, head_dim 64, fp16, density 0.5."""
    d = synth.make("bsr_tiny")
    st, p = _bsr_case(cuda, d, torch.float16)
    print("bsr tiny:", st)


BSR_CASES = [
    # M, N, R, C, Hq, Hkv, D, dtype, pattern, causal
    (100, 96, 16, 16, 4, 2, 64, torch.float16, "random", False),    # ragged last row block
    (130, 130, 13, 10, 6, 3, 128, torch.bfloat16, "random", True),  # odd R and C
    (64, 256, 32, 64, 8, 2, 128, torch.float16, "random", True),    # M < N, bottom-right causal
    (256, 256, 64, 64, 8, 8, 128, torch.float16, "diag_lower", True),  # g = 1
    (96, 96, 1, 1, 2, 1, 64, torch.float16, "random", False),       # R = C = 1
    (128, 128, 64, 32, 4, 1, 64, torch.bfloat16, "full", False),    # all blocks
]


@pytest.mark.parametrize("case", BSR_CASES)
def test_bsr_general(cuda, case):
    M, N, R, C, Hq, Hkv, D, dtype, pattern, causal = case
    d = synth.bsr_inputs(500 + M + R, M, N, R, C, Hq, Hkv, D, dtype=dtype, pattern=pattern,
                         causal=causal, density=0.4)
    _bsr_case(cuda, d, dtype)


def test_bsr_empty_row_blocks(cuda):
    d = synth.bsr_inputs(520, 64, 64, 16, 16, 4, 2, 64, pattern="random")
    indptr = torch.tensor([0, 0, 2, 2, 3], dtype=torch.int32)
    indices = torch.tensor([0, 3, 1], dtype=torch.int32)
    d.update(indptr=indptr, indices=indices)
    p = bskv.bskv_plan_bsr(indptr, indices, 64, 64, 16, 16, 4, 2, 64)
    out, lse = bskv.bskv_run_bsr(p, d["q"].to(cuda), d["k"].to(cuda), d["v"].to(cuda),
                                 return_lse=True)
    torch.cuda.synchronize()
    ref, ref_lse = att.bsr_attention(bits(d["q"]), bits(d["k"]), bits(d["v"]), "fp16",
                                     indptr.numpy(), indices.numpy(), 64, 64, 16, 16)
    assert_close(to64(out), ref, TOL, TOL, "out")
    lse = lse.cpu().numpy()
    assert np.isneginf(lse[:16]).all() and np.isneginf(lse[32:48]).all()
    assert (out[:16] == 0).all()
