"""GPU parity of variable-block sparse attention (per-kv-head block sizes and masks).

Gate: |gpu - oracle| <= 1e-2 + 1e-2 |oracle| on out and lse (fp16/bf16 inputs, fp32
accumulation); tensors head-major as on the page. head_dim 128 with 2 or 4 query heads per kv
head runs the tensor-core kernel (plan variant 4), other shapes the general kernel (variant
2); each case asserts which one it exercised.
"""

import json
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
HERE = os.path.dirname(os.path.abspath(__file__))


def _variant(d):
    g = d["num_qo_heads"] // d["num_kv_heads"]
    return 4 if d["head_dim"] == 128 and g in (2, 4) else 2


def _run(cuda, d, rows=None):
    p = bskv.bskv_plan_bsr_variable(d["block_mask_map"], d["block_row_sz"], d["block_col_sz"],
                                    d["num_qo_heads"], d["num_kv_heads"], d["head_dim"],
                                    causal=d["causal"], dtype=d["dtype"])
    assert p.metadata()[15] == _variant(d)
    bskv.bskv_get_device_status(reset=True)
    out, lse = bskv.bskv_run_bsr_variable(p, d["q"].to(cuda), d["k"].to(cuda), d["v"].to(cuda),
                                          return_lse=True)
    torch.cuda.synchronize()
    assert bskv.bskv_get_device_status() == 0
    dt = "bf16" if d["dtype"] == torch.bfloat16 else "fp16"
    ref, ref_lse = att.variable_block_attention(
        bits(d["q"]), bits(d["k"]), bits(d["v"]), dt, np.asarray(d["block_mask_map"]),
        np.asarray(d["block_row_sz"]), np.asarray(d["block_col_sz"]), causal=d["causal"],
        rows=rows)
    o = to64(out)
    l = lse.cpu().numpy().astype(np.float64)
    if rows is not None:
        o, l = o[:, rows], l[:, rows]
    st = assert_close(o, ref, TOL, TOL, "out")
    fin = np.isfinite(ref_lse)
    assert (np.isneginf(l) == ~fin).all()
    assert_close(l[fin], ref_lse[fin], TOL, TOL, "lse")
    return st


def test_variable_block_page_example(cuda):
    ex = json.load(open(os.path.join(HERE, "golden", "variable_block_example.json")))
    g = torch.Generator().manual_seed(3)
    L = ex["seq_len"]
    d = dict(q=torch.randn((1, L, 128), generator=g).half(),
             k=torch.randn((1, L, 128), generator=g).half(),
             v=torch.randn((1, L, 128), generator=g).half(),
             block_mask_map=np.array(ex["block_mask_map"], bool),
             block_row_sz=ex["block_row_sz"], block_col_sz=ex["block_col_sz"],
             num_qo_heads=1, num_kv_heads=1, head_dim=128, causal=False, dtype=torch.float16)
    _run(cuda, d)


@pytest.mark.parametrize("Hq,Hkv,D,MB,NB,L,Lk,dtype,causal", [
    (8, 4, 64, 5, 7, 300, 400, torch.float16, False),      # general (head_dim 64)
    (8, 4, 128, 6, 9, 513, 700, torch.bfloat16, True),     # tensor cores, g = 2
    (4, 4, 128, 3, 3, 77, 77, torch.float16, True),        # general (g = 1)
    (16, 4, 128, 5, 6, 700, 900, torch.float16, False),    # tensor cores, g = 4, runs > 128 keys
    (16, 4, 128, 9, 4, 1000, 600, torch.bfloat16, True),   # tensor cores, g = 4, qo > kv
    (8, 2, 128, 40, 40, 640, 640, torch.float16, True),    # tensor cores, small blocks (~16)
])
def test_variable_block_random(cuda, Hq, Hkv, D, MB, NB, L, Lk, dtype, causal):
    d = synth.variable_block_inputs(40 + MB, Hq, Hkv, D, MB, NB, L, Lk, density=0.5,
                                    dtype=dtype, causal=causal)
    _run(cuda, d)


@pytest.mark.parametrize("D", [64, 128])
def test_variable_block_rows_that_see_nothing(cuda, D):
    d = synth.variable_block_inputs(50, 8, 2, D, 4, 5, 200, 260, density=0.6,
                                    empty_row_block=2)
    _run(cuda, d)


def test_variable_block_full_workload_sampled(cuda):
    """The benchmark's workload (16384 tokens, 32/8 heads, D 128, fp16, 128 x 128 random-size
    blocks per kv head, 10 % kept, causal) in the launch configuration it times, checked on
    1024 sampled query tokens of every head (the oracle computes only those rows)."""
    d = synth.make("bsr_variable")
    rows = sorted(torch.randperm(d["qo_len"], generator=torch.Generator().manual_seed(5))[:1024].tolist())
    st = _run(cuda, d, rows=rows)
    print("variable blocks full workload sampled:", st)


def test_variable_block_rejects_other_entry_points(cuda):
    d = synth.variable_block_inputs(51, 4, 2, 64, 2, 2, 64, 64)
    p = bskv.bskv_plan_bsr_variable(d["block_mask_map"], d["block_row_sz"], d["block_col_sz"],
                                    4, 2, 64)
    with pytest.raises(bskv.BskvError) as e:
        bskv.bskv_run_bsr(p, d["q"].to(cuda), d["k"].to(cuda), d["v"].to(cuda))
    assert e.value.status == "ERR_INVALID_ARG"
