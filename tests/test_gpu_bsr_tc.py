"""GPU parity of the tensor-core (tcgen05) BSR kernel against the oracle.

Shapes with R = C = 64, head_dim 128 and 2 or 4 query heads per kv head take the
tensor-core path (the plan's variant 1). Gate: |gpu - oracle| <= 1e-2 + 1e-2 |oracle|.
"""

import numpy as np
import pytest
import torch

import block_sparse_kv_gb300 as bskv
import synth
from oracle import attention as att
from gpu_util import assert_close, bits, to64

pytestmark = pytest.mark.gpu
TOL = 1e-2


def _run(cuda, d, dtype, rows=None, repeat=False):
    dt = "bf16" if dtype == torch.bfloat16 else "fp16"
    p = bskv.bskv_plan_bsr(d["indptr"], d["indices"], d["M"], d["N"], d["R"], d["C"],
                           d["num_qo_heads"], d["num_kv_heads"], d["head_dim"],
                           causal=d["causal"], dtype=dtype)
    assert p.metadata()[15] == 1, "expected the tensor-core variant"
    q, k, v = d["q"].to(cuda), d["k"].to(cuda), d["v"].to(cuda)
    out, lse = bskv.bskv_run_bsr(p, q, k, v, return_lse=True)
    if repeat:
        out2 = bskv.bskv_run_bsr(p, q, k, v)
        torch.cuda.synchronize()
        assert torch.equal(out, out2)
    torch.cuda.synchronize()
    assert bskv.STATUS[bskv.bskv_get_device_status()] == "OK"
    hq = d["q"].cpu() if rows is None else d["q"].cpu()
    ref, ref_lse = att.bsr_attention(bits(hq), bits(d["k"]), bits(d["v"]), dt,
                                     d["indptr"].numpy(), d["indices"].numpy(), d["M"], d["N"],
                                     d["R"], d["C"], d["sm_scale"], d["causal"], rows)
    sel = slice(None) if rows is None else torch.as_tensor(rows)
    st = assert_close(to64(out[sel]), ref, TOL, TOL, "out")
    assert_close(lse[sel].cpu().numpy(), ref_lse, TOL, TOL, "lse")
    fin = np.isfinite(ref_lse)
    got = lse[sel].cpu().numpy().astype(np.float64)
    st["max_lse_err"] = float(np.abs(got[fin] - ref_lse[fin]).max()) if fin.any() else 0.0
    return st


CASES = [
    # M, N, Hq, Hkv, dtype, pattern, causal
    (256, 256, 8, 2, torch.float16, "diag_lower", True),    # g = 4: two M tiles
    (256, 256, 4, 2, torch.bfloat16, "diag_lower", True),   # g = 2: one M tile, bf16
    (320, 384, 16, 4, torch.float16, "random", False),      # several kv heads, random blocks
    (200, 256, 8, 2, torch.float16, "random", True),        # ragged M, bottom-right causal
    (512, 512, 8, 4, torch.bfloat16, "full", True),         # every block, dense causal
    (384, 384, 16, 4, torch.bfloat16, "random", True),      # g = 4 in bf16
]


@pytest.mark.parametrize("case", CASES)
def test_bsr_tc_small(cuda, case):
    M, N, Hq, Hkv, dtype, pattern, causal = case
    d = synth.bsr_inputs(600 + M + Hq, M, N, 64, 64, Hq, Hkv, 128, dtype=dtype, pattern=pattern,
                         causal=causal, density=0.5, p_off=0.3)
    _run(cuda, d, dtype, repeat=True)


def test_bsr_tc_sharp_softmax_rescales(cuda):
    """q x 8 makes the running max grow block after block (lazy O rescaling in TMEM)."""
    d = synth.bsr_inputs(650, 512, 512, 64, 64, 8, 2, 128, pattern="full", causal=False,
                         q_scale=8.0)
    st = _run(cuda, d, torch.float16)
    print("bsr tc sharp:", st)


def test_bsr_tc_empty_row_blocks(cuda):
    d = synth.bsr_inputs(651, 256, 256, 64, 64, 8, 2, 128, pattern="random")
    d["indptr"] = torch.tensor([0, 0, 2, 2, 3], dtype=torch.int32)
    d["indices"] = torch.tensor([0, 3, 1], dtype=torch.int32)
    _run(cuda, d, torch.float16)


def test_bsr_tc_full_prefill_workload_sampled_rows(cuda):
    """M = N = 16384, 32/8 heads, diagonal + 10% lower blocks, causal; about 1024 sampled rows
    (every row of 8 whole row blocks, spread over the sequence, plus 512 random rows).

    The fp16 kernel sums each row's softmax weights in packed f16 partials of at most 16
    values per 128-key step, converted to fp32 per step; every f16 addition rounds to 11
    significant bits, so the row sum l carries at most 15 * 2^-11 relative error from the
    additions, plus at most 2^-9 ln 2 + 2^-10 + 2^-11 from each weight (its f16 argument, the
    f16 exponential, its f16 value). The LSE error ln(l_gpu / l) measures it directly: here
    it must stay within that sum (0.0102), and it is reported."""
    d = synth.make("bsr_prefill", device=cuda)
    g = torch.Generator().manual_seed(5)
    blocks = [0, 1, 37, 100, 128, 200, 254, 255]
    whole = {b * 64 + r for b in blocks for r in range(64)}
    rows = sorted(set(torch.randint(0, 16384, (512,), generator=g).tolist()) | whole)
    st = _run(cuda, d, torch.float16, rows=np.array(rows), repeat=True)
    print("bsr prefill sampled rows:", st)
    assert st["max_lse_err"] <= 15 * 2.0 ** -11 + 2.0 ** -9 * np.log(2) + 2.0 ** -10 + 2.0 ** -11


def test_bsr_tc_forced_timeout_is_reported_and_recovers(cuda):
    """Every bounded wait of the tensor-core kernel gives up at once under the testing hook:
    the producer, the MMA issuer and both softmax warpgroups leave through the abort path
    (the issuer drains its MMAs), the status reads TIMEOUT, and the next run is correct."""
    d = synth.bsr_inputs(652, 256, 256, 64, 64, 8, 2, 128, pattern="random", causal=True)
    bskv.bskv_get_device_status(reset=True)
    bskv.bskv_set_debug_force_timeout(True)
    try:
        p = bskv.bskv_plan_bsr(d["indptr"], d["indices"], d["M"], d["N"], d["R"], d["C"],
                               d["num_qo_heads"], d["num_kv_heads"], d["head_dim"],
                               causal=d["causal"], dtype=torch.float16)
        bskv.bskv_run_bsr(p, d["q"].to(cuda), d["k"].to(cuda), d["v"].to(cuda))
        torch.cuda.synchronize()
    finally:
        bskv.bskv_set_debug_force_timeout(False)
    assert bskv.STATUS[bskv.bskv_get_device_status(reset=True)] == "ERR_TIMEOUT"
    _run(cuda, d, torch.float16)
