"""GPU parity of batch prefill over a paged KV cache.

Gate: |gpu - oracle| <= 1e-2 + 1e-2 |oracle| on out and lse (bf16/fp16 inputs, fp32
accumulation). The cache holds NaN in every slot no request owns (past each request's last
token and in spare pages), so a read outside the page table, or a garbage slot reaching the
PV product, poisons the output. head_dim 128 with 2 or 4 query heads per kv head and
page_size 8 .. 128 runs the tensor-core kernel (plan variant 5), other shapes the general
kernel (variant 3); each case asserts which one it exercised.
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


def _run(cuda, d, causal=True, requests=None):
    dtype = d["dtype"]
    p = bskv.bskv_plan_prefill_paged(d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                                     d["kv_last_page_len"], d["num_pages"], d["page_size"],
                                     d["num_qo_heads"], d["num_kv_heads"], d["head_dim"],
                                     causal=causal, dtype=dtype)
    g = d["num_qo_heads"] // d["num_kv_heads"]
    tc = d["head_dim"] == 128 and g in (2, 4) and d["page_size"] in (8, 16, 32, 64, 128)
    assert p.metadata()[15] == (5 if tc else 3)
    bskv.bskv_get_device_status(reset=True)
    out, lse = bskv.bskv_run_prefill_paged(p, d["q"].to(cuda), d["kv_cache"].to(cuda),
                                           return_lse=True)
    torch.cuda.synchronize()
    assert bskv.bskv_get_device_status() == 0
    dt = "bf16" if dtype == torch.bfloat16 else "fp16"
    qi = d["qo_indptr"].numpy()
    ref, ref_lse = att.paged_prefill(bits(d["q"]), bits(d["kv_cache"]), dt, qi,
                                     d["kv_indptr"].numpy(), d["kv_indices"].numpy(),
                                     d["kv_last_page_len"].numpy(), d["page_size"],
                                     causal=causal, requests=requests)
    o = to64(out)
    l = lse.cpu().numpy().astype(np.float64)
    if requests is not None:
        rows = np.concatenate([np.arange(qi[b], qi[b + 1]) for b in requests])
        o, l = o[rows], l[rows]
    st = assert_close(o, ref, TOL, TOL, "out")
    fin = np.isfinite(ref_lse)
    assert (np.isneginf(l) == ~fin).all()
    assert_close(l[fin], ref_lse[fin], TOL, TOL, "lse")
    return st


@pytest.mark.parametrize("lengths,qo,ps,Hq,Hkv,D,dtype,causal", [
    ([1, 17, 40, 90, 0], [1, 17, 3, 64, 0], 16, 8, 2, 128, torch.bfloat16, True),
    ([300, 129, 64], [300, 100, 1], 64, 32, 8, 128, torch.bfloat16, True),
    ([77, 200], [20, 200], 7, 4, 4, 64, torch.float16, True),
    ([150, 33], [40, 33], 16, 8, 1, 128, torch.float16, False),
    ([1000, 77, 0, 129], [257, 77, 0, 1], 8, 8, 4, 128, torch.float16, True),
    ([700, 300], [700, 100], 128, 16, 4, 128, torch.bfloat16, False),
    ([513, 64, 1], [200, 64, 1], 32, 8, 2, 128, torch.bfloat16, True),
    ([130, 2000], [130, 65], 64, 8, 4, 128, torch.float16, True),
])
def test_prefill_paged_small(cuda, lengths, qo, ps, Hq, Hkv, D, dtype, causal):
    d = synth.paged_prefill_inputs(90 + ps, len(lengths), Hq, Hkv, D, ps, 0, 0, 0, 0,
                                   dtype=dtype, lengths=lengths, qo_lens=qo)
    _run(cuda, d, causal)


def test_prefill_paged_full_workload(cuda):
    """The benchmark's workload (16 requests of 2048-8192 tokens, 1024 new, page 16), in the
    launch configuration the benchmark times; every request checked."""
    d = synth.make("prefill_paged", device="cuda")
    st = _run(cuda, d, True)
    print("prefill paged full workload:", st)


def test_prefill_paged_rejects_other_entry_points(cuda):
    d = synth.paged_prefill_inputs(95, 2, 4, 2, 64, 16, 0, 0, 0, 0, lengths=[20, 5],
                                   qo_lens=[4, 5])
    p = bskv.bskv_plan_prefill_paged(d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                                     d["kv_last_page_len"], d["num_pages"], 16, 4, 2, 64)
    q = d["q"].to(cuda)
    with pytest.raises(bskv.BskvError) as e:
        bskv.bskv_run_bsr(p, q, q, q)
    assert e.value.status == "ERR_INVALID_ARG"
