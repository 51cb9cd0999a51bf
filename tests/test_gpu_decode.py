"""GPU parity of the paged-KV decode (with split-KV + merge) against the oracle.

Gate: |gpu - oracle| <= 1e-2 + 1e-2 |oracle| for bf16/fp16 outputs (and the LSE). Inputs
carry NaN canaries in every pool page outside the page table and in every slot past a
request's last valid token, so a read outside the page table fails the test.
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


def _plan(d, dtype, max_workers=0):
    return bskv.bskv_plan_decode(d["kv_indptr"], d["kv_indices"], d["kv_last_page_len"],
                                 d["num_pages"], d["page_size"], d["num_qo_heads"],
                                 d["num_kv_heads"], d["head_dim"], dtype, max_workers=max_workers)


def _oracle(d, dt, requests=None):
    return att.paged_decode(bits(d["q"]), bits(d["kv_cache"]), dt, d["kv_indptr"].numpy(),
                            d["kv_indices"].numpy(), d["kv_last_page_len"].numpy(),
                            d["page_size"], d["sm_scale"], requests)


CASES = [
    # batch, Hq, Hkv, D, page_size, len_lo, len_hi, dtype, max_workers
    (4, 8, 2, 128, 16, 1, 200, torch.bfloat16, 0),
    (4, 8, 2, 128, 16, 1, 200, torch.bfloat16, 7),    # forced splits -> merge kernel
    (3, 32, 8, 128, 64, 100, 700, torch.bfloat16, 5),
    (5, 16, 1, 64, 16, 3, 300, torch.float16, 9),      # g = 16, D = 64, fp16
    (6, 4, 4, 128, 8, 1, 90, torch.bfloat16, 4),       # g = 1, page size 8
    (2, 12, 4, 64, 32, 33, 97, torch.float16, 3),      # g = 3 (not a power of two)
    (3, 32, 16, 64, 16, 20, 300, torch.float16, 6),    # two groups of 8 kv heads per request
    (2, 24, 12, 128, 16, 10, 200, torch.bfloat16, 4),  # 12 kv heads: per-kv-head variant
    (4, 64, 8, 128, 8, 1, 200, torch.bfloat16, 5),     # g = 8, page size 8, 8 kv heads
]


@pytest.mark.parametrize("case", CASES)
def test_decode_small(cuda, case):
    B, Hq, Hkv, D, ps, lo, hi, dtype, mw = case
    d = synth.paged_decode_inputs(200 + B + Hq + ps, B, Hq, Hkv, D, ps, lo, hi, dtype=dtype)
    p = _plan(d, dtype, mw)
    q, kv = d["q"].to(cuda), d["kv_cache"].to(cuda)
    out, lse = bskv.bskv_run_decode(p, q, kv, return_lse=True)
    torch.cuda.synchronize()
    assert bskv.bskv_get_device_status() == 0
    dt = "bf16" if dtype == torch.bfloat16 else "fp16"
    ref, ref_lse = _oracle(d, dt)
    assert_close(to64(out), ref, TOL, TOL, "out")
    assert_close(lse.cpu().numpy(), ref_lse, TOL, TOL, "lse")


@pytest.mark.parametrize("case", [
    (4, 8, 2, 128, 16, 1, 400, torch.bfloat16, 7),     # page-major variant, fused merges
    (3, 32, 8, 128, 64, 100, 700, torch.bfloat16, 5),  # per-kv-head variant, fused merges
    (5, 16, 1, 64, 8, 0, 300, torch.float16, 9),       # page 8, some empty requests
    (2, 16, 2, 128, 16, 900, 1000, torch.bfloat16, 20),  # > 8 pieces per unit: two kernels
])
def test_fused_merge_matches_two_kernel_path(cuda, case):
    """bskv_run_decode merges split units inside the attention kernel (the last worker of a
    unit merges it); bskv_run_decode_partial + bskv_decode_merge do it in two kernels.
    Both apply the same arithmetic in the same order, so they agree bit for bit, and a
    second fused run (merge counters reset by the first) gives the same bits again."""
    B, Hq, Hkv, D, ps, lo, hi, dtype, mw = case
    d = synth.paged_decode_inputs(400 + B + ps, B, Hq, Hkv, D, ps, lo, hi, dtype=dtype)
    p = _plan(d, dtype, mw)
    assert p.metadata()[6] > 0, "expected split units"
    q, kv = d["q"].to(cuda), d["kv_cache"].to(cuda)
    fused, fused_lse = bskv.bskv_run_decode(p, q, kv, return_lse=True)
    again, again_lse = bskv.bskv_run_decode(p, q, kv, return_lse=True)
    two = torch.full_like(fused, float("nan"))
    two_lse = torch.full_like(fused_lse, float("nan"))
    bskv.bskv_run_decode_partial(p, q, kv, out=two, lse=two_lse)
    bskv.bskv_decode_merge(p, two, two_lse)
    torch.cuda.synchronize()
    assert bskv.bskv_get_device_status() == 0
    assert torch.equal(fused, again) and torch.equal(fused_lse, again_lse)
    assert torch.equal(fused, two) and torch.equal(fused_lse, two_lse)
    dt = "bf16" if dtype == torch.bfloat16 else "fp16"
    ref, ref_lse = _oracle(d, dt)
    assert_close(to64(fused), ref, TOL, TOL, "out")


def test_decode_zero_length_requests(cuda):
    d = synth.paged_decode_inputs(301, 5, 8, 2, 128, 16, 0, 0, lengths=[0, 37, 0, 1, 300])
    p = _plan(d, torch.bfloat16, 3)
    out, lse = bskv.bskv_run_decode(p, d["q"].to(cuda), d["kv_cache"].to(cuda), return_lse=True)
    torch.cuda.synchronize()
    ref, ref_lse = _oracle(d, "bf16")
    assert_close(to64(out), ref, TOL, TOL, "out")
    lse = lse.cpu().numpy()
    assert np.isneginf(lse[[0, 2]]).all()
    assert_close(lse[[1, 3, 4]], ref_lse[[1, 3, 4]], TOL, TOL, "lse")


def test_decode_strided_views(cuda):
    """q / out as strided views and an NHD-style kv view (token stride != head_dim)."""
    d = synth.paged_decode_inputs(302, 3, 8, 2, 128, 16, 10, 100)
    q_big = torch.zeros((3, 16, 128), dtype=torch.bfloat16, device=cuda)
    q_big[:, ::2] = d["q"].to(cuda)
    q = q_big[:, ::2]
    kv = d["kv_cache"].to(cuda)
    nhd = torch.empty((kv.shape[0], 2, 16, 2, 128), dtype=kv.dtype, device=cuda)
    nhd.copy_(kv.permute(0, 1, 3, 2, 4))
    kv_view = nhd.permute(0, 1, 3, 2, 4)  # logical (page, 2, head, token, d), NHD storage
    out_big = torch.zeros((3, 8, 256), dtype=torch.bfloat16, device=cuda)
    out = out_big[:, :, :128]
    p = _plan(d, torch.bfloat16)
    bskv.bskv_run_decode(p, q, kv_view, out=out)
    torch.cuda.synchronize()
    ref, _ = _oracle(d, "bf16")
    assert_close(to64(out), ref, TOL, TOL, "out")
    assert (out_big[:, :, 128:] == 0).all()


def test_decode_full_workload_and_determinism(cuda):
    """Batch 64, 32/8 heads, head_dim 128, page 16, lengths U[512, 4096]; every request."""
    d = synth.make("paged_decode", device=cuda)
    p = _plan(d, torch.bfloat16)
    out, lse = bskv.bskv_run_decode(p, d["q"], d["kv_cache"], return_lse=True)
    out2 = bskv.bskv_run_decode(p, d["q"], d["kv_cache"])
    torch.cuda.synchronize()
    assert torch.equal(out, out2)  # run-to-run bitwise
    host = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in d.items()}
    ref, ref_lse = _oracle(host, "bf16")
    st = assert_close(to64(out), ref, TOL, TOL, "out")
    assert st["rel_fro"] < 1e-2, st
    assert_close(lse.cpu().numpy(), ref_lse, TOL, TOL, "lse")
    print("paged decode full:", st)


def test_decode_sharp_softmax(cuda):
    """q scaled by 8: a peaked softmax, so the tolerance is not met trivially."""
    d = synth.make("paged_decode", batch=8, q_scale=8.0, device=cuda)
    p = _plan(d, torch.bfloat16)
    out = bskv.bskv_run_decode(p, d["q"], d["kv_cache"])
    torch.cuda.synchronize()
    host = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in d.items()}
    ref, _ = _oracle(host, "bf16")
    st = assert_close(to64(out), ref, TOL, TOL, "out")
    print("sharp softmax:", st)


def test_split_kv_long_context(cuda):
    """Batch 8 x 131072 tokens, page 64, 64/8 heads, in the launch configuration the benchmark
    times: every output row of every request, checked two requests at a time on the host."""
    d = synth.make("split_decode", device=cuda)
    p = _plan(d, torch.bfloat16)
    out, lse = bskv.bskv_run_decode(p, d["q"], d["kv_cache"], return_lse=True)
    torch.cuda.synchronize()
    assert bskv.bskv_get_device_status() == 0
    for reqs in ([0, 1], [2, 3], [4, 5], [6, 7]):
        pages = np.concatenate([d["kv_indices"][int(d["kv_indptr"][b]):int(d["kv_indptr"][b + 1])].numpy()
                                for b in reqs])
        # move only these requests' pages to the host, renumbered
        sub = d["kv_cache"][torch.from_numpy(pages).to(cuda).long()].cpu()
        n0 = int(d["kv_indptr"][reqs[0] + 1] - d["kv_indptr"][reqs[0]])
        indptr = np.array([0, n0, len(pages)])
        host = dict(q=d["q"][reqs].cpu(), kv_cache=sub, kv_indptr=torch.from_numpy(indptr),
                    kv_indices=torch.arange(len(pages), dtype=torch.int32),
                    kv_last_page_len=d["kv_last_page_len"][reqs].cpu(), page_size=64,
                    sm_scale=d["sm_scale"])
        ref, ref_lse = _oracle(host, "bf16")
        assert_close(to64(out[reqs]), ref, TOL, TOL, "out %s" % reqs)
        assert_close(lse[reqs].cpu().numpy(), ref_lse, TOL, TOL, "lse %s" % reqs)
        del sub


def test_forced_timeout_is_reported_and_recovers(cuda):
    """The testing hook makes every bounded wait give up: the run returns, the device
    status reads TIMEOUT, and after clearing it the same run is correct again."""
    d = synth.paged_decode_inputs(303, 4, 8, 2, 128, 16, 50, 400)
    p = _plan(d, torch.bfloat16, 5)
    q, kv = d["q"].to(cuda), d["kv_cache"].to(cuda)
    bskv.bskv_get_device_status(reset=True)
    bskv.bskv_set_debug_force_timeout(True)
    try:
        bskv.bskv_run_decode(p, q, kv)
        torch.cuda.synchronize()
    finally:
        bskv.bskv_set_debug_force_timeout(False)
    assert bskv.STATUS[bskv.bskv_get_device_status(reset=True)] == "ERR_TIMEOUT"
    out = bskv.bskv_run_decode(p, q, kv)
    torch.cuda.synchronize()
    assert bskv.bskv_get_device_status() == 0
    ref, _ = _oracle(d, "bf16")
    assert_close(to64(out), ref, TOL, TOL, "out")
