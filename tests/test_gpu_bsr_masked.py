"""GPU parity of BSR attention with a per-block token mask (general and tensor-core kernels).

Gate: |gpu - oracle| <= 1e-2 + 1e-2 |oracle| on out and lse (fp16/bf16 inputs, fp32
accumulation). The mask is drawn per pair, packed with numpy.packbits(bitorder="little"),
and handed to the kernel as device bytes; the oracle reads the unpacked boolean mask.
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


def _run_case(cuda, d, dtype, bm):
    p = bskv.bskv_plan_bsr_masked(d["indptr"], d["indices"], d["M"], d["N"], d["R"], d["C"],
                                  d["num_qo_heads"], d["num_kv_heads"], d["head_dim"], dtype)
    packed = torch.from_numpy(np.packbits(bm.reshape(-1), bitorder="little").copy()).to(cuda)
    q, k, v = d["q"].to(cuda), d["k"].to(cuda), d["v"].to(cuda)
    bskv.bskv_get_device_status(reset=True)
    out, lse = bskv.bskv_run_bsr_masked(p, q, k, v, packed, return_lse=True)
    torch.cuda.synchronize()
    assert bskv.bskv_get_device_status() == 0
    dt = "bf16" if dtype == torch.bfloat16 else "fp16"
    ref, ref_lse = att.bsr_attention(bits(d["q"]), bits(d["k"]), bits(d["v"]), dt, d["indptr"],
                                     d["indices"], d["M"], d["N"], d["R"], d["C"],
                                     block_mask=bm)
    assert_close(to64(out), ref, TOL, TOL, "out")
    l = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert (np.isneginf(l) == ~fin).all()
    assert_close(l[fin], ref_lse[fin], TOL, TOL, "lse")


def _mask(d, p_keep, seed, blank_row=None):
    nnz = int(d["indptr"][-1])
    g = torch.Generator().manual_seed(seed)
    bm = (torch.rand((nnz, d["R"], d["C"]), generator=g) < p_keep).numpy()
    if blank_row is not None:
        bm[:, blank_row, :] = False  # that row of every block: its queries see nothing
    return bm


@pytest.mark.parametrize("M,N,R,C,Hq,Hkv,D,dtype", [
    (64, 64, 16, 16, 4, 2, 64, torch.float16),      # the tiny BSR shape
    (200, 256, 64, 64, 32, 8, 128, torch.float16),  # tensor-core, two M tiles, ragged last rows
    (256, 320, 64, 64, 16, 8, 128, torch.bfloat16),  # tensor-core, one M tile
    (96, 160, 32, 16, 8, 8, 128, torch.bfloat16),   # no GQA, bf16
])
def test_bsr_masked(cuda, M, N, R, C, Hq, Hkv, D, dtype):
    d = synth.bsr_inputs(90 + R, M, N, R, C, Hq, Hkv, D, dtype=dtype, pattern="random",
                         density=0.5)
    _run_case(cuda, d, dtype, _mask(d, 0.5, 3))


def test_bsr_masked_rows_that_see_nothing(cuda):
    d = synth.bsr_inputs(97, 64, 64, 16, 16, 4, 2, 64, pattern="random", density=0.7)
    _run_case(cuda, d, torch.float16, _mask(d, 0.4, 4, blank_row=5))


def test_bsr_masked_rejects_missing_or_short_mask(cuda):
    d = synth.bsr_inputs(98, 64, 64, 16, 16, 4, 2, 64, pattern="random", density=0.7)
    p = bskv.bskv_plan_bsr_masked(d["indptr"], d["indices"], 64, 64, 16, 16, 4, 2, 64)
    q, k, v = d["q"].to(cuda), d["k"].to(cuda), d["v"].to(cuda)
    short = torch.zeros(1, dtype=torch.uint8, device=cuda)
    with pytest.raises(bskv.BskvError) as e:
        bskv.bskv_run_bsr_masked(p, q, k, v, short)
    assert e.value.status == "ERR_INVALID_ARG"
    with pytest.raises(bskv.BskvError) as e:
        bskv.bskv_run_bsr(p, q, k, v)   # a masked plan needs its mask
    assert e.value.status == "ERR_INVALID_ARG"
