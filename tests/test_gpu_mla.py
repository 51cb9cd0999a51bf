"""GPU parity of the sparse MLA FP8 decode (and the full RoPE+FP8 -> decode pipeline).

Gate: |gpu - oracle| <= 3e-2 + 3e-2 |oracle| on the bf16 output and the LSE, on every input
here (lists of 1 key to full workloads, a peaked softmax, two clusters of keys with opposite
values). The E4M3 rows the decode reads come either from the oracle's own prologue
(decode-only tests) or, for the pipeline tests, each side builds its own rows (GPU prologue vs
oracle prologue).
"""

import math

import numpy as np
import pytest
import torch

import block_sparse_kv_gb300 as bskv
import synth
from oracle import attention as att
from oracle import rope
from gpu_util import assert_close, bits, to64

pytestmark = pytest.mark.gpu
TOL = 3e-2
SCALE = 1.0 / math.sqrt(576)


def _oracle_rows(m, sq=1.0, skv=1.0):
    qr, kr, qn, kn = rope.mla_rope_quantize_fp8(
        bits(m["q_rope"]), bits(m["k_rope"]), bits(m["q_nope"]), bits(m["k_nope"]),
        m["cos_sin"].cpu().numpy(), m["pos_q"].numpy(), m["pos_k"].numpy(), True, sq, skv)
    B, T, H = m["batch"], m["q_len"], m["heads"]
    query = np.concatenate([qn, qr], axis=-1).reshape(B, T, H, 576)
    kv = np.concatenate([kn, kr], axis=-1)
    return query, kv


def _decode(cuda, m, query, kv, seq_lens, bmm1=SCALE, bmm2=1.0, repeat=False):
    B, T, H, K = m["batch"], m["q_len"], m["heads"], m["top_k"]
    p = bskv.bskv_plan_mla_sparse(seq_lens, B, T, H, K)
    q_d = torch.from_numpy(np.ascontiguousarray(query)).to(cuda) if isinstance(query, np.ndarray) else query
    kv_d = torch.from_numpy(np.ascontiguousarray(kv)).to(cuda) if isinstance(kv, np.ndarray) else kv
    idx = m["indices"].to(cuda)
    out, lse = bskv.bskv_run_mla_sparse(p, q_d, kv_d, idx, bmm1, bmm2, return_lse=True)
    if repeat:
        out2 = bskv.bskv_run_mla_sparse(p, q_d, kv_d, idx, bmm1, bmm2)
        torch.cuda.synchronize()
        assert torch.equal(out, out2)
    torch.cuda.synchronize()
    return out, lse


def _check(out, lse, ref, ref_lse, sel=None):
    o = to64(out).reshape(-1, out.shape[-2], 512)
    l = lse.reshape(-1, lse.shape[-1]).cpu().numpy()
    if sel is not None:
        o, l = o[sel], l[sel]
    st = assert_close(o, ref, TOL, TOL, "out")
    fin = np.isfinite(ref_lse)
    assert (np.isneginf(l) == ~fin).all()
    assert_close(l[fin], ref_lse[fin], TOL, TOL, "lse")
    return st


@pytest.mark.parametrize("heads,q_len,top_k,seq", [
    (128, 1, 128, [128, 70, 0]),      # ragged tail and an empty request
    (16, 2, 192, [192, 64]),          # fewer heads, two query tokens per request
    (128, 1, 1024, [1024, 1000]),     # several tiles per query: split-KV pieces + merge
])
def test_mla_decode_small(cuda, heads, q_len, top_k, seq):
    B = len(seq)
    m = synth.mla_inputs(800 + heads + top_k, batch=B, heads=heads, top_k=top_k, pool_rows=4096,
                         ctx_lo=top_k, ctx_hi=4096, q_len=q_len, max_seq_len=4096)
    query, kv = _oracle_rows(m)
    out, lse = _decode(cuda, m, query, kv, seq, repeat=True)
    assert bskv.bskv_get_device_status() == 0
    ref, ref_lse = att.mla_sparse_decode(query, kv, m["indices"].numpy(), np.array(seq), SCALE, 1.0)
    _check(out, lse, ref, ref_lse)


def test_mla_decode_short_lists(cuda):
    """Queries with a handful of keys (1 to 63), where no rounding averages out: the weights
    enter PV as two E4M3 terms, so the plain gate holds."""
    seq = [1, 5, 17, 63]
    B, K = len(seq), 64
    m = synth.mla_inputs(880, batch=B, heads=128, top_k=K, pool_rows=1024, ctx_lo=K,
                         ctx_hi=1024, max_seq_len=1024)
    query, kv = _oracle_rows(m)
    out, lse = _decode(cuda, m, query, kv, seq, repeat=True)
    assert bskv.bskv_get_device_status() == 0
    ref, ref_lse = att.mla_sparse_decode(query, kv, m["indices"].numpy(), np.array(seq), SCALE, 1.0)
    st = _check(out, lse, ref, ref_lse)
    print("mla short lists:", st)


def _e4m3(x):
    return torch.as_tensor(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_mla_two_clusters_of_keys(cuda):
    """Half of a query's 64 listed rows have logit 0 and V = +4, the other half logit
    -c_h * 2.25 / 24 and V = -4, so the output is a difference of two large terms and every
    error in the weight ratio shows directly. c_h (the query's one nonzero value, in the
    rotated tail) varies over the heads; for c_h = 1 the weight 0.9105 falls next to the
    midpoint of two E4M3 codes (0.875, 0.9375), where one code alone would move the output
    by about 0.06, twice the gate."""
    H, K = 128, 64
    c = np.array([0.5, 0.625, 0.75, 0.875, 1.0, 1.125, 1.25, 1.5] * (H // 8), np.float32)
    q = np.zeros((1, 1, H, 576), np.float32)
    q[0, 0, :, 512] = c
    rows = np.zeros((2, 576), np.float32)
    rows[0, :512] = 4.0
    rows[1, :512] = -4.0
    rows[1, 512] = -2.25
    query, kv = _e4m3(q), _e4m3(rows)
    idx = torch.tensor([0, 1] * (K // 2), dtype=torch.int32).view(1, 1, K)
    m = dict(batch=1, q_len=1, heads=H, top_k=K, indices=idx)
    out, lse = _decode(cuda, m, query, kv, [K], repeat=True)
    assert bskv.bskv_get_device_status() == 0
    ref, ref_lse = att.mla_sparse_decode(query, kv, idx.numpy(), np.array([K]), SCALE, 1.0)
    st = _check(out, lse, ref, ref_lse)
    print("mla two clusters:", st)


def test_mla_duplicate_indices(cuda):
    """A row listed several times in a query's index list counts once per listing (list
    semantics, as in the oracle): the second half of each list repeats its first half, and
    a few single rows repeat further, across tile boundaries and split pieces."""
    m = synth.mla_inputs(860, batch=3, heads=128, top_k=512, pool_rows=2048, ctx_lo=512,
                         ctx_hi=2048, max_seq_len=2048)
    idx = m["indices"].clone()
    idx[:, :, 256:] = idx[:, :, :256]
    idx[:, :, 300:310] = idx[:, :, 5:6]
    m["indices"] = idx
    query, kv = _oracle_rows(m)
    seq = [512, 400, 137]
    out, lse = _decode(cuda, m, query, kv, seq)
    assert bskv.bskv_get_device_status() == 0
    ref, ref_lse = att.mla_sparse_decode(query, kv, idx.numpy(), np.array(seq), SCALE, 1.0)
    _check(out, lse, ref, ref_lse)


def test_mla_sharp_softmax(cuda):
    """q x 6: a peaked softmax dominated by a few keys per head, under the plain gate."""
    m = synth.mla_inputs(850, batch=2, heads=128, top_k=512, pool_rows=2048, ctx_lo=512,
                         ctx_hi=2048, max_seq_len=2048, q_scale=6.0)
    query, kv = _oracle_rows(m)
    out, lse = _decode(cuda, m, query, kv, [512, 512])
    ref, ref_lse = att.mla_sparse_decode(query, kv, m["indices"].numpy(), np.array([512, 512]), SCALE, 1.0)
    st = _check(out, lse, ref, ref_lse)
    print("mla sharp:", st)


def test_mla_pipeline_with_scale_folding(cuda):
    """Prologue with non-unit quant scales and decode with the folded scales, end to end."""
    sq, skv = 2.0, 0.5
    m = synth.mla_inputs(851, batch=3, heads=128, top_k=256, pool_rows=2048, ctx_lo=256,
                         ctx_hi=2048, max_seq_len=2048)
    g = {k: (v.to(cuda) if torch.is_tensor(v) else v) for k, v in m.items()}
    query = torch.empty((3, 1, 128, 576), dtype=torch.uint8, device=cuda)
    pool = torch.empty((2048, 576), dtype=torch.uint8, device=cuda)
    bskv.bskv_rope_quantize_fp8(g["q_rope"], g["k_rope"], g["q_nope"], g["k_nope"], g["cos_sin"],
                                g["pos_q"], True, sq, skv, q_rope_out=query[:, 0, :, 512:],
                                k_rope_out=pool[:, 512:], q_nope_out=query[:, 0, :, :512],
                                k_nope_out=pool[:, :512], pos_ids_k=g["pos_k"])
    bmm1, bmm2 = SCALE / (sq * skv), 1.0 / skv
    out, lse = _decode(cuda, m, query, pool, [256, 256, 256], bmm1, bmm2)
    oq, okv = _oracle_rows(m, sq, skv)
    ref, ref_lse = att.mla_sparse_decode(oq, okv, m["indices"].numpy(), np.array([256] * 3), bmm1, bmm2)
    _check(out, lse, ref, ref_lse)


def test_mla_full_workload_pipeline(cuda):
    """128 queries x 128 heads x 2048 rows over a 65536-row pool built by the prologue, in
    the launch configuration the benchmark times; every query checked against the oracle's
    own prologue + decode."""
    m = synth.make("mla_decode", device=cuda)
    query = torch.empty((128, 1, 128, 576), dtype=torch.uint8, device=cuda)
    pool = torch.empty((65536, 576), dtype=torch.uint8, device=cuda)
    bskv.bskv_rope_quantize_fp8(m["q_rope"], m["k_rope"], m["q_nope"], m["k_nope"], m["cos_sin"],
                                m["pos_q"].to(cuda), True, q_rope_out=query[:, 0, :, 512:],
                                k_rope_out=pool[:, 512:], q_nope_out=query[:, 0, :, :512],
                                k_nope_out=pool[:, :512], pos_ids_k=m["pos_k"].to(cuda))
    out, lse = _decode(cuda, m, query, pool, m["seq_lens"], repeat=True)
    assert bskv.bskv_get_device_status() == 0
    host = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in m.items()}
    oq, okv = _oracle_rows(host)
    ref, ref_lse = att.mla_sparse_decode(oq, okv, host["indices"].numpy(), host["seq_lens"].numpy(),
                                         SCALE, 1.0)
    st = _check(out, lse, ref, ref_lse)
    print("mla full workload:", st)


def test_mla_bad_index_is_reported(cuda):
    m = synth.mla_inputs(852, batch=1, heads=128, top_k=64, pool_rows=512, ctx_lo=64, ctx_hi=512,
                         max_seq_len=512)
    query, kv = _oracle_rows(m)
    m["indices"][0, 0, 5] = 512  # one past the last row
    bskv.bskv_get_device_status(reset=True)
    _decode(cuda, m, query, kv, [64])
    assert bskv.STATUS[bskv.bskv_get_device_status(reset=True)] == "ERR_DEVICE_INDEX"


def test_mla_forced_timeout_is_reported_and_recovers(cuda):
    """The testing hook makes every bounded wait of the cluster kernel give up at once: both
    CTAs of each pair leave through the abort path, the device status reads TIMEOUT, and once
    the hook is cleared the same run is correct."""
    m = synth.mla_inputs(870, batch=3, heads=128, top_k=256, pool_rows=2048, ctx_lo=256,
                         ctx_hi=2048, max_seq_len=2048)
    query, kv = _oracle_rows(m)
    seq = [256, 200, 130]
    bskv.bskv_get_device_status(reset=True)
    bskv.bskv_set_debug_force_timeout(True)
    try:
        _decode(cuda, m, query, kv, seq)
    finally:
        bskv.bskv_set_debug_force_timeout(False)
    assert bskv.STATUS[bskv.bskv_get_device_status(reset=True)] == "ERR_TIMEOUT"
    out, lse = _decode(cuda, m, query, kv, seq)
    assert bskv.bskv_get_device_status() == 0
    ref, ref_lse = att.mla_sparse_decode(query, kv, m["indices"].numpy(), np.array(seq), SCALE, 1.0)
    _check(out, lse, ref, ref_lse)
