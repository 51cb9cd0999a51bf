"""GPU parity of bskv_rope_quantize_fp8 against the oracle (E4M3 bytes).

Gate: bytes identical except for at most 1 E4M3 ulp on at most 0.1% of them; with unit
scales the NoPE bytes are identical. Outputs are written into slices of 576-byte rows
whose neighbouring bytes are sentinels that must survive.
"""

import numpy as np
import pytest
import torch

import block_sparse_kv_gb300 as bskv
import synth
from oracle import numerics as nx
from oracle import rope
from gpu_util import bits, u8

pytestmark = pytest.mark.gpu


def _check_bytes(got, ref, exact=False, what=""):
    d = nx.e4m3_ulp_distance(got, ref)
    frac = float((d > 0).mean()) if d.size else 0.0
    assert d.max(initial=0) <= (0 if exact else 1), (what, int(d.max()))
    assert frac <= 1e-3, (what, frac)
    return frac


def _run(cuda, seed, nq, H, nk, max_seq, neox, cache_dtype, pos_dtype, sq=1.0, skv=1.0):
    d = synth.mla_inputs(seed, batch=nq, heads=H, top_k=64, pool_rows=nk, ctx_lo=64,
                         ctx_hi=nk, max_seq_len=max_seq, cache_dtype=cache_dtype)
    g = torch.Generator().manual_seed(seed + 5)
    pos_k = torch.randint(0, max_seq, (nk,), generator=g, dtype=torch.int64).to(pos_dtype)
    pos_q = d["pos_q"].to(pos_dtype)
    dev = {k: (v.to(cuda) if torch.is_tensor(v) else v) for k, v in d.items()}
    # merged 576-byte rows with sentinel padding on both sides of every row
    SENT = 0xA5
    qbuf = torch.full((nq, H, 576 + 32), SENT, dtype=torch.uint8, device=cuda)
    kbuf = torch.full((nk, 576 + 32), SENT, dtype=torch.uint8, device=cuda)
    q_view, k_view = qbuf[..., 16:16 + 576], kbuf[:, 16:16 + 576]
    bskv.bskv_rope_quantize_fp8(dev["q_rope"], dev["k_rope"], dev["q_nope"], dev["k_nope"],
                                dev["cos_sin"], pos_q.to(cuda), neox, sq, skv,
                                q_rope_out=q_view[..., 512:], k_rope_out=k_view[:, 512:],
                                q_nope_out=q_view[..., :512], k_nope_out=k_view[:, :512],
                                pos_ids_k=pos_k.to(cuda))
    torch.cuda.synchronize()
    assert bskv.bskv_get_device_status() == 0
    qb, kb = u8(qbuf), u8(kbuf)
    assert (qb[..., :16] == SENT).all() and (qb[..., -16:] == SENT).all()
    assert (kb[:, :16] == SENT).all() and (kb[:, -16:] == SENT).all()
    cache = d["cos_sin"].numpy() if cache_dtype == torch.float32 else bits(d["cos_sin"])
    ref = rope.mla_rope_quantize_fp8(bits(d["q_rope"]), bits(d["k_rope"]), bits(d["q_nope"]),
                                     bits(d["k_nope"]), cache, pos_q.numpy(), pos_k.numpy(),
                                     neox, sq, skv,
                                     "f32" if cache_dtype == torch.float32 else "bf16")
    fr = []
    fr.append(_check_bytes(qb[..., 16 + 512:16 + 576], ref[0], what="q_rope"))
    fr.append(_check_bytes(kb[:, 16 + 512:16 + 576], ref[1], what="k_rope"))
    unit = sq == 1.0 and skv == 1.0
    fr.append(_check_bytes(qb[..., 16:16 + 512], ref[2], exact=unit, what="q_nope"))
    fr.append(_check_bytes(kb[:, 16:16 + 512], ref[3], exact=unit, what="k_nope"))
    return fr


@pytest.mark.parametrize("neox", [True, False])
@pytest.mark.parametrize("cache_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("pos_dtype", [torch.int32, torch.int64])
def test_rope_quantize_small(cuda, neox, cache_dtype, pos_dtype):
    _run(cuda, 70, nq=9, H=5, nk=300, max_seq=4096, neox=neox, cache_dtype=cache_dtype,
         pos_dtype=pos_dtype)


def test_rope_quantize_nonunit_scales(cuda):
    _run(cuda, 71, nq=6, H=16, nk=513, max_seq=2048, neox=True, cache_dtype=torch.float32,
         pos_dtype=torch.int32, sq=3.7, skv=0.3)


def test_rope_quantize_full_mla_prologue(cuda):
    """The MLA workload's prologue: 65536 key rows and 128 x 128 query rows."""
    fr = _run(cuda, 1003, nq=128, H=128, nk=65536, max_seq=65536, neox=True,
              cache_dtype=torch.float32, pos_dtype=torch.int32)
    print("ulp-off fractions (q_rope, k_rope, q_nope, k_nope):", fr)


def test_rope_position_out_of_range_is_reported(cuda):
    d = synth.mla_inputs(72, batch=2, heads=2, top_k=64, pool_rows=64, ctx_lo=64, ctx_hi=64,
                         max_seq_len=64)
    dev = {k: (v.to(cuda) if torch.is_tensor(v) else v) for k, v in d.items()}
    bskv.bskv_get_device_status(reset=True)
    pos = torch.tensor([3, 64], dtype=torch.int32, device=cuda)
    bskv.bskv_rope_quantize_fp8(dev["q_rope"], None, dev["q_nope"], None, dev["cos_sin"], pos)
    torch.cuda.synchronize()
    assert bskv.STATUS[bskv.bskv_get_device_status(reset=True)] == "ERR_DEVICE_INDEX"
    assert bskv.bskv_get_device_status() == 0


# ---------------------------------------------------------------------------------------
# RoPE + FP8 appended into a paged latent cache
# ---------------------------------------------------------------------------------------

def _append(cuda, d, neox=True, skv=1.0, batch_indices=None, positions=None):
    cache = d["kv_pages"].to(cuda).clone()
    bi = d["batch_indices"] if batch_indices is None else batch_indices
    pos = d["positions"] if positions is None else positions
    bskv.bskv_rope_quantize_fp8_append_paged(
        d["k_rope"].to(cuda), d["k_nope"].to(cuda), d["pos_k"].to(cuda), d["cos_sin"].to(cuda),
        bi.to(cuda), pos.to(cuda), d["kv_indptr"].to(cuda), d["kv_indices"].to(cuda), cache,
        is_neox=neox, quant_scale_kv=skv)
    torch.cuda.synchronize()
    return u8(cache)


def _append_ref(d, neox=True, skv=1.0):
    return rope.rope_quantize_fp8_append_paged(
        bits(d["k_rope"]), bits(d["k_nope"]), d["cos_sin"].cpu().numpy(), d["pos_k"].numpy(),
        d["batch_indices"].numpy(), d["positions"].numpy(), d["kv_indptr"].numpy(),
        d["kv_indices"].numpy(), u8(d["kv_pages"]), d["page_size"], neox, skv)


def _check_append(got, ref, d, exact_nope):
    """Untouched cache bytes identical; appended rows under the prologue's byte gate."""
    ps = d["page_size"]
    ip, ix = d["kv_indptr"].numpy(), d["kv_indices"].numpy()
    bi, pos = d["batch_indices"].numpy(), d["positions"].numpy()
    pages = ix[ip[bi] + pos // ps]
    slots = pos % ps
    touched = np.zeros(got.shape[:2], bool)
    touched[pages, slots] = True
    np.testing.assert_array_equal(got[~touched], ref[~touched])
    _check_bytes(got[pages, slots, 512:], ref[pages, slots, 512:], what="k_rope")
    _check_bytes(got[pages, slots, :512], ref[pages, slots, :512], exact=exact_nope, what="k_nope")


@pytest.mark.parametrize("ps,neox,skv", [(16, True, 1.0), (64, False, 1.0), (7, True, 0.75)])
def test_rope_append_paged_small(cuda, ps, neox, skv):
    d = synth.mla_append_inputs(31, batch=4, page_size=ps, len_lo=0, len_hi=0, new_tokens=9,
                                lens=[0, 15, 64, 200], max_seq_len=512)
    bskv.bskv_get_device_status(reset=True)
    got = _append(cuda, d, neox, skv)
    assert bskv.bskv_get_device_status() == 0
    _check_append(got, _append_ref(d, neox, skv), d, exact_nope=skv == 1.0)


def test_rope_append_paged_full_workload(cuda):
    """The benchmark's append: 128 requests x 512 new tokens into the page-64 cache."""
    d = synth.make("mla_append", device="cuda")
    bskv.bskv_get_device_status(reset=True)
    got = _append(cuda, d)
    assert bskv.bskv_get_device_status() == 0
    _check_append(got, _append_ref(d), d, exact_nope=True)


def test_rope_append_paged_bad_destination_is_reported(cuda):
    d = synth.mla_append_inputs(32, batch=2, page_size=16, len_lo=0, len_hi=0, new_tokens=4,
                                lens=[3, 20], max_seq_len=256)
    pos = d["positions"].clone()
    bi = d["batch_indices"].clone()
    pos[1] = 10 ** 6            # past the request's pages
    bi[5] = 7                   # no such request
    bskv.bskv_get_device_status(reset=True)
    got = _append(cuda, d, batch_indices=bi, positions=pos)
    assert bskv.STATUS[bskv.bskv_get_device_status(reset=True)] == "ERR_DEVICE_INDEX"
    ref = _append_ref(d)
    keep = [i for i in range(len(pos)) if i not in (1, 5)]
    ps = 16
    ip, ix = d["kv_indptr"].numpy(), d["kv_indices"].numpy()
    b0, p0 = d["batch_indices"].numpy(), d["positions"].numpy()
    for i in keep:   # the valid rows were written as usual
        pg, sl = ix[ip[b0[i]] + p0[i] // ps], p0[i] % ps
        _check_bytes(got[pg, sl], ref[pg, sl], what="row %d" % i)
    for i in (1, 5):  # the rejected rows' own slots keep their old bytes
        pg, sl = ix[ip[b0[i]] + p0[i] // ps], p0[i] % ps
        np.testing.assert_array_equal(got[pg, sl], u8(d["kv_pages"])[pg, sl])
