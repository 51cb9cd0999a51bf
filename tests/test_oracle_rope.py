"""Pins of the oracle's RoPE + FP8 quantisation (CPU only).

Pins: position 0 is the identity rotation (bytes equal the plain cast); the two layouts
differ by a fixed permutation of the 64 tail values; each rotated pair keeps its norm;
the rotation equals multiplication by exp(i*angle) on the complex pair (closed form
from the cache's own angle definition); quant scales act as plain multipliers. The paged
append places exactly the prologue's key rows: read back through the page table in token
order they sit at their positions, every other cache byte is unchanged, and with
page_size 1 and pages in order the cache is the prologue's row array.
"""

import numpy as np
import pytest
import torch

import synth
from oracle import numerics as nx
from oracle import rope


def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def _inputs(seed=3, nq=5, H=3, nk=7, max_seq=64):
    d = synth.mla_inputs(seed, batch=nq, heads=H, top_k=64, pool_rows=max_seq, ctx_lo=64,
                         ctx_hi=64, max_seq_len=max_seq)
    return d


def test_position_zero_is_identity():
    d = _inputs()
    nq = d["q_rope"].shape[0]
    pos = np.zeros(nq, np.int64)
    qr, kr, qn, kn = rope.mla_rope_quantize_fp8(
        _bits(d["q_rope"]), _bits(d["k_rope"]), _bits(d["q_nope"]), _bits(d["k_nope"]),
        d["cos_sin"].numpy(), pos, np.zeros(d["k_rope"].shape[0], np.int64), True)
    np.testing.assert_array_equal(qr, nx.e4m3_encode(nx.bf16_bits_to_f64(_bits(d["q_rope"]))))
    np.testing.assert_array_equal(kr, nx.e4m3_encode(nx.bf16_bits_to_f64(_bits(d["k_rope"]))))
    np.testing.assert_array_equal(qn, nx.e4m3_encode(nx.bf16_bits_to_f64(_bits(d["q_nope"]))))
    # the plain cast agrees with torch's cast of the same bf16 values (in range here)
    np.testing.assert_array_equal(
        kn, d["k_nope"].to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def test_neox_and_interleaved_are_permutations_of_each_other():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((11, 64))
    ang = rng.uniform(0, 7, (11, 32))
    c, s = np.cos(ang), np.sin(ang)
    perm = np.empty(64, np.int64)  # neox position -> interleaved position
    perm[:32] = 2 * np.arange(32)
    perm[32:] = 2 * np.arange(32) + 1
    y_neox = rope.rotate(x, c, s, True)
    x_int = np.empty_like(x)
    x_int[:, perm] = x
    y_int = rope.rotate(x_int, c, s, False)
    np.testing.assert_allclose(y_int[:, perm], y_neox, rtol=0, atol=1e-15)


@pytest.mark.parametrize("neox", [True, False])
def test_rotation_scales_pair_norm_and_matches_complex_product(neox):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((9, 64))
    pos = rng.integers(0, 5000, 9)
    cache = synth.rope_cos_sin_cache(5000).numpy()
    c, s = rope.cache_rows(cache, pos)
    y = rope.rotate(x, c, s, neox)
    if neox:
        a, b, ya, yb = x[:, :32], x[:, 32:], y[:, :32], y[:, 32:]
    else:
        a, b, ya, yb = x[:, 0::2], x[:, 1::2], y[:, 0::2], y[:, 1::2]
    np.testing.assert_allclose(ya ** 2 + yb ** 2, (a ** 2 + b ** 2) * (c ** 2 + s ** 2), rtol=1e-12)
    # closed form: (a + ib) * exp(i*theta) with theta the angle stored in the cache
    theta = np.arctan2(s, c)
    z = (a + 1j * b) * np.exp(1j * theta) * np.hypot(c, s)
    np.testing.assert_allclose(ya, z.real, atol=1e-12)
    np.testing.assert_allclose(yb, z.imag, atol=1e-12)


def test_quant_scale_is_a_multiplier():
    d = _inputs(seed=9)
    pos_q = d["pos_q"].numpy()
    pos_k = d["pos_k"].numpy()
    a = rope.mla_rope_quantize_fp8(_bits(d["q_rope"]), _bits(d["k_rope"]), _bits(d["q_nope"]),
                                   _bits(d["k_nope"]), d["cos_sin"].numpy(), pos_q, pos_k,
                                   True, 0.5, 0.25)
    # scaling by a power of two commutes exactly with the rounding away from the ends
    b = rope.mla_rope_quantize_fp8(_bits(d["q_rope"]), _bits(d["k_rope"]), _bits(d["q_nope"]),
                                   _bits(d["k_nope"]), d["cos_sin"].numpy(), pos_q, pos_k,
                                   True, 1.0, 1.0)
    for x, y, sc in zip(a, b, (0.5, 0.25, 0.5, 0.25)):
        xv, yv = nx.e4m3_decode(x), nx.e4m3_decode(y)
        normal = np.abs(yv) >= 2.0 ** -4  # both far from the subnormal range
        np.testing.assert_array_equal(xv[normal], yv[normal] * sc)


def test_bad_position_rejected():
    d = _inputs()
    with pytest.raises(ValueError):
        rope.cache_rows(d["cos_sin"].numpy(), np.array([64]))


def _logical_rows(cache, indptr, indices, b, ps, n):
    """Rows [0, n) of request b in token order, gathered through the page table."""
    return np.stack([cache[indices[indptr[b] + t // ps], t % ps] for t in range(n)])


@pytest.mark.parametrize("ps,neox", [(16, True), (7, False)])
def test_paged_append_places_the_prologue_rows(ps, neox):
    d = synth.mla_append_inputs(21, batch=3, page_size=ps, len_lo=0, len_hi=0, new_tokens=5,
                                lens=[9, 0, 40], max_seq_len=128)
    cache0 = d["kv_pages"].numpy()
    ip, ix = d["kv_indptr"].numpy(), d["kv_indices"].numpy()
    bi, pos = d["batch_indices"].numpy(), d["positions"].numpy()
    new = rope.rope_quantize_fp8_append_paged(
        _bits(d["k_rope"]), _bits(d["k_nope"]), d["cos_sin"].numpy(), d["pos_k"].numpy(), bi, pos,
        ip, ix, cache0, ps, neox)
    _, kr, _, kn = rope.mla_rope_quantize_fp8(None, _bits(d["k_rope"]), None, _bits(d["k_nope"]),
                                              d["cos_sin"].numpy(), None, d["pos_k"].numpy(), neox)
    touched = np.zeros(cache0.shape[:2], bool)
    for b in range(3):
        n = int(pos[bi == b].max()) + 1 if (bi == b).any() else 0
        rows = _logical_rows(new, ip, ix, b, ps, n)
        old = _logical_rows(cache0, ip, ix, b, ps, n)
        for i in np.nonzero(bi == b)[0]:
            np.testing.assert_array_equal(rows[pos[i], :512], kn[i])
            np.testing.assert_array_equal(rows[pos[i], 512:], kr[i])
            touched[ix[ip[b] + pos[i] // ps], pos[i] % ps] = True
        keep = np.setdiff1d(np.arange(n), pos[bi == b])
        np.testing.assert_array_equal(rows[keep], old[keep])
    np.testing.assert_array_equal(new[~touched], cache0[~touched])


def test_paged_append_page_size_one_in_order_is_the_row_array():
    d = synth.mla_append_inputs(22, batch=2, page_size=1, len_lo=0, len_hi=0, new_tokens=3,
                                lens=[2, 4], max_seq_len=64)
    n_pages = d["num_pages"]
    ip = d["kv_indptr"].numpy()
    ix = np.arange(int(ip[-1]), dtype=np.int32)      # pages in order: row = indptr[b] + t
    cache0 = d["kv_pages"].numpy()
    bi, pos = d["batch_indices"].numpy(), d["positions"].numpy()
    new = rope.rope_quantize_fp8_append_paged(
        _bits(d["k_rope"]), _bits(d["k_nope"]), d["cos_sin"].numpy(), d["pos_k"].numpy(), bi, pos,
        ip, ix, cache0, 1)
    _, kr, _, kn = rope.mla_rope_quantize_fp8(None, _bits(d["k_rope"]), None, _bits(d["k_nope"]),
                                              d["cos_sin"].numpy(), None, d["pos_k"].numpy(), True)
    flat = new.reshape(n_pages, 576)
    for i in range(len(bi)):
        r = int(ip[bi[i]]) + int(pos[i])
        np.testing.assert_array_equal(flat[r], np.concatenate([kn[i], kr[i]]))
