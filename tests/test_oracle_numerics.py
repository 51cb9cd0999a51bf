"""Pins of the oracle's number decoding and its E4M3 codec (CPU only).

The E4M3 encoder is pinned against a library routine (torch's float8_e4m3fn cast, which
rounds to nearest even and returns NaN past the range) wherever the two definitions
agree, and by the format's own invariants elsewhere.
"""

import numpy as np
import pytest
import torch

from oracle import numerics as nx


def test_bf16_decode_matches_torch():
    g = torch.Generator().manual_seed(1)
    x = torch.randn(100000, generator=g) * torch.exp(torch.randn(100000, generator=g) * 8)
    b = x.to(torch.bfloat16)
    bits = b.view(torch.int16).numpy().view(np.uint16)
    ref = b.to(torch.float64).numpy()
    np.testing.assert_array_equal(nx.bf16_bits_to_f64(bits), ref)


def test_fp16_decode_matches_numpy_every_code():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = nx.fp16_bits_to_f64(bits)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_e4m3_decode_all_codes_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = nx.e4m3_decode(codes)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()
    assert nx.e4m3_decode(np.array([0x7E], np.uint8))[0] == 448.0
    assert nx.e4m3_decode(np.array([0x01], np.uint8))[0] == 2.0 ** -9


def test_e4m3_roundtrip_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    vals = nx.e4m3_decode(codes)
    back = nx.e4m3_encode(vals)
    finite = ~np.isnan(vals)
    np.testing.assert_array_equal(nx.e4m3_decode(back)[finite], vals[finite])
    assert np.all((back[~finite] & 0x7F) == 0x7F)


def _torch_cast(x):
    return torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_matches_torch_dense_sweep_and_ties():
    g = np.random.default_rng(5)
    x = np.concatenate([
        g.standard_normal(200000) * np.exp2(g.uniform(-12, 9, 200000)),
        # every midpoint between adjacent representable magnitudes (ties to even)
        (lambda v: (v[:-1] + v[1:]) / 2)(np.unique(np.abs(nx.e4m3_decode(np.arange(0x7F, dtype=np.uint8))))),
        np.linspace(-448, 448, 20001),
    ])
    x = x[np.abs(x) <= 448]
    x = x.astype(np.float32).astype(np.float64)  # values torch can take exactly
    np.testing.assert_array_equal(nx.e4m3_encode(x), _torch_cast(x))


def test_e4m3_saturation_and_specials():
    x = np.array([449.0, 463.9, 464.0, 470.0, 1e9, np.inf, -1e9, -np.inf, np.nan, -0.0, 0.0])
    got = nx.e4m3_encode(x)
    assert list(got[:6]) == [0x7E] * 6
    assert list(got[6:8]) == [0xFE] * 2
    assert got[8] & 0x7F == 0x7F
    assert got[9] == 0x80 and got[10] == 0x00


def test_e4m3_ulp_distance():
    a = np.array([0x00, 0x80, 0x01, 0x81, 0x38, 0x7E], np.uint8)
    b = np.array([0x80, 0x00, 0x81, 0x01, 0x39, 0x7D], np.uint8)
    assert list(nx.e4m3_ulp_distance(a, b)) == [0, 0, 2, 2, 1, 1]


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_bits_dispatch(dt):
    t = torch.tensor([1.5, -2.25], dtype=torch.bfloat16 if dt == "bf16" else torch.float16)
    bits = t.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(nx.bits_to_f64(bits, dt), [1.5, -2.25])
