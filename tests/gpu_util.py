"""Helpers shared by the GPU parity tests (comparison against the oracle)."""

import numpy as np
import torch


def bits(t):
    """Raw 16-bit patterns of a bf16/fp16 tensor as a host uint16 array."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def u8(t):
    return t.detach().contiguous().cpu().view(torch.uint8).numpy()


def to64(t):
    return t.detach().float().cpu().double().numpy()


def assert_close(got, ref, atol, rtol, what=""):
    """|got - ref| <= atol + rtol |ref| element-wise; returns error statistics."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    both_inf = np.isinf(ref) & (got == ref)
    with np.errstate(invalid="ignore"):
        err = np.where(both_inf, 0.0, np.abs(got - ref))
    bad = ~(err <= atol + rtol * np.abs(np.where(both_inf, 0.0, ref)))
    stats = dict(max_abs=float(np.nanmax(err)) if err.size else 0.0,
                 rel_fro=float(np.linalg.norm(np.nan_to_num(err)) / max(np.linalg.norm(np.nan_to_num(np.where(both_inf, 0, ref))), 1e-300)),
                 n_bad=int(bad.sum()), n=int(err.size))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d/%d outside tolerance (atol=%g rtol=%g); first %s got %s ref %s; %s"
                             % (what, bad.sum(), bad.size, atol, rtol, idx.tolist(),
                                got[tuple(idx.T)].tolist(), ref[tuple(idx.T)].tolist(), stats))
    return stats
