"""Comparison helpers for the GPU parity tests (device result vs fp64 oracle).

Tolerances: the benchmark spec's bounds are max-abs <= 1e-4 (fp32 path) or <= 2e-2
(bf16 path) on Z, Y (and, by the same bf16 reading, on dQ, dK, dV), and
<= 1e-3 on L. Because many outputs here are much smaller than 2e-2 (Z is an
average over tens of thousands of tokens), each check also bounds the error
relative to the largest reference magnitude, so a wrong result cannot pass
by being small: rel 1e-4 (fp32) or 2e-2 (bf16). L, a log-normaliser of
magnitude ~10, is held to its absolute 1e-3.
"""
import numpy as np
import torch

ATOL = {"f32": 1e-4, "bf16": 2e-2}
REL = {"f32": 1e-4, "bf16": 2e-2}
L_ATOL = 1e-3


def to_np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().float().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def max_err(dev, ref):
    d, r = to_np(dev), to_np(ref)
    assert d.shape == r.shape, (d.shape, r.shape)
    ninf_r, ninf_d = np.isneginf(r), np.isneginf(d)
    assert np.array_equal(ninf_r, ninf_d), "-inf pattern differs"
    assert not np.isnan(d).any(), "NaN in device result"
    fin = ~ninf_r
    if not fin.any():
        return 0.0, 0.0
    return float(np.abs(d[fin] - r[fin]).max()), float(np.abs(r[fin]).max())


def assert_close(name, dev, ref, dtype, atol=None, rel=None):
    err, scale = max_err(dev, ref)
    atol = ATOL[dtype] if atol is None else atol
    rel = REL[dtype] if rel is None else rel
    assert err <= atol, f"{name}: max abs err {err:.3e} > {atol:.1e}"
    assert err <= rel * scale + 1e-30, f"{name}: max abs err {err:.3e} > {rel:.1e} x {scale:.3e}"
    return err


def assert_L_close(name, dev, ref):
    err, _ = max_err(dev, ref)
    assert err <= L_ATOL, f"{name}: max abs err {err:.3e} > {L_ATOL:.1e}"
    return err
