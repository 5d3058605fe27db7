"""Pins for the oracle's global-normaliser encoder backward (backward paragraphs of
the FLARE++ context-parallel appendix), CPU only: central finite differences,
torch autograd of the plain forward (a library routine), and invariants."""
import math

import numpy as np
import pytest
import torch

import oracle


def _problem(rng, B=2, H=2, M=3, N=12, D=4, pad=0.25):
    Q = rng.standard_normal((H, M, D))
    K = rng.standard_normal((B, N, H, D))
    V = rng.standard_normal((B, N, H, D))
    mask = (rng.random((B, N)) > pad).astype(np.uint8)
    dZ = rng.standard_normal((B, H, M, D))
    return Q, K, V, mask, dZ


def test_finite_differences():
    rng = np.random.default_rng(0)
    Q, K, V, mask, dZ = _problem(rng, B=1, N=7)
    Qb = np.broadcast_to(Q, (1,) + Q.shape).copy()          # per-batch query
    Z, L = oracle.encode(Qb, K, V, mask)
    dQ, dK, dV = oracle.encode_bwd(Qb, K, V, mask, Z, L, dZ)

    def J(q, k, v):
        return float((oracle.encode(q, k, v, mask)[0] * dZ).sum())

    eps = 1e-6
    for name, X, G in (("Q", Qb, dQ), ("K", K, dK), ("V", V, dV)):
        num = np.zeros_like(X)
        it = np.nditer(X, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            args = {"Q": (Qb, K, V), "K": (Qb, K, V), "V": (Qb, K, V)}[name]
            ap = [Xp if a is X else a for a in args]
            am = [Xm if a is X else a for a in args]
            num[idx] = (J(*ap) - J(*am)) / (2 * eps)
        np.testing.assert_allclose(G, num, atol=1e-7, err_msg=name)


def test_against_torch_autograd():
    rng = np.random.default_rng(1)
    B, H, M, N, D = 2, 3, 5, 40, 8
    Q, K, V, mask, dZ = _problem(rng, B, H, M, N, D)
    mask[1, :] = 0
    mask[1, 3] = 1                        # one valid key in batch element 1
    s = 1 / math.sqrt(D)
    Z, L = oracle.encode(Q, K, V, mask)
    dQ, dK, dV = oracle.encode_bwd(Q, K, V, mask, Z, L, dZ)

    q = torch.from_numpy(np.broadcast_to(Q, (B, H, M, D)).copy()).requires_grad_()
    k = torch.from_numpy(K).requires_grad_()
    v = torch.from_numpy(V).requires_grad_()
    am = torch.from_numpy(mask.astype(bool))[:, None, None, :]
    sc = (q @ k.permute(0, 2, 3, 1)) * s                  # [B,H,M,N]
    p = torch.softmax(sc.masked_fill(~am, -math.inf), dim=-1)
    z = p @ v.permute(0, 2, 1, 3)
    (z * torch.from_numpy(dZ)).sum().backward()
    np.testing.assert_allclose(dQ, q.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dK, k.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dV, v.grad.numpy(), atol=1e-12)


def test_gradient_invariants():
    """sum_n dS_mn = 0 per row, hence sum_n dK_n = 0 per (b, h); and by row
    stochasticity sum_n dV_n = sum over non-empty rows of dZ_m."""
    rng = np.random.default_rng(2)
    Q, K, V, mask, dZ = _problem(rng, B=2, H=2, M=4, N=30, D=5)
    mask[0, :] = 0                         # batch element 0: every row empty
    Z, L = oracle.encode(Q, K, V, mask)
    dQ, dK, dV = oracle.encode_bwd(Q, K, V, mask, Z, L, dZ)
    np.testing.assert_allclose(dK.sum(1), 0.0, atol=1e-12)
    expect = np.where(np.isfinite(L)[..., None], dZ, 0.0).sum(2)       # [B,H,D]
    np.testing.assert_allclose(dV.sum(1), expect, atol=1e-12)
    assert np.all(dQ[0] == 0) and np.all(dK[0] == 0) and np.all(dV[0] == 0)
    # masked tokens receive no gradient
    assert np.all(dK[mask == 0] == 0) and np.all(dV[mask == 0] == 0)


def test_shard_local_gradients_with_global_statistics_are_exact():
    """With the global Z, L each shard's dK_r, dV_r is the slice of the global
    gradient and dQ is the sum of the shards' contributions."""
    rng = np.random.default_rng(3)
    Q, K, V, mask, dZ = _problem(rng, N=40)
    Z, L = oracle.encode(Q, K, V, mask)
    dQ, dK, dV = oracle.encode_bwd(Q, K, V, mask, Z, L, dZ)
    off = [0, 9, 9, 31, 40]
    dQ_sum = np.zeros_like(dQ)
    for r in range(4):
        shard = np.zeros_like(mask)
        shard[:, off[r]:off[r + 1]] = mask[:, off[r]:off[r + 1]]
        dQr, dKr, dVr = oracle.encode_bwd(Q, K, V, shard, Z, L, dZ)
        np.testing.assert_allclose(dKr[:, off[r]:off[r + 1]], dK[:, off[r]:off[r + 1]], atol=1e-13)
        np.testing.assert_allclose(dVr[:, off[r]:off[r + 1]], dV[:, off[r]:off[r + 1]], atol=1e-13)
        dQ_sum += dQr
    np.testing.assert_allclose(dQ_sum, dQ, atol=1e-12)


def test_local_normaliser_backward_is_wrong():
    """A conventional per-shard SDPA backward (local L_r, local c_r) misses the
    between-shard term and must not reproduce the global gradient."""
    rng = np.random.default_rng(4)
    Q, K, V, mask, dZ = _problem(rng, N=40, pad=0.0)
    Z, L = oracle.encode(Q, K, V, mask)
    dQ, dK, dV = oracle.encode_bwd(Q, K, V, mask, Z, L, dZ)
    off = [0, 13, 40]
    O_r, L_r = oracle.encode_shards(Q, K, V, mask, off)
    dK_loc = np.zeros_like(dK)
    for r in range(2):
        shard = np.zeros_like(mask)
        shard[:, off[r]:off[r + 1]] = 1
        _, dKr, _ = oracle.encode_bwd(Q, K, V, shard, O_r[r], L_r[r], dZ)
        dK_loc[:, off[r]:off[r + 1]] = dKr[:, off[r]:off[r + 1]]
    assert np.abs(dK_loc - dK).max() > 1e-3
