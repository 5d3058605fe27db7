"""Pins for the oracle's mixer backward passes (FLARE and FLARE++), CPU only.

The chain is the one of the appendix's backward paragraphs (the decode's
gradient of Z summed first, then the encoder with its own saved statistics;
for FLARE++ the decode's and the physical-value encoder's gradients of Q(X)
summed and sent through the query-synthesis encoder). It is pinned against
central finite differences of <dY, Y> through the oracle's own forward, and
against torch autograd of a plain torch mixer (a library routine), both with a
padding mask so that padded tokens (which still decode) are covered."""
import math

import numpy as np
import torch

import oracle


def _fd(J, X, eps=1e-6):
    num = np.zeros_like(X)
    it = np.nditer(X, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        Xp, Xm = X.copy(), X.copy()
        Xp[idx] += eps
        Xm[idx] -= eps
        num[idx] = (J(Xp) - J(Xm)) / (2 * eps)
    return num


def _mask(B, N, rng):
    m = (rng.random((B, N)) > 0.25).astype(np.uint8)
    m[:, 0] = 1
    return m


def test_flare_bwd_finite_differences():
    rng = np.random.default_rng(40)
    B, H, M, N, D = 2, 1, 3, 6, 2
    Q = rng.standard_normal((B, H, M, D))
    K = rng.standard_normal((B, N, H, D))
    V = rng.standard_normal((B, N, H, D))
    dY = rng.standard_normal((B, N, H, D))
    mask = _mask(B, N, rng)
    Z, L, _ = oracle.flare_fwd(Q, K, V, mask)
    dQ, dK, dV = oracle.flare_bwd(Q, K, V, mask, Z, L, dY)

    def J(q, k, v):
        return float((oracle.flare_fwd(q, k, v, mask)[2] * dY).sum())

    np.testing.assert_allclose(dQ, _fd(lambda x: J(x, K, V), Q), atol=1e-7)
    np.testing.assert_allclose(dK, _fd(lambda x: J(Q, x, V), K), atol=1e-7)
    np.testing.assert_allclose(dV, _fd(lambda x: J(Q, K, x), V), atol=1e-7)
    # padded tokens carry no value gradient but keep the decode's key gradient
    pad = mask == 0
    assert pad.any()
    np.testing.assert_allclose(dV[pad], 0.0, atol=1e-12)
    assert np.abs(dK[pad]).max() > 1e-6


def _torch_encode(q, k, v, mask, s):
    # q [B,H,M,D] or [H,M,D]; k, v [B,N,H,D]
    kk, vv = k.permute(0, 2, 1, 3), v.permute(0, 2, 1, 3)
    t = (q @ kk.transpose(-1, -2)) * s                          # [B,H,M,N]
    if mask is not None:
        t = t.masked_fill(~mask.bool()[:, None, None, :], float("-inf"))
    return torch.softmax(t, dim=-1) @ vv


def _torch_decode(q, z, k, s):
    kk = k.permute(0, 2, 1, 3)                                  # [B,H,N,D]
    a = torch.softmax((kk @ q.transpose(-1, -2)) * s, dim=-1)   # [B,H,N,M]
    return (a @ z).permute(0, 2, 1, 3)                          # [B,N,H,D]


def test_flare_bwd_against_torch_autograd():
    rng = np.random.default_rng(41)
    B, H, M, N, D = 2, 3, 5, 40, 8
    s = 1 / math.sqrt(D)
    Q = rng.standard_normal((H, M, D))
    K = rng.standard_normal((B, N, H, D))
    V = rng.standard_normal((B, N, H, D))
    dY = rng.standard_normal((B, N, H, D))
    mask = _mask(B, N, rng)
    Z, L, _ = oracle.flare_fwd(Q, K, V, mask)
    dQ, dK, dV = oracle.flare_bwd(Q, K, V, mask, Z, L, dY)
    q, k, v = (torch.from_numpy(x).requires_grad_() for x in (Q, K, V))
    tm = torch.from_numpy(mask)
    y = _torch_decode(q, _torch_encode(q, k, v, tm, s), k, s)
    (y * torch.from_numpy(dY)).sum().backward()
    # a replicated Q's gradient is returned per batch element
    np.testing.assert_allclose(dQ.sum(0), q.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dK, k.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dV, v.grad.numpy(), atol=1e-11)


def test_flare_pp_bwd_finite_differences():
    rng = np.random.default_rng(42)
    B, H, M, N, D = 2, 1, 3, 5, 2
    Qs = rng.standard_normal((H, M, D))
    Kt, Vt, K, V, dY = (rng.standard_normal((B, N, H, D)) for _ in range(5))
    mask = _mask(B, N, rng)
    Qd, L1, Z, L2, _ = oracle.flare_pp_fwd(Qs, Kt, Vt, K, V, mask)
    dQs, dKt, dVt, dK, dV, dQd = oracle.flare_pp_bwd(Qs, Kt, Vt, K, V, mask, Qd, L1, Z, L2, dY)

    def J(qs, kt, vt, k, v):
        return float((oracle.flare_pp_fwd(qs, kt, vt, k, v, mask)[4] * dY).sum())

    args = [Qs, Kt, Vt, K, V]
    for i, G in enumerate((dQs, dKt, dVt, dK, dV)):
        def Ji(x, i=i):
            a = list(args)
            a[i] = x
            return J(*a)
        num = _fd(Ji, args[i])
        got = G.sum(0) if i == 0 else G          # per batch element -> replicated seeds
        np.testing.assert_allclose(got, num, atol=1e-7, err_msg=str(i))


def test_flare_pp_bwd_against_torch_autograd():
    rng = np.random.default_rng(43)
    B, H, M, N, D = 2, 2, 4, 30, 8
    s = 1 / math.sqrt(D)
    Qs = 0.3 * rng.standard_normal((H, M, D))
    Kt, Vt, K, V, dY = (rng.standard_normal((B, N, H, D)) for _ in range(5))
    mask = _mask(B, N, rng)
    Qd, L1, Z, L2, _ = oracle.flare_pp_fwd(Qs, Kt, Vt, K, V, mask)
    dQs, dKt, dVt, dK, dV, dQd = oracle.flare_pp_bwd(Qs, Kt, Vt, K, V, mask, Qd, L1, Z, L2, dY)
    ts = [torch.from_numpy(x).requires_grad_() for x in (Qs, Kt, Vt, K, V)]
    tm = torch.from_numpy(mask)
    qd = _torch_encode(ts[0], ts[1], ts[2], tm, s)
    qd.retain_grad()
    z = _torch_encode(qd, ts[3], ts[4], tm, s)
    y = _torch_decode(qd, z, ts[3], s)
    (y * torch.from_numpy(dY)).sum().backward()
    np.testing.assert_allclose(dQs.sum(0), ts[0].grad.numpy(), atol=1e-11)
    for G, t in zip((dKt, dVt, dK, dV), ts[1:]):
        np.testing.assert_allclose(G, t.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dQd, qd.grad.numpy(), atol=1e-11)


def test_flare_pp_bwd_needs_both_query_gradient_shares():
    """Dropping either share of dQ(X) (the decode's or the physical-value
    encoder's) changes the seeds' and K~, V~ gradients: both terms matter."""
    rng = np.random.default_rng(44)
    B, H, M, N, D = 1, 1, 3, 12, 4
    Qs = rng.standard_normal((H, M, D))
    Kt, Vt, K, V, dY = (rng.standard_normal((B, N, H, D)) for _ in range(5))
    Qd, L1, Z, L2, _ = oracle.flare_pp_fwd(Qs, Kt, Vt, K, V)
    full = oracle.flare_pp_bwd(Qs, Kt, Vt, K, V, None, Qd, L1, Z, L2, dY)
    dQX_dec, dZ, _ = oracle.decode_bwd(Qd, Z, K, dY)
    dQX_enc, _, _ = oracle.encode_bwd(Qd, K, V, None, Z, L2, dZ)
    np.testing.assert_allclose(full[5], dQX_dec + dQX_enc, atol=1e-12)
    for part in (dQX_dec, dQX_enc):
        dQs_part = oracle.encode_bwd(Qs, Kt, Vt, None, Qd, L1, part)[0]
        assert np.abs(dQs_part - full[0]).max() > 1e-3
