"""Pins for the oracle's decode backward (the chain rule of the FLARE local
decode, whose formula the pages leave stripped), CPU only: central finite
differences of <dY, Y>, torch autograd of a plain decode (a library routine),
and the invariants the softmax over the latents fixes."""
import math

import numpy as np
import torch

import oracle


def _problem(rng, B=1, H=2, M=5, N=7, D=3):
    Q = rng.standard_normal((B, H, M, D))
    Z = rng.standard_normal((B, H, M, D))
    K = rng.standard_normal((B, N, H, D))
    dY = rng.standard_normal((B, N, H, D))
    return Q, Z, K, dY


def test_finite_differences():
    rng = np.random.default_rng(20)
    Q, Z, K, dY = _problem(rng)
    dQ, dZ, dK = oracle.decode_bwd(Q, Z, K, dY)

    def J(q, z, k):
        return float((oracle.decode(q, z, k) * dY).sum())

    eps = 1e-6
    for name, X, G in (("Q", Q, dQ), ("Z", Z, dZ), ("K", K, dK)):
        num = np.zeros_like(X)
        it = np.nditer(X, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            ap = [Xp if a is X else a for a in (Q, Z, K)]
            am = [Xm if a is X else a for a in (Q, Z, K)]
            num[idx] = (J(*ap) - J(*am)) / (2 * eps)
        np.testing.assert_allclose(G, num, atol=1e-7, err_msg=name)


def test_against_torch_autograd():
    rng = np.random.default_rng(21)
    B, H, M, N, D = 2, 3, 6, 30, 8
    Q, Z, K, dY = _problem(rng, B, H, M, N, D)
    s = 1 / math.sqrt(D)
    dQ, dZ, dK = oracle.decode_bwd(Q, Z, K, dY)
    q = torch.from_numpy(Q).requires_grad_()
    z = torch.from_numpy(Z).requires_grad_()
    k = torch.from_numpy(K).requires_grad_()
    t = (k.permute(0, 2, 1, 3) @ q.transpose(-1, -2)) * s        # [B,H,N,M]
    y = torch.softmax(t, dim=-1) @ z                               # [B,H,N,D]
    (y * torch.from_numpy(dY).permute(0, 2, 1, 3)).sum().backward()
    np.testing.assert_allclose(dQ, q.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dZ, z.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dK, k.grad.numpy(), atol=1e-12)


def test_invariants():
    """Softmax weights sum to one over the latents: sum_m dZ_m = sum_n dY_n;
    moving every latent query by the same vector leaves Y unchanged:
    sum_m dQ_m = 0; a constant dY (the same for all latents' outputs) meets
    equal Z rows and gives no score gradient: dK = dQ = 0."""
    rng = np.random.default_rng(22)
    Q, Z, K, dY = _problem(rng, B=2, H=2, M=7, N=25, D=5)
    dQ, dZ, dK = oracle.decode_bwd(Q, Z, K, dY)
    np.testing.assert_allclose(dZ.sum(2), dY.sum(1), atol=1e-12)
    np.testing.assert_allclose(dQ.sum(2), 0.0, atol=1e-12)
    Zc = np.broadcast_to(Z[:, :, :1], Z.shape).copy()              # equal Z rows
    dQc, dZc, dKc = oracle.decode_bwd(Q, Zc, K, dY)
    np.testing.assert_allclose(dKc, 0.0, atol=1e-12)
    np.testing.assert_allclose(dQc, 0.0, atol=1e-12)


def test_replicated_query_and_bf16_inputs():
    """A replicated [H,M,D] query gives the per-batch slices of the broadcast
    one; bf16 bit patterns are read exactly."""
    rng = np.random.default_rng(23)
    B, H, M, N, D = 2, 2, 4, 9, 4
    Q = rng.standard_normal((H, M, D))
    Z = rng.standard_normal((B, H, M, D))
    K = torch.randn((B, N, H, D), generator=torch.Generator().manual_seed(3)).bfloat16()
    dY = torch.randn((B, N, H, D), generator=torch.Generator().manual_seed(4)).bfloat16()
    a = oracle.decode_bwd(Q, Z, K, dY)
    b = oracle.decode_bwd(np.broadcast_to(Q, (B, H, M, D)).copy(), Z, K.double(), dY.double())
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, atol=1e-12)
