"""Pins for the oracle's local decode and the FLARE / FLARE++ compositions
(FLARE decode and FLARE++ paragraphs of the context-parallel appendix), CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle


def _brute_decode(Q, Z, K, s):
    B, N, H, D = K.shape
    M = Q.shape[-2]
    Y = np.zeros((B, N, H, D))
    for b in range(B):
        for n in range(N):
            for h in range(H):
                q = Q[h] if Q.ndim == 3 else Q[b, h]
                w = [math.exp(s * sum(K[b, n, h, d] * q[m, d] for d in range(D))) for m in range(M)]
                tot = sum(w)
                for m in range(M):
                    for d in range(D):
                        Y[b, n, h, d] += w[m] / tot * Z[b, h, m, d]
    return Y


def test_brute_force_tiny():
    rng = np.random.default_rng(0)
    B, H, M, N, D = 2, 2, 3, 5, 4
    Q = rng.standard_normal((H, M, D))
    Z = rng.standard_normal((B, H, M, D))
    K = rng.standard_normal((B, N, H, D))
    Y = oracle.decode(Q, Z, K)
    np.testing.assert_allclose(Y, _brute_decode(Q, Z, K, 0.5), atol=1e-13)


@pytest.mark.parametrize("replicated", [True, False])
def test_against_library_sdpa(replicated):
    """Decode = SDPA with the token keys as queries, Q as keys and Z as values."""
    rng = np.random.default_rng(1)
    B, H, M, N, D = 2, 3, 7, 50, 16
    Q = rng.standard_normal((H, M, D) if replicated else (B, H, M, D))
    Z = rng.standard_normal((B, H, M, D))
    K = rng.standard_normal((B, N, H, D)) * 2
    Y = oracle.decode(Q, Z, K)
    q = torch.from_numpy(K).permute(0, 2, 1, 3)                 # [B,H,N,D] as queries
    k = torch.from_numpy(Q)
    k = k.expand(B, *k.shape) if k.dim() == 3 else k              # [B,H,M,D] as keys
    yt = torch.nn.functional.scaled_dot_product_attention(q, k, torch.from_numpy(Z))
    np.testing.assert_allclose(Y, yt.permute(0, 2, 1, 3).numpy(), atol=1e-12)


def test_equal_latent_values_pass_through():
    rng = np.random.default_rng(2)
    B, H, M, N, D = 1, 2, 6, 20, 8
    Q = rng.standard_normal((H, M, D)) * 3
    z = rng.standard_normal((B, H, 1, D))
    Z = np.broadcast_to(z, (B, H, M, D)).copy()
    K = rng.standard_normal((B, N, H, D))
    Y = oracle.decode(Q, Z, K)
    for n in range(N):
        np.testing.assert_allclose(Y[0, n], z[0, :, 0], atol=1e-14)


def test_zero_query_gives_latent_mean():
    rng = np.random.default_rng(3)
    B, H, M, N, D = 2, 2, 5, 9, 4
    Z = rng.standard_normal((B, H, M, D))
    K = rng.standard_normal((B, N, H, D))
    Y = oracle.decode(np.zeros((H, M, D)), Z, K)
    for b in range(B):
        for n in range(N):
            np.testing.assert_allclose(Y[b, n], Z[b].mean(1), atol=1e-14)


def test_weights_are_stochastic():
    """With Z_m = e_m the decode output is the decode softmax row."""
    rng = np.random.default_rng(4)
    B, H, M, N = 1, 2, 6, 10
    D = M
    Q = rng.standard_normal((H, M, D)) * 4
    K = rng.standard_normal((B, N, H, D))
    Z = np.broadcast_to(np.eye(M), (B, H, M, D)).copy()
    Y = oracle.decode(Q, Z, K)
    assert (Y >= 0).all()
    np.testing.assert_allclose(Y.sum(-1), 1.0, atol=1e-14)


def test_token_subset_matches_full():
    rng = np.random.default_rng(5)
    B, H, M, N, D = 2, 2, 4, 30, 4
    Q = rng.standard_normal((H, M, D))
    Z = rng.standard_normal((B, H, M, D))
    K = rng.standard_normal((B, N, H, D))
    Y = oracle.decode(Q, Z, K)
    toks = np.array([0, 5, 29, 30, 59])
    Ys = oracle.decode(Q, Z, K, tokens=toks)
    np.testing.assert_array_equal(Ys, Y.reshape(B * N, H, D)[toks])


def test_flare_pp_composition_against_library():
    """FLARE++ = encoder(seeds) -> encoder(Q(X)) -> decode, each step a library SDPA."""
    rng = np.random.default_rng(6)
    B, H, M, N, D = 2, 2, 4, 40, 8
    Qs = rng.standard_normal((H, M, D))
    Kt, Vt, K, V = (rng.standard_normal((B, N, H, D)) for _ in range(4))
    mask = (rng.random((B, N)) > 0.2).astype(np.uint8)
    Qd, L1, Z, L2, Y = oracle.flare_pp_fwd(Qs, Kt, Vt, K, V, mask)

    def sdpa(q, k, v, am=None):
        return torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=am)

    t = lambda x: torch.from_numpy(x).permute(0, 2, 1, 3)        # [B,N,H,D] -> [B,H,N,D]
    am = torch.from_numpy(mask.astype(bool))[:, None, None, :]
    qd = sdpa(torch.from_numpy(Qs).expand(B, H, M, D), t(Kt), t(Vt), am)
    z = sdpa(qd, t(K), t(V), am)
    y = sdpa(t(K), qd, z).permute(0, 2, 1, 3)
    np.testing.assert_allclose(Qd, qd.numpy(), atol=1e-12)
    np.testing.assert_allclose(Z, z.numpy(), atol=1e-12)
    np.testing.assert_allclose(Y, y.numpy(), atol=1e-12)
    assert L1.shape == L2.shape == (B, H, M)


def test_shared_projection_flare_pp_reuses_tokens():
    """With K~ = K, V~ = V both encoders read the same tokens (shared-projection variant)."""
    rng = np.random.default_rng(7)
    B, H, M, N, D = 1, 2, 3, 25, 4
    Qs = rng.standard_normal((H, M, D))
    K, V = rng.standard_normal((B, N, H, D)), rng.standard_normal((B, N, H, D))
    Qd, L1, Z, L2, Y = oracle.flare_pp_fwd(Qs, K, V, K, V)
    Qd2, L1b = oracle.encode(Qs, K, V)
    np.testing.assert_array_equal(Qd, Qd2)
    np.testing.assert_array_equal(L1, L1b)
    Z2, L2b = oracle.encode(Qd, K, V)
    np.testing.assert_array_equal(Z, Z2)
