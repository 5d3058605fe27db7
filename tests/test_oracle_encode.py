"""Pins for the oracle's encoder (eq. 18 of the FLARE++ context-parallel appendix)
and its per-shard form, CPU only: brute force, a library routine, closed forms
and invariants. None of them re-uses the oracle's own code."""
import math

import numpy as np
import pytest
import torch

import oracle


def _brute_encode(Q, K, V, mask, s):
    """Naive softmax without max subtraction, pure Python, tiny inputs only."""
    B, N, H, D = K.shape
    M = Q.shape[-2]
    Z = np.zeros((B, H, M, D))
    L = np.zeros((B, H, M))
    for b in range(B):
        for h in range(H):
            q = Q[h] if Q.ndim == 3 else Q[b, h]
            for m in range(M):
                w = []
                for n in range(N):
                    if mask is not None and not mask[b, n]:
                        continue
                    w.append((math.exp(s * sum(q[m, d] * K[b, n, h, d] for d in range(D))), n))
                tot = sum(x for x, _ in w)
                if not w:
                    L[b, h, m] = -math.inf
                    continue
                L[b, h, m] = math.log(tot)
                for x, n in w:
                    for d in range(D):
                        Z[b, h, m, d] += x / tot * V[b, n, h, d]
    return Z, L


@pytest.mark.parametrize("seed", range(5))
def test_brute_force_tiny(seed):
    rng = np.random.default_rng(seed)
    B, H = 2, 2
    M, N, D = int(rng.integers(1, 4)), int(rng.integers(1, 9)), int(rng.integers(1, 5))
    Q = rng.standard_normal((H, M, D))
    K = rng.standard_normal((B, N, H, D))
    V = rng.standard_normal((B, N, H, D))
    mask = (rng.random((B, N)) > 0.3).astype(np.uint8)
    mask[0, :] = 0                  # an empty batch element
    s = 1 / math.sqrt(D)
    Z, L = oracle.encode(Q, K, V, mask)
    Zb, Lb = _brute_encode(Q, K, V, mask, s)
    np.testing.assert_allclose(Z, Zb, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, Lb, rtol=0, atol=1e-12)


def _torch_sdpa_reference(Q, K, V, mask, s):
    """torch's scaled_dot_product_attention (math backend, fp64) as a library pin,
    plus torch.logsumexp of the masked scores."""
    B, N, H, D = K.shape
    q = torch.from_numpy(Q)
    q = q.expand(B, *q.shape) if q.dim() == 3 else q                   # [B,H,M,D]
    k = torch.from_numpy(K).permute(0, 2, 1, 3)                         # [B,H,N,D]
    v = torch.from_numpy(V).permute(0, 2, 1, 3)
    am = torch.from_numpy(mask.astype(bool))[:, None, None, :]          # [B,1,1,N]
    z = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=am, scale=s)
    sc = (q @ k.transpose(-1, -2)) * s
    lse = torch.logsumexp(sc.masked_fill(~am, -math.inf), dim=-1)
    return z.numpy(), lse.numpy()


@pytest.mark.parametrize("replicated", [True, False])
def test_against_library_sdpa(replicated):
    rng = np.random.default_rng(21)
    B, H, M, N, D = 2, 3, 5, 300, 16
    Q = rng.standard_normal((H, M, D) if replicated else (B, H, M, D)) * 2
    K = rng.standard_normal((B, N, H, D))
    V = rng.standard_normal((B, N, H, D))
    mask = (rng.random((B, N)) > 0.25).astype(np.uint8)
    s = 0.3
    Z, L = oracle.encode(Q, K, V, mask, scale=s)
    Zt, Lt = _torch_sdpa_reference(Q, K, V, mask, s)
    np.testing.assert_allclose(Z, Zt, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, Lt, rtol=0, atol=1e-12)


def test_default_scale_is_inverse_sqrt_d():
    rng = np.random.default_rng(2)
    Q = rng.standard_normal((1, 2, 9))
    K = rng.standard_normal((1, 7, 1, 9))
    V = rng.standard_normal((1, 7, 1, 9))
    Z1, L1 = oracle.encode(Q, K, V)
    Z2, L2 = oracle.encode(Q, K, V, scale=1 / 3)
    np.testing.assert_array_equal(Z1, Z2)
    np.testing.assert_array_equal(L1, L2)


def test_zero_query_gives_mean_of_valid_values():
    rng = np.random.default_rng(3)
    B, H, M, N, D = 2, 2, 3, 50, 4
    Q = np.zeros((H, M, D))
    K = rng.standard_normal((B, N, H, D))
    V = rng.standard_normal((B, N, H, D))
    mask = (rng.random((B, N)) > 0.4).astype(np.uint8)
    Z, L = oracle.encode(Q, K, V, mask)
    for b in range(B):
        valid = mask[b].astype(bool)
        for h in range(H):
            for m in range(M):
                np.testing.assert_allclose(Z[b, h, m], V[b, valid, h].mean(0), atol=1e-13)
                assert L[b, h, m] == pytest.approx(math.log(valid.sum()), abs=1e-13)


def test_single_valid_key_returns_its_value_and_score():
    rng = np.random.default_rng(4)
    B, H, M, N, D = 1, 1, 4, 10, 8
    Q = rng.standard_normal((H, M, D))
    K = rng.standard_normal((B, N, H, D))
    V = rng.standard_normal((B, N, H, D))
    mask = np.zeros((B, N), np.uint8)
    mask[0, 6] = 1
    Z, L = oracle.encode(Q, K, V, mask)
    s = 1 / math.sqrt(D)
    for m in range(M):
        np.testing.assert_allclose(Z[0, 0, m], V[0, 6, 0], atol=1e-15)
        assert L[0, 0, m] == pytest.approx(s * Q[0, m] @ K[0, 6, 0], abs=1e-13)


def test_identical_keys_give_uniform_weights():
    rng = np.random.default_rng(5)
    B, H, M, N, D = 1, 2, 3, 33, 6
    Q = rng.standard_normal((H, M, D))
    K = np.broadcast_to(rng.standard_normal((1, 1, H, D)), (B, N, H, D)).copy()
    V = rng.standard_normal((B, N, H, D))
    Z, L = oracle.encode(Q, K, V)
    s = 1 / math.sqrt(D)
    for h in range(H):
        for m in range(M):
            np.testing.assert_allclose(Z[0, h, m], V[0, :, h].mean(0), atol=1e-13)
            assert L[0, h, m] == pytest.approx(s * Q[h, m] @ K[0, 0, h] + math.log(N), abs=1e-12)


def test_rows_are_stochastic():
    """With V_n = e_n the encoder output row is the attention row: >= 0, sums to 1."""
    rng = np.random.default_rng(6)
    B, H, M, N = 2, 2, 4, 24
    D = N
    Q = rng.standard_normal((H, M, D)) * 3
    K = rng.standard_normal((B, N, H, D))
    V = np.zeros((B, N, H, D))
    for n in range(N):
        V[:, n, :, n] = 1.0
    mask = (rng.random((B, N)) > 0.3).astype(np.uint8)
    Z, _ = oracle.encode(Q, K, V, mask)
    assert (Z >= 0).all()
    np.testing.assert_allclose(Z.sum(-1), 1.0, atol=1e-13)
    # padded tokens get no weight
    for b in range(B):
        assert np.abs(Z[b][..., mask[b] == 0]).max(initial=0.0) == 0.0


def test_token_permutation_invariance():
    rng = np.random.default_rng(7)
    B, H, M, N, D = 2, 2, 3, 64, 8
    Q = rng.standard_normal((H, M, D))
    K = rng.standard_normal((B, N, H, D))
    V = rng.standard_normal((B, N, H, D))
    mask = (rng.random((B, N)) > 0.2).astype(np.uint8)
    perm = rng.permutation(N)
    Z, L = oracle.encode(Q, K, V, mask)
    Zp, Lp = oracle.encode(Q, K[:, perm], V[:, perm], mask[:, perm])
    np.testing.assert_allclose(Zp, Z, atol=1e-13)
    np.testing.assert_allclose(Lp, L, atol=1e-13)


def test_empty_rows_give_minus_inf_and_zero_not_nan():
    rng = np.random.default_rng(8)
    Q = rng.standard_normal((2, 3, 4))
    K = rng.standard_normal((2, 5, 2, 4))
    V = rng.standard_normal((2, 5, 2, 4))
    mask = np.ones((2, 5), np.uint8)
    mask[1] = 0
    Z, L = oracle.encode(Q, K, V, mask)
    assert np.all(L[1] == -np.inf) and np.all(Z[1] == 0)
    assert np.isfinite(L[0]).all()
    # an empty token range (an empty shard)
    Z, L = oracle.encode(Q, K, V, None, n_range=(3, 3))
    assert np.all(L == -np.inf) and np.all(Z == 0)


def test_large_scores_stay_finite_and_match_library():
    rng = np.random.default_rng(9)
    B, H, M, N, D = 1, 1, 4, 40, 8
    Q = rng.standard_normal((H, M, D)) * 60
    K = rng.standard_normal((B, N, H, D)) * 60
    V = rng.standard_normal((B, N, H, D))
    mask = np.ones((B, N), np.uint8)
    Z, L = oracle.encode(Q, K, V, mask)
    assert np.isfinite(Z).all() and np.isfinite(L).all()
    Zt, Lt = _torch_sdpa_reference(Q, K, V, mask, 1 / math.sqrt(D))
    np.testing.assert_allclose(Z, Zt, atol=1e-10)
    np.testing.assert_allclose(L, Lt, rtol=1e-14)


def test_bf16_and_f32_inputs_are_read_exactly():
    rng = np.random.default_rng(10)
    Q = torch.from_numpy(rng.standard_normal((2, 3, 8))).to(torch.bfloat16)
    K = torch.from_numpy(rng.standard_normal((1, 20, 2, 8))).to(torch.bfloat16)
    V = torch.from_numpy(rng.standard_normal((1, 20, 2, 8))).to(torch.bfloat16)
    Z1, L1 = oracle.encode(Q, K, V)
    Z2, L2 = oracle.encode(Q.double().numpy(), K.double().numpy(), V.double().numpy())
    Z3, L3 = oracle.encode(Q.float(), K.float(), V.float())
    np.testing.assert_array_equal(Z1, Z2)
    np.testing.assert_array_equal(L1, L2)
    np.testing.assert_array_equal(Z1, Z3)
    np.testing.assert_array_equal(L1, L3)


def test_row_subset_matches_full():
    rng = np.random.default_rng(12)
    Q = rng.standard_normal((2, 5, 4))
    K = rng.standard_normal((2, 30, 2, 4))
    V = rng.standard_normal((2, 30, 2, 4))
    Z, L = oracle.encode(Q, K, V)
    rows = np.array([0, 7, 13, 19])
    Zs, Ls = oracle.encode(Q, K, V, rows=rows)
    np.testing.assert_array_equal(Zs.reshape(-1, 4)[rows], Z.reshape(-1, 4)[rows])
    np.testing.assert_array_equal(Ls.reshape(-1)[rows], L.reshape(-1)[rows])
