"""Pins for the oracle's merges (CPU only).

The normaliser merge follows "Ring vs. Tree Attention" (the online-softmax
merge and its Proposition); the vector log-sum-exp merge follows eq. 23 and
the cross-rank log-sum-exp paragraph of the FLARE++ context-parallel appendix.
"""
import math
import os
import random

import numpy as np
import pytest

import oracle
from oracle import normalizer as nz

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "ring_tree_merge_exercise.txt")


def _read_exercise():
    fields = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            fields[key.strip()] = val.strip()
    states = [tuple(float(t) for t in s.split()) for s in fields["states"].split("|")]
    terms = {int(k): float(c) for k, c in (t.split(":") for t in fields["expected_l_terms"].split())}
    return states, float(fields["expected_m"]), terms


def test_page_exercise_ring_equals_tree_equals_closed_form():
    states, m_exp, terms = _read_exercise()
    assert len(states) == 8
    l_exp = sum(c * math.exp(-k) for k, c in terms.items())
    ring = nz.fold_left(states)
    tree = nz.fold_tree(states)
    assert ring[0] == m_exp and tree[0] == m_exp
    assert ring[1] == pytest.approx(l_exp, rel=1e-14)
    assert tree[1] == pytest.approx(l_exp, rel=1e-14)
    assert l_exp == pytest.approx(2.6889516522, abs=1e-10)


def test_state_of_matches_direct_log_sum_exp():
    rng = random.Random(3)
    s = [rng.uniform(-30, 30) for _ in range(50)]
    direct = math.log(sum(math.exp(x) for x in s))
    assert nz.log_normaliser(nz.state_of(s)) == pytest.approx(direct, rel=1e-14)


@pytest.mark.parametrize("seed", range(8))
def test_any_partition_any_order_any_tree(seed):
    rng = random.Random(seed)
    scores = [rng.gauss(0, 5) for _ in range(rng.randint(1, 200))]
    whole = nz.state_of(scores)
    # random disjoint partition (some parts empty)
    parts = [[] for _ in range(rng.randint(1, 12))]
    for x in scores:
        parts[rng.randrange(len(parts))].append(x)
    states = [nz.state_of(p) for p in parts]
    rng.shuffle(states)
    for res in (nz.fold_left(states), nz.fold_tree(states), _random_tree(states, rng)):
        assert res[0] == whole[0]
        assert res[1] == pytest.approx(whole[1], rel=1e-12)


def _random_tree(states, rng):
    pool = list(states)
    while len(pool) > 1:
        i = rng.randrange(len(pool) - 1)
        pool[i:i + 2] = [nz.merge(pool[i], pool[i + 1])]
    return pool[0]


def test_merge_commutes_and_empty_is_identity():
    a, b = (1.5, 2.0), (-0.25, 7.0)
    assert nz.merge(a, b) == nz.merge(b, a)
    assert nz.merge(a, nz.EMPTY) == a
    assert nz.merge(nz.EMPTY, nz.EMPTY) == nz.EMPTY


def test_double_counting_changes_the_state():
    # failure mode on the page: a score counted on two shards corrupts (m, l)
    scores = [0.3, 1.2, -0.7, 2.2]
    good = nz.fold_left([nz.state_of(scores[:2]), nz.state_of(scores[2:])])
    bad = nz.fold_left([nz.state_of(scores[:3]), nz.state_of(scores[2:])])
    assert bad[1] != pytest.approx(good[1], rel=1e-6)


# ---- vector merge, eq. 23 ------------------------------------------------------------

def _random_problem(rng, B=2, H=2, M=3, N=40, D=5, pad=0.2):
    Q = rng.standard_normal((H, M, D))
    K = rng.standard_normal((B, N, H, D))
    V = rng.standard_normal((B, N, H, D))
    mask = (rng.random((B, N)) > pad).astype(np.uint8)
    return Q, K, V, mask


def _random_offsets(rng, N, R):
    cuts = np.sort(rng.integers(0, N + 1, size=R - 1))
    return [0] + [int(c) for c in cuts] + [N]


@pytest.mark.parametrize("seed", range(6))
def test_split_encoder_equals_unsplit(seed):
    """eq. 18 == eq. 23: per-shard (O_r, L_r) merged equals the global encoder."""
    rng = np.random.default_rng(seed)
    Q, K, V, mask = _random_problem(rng)
    R = int(rng.integers(1, 9))
    off = _random_offsets(rng, K.shape[1], R)
    Z, L = oracle.encode(Q, K, V, mask)
    O_r, L_r = oracle.encode_shards(Q, K, V, mask, off)
    Zm, Lm = oracle.lse_merge(O_r, L_r)
    np.testing.assert_allclose(Zm, Z, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Lm, L, rtol=0, atol=1e-12)
    # shard order does not matter
    perm = rng.permutation(R)
    Zp, Lp = oracle.lse_merge(O_r[perm], L_r[perm])
    np.testing.assert_allclose(Zp, Z, rtol=0, atol=1e-12)
    np.testing.assert_allclose(Lp, L, rtol=0, atol=1e-12)


def test_vector_merge_normaliser_agrees_with_page_merge():
    """The L of eq. 23 is the log-normaliser of the page-3 merge of (L_r, 1)."""
    rng = np.random.default_rng(11)
    L_r = rng.normal(0, 4, size=(7, 1))
    O_r = rng.standard_normal((7, 1, 3))
    _, L = oracle.lse_merge(O_r, L_r)
    st = nz.fold_tree([(float(l), 1.0) for l in L_r[:, 0]])
    assert L[0] == pytest.approx(nz.log_normaliser(st), rel=1e-14)


def test_merge_of_one_shard_is_identity():
    rng = np.random.default_rng(5)
    O = rng.standard_normal((1, 4, 6))
    Lr = rng.standard_normal((1, 4))
    Z, L = oracle.lse_merge(O, Lr)
    np.testing.assert_array_equal(Z, O[0])
    np.testing.assert_array_equal(L, Lr[0])


def test_empty_shards_carry_no_mass_and_all_empty_is_empty():
    rng = np.random.default_rng(6)
    O = rng.standard_normal((3, 2, 4))
    Lr = rng.standard_normal((3, 2))
    O[1] = 0.0
    Lr[1] = -np.inf
    Z, L = oracle.lse_merge(O, Lr)
    Z2, L2 = oracle.lse_merge(O[[0, 2]], Lr[[0, 2]])
    np.testing.assert_allclose(Z, Z2, atol=1e-15)
    np.testing.assert_allclose(L, L2, atol=1e-15)
    Lr[:] = -np.inf
    O[:] = 0.0
    Z, L = oracle.lse_merge(O, Lr)
    assert np.all(L == -np.inf) and np.all(Z == 0.0) and not np.isnan(Z).any()


def test_double_counted_shard_changes_the_merge():
    rng = np.random.default_rng(8)
    Q, K, V, mask = _random_problem(rng, pad=0.0)
    off = [0, 15, 40]
    O_r, L_r = oracle.encode_shards(Q, K, V, mask, off)
    Z, L = oracle.lse_merge(O_r, L_r)
    Zd, Ld = oracle.lse_merge(O_r[[0, 1, 1]], L_r[[0, 1, 1]])
    assert np.abs(Ld - L).max() > 1e-3
    assert np.abs(Zd - Z).max() > 1e-3
