"""Online-softmax normaliser state and its merge -- test infrastructure.

Source: "Ring vs. Tree Attention", section "The shared building block: the
online-softmax merge" and the Proposition that the merge is a commutative
semigroup. A state (m, l) stands for a set of scores s_i with running maximum
m and l = sum_i exp(s_i - m). Two states of disjoint score sets combine as
m = max(m1, m2), l = l1 exp(m1 - m) + l2 exp(m2 - m).

The empty set is the state (-inf, 0); it is the identity of the merge (a
reading: the page does not name an identity, but it is what the definition of
l gives for no scores). Pure Python floats, used by the merge tests only.
"""
from __future__ import annotations

import math
from typing import Iterable, Sequence, Tuple

State = Tuple[float, float]
EMPTY: State = (-math.inf, 0.0)


def state_of(scores: Iterable[float]) -> State:
    """The (m, l) state of a finite set of scores, straight from its definition."""
    scores = list(scores)
    if not scores:
        return EMPTY
    m = max(scores)
    return m, sum(math.exp(x - m) for x in scores)


def merge(a: State, b: State) -> State:
    """Combine two states of disjoint score sets (page's merge rule)."""
    m1, l1 = a
    m2, l2 = b
    m = max(m1, m2)
    if m == -math.inf:
        return EMPTY
    w1 = 0.0 if m1 == -math.inf else l1 * math.exp(m1 - m)
    w2 = 0.0 if m2 == -math.inf else l2 * math.exp(m2 - m)
    return m, w1 + w2


def fold_left(states: Sequence[State]) -> State:
    """Ring schedule: merge the states one after another, left to right."""
    acc = EMPTY
    for s in states:
        acc = merge(acc, s)
    return acc


def fold_tree(states: Sequence[State]) -> State:
    """Tree schedule: merge neighbouring pairs, round after round."""
    level = list(states) or [EMPTY]
    while len(level) > 1:
        nxt = [merge(level[i], level[i + 1]) for i in range(0, len(level) - 1, 2)]
        if len(level) % 2:
            nxt.append(level[-1])
        level = nxt
    return level[0]


def log_normaliser(state: State) -> float:
    """log sum_i exp(s_i) of the state's scores (m + log l)."""
    m, l = state
    return -math.inf if l == 0.0 else m + math.log(l)
