"""Expert residency policy (DynaExq page, sections 2.5 and 3.5): the
oracle's hotness update and selection with hysteresis pinned to their
definitions and closed forms, and the library's host-side selection compared
with the oracle.  CPU only."""
import itertools

import numpy as np
import pytest

import oracle

moe = pytest.importorskip("aware_expert_routing_gb300")


@pytest.fixture(scope="module")
def lib():
    from aware_expert_routing_gb300 import build as b
    b.build()
    return moe.load()


def test_ema_closed_form():
    """S_e <- alpha S_e + (1 - alpha) c_e from S = 0 with a constant count c
    gives S_t = c (1 - alpha^t)."""
    c = np.array([0.0, 1.0, 4.0, 9.0])
    S = np.zeros(4)
    for t in range(1, 30):
        S = oracle.ema_update(S, c, 0.9)
        assert np.allclose(S, c * (1 - 0.9 ** t), rtol=0, atol=1e-12)
    # one step from arbitrary scores: a convex combination
    S0 = np.array([5.0, 2.0, 0.0, 7.0])
    assert np.allclose(oracle.ema_update(S0, c, 0.25), 0.25 * S0 + 0.75 * c)


def by_pairing(S, in_hot, margin):
    """The selection stated another way: outsiders by score descending (ties
    to the lower id), members by score ascending (ties to the higher id);
    the leading pairs whose outsider scores more than `margin` above its
    member swap."""
    N = len(S)
    out = sorted((e for e in range(N) if not in_hot[e]), key=lambda e: (-S[e], e))
    ins = sorted((e for e in range(N) if in_hot[e]), key=lambda e: (S[e], -e))
    pro, dem = [], []
    for o, i in zip(out, ins):
        if not S[o] > S[i] + margin:
            break
        pro.append(o)
        dem.append(i)
    h = np.array(in_hot, bool).copy()
    h[pro] = True
    h[dem] = False
    return h, pro, dem


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("margin", [0.0, 0.5, 2.0])
def test_selection_matches_pairing(seed, margin):
    rng = np.random.default_rng(seed)
    N = 24
    S = (rng.integers(0, 8, N).astype(float) if seed % 3 == 0 else rng.exponential(3.0, N))   # ties when integer
    hot = np.zeros(N, bool)
    hot[rng.choice(N, 7, replace=False)] = True
    h, pro, dem = oracle.hot_select(S, hot, margin)
    h2, pro2, dem2 = by_pairing(S, hot, margin)
    assert np.array_equal(h, h2) and pro == pro2 and dem == dem2
    assert h.sum() == hot.sum()                                       # the budget holds
    assert set(pro) <= set(np.nonzero(~hot)[0]) and set(dem) <= set(np.nonzero(hot)[0])
    # afterwards no outsider scores more than the margin above a member
    assert S[~h].max() <= S[h].min() + margin


def test_margin_zero_gives_the_top_n():
    rng = np.random.default_rng(3)
    for _ in range(20):
        S = rng.normal(size=16)
        hot = np.zeros(16, bool)
        hot[rng.choice(16, 5, replace=False)] = True
        h, _, _ = oracle.hot_select(S, hot, 0.0)
        assert set(np.nonzero(h)[0]) == set(np.argsort(-S)[:5])


def test_worked_example_and_hysteresis():
    """Scores 5, 1, 3, 9, 2, 7 with members {0, 1, 2}: with margin 2.5,
    9 replaces 1 (9 > 1 + 2.5), 7 replaces 3 (7 > 3 + 2.5), and 3 does not
    replace 5 (3 < 5 + 2.5).  Scores within the margin of the set's edge
    move nothing."""
    S = np.array([5.0, 1.0, 3.0, 9.0, 2.0, 7.0])
    h, pro, dem = oracle.hot_select(S, [1, 1, 1, 0, 0, 0], 2.5)
    assert pro == [3, 5] and dem == [1, 2] and list(np.nonzero(h)[0]) == [0, 3, 5]
    base = np.array([4.0, 4.0, 4.0, 4.0, 4.0, 4.0])
    rng = np.random.default_rng(0)
    for _ in range(50):   # fluctuations of +-0.4 with a margin of 1: no swap ever
        h, pro, _ = oracle.hot_select(base + rng.uniform(-0.4, 0.4, 6), [1, 1, 0, 0, 1, 0], 1.0)
        assert pro == [] and list(np.nonzero(h)[0]) == [0, 1, 4]


def test_every_member_set_on_tiny_cases():
    """All 2-of-5 member sets of a few score vectors: the result is the one
    the pairing gives, and the budget holds."""
    for S in ([3, 1, 4, 1, 5], [2, 2, 2, 2, 2], [0, 9, 0, 9, 1]):
        S = np.array(S, float)
        for members in itertools.combinations(range(5), 2):
            hot = np.zeros(5, bool)
            hot[list(members)] = True
            for m in (0.0, 1.0):
                assert oracle.hot_select(S, hot, m)[1:] == by_pairing(S, hot, m)[1:]


@pytest.mark.parametrize("seed", range(10))
def test_library_selection_matches_oracle(lib, seed):
    rng = np.random.default_rng(100 + seed)
    N = 128
    S = rng.integers(0, 20, N).astype(float) if seed % 2 else rng.exponential(5.0, N)
    hot = np.zeros(N, bool)
    hot[rng.choice(N, 32, replace=False)] = True
    for margin in (0.0, 1.0, 4.0):
        h1, p1, d1 = moe.moe_residency_select(S, hot, margin)
        h2, p2, d2 = oracle.hot_select(S, hot, margin)
        assert np.array_equal(h1, h2) and p1 == p2 and d1 == d2
