"""The EMA hot-set selection (DynaExq page, section 2.5: per-expert counts,
S <- alpha*S + (1-alpha)*c every update, top-n_hi by S).  CPU only."""
import numpy as np

import aware_expert_routing_gb300 as moe


def test_ema_matches_closed_form_and_ties():
    rng = np.random.default_rng(0)
    c = rng.integers(0, 6, size=(200, 32)).astype(np.float64)
    T = c.shape[0]
    S = sum(0.1 * 0.9 ** (T - 1 - t) * c[t] for t in range(T))       # unrolled recurrence
    want = sorted(sorted(range(32), key=lambda e: (-S[e], e))[:8])
    assert list(moe.ema_hot_set(c, 8)) == want
    # equal scores: lower ids win
    flat = np.ones((5, 10))
    assert list(moe.ema_hot_set(flat, 3)) == [0, 1, 2]
    # recent counts weigh more than old ones
    c2 = np.zeros((3, 4))
    c2[0, 0] = 10
    c2[2, 1] = 10
    assert list(moe.ema_hot_set(c2, 1)) == [1]
