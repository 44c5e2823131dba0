"""Pins of the oracle's routing against what the OEA page and plain
mathematics fix: brute-force enumeration, closed forms, invariants and
special cases.  CPU only."""
import itertools
import math

import numpy as np
import pytest

import oracle
from conftest import read_golden

TOPK, OEA = oracle.TOPK, oracle.OEA


def dominates(l, a, b):
    """a must be ranked before b: larger score, or equal score and lower id."""
    return l[a] > l[b] or (l[a] == l[b] and a < b)


def brute_top(l, candidates, m):
    """The unique m-subset of `candidates` whose members all dominate the rest,
    found by enumerating every m-subset."""
    candidates = list(candidates)
    found = []
    for sub in itertools.combinations(candidates, m):
        rest = [e for e in candidates if e not in sub]
        if all(dominates(l, a, b) for a in sub for b in rest):
            found.append(set(sub))
    assert len(found) == 1
    return found[0]


def tied_logits(rng, B, N, levels=5):
    """Scores on a coarse grid so that ties are frequent."""
    return rng.integers(0, levels, size=(B, N)).astype(np.float32) * np.float32(0.25)


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_brute_force_with_ties(seed):
    rng = np.random.default_rng(seed)
    B, N, k = 5, 16, 4
    lg = tied_logits(rng, B, N) if seed % 2 else rng.standard_normal((B, N)).astype(np.float32)
    r = oracle.route(lg, TOPK, k)
    for i in range(B):
        want = brute_top(lg[i], range(N), k)
        assert set(r["idx"][i]) == want
        # slots are in ranked order
        for j in range(k - 1):
            assert dominates(lg[i], r["idx"][i][j], r["idx"][i][j + 1])


def softmax_prefix_count_fp64(l, p):
    """t_i by a different route: fp64 probabilities sorted by value; also
    returns the prefix sums so that callers can spot near-ties."""
    P = np.exp(l.astype(np.float64) - l.max())
    P /= P.sum()
    c = np.cumsum(np.sort(P)[::-1])
    if p >= 1:
        return len(l), c
    return int(np.searchsorted(c, p, side="left") + 1), c


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("k0,p,maxP,kmax", [(2, 0.5, 16, 4), (3, 1.0, 16, 4), (1, 0.3, 16, 4),
                                            (2, 0.7, 6, 4), (2, 1.0, 16, 6), (2, 0.6, 5, 5)])
def test_oea_matches_brute_force(seed, k0, p, maxP, kmax):
    """Phase 1 / union / phase 2 rebuilt from the OEA page's definitions
    (section 2 Q2, section 3) with subset enumeration."""
    rng = np.random.default_rng(100 + seed)
    B, N, k = 4, 12, 4
    lg = (tied_logits(rng, B, N, 6) if seed % 3 == 0
          else (rng.standard_normal((B, N)) * 1.5).astype(np.float32))
    r = oracle.route(lg, OEA, k, k0, p, maxP, kmax)
    # phase 1
    n = []
    for i in range(B):
        t, cum = softmax_prefix_count_fp64(lg[i], p)
        if p < 1 and np.min(np.abs(cum - p)) < 1e-4:
            pytest.skip("prefix within 1e-4 of p: decided by rounding")
        n.append(min(k0, t))
    assert list(r["nbase"]) == n
    check_union_and_phase2(lg, r, n, maxP, kmax)


def check_union_and_phase2(lg, r, n, maxP, kmax):
    """The union of the top-n_i baselines and the phase-2 picks, rebuilt
    from the OEA page's definitions (section 2 Q2, section 3) by subset
    enumeration, for given baseline sizes n_i."""
    B, N = lg.shape
    base = [brute_top(lg[i], range(N), n[i]) for i in range(B)]
    S_base = set().union(*base)
    assert r["T"] == len(S_base)
    # phase 2: candidates are in-union experts within rank maxP
    for i in range(B):
        depth_set = brute_top(lg[i], range(N), min(maxP, N)) | base[i]
        cand = (S_base & depth_set) - base[i]
        m = min(kmax - n[i], len(cand))
        want = base[i] | (brute_top(lg[i], cand, m) if m > 0 else set())
        got = [e for e in r["idx"][i] if e >= 0]
        assert set(got) == want and len(got) == len(want)
        # the token's top-n_i come first, in rank order
        assert set(got[:n[i]]) == base[i]


def test_topk_invariants_and_grouping():
    """cnt_e <= B, T <= N, sum cnt_e = B*k (OEA page, section 4, check 3);
    the per-expert grouping lists each (token, slot) exactly once."""
    rng = np.random.default_rng(7)
    for B in (1, 3, 16, 37):
        lg = rng.standard_normal((B, 128)).astype(np.float32)
        r = oracle.route(lg, TOPK, 8)
        cnt = r["counts"]
        assert cnt.max() <= B and r["T"] <= 128 and cnt.sum() == B * 8
        assert r["T"] == (cnt > 0).sum() == len(set(r["idx"].ravel()))
        assert list(r["active"]) == sorted(np.nonzero(cnt)[0])
        assert sorted(r["perm"]) == list(range(B * 8))
        for e in range(128):
            seg = r["perm"][r["offsets"][e]:r["offsets"][e + 1]]
            assert all(r["idx"].ravel()[q] == e for q in seg)
            assert list(seg // 8) == sorted(seg // 8)


@pytest.mark.parametrize("k0,p", [(3, 1.0), (5, 1.0), (5, 0.7), (2, 0.5)])
def test_oea_invariants(k0, p):
    """OEA page, section 2 Q2: phase 2 leaves T = |S_base| unchanged, every
    token keeps its top-n_i, picks only from S_base, keeps min(k, T) experts
    when maxP = N, and its renormalised weights sum to 1."""
    rng = np.random.default_rng(11)
    N, k = 128, 8
    for B in (1, 2, 16, 64):
        lg = rng.standard_normal((B, N)).astype(np.float32)
        r = oracle.route(lg, OEA, k, k0, p)
        base_union = set()
        for i in range(B):
            order = sorted(range(N), key=lambda e: (-lg[i][e], e))
            base_union |= set(order[:r["nbase"][i]])
        assert r["T"] == len(base_union)
        vt = oracle.route(lg, TOPK, k)
        assert r["T"] <= vt["T"]
        for i in range(B):
            order = sorted(range(N), key=lambda e: (-lg[i][e], e))
            got = [e for e in r["idx"][i] if e >= 0]
            assert got[:r["nbase"][i]] == order[:r["nbase"][i]]
            assert set(got) <= base_union
            assert len(got) == min(k, r["T"])
            assert abs(r["w"][i].sum() - 1.0) < 1e-12
        assert r["counts"].sum() == sum(min(k, r["T"]) for _ in range(B))


def test_weights_are_renormalised_scores():
    """Kept scores renormalised (OEA page, section 2 Q2): positive, summing to
    one, with ratios exp(l_a - l_b).  Worked case: kept scores ln 3 and ln 1
    give weights 3/4 and 1/4."""
    lg = np.full((1, 6), -50.0, np.float32)
    lg[0, 4], lg[0, 1] = math.log(3.0), 0.0
    r = oracle.route(lg, TOPK, 2)
    assert list(r["idx"][0]) == [4, 1]
    assert abs(r["w"][0][0] - 0.75) < 1e-7 and abs(r["w"][0][1] - 0.25) < 1e-7
    rng = np.random.default_rng(3)
    lg = rng.standard_normal((8, 32)).astype(np.float32)
    r = oracle.route(lg, OEA, 6, 3, 0.8)
    for i in range(8):
        ids = [e for e in r["idx"][i] if e >= 0]
        ws = r["w"][i][:len(ids)]
        assert (ws > 0).all() and abs(ws.sum() - 1) < 1e-12
        for a in range(len(ids)):
            assert abs(ws[a] / ws[0] - math.exp(float(lg[i][ids[a]]) - float(lg[i][ids[0]]))) < 1e-9


def test_top_p_worked_example():
    """Adaptive top-p count t_i (OEA page, section 2 Q2), worked by hand: softmax
    probabilities 0.5, 0.3, 0.2 (other experts negligible) have prefixes
    0.5, 0.8, 1.0, so t = 1 for p <= 0.5, t = 2 for 0.5 < p <= 0.8, t = 3 above.
    With k0 = 8 the baseline size n = t."""
    lg = np.full((1, 16), -1.0e4, np.float32)
    lg[0, 9], lg[0, 2], lg[0, 14] = math.log(0.5), math.log(0.3), math.log(0.2)
    for p, t in [(0.2, 1), (0.49, 1), (0.51, 2), (0.7, 2), (0.79, 2), (0.81, 3), (0.95, 3)]:
        r = oracle.route(lg, OEA, 8, 8, p)
        assert r["nbase"][0] == t, (p, t)
        assert list(r["idx"][0][:t]) == [9, 2, 14][:t]


def test_special_cases_reduce_to_known_routers():
    rng = np.random.default_rng(5)
    lg = rng.standard_normal((16, 64)).astype(np.float32)
    # k0 = k, top-p off: OEA is plain top-k (definitions in section 2 Q2 and section 5)
    a, b = oracle.route(lg, OEA, 8, 8, 1.0), oracle.route(lg, TOPK, 8)
    assert (a["idx"] == b["idx"]).all() and np.allclose(a["w"], b["w"])
    # B = 1: piggybacking adds nothing beyond the token's own top-n (section 7, detail 2)
    for k0 in (1, 3, 5):
        one = oracle.route(lg[:1], OEA, 8, k0, 1.0)
        pr = oracle.route(lg[:1], TOPK, k0)
        assert one["T"] == k0 and list(one["idx"][0][:k0]) == list(pr["idx"][0])
        assert (one["idx"][0][k0:] == -1).all()
    # p -> 0+: every baseline is the token's top-1
    r = oracle.route(lg, OEA, 8, 5, 1e-6)
    assert (r["nbase"] == 1).all()
    assert r["T"] == len(set(int(np.argmax(lg[i])) for i in range(16)))
    # identical tokens: the union is one token's top-k0, so T = k0 and all equal
    same = np.repeat(lg[:1], 8, axis=0)
    r = oracle.route(same, OEA, 8, 3, 1.0)
    assert r["T"] == 3 and (r["idx"] == r["idx"][0]).all()
    r = oracle.route(same, TOPK, 8)
    assert r["T"] == 8


def test_padding_tokens_select_nothing():
    """Padding mask (OEA page, section 7, detail 1): tokens past B_valid add
    no expert to the union and get no slot."""
    rng = np.random.default_rng(9)
    lg = rng.standard_normal((10, 32)).astype(np.float32)
    for mode in (TOPK, OEA):
        full = oracle.route(lg[:6], mode, 4, 2, 1.0)
        pad = oracle.route(lg, mode, 4, 2, 1.0, B_valid=6)
        assert pad["T"] == full["T"]
        assert (pad["idx"][:6] == full["idx"]).all() and (pad["idx"][6:] == -1).all()
        assert (pad["w"][6:] == 0).all() and (pad["counts"] == full["counts"]).all()


def expected_union(N, k, B):
    return N * (1.0 - (1.0 - k / N) ** B)


def test_uniform_union_closed_form_printed_value():
    g = read_golden("uniform_union.txt")
    N, k, B = int(g["N"]), int(g["k"]), int(g["B"])
    assert round(expected_union(N, k, B)) == int(g["expected_T_approx"])
    assert round(expected_union(N, k, B) / expected_union(N, k, 1)) == int(g["ratio_to_B1_approx"])


@pytest.mark.parametrize("B", [1, 4, 16, 64])
@pytest.mark.parametrize("mode,kk", [(TOPK, 8), (OEA, 3), (OEA, 5)])
def test_union_size_monte_carlo(B, mode, kk):
    """E[T] = N (1 - (1 - k/N)^B) under uniform routing (OEA page, section 4);
    for simplified OEA (top-p off, k^max = k) the union is that of the top-k0
    sets, so k0 replaces k.  i.i.d. scores make each token's ranking a
    uniformly random permutation."""
    rng = np.random.default_rng(1000 * B + kk)
    N, k = 128, 8
    trials = 300
    Ts = []
    for _ in range(trials):
        lg = rng.standard_normal((B, N)).astype(np.float32)
        r = oracle.route(lg, mode, k, kk if mode == OEA else None, 1.0)
        Ts.append(r["T"])
    Ts = np.array(Ts, np.float64)
    want = expected_union(N, kk if mode == OEA else k, B)
    se = max(Ts.std(ddof=1) / math.sqrt(trials), 1e-9)
    assert abs(Ts.mean() - want) < 4.5 * se + 1e-9, (Ts.mean(), want, se)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("k0,maxP,kmax", [(2, 12, 4), (3, 6, 4), (3, 12, 6)])
def test_given_baseline_sizes_follow_the_definitions(seed, k0, maxP, kmax):
    """Phase 1 with the baseline sizes n_i given (the n_base input): the
    union and phase 2 follow the definitions for those n_i, and passing the
    oracle's own n_i reproduces its routing exactly."""
    rng = np.random.default_rng(300 + seed)
    B, N, k = 5, 12, 4
    lg = (tied_logits(rng, B, N, 6) if seed % 3 == 0
          else (rng.standard_normal((B, N)) * 1.5).astype(np.float32))
    nb = rng.integers(1, k0 + 1, size=B).astype(np.int32)
    r = oracle.route(lg, OEA, k, k0, 0.6, maxP, kmax, nbase=nb)
    assert list(r["nbase"]) == list(nb)
    check_union_and_phase2(lg, r, list(nb), maxP, kmax)
    own = oracle.route(lg, OEA, k, k0, 0.6, maxP, kmax)
    again = oracle.route(lg, OEA, k, k0, 0.6, maxP, kmax, nbase=own["nbase"])
    for key in ("idx", "nbase", "counts", "offsets", "active", "perm"):
        assert np.array_equal(own[key], again[key])
    assert own["T"] == again["T"] and np.array_equal(own["w"], again["w"])
    with pytest.raises(ValueError):
        oracle.route(lg, OEA, k, k0, 0.6, maxP, kmax, nbase=np.full(B, k0 + 1, np.int32))


def test_batch_size_policy():
    """Batch-size-dependent k0 (OEA page, section 7, implementation detail 2):
    piggybacking adds nothing for one token, so OEA is off there (plain
    top-k, top-p off); smaller batches keep a larger, safer k0 than larger
    ones; for k = 8 the two values are the page's settings k0 = 5 and
    k0 = 3.  k0 <= 0 in a routing call applies the policy."""
    for k in (1, 4, 8, 16):
        assert oracle.policy_k0(1, k, 0.7) == (k, 1.0)
        assert oracle.policy_k0(0, k, 0.7) == (k, 1.0)
        ks = [oracle.policy_k0(B, k, 0.7)[0] for B in range(1, 257)]
        assert all(a >= b for a, b in zip(ks, ks[1:])) and all(1 <= x <= k for x in ks)
    assert {oracle.policy_k0(B, 8)[0] for B in range(2, 16)} == {5}
    assert {oracle.policy_k0(B, 8)[0] for B in range(16, 257)} == {3}
    k0, p = oracle.policy_k0(4, 8, 0.7)
    assert abs(p - 0.7) < 1e-7
    rng = np.random.default_rng(17)
    lg = rng.standard_normal((64, 128)).astype(np.float32)
    one = oracle.route(lg[:1], OEA, 8, 0, 0.7)
    plain = oracle.route(lg[:1], TOPK, 8)
    assert one["T"] == 8 and np.array_equal(one["idx"], plain["idx"])
    assert np.allclose(one["w"], plain["w"], rtol=0, atol=1e-15)
    padded = oracle.route(lg[:5], OEA, 8, 0, 1.0, B_valid=1)   # one real token, four padding
    assert padded["T"] == 8 and np.array_equal(padded["idx"][0], plain["idx"][0])
    for B in (2, 4, 15, 16, 64):
        k0, _ = oracle.policy_k0(B, 8, 0.9)
        a, b = oracle.route(lg[:B], OEA, 8, 0, 0.9), oracle.route(lg[:B], OEA, 8, k0, 0.9)
        assert np.array_equal(a["idx"], b["idx"]) and a["T"] == b["T"]
        assert (a["nbase"] <= k0).all()


def test_invalid_arguments_rejected():
    lg = np.zeros((2, 8), np.float32)
    with pytest.raises(ValueError):
        oracle.route(lg, TOPK, 9)
    with pytest.raises(ValueError):
        oracle.route(lg, OEA, 4, 5, 1.0)
    with pytest.raises(ValueError):
        oracle.route(lg, OEA, 4, 2, 0.0)
    with pytest.raises(ValueError):
        oracle.route(lg, OEA, 4, 2, 1.0, nbase=np.zeros(2, np.int32))
