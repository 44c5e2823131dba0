"""The latency-vs-T fit of bench.py (CPU): exact data gives the planted
coefficients and R^2 = 1; noise lowers R^2."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_linear_fit_recovers_plane():
    rng = np.random.default_rng(3)
    sum_cnt = rng.integers(1, 512, 40).astype(float)
    T = rng.integers(1, 128, 40).astype(float)
    y = 0.05 * sum_cnt + 1.4 * T + 9.0
    X = np.stack([sum_cnt, T, np.ones_like(T)], axis=1)
    f = bench.linear_fit(X, y)
    assert np.allclose(f["coef"], [0.05, 1.4, 9.0], rtol=1e-9, atol=1e-9)
    assert abs(f["r2"] - 1.0) < 1e-12
    g = bench.linear_fit(X, y + rng.normal(0, 5.0, 40))
    assert 0.5 < g["r2"] < 1.0


def test_linearity_points_are_distinct():
    """One token keeps at most k experts, so at B = 1 only T <= k is a new
    point: no (B, k, T) point repeats."""
    for B in (1, 4, 16, 64):
        pts = bench.linearity_points(8, 128, B)
        assert len(set(pts)) == len(pts)
        if B == 1:
            assert max(pts) <= 8
        else:
            assert max(pts) == 128


def test_strip_comments_keeps_code_and_literals():
    """The ncu record's source hash ignores comments and layout but not
    code: comment markers inside string or character literals are code."""
    src = ('int a = 1;  // one\n/* two\n   lines */ const char* s = "x // y /* z */";\n'
           "char q = '/'; char e = '\\''; const char* t = \"esc \\\" // still\";\n")
    got = bench.strip_comments(src)
    assert got == ('int a = 1; const char* s = "x // y /* z */"; char q = \'/\'; char e = \'\\\'\'; '
                   'const char* t = "esc \\" // still";')
    assert bench.strip_comments("a  =\n b; // c") == bench.strip_comments("a =  b;")
    assert bench.strip_comments("a = b;") != bench.strip_comments("a = c;")
    assert "record" not in bench.strip_comments("x = 1; // record\ny = 2;")
