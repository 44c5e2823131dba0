"""Pins of the oracle's expert FFN, combine and INT4 dequantisation: a worked
example, an independent library computation (torch fp64), algebraic
invariants and a closed form.  CPU only."""
import numpy as np
import pytest
import torch

import oracle
import synth
from conftest import read_golden


def _vec(s):
    return np.array([float(v) for v in s.split()], np.float64)


def test_swiglu_worked_example():
    g = read_golden("swiglu_hand.txt")
    x = _vec(g["x"])
    wg = _vec(g["w_gate"]).reshape(2, 3)
    wu = _vec(g["w_up"]).reshape(2, 3)
    wd = _vec(g["w_down"]).reshape(3, 2)
    y = oracle.expert_ffn(x, wg, wu, wd)
    assert np.allclose(y, _vec(g["y"]), rtol=0, atol=1e-15)


def torch_expert(x, wg, wu, wd):
    """The same expert through torch's fp64 matmul and SiLU (a library routine)."""
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))
    h = torch.nn.functional.silu(t(wg) @ t(x)) * (t(wu) @ t(x))
    return (t(wd) @ h).numpy()


@pytest.mark.parametrize("d,F", [(8, 5), (64, 128), (96, 40)])
def test_expert_matches_library_fp64(d, F):
    rng = np.random.default_rng(d * F)
    x = rng.standard_normal(d).astype(np.float32)
    wg, wu = (rng.standard_normal((2, F, d)) / np.sqrt(d)).astype(np.float32)
    wd = (rng.standard_normal((d, F)) / np.sqrt(F)).astype(np.float32)
    y = oracle.expert_ffn(x, wg, wu, wd)
    ref = torch_expert(x, wg, wu, wd)
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-13)


def test_expert_algebra():
    """Linear in W_down and in W_up, not in W_gate; invariant under a shared
    permutation of the hidden units; W_down = I gives silu(g) * u."""
    rng = np.random.default_rng(1)
    d, F = 24, 24
    x = rng.standard_normal(d).astype(np.float32)
    wg, wu = rng.standard_normal((2, F, d)).astype(np.float32) * 0.2
    wd = rng.standard_normal((d, F)).astype(np.float32) * 0.2
    y = oracle.expert_ffn(x, wg, wu, wd)
    assert np.allclose(oracle.expert_ffn(x, wg, wu * 2, wd), 2 * y, rtol=1e-12, atol=1e-14)
    assert np.allclose(oracle.expert_ffn(x, wg, wu, wd * 4), 4 * y, rtol=1e-12, atol=1e-14)
    assert not np.allclose(oracle.expert_ffn(x, wg * 2, wu, wd), 2 * y, rtol=1e-3)
    pf = rng.permutation(F)
    assert np.allclose(oracle.expert_ffn(x, wg[pf], wu[pf], wd[:, pf]), y, rtol=1e-12, atol=1e-14)
    g = wg.astype(np.float64) @ x
    u = wu.astype(np.float64) @ x
    eye = np.eye(d, dtype=np.float32)
    closed = g / (1.0 + np.exp(-g)) * u
    assert np.allclose(oracle.expert_ffn(x, wg, wu, eye), closed, rtol=1e-12, atol=1e-14)


def test_combine_is_weighted_sum_in_slot_order():
    """out_i = sum_j w_ij y_{e_ij}(x_i) (kept, renormalised scores weight the
    expert outputs; OEA page, section 2 Q2); unused slots (-1) add nothing."""
    rng = np.random.default_rng(2)
    B, N, d, F = 3, 5, 16, 12
    x = rng.standard_normal((B, d)).astype(np.float32)
    wg, wu = rng.standard_normal((2, N, F, d)).astype(np.float32) * 0.3
    wd = rng.standard_normal((N, d, F)).astype(np.float32) * 0.3
    idx = np.array([[4, 0, -1], [1, 1, 2], [3, -1, -1]], np.int32)
    w = np.array([[0.7, 0.3, 0.0], [0.5, 0.25, 0.25], [1.0, 0.0, 0.0]])
    out = oracle.moe_experts(x, wg, wu, wd, idx, w)
    for i in range(B):
        ref = np.zeros(d)
        for j in range(3):
            if idx[i, j] >= 0:
                e = idx[i, j]
                ref += w[i, j] * torch_expert(x[i], wg[e], wu[e], wd[e])
        assert np.allclose(out[i], ref, rtol=1e-12, atol=1e-14)


def test_router_logits_match_library():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((7, 40)).astype(np.float32)
    wr = rng.standard_normal((9, 40)).astype(np.float32)
    b = rng.standard_normal(9).astype(np.float32)
    lg = oracle.router_logits(x, wr, b)
    ref = (torch.from_numpy(x.astype(np.float64)) @ torch.from_numpy(wr.astype(np.float64)).T
           + torch.from_numpy(b.astype(np.float64))).numpy()
    assert np.allclose(lg, ref, rtol=1e-13, atol=1e-13)
    assert np.allclose(oracle.router_logits(x, wr), ref - b, rtol=1e-13, atol=1e-13)


def pack_by_definition(q, s, rb):
    """The packed format built byte by byte from its definition (a second,
    independent construction): chunks of rb rows x 128 columns (one scale
    group), codes then one bf16 scale per row."""
    R, K = q.shape
    out = bytearray()
    for rbi in range(R // rb):
        for kb in range(K // 128):
            codes = bytearray(rb * 64)
            for rr in range(rb):
                r = rbi * rb + rr
                for cl in range(128):
                    o = cl % 8
                    bit = 4 * (o // 2) + 16 * (o % 2)
                    word_off = rr * 64 + (cl // 8) * 4
                    v = (int(q[r, kb * 128 + cl]) + 8) << bit
                    for byte in range(4):
                        codes[word_off + byte] |= (v >> (8 * byte)) & 0xFF
            scales = bytearray()
            for rr in range(rb):
                group = kb
                bits = int(synth.to_bf16_bits(np.array([s[rbi * rb + rr, group]], np.float32))[0])
                scales += bytes([bits & 0xFF, bits >> 8])
            out += codes + scales
    return np.frombuffer(bytes(out), np.uint8)


def test_dequant_int4_codes_and_layout():
    """Every code -7..7 at every nibble position, four 128-column groups per
    row with their own scales, several row and column chunks: w = q * s
    (DynaExq page, section 3.2, INT4 tier)."""
    rng = np.random.default_rng(6)
    rows, cols, rb = 32, 512, 16
    q = rng.integers(-7, 8, size=(rows, cols)).astype(np.int8)
    q[0, :15] = np.arange(-7, 8)
    s = synth.round_bf16(rng.uniform(0.01, 2.0, size=(rows, cols // 128)).astype(np.float32))
    packed = pack_by_definition(q, s, rb)
    assert np.array_equal(packed, synth.pack_int4_tiles(q, s, rb))
    out = oracle.dequant_int4(packed, rows, cols, rb)
    assert np.array_equal(out, (q * np.repeat(s, 128, axis=1)).astype(np.float32))


def test_int4_expert_bytes_are_half_a_byte_per_weight_plus_group_scales():
    """One expert at the Qwen3-30B-A3B shapes: 3 d d_ff / 2 code bytes and
    one bf16 scale per row and 128-column group, 2,433,024 bytes."""
    d, F = 2048, 768
    assert synth.int4_expert_bytes(d, F) == 3 * (d * F // 2 + d * F // 128 * 2) == 2_433_024
    rng = np.random.default_rng(1)
    g, u = (synth.round_bf16(rng.standard_normal((128, 256)).astype(np.float32)) for _ in range(2))
    dn = synth.round_bf16(rng.standard_normal((256, 128)).astype(np.float32))
    (pg, pu, pd), _ = synth.pack_int4_expert(g, u, dn)
    assert pg.size + pu.size + pd.size == synth.int4_expert_bytes(256, 128)


def test_int4_round_trip_within_half_step():
    """quantise -> pack -> dequantise reproduces each weight within half a
    quantisation step, and exactly where the weight is a multiple of it."""
    w = synth.normal(12, (64, 768), 0.03, True)
    q, s = synth.quantize_int4(w)
    out = oracle.dequant_int4(synth.pack_int4_tiles(q, s, 32), 64, 768, 32)
    step = np.repeat(s, 128, axis=1)
    assert (np.abs(out - w) <= step / 2 + 1e-12).all()
    assert (np.abs(q) <= 7).all() and (np.abs(q) == 7).any()
