"""Parity of the CUDA path with the CPU oracle, through the C ABI.

Routing is compared bit-exactly against the oracle run on the GPU's own fp32
router scores; scores, weights and outputs within the stated tolerances.
Sizes are small enough for the oracle to finish in seconds but span several
tiles with ragged tails; the full-size workloads are checked on sampled
tokens."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("aware_expert_routing_gb300")
import gpu_util as gu  # noqa: E402

TOPK, OEA = 0, 1


@pytest.fixture(scope="module", autouse=True)
def built():
    from aware_expert_routing_gb300 import build as b
    b.build()
    oracle.build()
    assert torch.cuda.is_available()
    moe.load()


def W(name, **kw):
    base = dict(N=128, k=8, d=512, F=256, B=16, seed=11)
    base.update(kw)
    return synth.Workload(name, **base)


def run_case(w, B, mode, k0=None, p=1.0, maxP=0, kmax=0, B_valid=-1, L=None, check_e2e=True, alias_up=False):
    L = L if L is not None else synth.make_layer(w, 0, B)
    if alias_up:   # W_up is W_gate's own device buffer
        L = dict(L, w_up=L["w_gate"])
    D = gu.device_inputs(L, w.bf16)
    if alias_up:
        D["w_up"] = D["w_gate"]
    prm = gu.params_for(w, B, mode, k0, p, maxP, kmax, B_valid)
    r, out, ws, flags = gu.run_layer(w, D, prm)
    assert flags == 0, f"device flags {flags:#x}"
    g = gu.to_np(r)
    bv = B if B_valid < 0 else B_valid
    lg_ref = oracle.router_logits(L["x"], L["w_router"], L["bias"])
    if B:
        tol = (1e-3 if w.bf16 else 1e-5) * np.abs(lg_ref).max()
        assert np.abs(g["logits"] - lg_ref).max() <= tol
    ref = gu.check_routing(g, prm, bv)
    o = oracle.moe_experts(L["x"], L["w_gate"], L["w_up"], L["w_down"], g["expert_idx"],
                           g["weights"].astype(np.float64))
    if B:
        gu.check_output(out, o, w.bf16)
        if B_valid >= 0:
            assert (out[B_valid:].float() == 0).all()
    if check_e2e and B:
        # The oracle's own scores (fp64 sums rounded to fp32) give the same
        # routing whenever every token's top-(kmax+1) order is the same.
        own = oracle.route(lg_ref.astype(np.float32), OEA if mode == OEA else TOPK, prm.k, prm.k0,
                           prm.p, prm.maxP if 0 < prm.maxP < prm.N else prm.N,
                           prm.kmax if prm.kmax > 0 else prm.k, bv)
        depth = (prm.kmax if prm.kmax > 0 else prm.k) + 1
        same = all(np.array_equal(np.argsort(-g["logits"][i], kind="stable")[:depth],
                                  np.argsort(-lg_ref[i].astype(np.float32), kind="stable")[:depth])
                   for i in range(B))
        k0r, pr = gu.resolved_k0_p(prm, bv)
        if same and not gu.near_tie_tokens(lg_ref, pr, k0r, bv):
            assert own["T"] == g["T"] and np.array_equal(own["idx"], g["expert_idx"])
    return g, out, ref


# ---- the tiny fp32 layer (N=16, k=4, d=64, d_ff=128, B=4) -------------------
@pytest.mark.parametrize("mode,k0,p", [(TOPK, 4, 1.0), (OEA, 2, 0.5)])
def test_tiny_fp32_layer(mode, k0, p):
    w = synth.WORKLOADS["tiny_fp32_n16_k4_d64_f128_b4"]
    run_case(w, w.B, mode, k0, p)


# ---- bf16 layers at test sizes ------------------------------------------------
@pytest.mark.parametrize("mode,k0,p,zipf", [
    (TOPK, 8, 1.0, False), (OEA, 3, 1.0, False), (OEA, 5, 1.0, False), (OEA, 5, 0.7, True),
    (TOPK, 8, 1.0, True), (OEA, 1, 1.0, False), (OEA, 8, 1.0, False), (OEA, 4, 0.5, True)])
def test_bf16_layer_modes(mode, k0, p, zipf):
    w = W("t_modes", zipf=zipf)
    run_case(w, w.B, mode, k0, p)


@pytest.mark.parametrize("B", [1, 7, 37, 64, 256])
def test_bf16_ragged_batches(B):
    w = W("t_ragged", N=64, d=256, F=128, seed=12, zipf=True)
    run_case(w, B, OEA, 3, 0.7)
    run_case(w, B, TOPK)


@pytest.mark.parametrize("B", [16, 17, 32, 33, 48, 64, 65])
def test_whole_batch_boundaries(B):
    # Up to 64 tokens the whole batch is the phase-A operand: one chunk per
    # expert, each expert's tokens from the routing's two 32-token words,
    # and with OEA the early start.  65 tokens take the expert-grouped copy.
    # N = 512 keeps the routing kernel busy long enough for phase-B tiles to
    # be posted before it completes, when their MMA width (the chunk's token
    # count) is not yet known; Zipf routing gives chunks of many tokens.
    w = W("t_whole", N=512, k=8, d=512, F=256, seed=100 + B, zipf=True)
    run_case(w, B, OEA, 4, 1.0)
    run_case(w, B, TOPK)


@pytest.mark.parametrize("B,d,F", [(8, 512, 256), (16, 384, 128), (32, 512, 256), (48, 256, 384), (65, 512, 256),
                                   (130, 320, 192)])
def test_separate_gate_up_maps(B, d, F):
    # W_gate and W_up share one interleaving 5D tensor map when they lie
    # less than 2^40 bytes apart and not at the same address; otherwise
    # (separate allocations in distant address ranges, or here W_up passed
    # as W_gate's own buffer) the kernel loads each 8-row group of both
    # through 8-row maps, all of a stage's K blocks per load.  Stages of 4
    # (B=8), 2 and 1 (d=320, F=192) blocks; whole batches and the
    # expert-grouped copy.
    w = W("t_sep_gu", N=64, k=8, d=d, F=F, seed=300 + B, zipf=True)
    run_case(w, B, OEA, 3, 1.0, alias_up=True)
    run_case(w, B, TOPK, alias_up=True)


@pytest.mark.parametrize("N,k,d,F", [(16, 4, 64, 64), (160, 6, 320, 192), (1024, 8, 128, 64),
                                     (256, 16, 192, 320), (32, 32, 64, 128)])
def test_bf16_shapes(N, k, d, F):
    w = W("t_shapes", N=N, k=k, d=d, F=F, seed=N + d)
    run_case(w, 29, OEA, max(1, k // 2), 1.0)
    run_case(w, 29, TOPK)


@pytest.mark.parametrize("N", [128, 1024])
@pytest.mark.parametrize("maxP,p", [(0, 1.0), (5, 0.8)])
def test_route_full_cluster(N, maxP, p):
    # The largest batch: eight CTAs of 32 tokens (one or two per warp),
    # S_base and the per-expert counts gathered across all of them.
    w = W("t_cluster", N=N, k=8, d=128, F=64, seed=N + maxP, zipf=True)
    run_case(w, 256, OEA, 3, p, maxP=maxP, kmax=10, B_valid=250)
    run_case(w, 256, TOPK)


@pytest.mark.parametrize("N,k,d,F", [(32, 4, 320, 192), (64, 8, 384, 128), (128, 8, 512, 256),
                                     (16, 4, 256, 768)])
@pytest.mark.parametrize("B", [1, 6, 16])
def test_small_batch_stage_widths(N, k, d, F, B):
    # Batches of up to 16 tokens stream 1, 2 or 4 column blocks per stage
    # (the most that divides both d / 64 and d_ff / 64): every width, a
    # single token, a partial and a full batch.
    w = W("t_widths", N=N, k=k, d=d, F=F, seed=d + F + B)
    run_case(w, B, OEA, max(1, k // 2), 1.0)
    run_case(w, B, TOPK)


@pytest.mark.parametrize("maxP,kmax", [(6, 8), (12, 8), (128, 11), (10, 10), (3, 5)])
def test_general_oea_knobs(maxP, kmax):
    w = W("t_knobs", seed=21)
    run_case(w, 24, OEA, 3, 0.8, maxP=maxP, kmax=kmax)


@pytest.mark.parametrize("N", [32, 256, 512, 1024])
@pytest.mark.parametrize("B", [12, 48])
@pytest.mark.parametrize("maxP,p", [(0, 1.0), (0, 0.6), (7, 1.0), (5, 0.8)])
def test_route_branches(N, B, maxP, p):
    # Every expert-count class of the routing kernel, with one token per warp
    # (picks kept in registers across the phases) and with more tokens than
    # warps (keys reloaded), both phase-2 forms and top-p on and off.
    w = W("t_branches", N=N, k=8, d=128, F=64, seed=N + B + maxP, zipf=True)
    run_case(w, B, OEA, 3, p, maxP=maxP, kmax=10, B_valid=B - 3)


@pytest.mark.parametrize("B", [1, 4, 16, 40])
@pytest.mark.parametrize("p", [1.0, 0.8])
def test_batch_size_policy(B, p):
    """k0 <= 0 chooses k0 from the batch (OEA page, section 7, implementation
    detail 2): a single token routes as plain top-k, smaller batches keep
    more experts per token.  The oracle applies its own copy of the rule."""
    w = W("t_policy", seed=23 + B, zipf=True)
    g, _, _ = run_case(w, B, OEA, 0, p)
    k0, _ = oracle.policy_k0(B, w.k, p)
    assert (g["n_base"][:B] <= k0).all()
    if B == 1:
        top, _, _ = run_case(w, 1, TOPK)
        assert np.array_equal(g["expert_idx"], top["expert_idx"]) and g["T"] == w.k
    # one real token among padding routes as plain top-k too
    g2, _, _ = run_case(w, B, OEA, 0, p, B_valid=1)
    assert g2["T"] == w.k


@pytest.mark.parametrize("mode", [TOPK, OEA])
def test_padding_tokens(mode):
    w = W("t_pad", seed=5)
    g, out, _ = run_case(w, 16, mode, 3, 1.0, B_valid=11)
    assert (g["expert_idx"][11:] == -1).all() and (g["weights"][11:] == 0).all()
    g2, _, _ = run_case(w, 11, mode, 3, 1.0, L={**synth.make_layer(w, 0, 16),
                                                "x": synth.make_layer(w, 0, 16)["x"][:11]})
    assert g2["T"] == g["T"]


@pytest.mark.parametrize("layout", ["up_above_gate", "up_below_gate", "gate_is_up"])
@pytest.mark.parametrize("B", [16, 37])
def test_gate_up_layouts(layout, B):
    """W_gate and W_up are read through one tensor map spanning both arrays
    when possible (lower address first), through two maps otherwise; every
    arrangement gives the oracle's result."""
    w = W("t_gu", N=32, d=256, F=192, seed=17)
    L = synth.make_layer(w, 0, B)
    if layout == "gate_is_up":
        L["w_up"] = L["w_gate"]
    D = gu.device_inputs(L, w.bf16)
    both = torch.empty((2,) + tuple(D["w_gate"].shape), dtype=D["w_gate"].dtype, device=gu.DEV)
    if layout == "up_above_gate":
        both[0], both[1] = D["w_gate"], D["w_up"]
        D["w_gate"], D["w_up"] = both[0], both[1]
    elif layout == "up_below_gate":
        both[0], both[1] = D["w_up"], D["w_gate"]
        D["w_gate"], D["w_up"] = both[1], both[0]
    else:
        D["w_up"] = D["w_gate"]
    for mode, k0 in ((TOPK, 8), (OEA, 3)):
        prm = gu.params_for(w, B, mode, k0, 1.0)
        r, out, ws, flags = gu.run_layer(w, D, prm)
        assert flags == 0, f"device flags {flags:#x}"
        g = gu.to_np(r)
        gu.check_routing(g, prm, B)
        o = oracle.moe_experts(L["x"], L["w_gate"], L["w_up"], L["w_down"], g["expert_idx"],
                               g["weights"].astype(np.float64))
        gu.check_output(out, o, w.bf16)


def test_hot_experts_many_tokens_per_expert():
    """Experts with more tokens than one 32-token pass (chunked tiles)."""
    w = W("t_hot", N=64, d=256, F=192, seed=3)
    L = synth.make_layer(w, 0, 100)
    bias = np.zeros(64, np.float32)
    bias[3], bias[7], bias[40] = 30.0, 20.0, 10.0   # gaps far above the score spread
    L["bias"] = bias
    g, _, _ = run_case(w, 100, TOPK, L=L)
    assert g["counts"][3] == 100 and g["counts"][7] == 100
    g, _, _ = run_case(w, 100, OEA, 2, 1.0, L=L)
    assert g["T"] == 2


def test_identical_tokens():
    w = W("t_same", seed=8)
    L = synth.make_layer(w, 0, 12)
    L["x"] = np.repeat(L["x"][:1], 12, axis=0)
    g, _, _ = run_case(w, 12, OEA, 3, 1.0, L=L)
    assert g["T"] == 3
    g, _, _ = run_case(w, 12, TOPK, L=L)
    assert g["T"] == 8


@pytest.mark.parametrize("N", [64, 128, 256])
def test_tied_scores(N):
    # Experts 2j and 2j+1 have the same router row (and no bias), so every
    # token scores them exactly alike: the ranking must put the lower id
    # first, and the selections must match the oracle's bit for bit.
    w = W("t_ties", N=N, k=8, d=256, F=128, seed=N + 3)
    L = synth.make_layer(w, 0, 24)
    L["w_router"] = np.repeat(L["w_router"][::2], 2, axis=0)
    L["bias"] = None if L["bias"] is None else np.zeros_like(L["bias"])
    g, _, _ = run_case(w, 24, OEA, 3, 1.0, L=L, check_e2e=False)
    assert (g["logits"][:, ::2] == g["logits"][:, 1::2]).all()
    run_case(w, 24, OEA, 5, 0.8, maxP=9, kmax=8, L=L, check_e2e=False)
    run_case(w, 24, TOPK, L=L, check_e2e=False)


def test_empty_batch():
    w = W("t_empty")
    run_case(w, 0, OEA, 3, 1.0)
    run_case(w, 0, TOPK)


def test_all_padding():
    w = W("t_allpad")
    g, out, _ = run_case(w, 5, OEA, 3, 1.0, B_valid=0)
    assert g["T"] == 0 and (out.float() == 0).all()


def test_deterministic_and_repeatable():
    """Same inputs -> same bits, across layer calls and across repeated expert
    calls on one routing (the in-kernel counters reset themselves)."""
    w = W("t_det", N=64, d=256, F=128, seed=9, zipf=True)
    L = synth.make_layer(w, 0, 48)
    D = gu.device_inputs(L, True)
    prm = gu.params_for(w, 48, OEA, 4, 0.9)
    r1, o1, ws, _ = gu.run_layer(w, D, prm)
    r2, o2, _, _ = gu.run_layer(w, D, prm, ws=ws)
    assert torch.equal(o1, o2) and torch.equal(r1.expert_idx, r2.expert_idx)
    assert torch.equal(r1.weights, r2.weights)
    o3 = torch.empty_like(o1)
    for _ in range(3):
        moe.moe_expert_ffn(D["x"], D["w_gate"], D["w_up"], D["w_down"], w.F, prm, r2, o3, ws)
        assert moe.moe_device_status(ws) == 0
        assert torch.equal(o1, o3)


@pytest.mark.parametrize("mode", [OEA, TOPK])
def test_early_union_follows_the_latest_routing(mode):
    """With OEA routing, batches of up to 16 start the expert kernel from
    S_base, which the routing kernel publishes after phase 1 tagged with the
    routing call's epoch.  An expert call must use the union of the latest
    routing call on its workspace -- also after routing calls that no expert
    call followed -- and expert calls after a host synchronisation (no
    overlap with the routing kernel) must give the same bits.  Top-k routing
    (which waits for the whole routing) must behave the same way."""
    w = W("t_epoch", N=128, d=512, F=256, seed=21)
    B = 12
    prm = gu.params_for(w, B, mode, 3 if mode == OEA else None, 1.0)
    Ls = [synth.make_layer(w, layer, B) for layer in range(3)]
    Ds = [gu.device_inputs(L, True) for L in Ls]
    g2, ref2, _ = run_case(w, B, mode, 3 if mode == OEA else None, 1.0, L=Ls[2])   # checked against the oracle
    Ts = [run_case(w, B, mode, 3 if mode == OEA else None, 1.0, L=L)[0]["active"] for L in Ls[:2]]
    assert any(not np.array_equal(t, g2["active"]) for t in Ts)   # the earlier unions differ
    ws = moe.alloc_workspace(prm, w.F, gu.DEV)
    r = moe.Routing(prm, gu.DEV, with_logits=True)
    out = torch.empty_like(ref2)
    for D in Ds[:2]:   # routing calls that no expert call follows
        moe.moe_route(D["x"], D["w_router"], D["bias"], prm, r, ws)
    D = Ds[2]
    moe.moe_route(D["x"], D["w_router"], D["bias"], prm, r, ws)
    moe.moe_expert_ffn(D["x"], D["w_gate"], D["w_up"], D["w_down"], w.F, prm, r, out, ws)
    assert moe.moe_device_status(ws) == 0
    assert torch.equal(out, ref2)
    torch.cuda.synchronize()
    for _ in range(2):
        out.fill_(float("nan"))
        moe.moe_expert_ffn(D["x"], D["w_gate"], D["w_up"], D["w_down"], w.F, prm, r, out, ws)
        assert moe.moe_device_status(ws) == 0
        assert torch.equal(out, ref2)


def test_wait_timeout_is_flagged_and_the_workspace_recovers():
    """A bounded in-kernel wait that runs out ends the call with
    MOE_FLAG_WAIT_TIMEOUT instead of hanging, and the context and the
    workspace stay usable.  With OEA routing of up to 16 tokens the expert
    kernel waits for the union that the preceding routing call publishes
    under its epoch.  Erasing the workspace after that routing call has
    completed (as if freshly zero-filled) means the awaited union never
    appears; with the bound set to 2 ms the wait gives up.  Nothing faults
    and nothing stalls the GPU: every CTA reaches the end of the kernel."""
    w = W("t_timeout", N=64, d=256, F=128, seed=31)
    B = 8
    L = synth.make_layer(w, 0, B)
    D = gu.device_inputs(L, True)
    prm = gu.params_for(w, B, OEA, 3, 1.0)
    r = moe.Routing(prm, gu.DEV, with_logits=True)
    ws = moe.alloc_workspace(prm, w.F, gu.DEV)
    out = torch.empty(B, w.d, dtype=torch.bfloat16, device=gu.DEV)
    moe.moe_route(D["x"], D["w_router"], D["bias"], prm, r, ws)
    torch.cuda.synchronize()
    ws.zero_()
    moe.moe_set_wait_timeout_us(2000)
    try:
        moe.moe_expert_ffn(D["x"], D["w_gate"], D["w_up"], D["w_down"], w.F, prm, r, out, ws)
        flags = moe.moe_device_status(ws)
    finally:
        moe.moe_set_wait_timeout_us(0)
    assert flags & moe.FLAG_WAIT_TIMEOUT
    # the next layer call on the same workspace is correct and raises nothing
    g, out2, ref = run_case(w, B, OEA, 3, 1.0, L=L)
    r2, out3, _, flags = gu.run_layer(w, D, prm, ws=ws)
    assert flags == 0 and torch.equal(out3, out2) and torch.equal(r2.expert_idx, r.expert_idx)


def test_nonfinite_scores_are_flagged():
    w = W("t_inf", N=32, d=128, F=64)
    L = synth.make_layer(w, 0, 4)
    L["x"][2, 5] = np.inf
    D = gu.device_inputs(L, True)
    prm = gu.params_for(w, 4, TOPK)
    _, _, _, flags = gu.run_layer(w, D, prm)
    assert flags & moe.FLAG_NONFINITE_SCORE


@pytest.mark.parametrize("bf16", [True, False])
def test_device_generator_matches_host(bf16):
    n, start, seed, std = 100_003, 12_345, synth.tensor_seed(4, 1, synth.T_GATE), 0.02
    t = torch.empty(n, dtype=torch.bfloat16 if bf16 else torch.float32, device=gu.DEV)
    moe.moe_synth_normal(t, seed, float(synth.scale_f32(std)), start)
    host = synth.normal(seed, (n,), std, bf16, start=start)
    assert np.array_equal(t.float().cpu().numpy(), host)


# ---- full-size workloads, every token against the oracle -------------------
def full_size_layer(w: synth.Workload, layer: int, B: int):
    """Weights generated on the device with the same generator as the host."""
    bf = torch.bfloat16
    D = {"x": torch.from_numpy(synth.make_tensor(w, layer, synth.T_X, B)).to(gu.DEV).to(bf).contiguous()}
    for name, tid in (("w_router", synth.T_ROUTER), ("w_gate", synth.T_GATE), ("w_up", synth.T_UP),
                      ("w_down", synth.T_DOWN)):
        t = torch.empty(synth.tensor_shape(w, tid, B), dtype=bf, device=gu.DEV)
        moe.moe_synth_normal(t, synth.tensor_seed(w.seed, layer, tid), float(synth.scale_f32(synth.tensor_std(w, tid))))
        D[name] = t
    b = synth.make_bias(w, layer)
    D["bias"] = torch.from_numpy(b).to(gu.DEV) if b is not None else None
    return D


@pytest.mark.parametrize("wname,B,runs", [
    ("qwen3_30b_a3b_uniform_b16", 16, [(TOPK, 8, 1.0), (OEA, 3, 1.0), (OEA, 5, 1.0)]),
    ("qwen3_30b_a3b_zipf_sweep", 1, [(TOPK, 8, 1.0), (OEA, 5, 0.7)]),
    ("qwen3_30b_a3b_zipf_sweep", 4, [(TOPK, 8, 1.0), (OEA, 5, 0.7), (OEA, 0, 0.7)]),
    ("qwen3_30b_a3b_zipf_sweep", 16, [(TOPK, 8, 1.0), (OEA, 5, 0.7)]),
    ("qwen3_30b_a3b_zipf_sweep", 64, [(TOPK, 8, 1.0), (OEA, 5, 0.7)]),
    ("qwen3_30b_a3b_zipf_sweep", 256, [(TOPK, 8, 1.0), (OEA, 5, 0.7)]),
    ("qwen3_235b_a22b_zipf_b64", 16, [(TOPK, 8, 1.0), (OEA, 5, 0.7)]),
    ("qwen3_235b_a22b_zipf_b64", 64, [(TOPK, 8, 1.0), (OEA, 5, 0.7)]),
    ("qwen3_235b_a22b_zipf_b64", 256, [(TOPK, 8, 1.0), (OEA, 5, 0.7)]),
])
def test_full_size_every_token(pool, wname, B, runs):
    """The benchmark workloads at full size: scores, the whole routing and
    every output element of every token against the oracle (which
    regenerates each activated expert from the seeded generator)."""
    w = synth.WORKLOADS[wname]
    D = full_size_layer(w, 0, B)
    x = synth.make_tensor(w, 0, synth.T_X, B)
    wr = synth.make_tensor(w, 0, synth.T_ROUTER)
    bias = synth.make_bias(w, 0)
    lg_ref = oracle.router_logits(x, wr, bias)
    res = []
    for mode, k0, p in runs:
        prm = gu.params_for(w, B, mode, k0, p)
        r, out, ws, flags = gu.run_layer(w, D, prm)
        assert flags == 0
        g = gu.to_np(r)
        assert np.abs(g["logits"] - lg_ref).max() <= 1e-3 * np.abs(lg_ref).max()
        gu.check_routing(g, prm, B)
        res.append((g, out))
    refs = pool.layer_outputs(w, 0, x, [(g["expert_idx"], g["weights"].astype(np.float64)) for g, _ in res])
    for (g, out), ref in zip(res, refs):
        gu.check_output(out, ref, True)
