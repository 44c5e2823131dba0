"""Mixed-precision experts on the GPU: hot experts bf16, cold experts INT4
(DynaExq page, section 3.2).  The oracle multiplies with the same packed
bytes decoded to w = q * s."""
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
    moe.load()


def build_mixed(w, L, hot, active=None, alias_up=False):
    """Device buffers of a mixed layer and the oracle's effective weights.
    Cold experts outside `active` (if given) get zero images (never read).
    alias_up: the hot experts' W_up is their W_gate buffer (separate 8-row
    gate/up maps in the kernel); L's w_up must then equal its w_gate."""
    N, d, F = w.N, w.d, w.F
    hot = list(hot)
    cold = [e for e in range(N) if e not in hot]
    slot = np.empty(N, np.int32)
    for i, e in enumerate(hot):
        slot[e] = i
    for i, e in enumerate(cold):
        slot[e] = -1 - i
    eff = {k: L[k].copy() for k in ("w_gate", "w_up", "w_down")}
    na, nd = moe.int4_image_bytes(F, d), moe.int4_image_bytes(d, F)   # codes + a scale per 128-column group
    qg = np.zeros((len(cold), na), np.uint8)
    qu = np.zeros((len(cold), na), np.uint8)
    qd = np.zeros((len(cold), nd), np.uint8)
    for i, e in enumerate(cold):
        if active is not None and e not in active:
            continue
        (pg, pu, pd), _ = synth.pack_int4_expert(L["w_gate"][e], L["w_up"][e], L["w_down"][e])
        qg[i], qu[i], qd[i] = pg, pu, pd
        eff["w_gate"][e] = oracle.dequant_int4(pg, F, d, synth.INT4_RB_GATE_UP)
        eff["w_up"][e] = oracle.dequant_int4(pu, F, d, synth.INT4_RB_GATE_UP)
        eff["w_down"][e] = oracle.dequant_int4(pd, d, F, synth.INT4_RB_DOWN)
    bf = torch.bfloat16
    dev = gu.DEV
    hot_w = {k: torch.from_numpy(L[k][hot]).to(dev).to(bf).contiguous() for k in ("w_gate", "w_up", "w_down")}
    if alias_up:
        assert np.array_equal(L["w_up"], L["w_gate"])
        hot_w["w_up"] = hot_w["w_gate"]
    mixed = moe.MixedExperts(torch.from_numpy(slot).to(dev),
                             torch.from_numpy(qg).to(dev), torch.from_numpy(qu).to(dev),
                             torch.from_numpy(qd).to(dev), len(hot), len(cold))
    return hot_w, mixed, eff


def run_mixed(w, L, D, hot_w, mixed, prm):
    r = moe.Routing(prm, gu.DEV, with_logits=True)
    ws = moe.alloc_workspace(prm, w.F, gu.DEV)
    out = torch.full((prm.B, w.d), float("nan"), dtype=torch.bfloat16, device=gu.DEV)
    moe.moe_route(D["x"], D["w_router"], D["bias"], prm, r, ws)
    moe.moe_expert_ffn_mixed(D["x"], hot_w["w_gate"], hot_w["w_up"], hot_w["w_down"], mixed, w.F, prm, r, out, ws)
    assert moe.moe_device_status(ws) == 0
    return r, out


@pytest.mark.parametrize("mode,k0,p,B", [(TOPK, 4, 1.0, 20), (OEA, 2, 0.7, 20), (OEA, 3, 1.0, 37),
                                         (OEA, 4, 1.0, 64), (TOPK, 4, 1.0, 64), (OEA, 3, 1.0, 65)])
def test_mixed_layer_parity(mode, k0, p, B):
    w = synth.Workload("t_mixed", N=32, k=4, d=512, F=256, B=B, seed=41, zipf=True)
    L = synth.make_layer(w, 0, B)
    hot = [0, 3, 4, 9, 10, 11, 17, 20, 25, 31]
    hot_w, mixed, eff = build_mixed(w, L, hot)
    D = gu.device_inputs(L, True)
    prm = gu.params_for(w, B, mode, k0, p)
    r, out = run_mixed(w, L, D, hot_w, mixed, prm)
    g = gu.to_np(r)
    gu.check_routing(g, prm, B)
    ref = oracle.moe_experts(L["x"], eff["w_gate"], eff["w_up"], eff["w_down"], g["expert_idx"],
                             g["weights"].astype(np.float64))
    gu.check_output(out, ref, True)
    # the INT4 path really differs from bf16 weights (the test would notice a mix-up)
    ref_bf16 = oracle.moe_experts(L["x"], L["w_gate"], L["w_up"], L["w_down"], g["expert_idx"],
                                  g["weights"].astype(np.float64))
    assert np.abs(ref - ref_bf16).max() > 1e-3 * np.abs(ref_bf16).max()


@pytest.mark.parametrize("mode,B", [(OEA, 8), (TOPK, 32), (OEA, 64), (TOPK, 80)])
def test_mixed_separate_gate_up_maps(mode, B):
    # Hot experts whose W_gate and W_up cannot share one 5D map (W_up passed
    # as W_gate's buffer): their stages load 8-row groups of each, K blocks
    # per load; INT4 stages are unchanged (decoded into shared or tensor
    # memory).
    w = synth.Workload("t_mixed_sep", N=32, k=4, d=512, F=256, B=B, seed=43 + B, zipf=True)
    L = synth.make_layer(w, 0, B)
    L = dict(L, w_up=L["w_gate"].copy())
    hot = [0, 3, 4, 9, 10, 11, 17, 20, 25, 31]
    hot_w, mixed, eff = build_mixed(w, L, hot, alias_up=True)
    D = gu.device_inputs(L, True)
    prm = gu.params_for(w, B, mode, 3 if mode == OEA else 4, 1.0)
    r, out = run_mixed(w, L, D, hot_w, mixed, prm)
    g = gu.to_np(r)
    gu.check_routing(g, prm, B)
    ref = oracle.moe_experts(L["x"], eff["w_gate"], eff["w_up"], eff["w_down"], g["expert_idx"],
                             g["weights"].astype(np.float64))
    gu.check_output(out, ref, True)


@pytest.mark.parametrize("d,F,B", [(512, 256, 8), (384, 128, 16), (512, 256, 1), (256, 384, 5)])
def test_mixed_small_batches(d, F, B):
    # Batches of up to 16 tokens: INT4 stages of 4, 2 or 1 column blocks,
    # each block converted from its own packed chunk.
    w = synth.Workload("t_mixed_small", N=32, k=4, d=d, F=F, B=B, seed=d + F + B, zipf=True)
    L = synth.make_layer(w, 0, B)
    hot = [1, 2, 5, 8, 13, 21, 30]
    hot_w, mixed, eff = build_mixed(w, L, hot)
    D = gu.device_inputs(L, True)
    prm = gu.params_for(w, B, OEA, 3, 1.0)
    r, out = run_mixed(w, L, D, hot_w, mixed, prm)
    g = gu.to_np(r)
    gu.check_routing(g, prm, B)
    ref = oracle.moe_experts(L["x"], eff["w_gate"], eff["w_up"], eff["w_down"], g["expert_idx"],
                             g["weights"].astype(np.float64))
    gu.check_output(out, ref, True)


@pytest.mark.parametrize("rows,cols,rb", [(64, 2048, 64), (256, 384, 128), (24, 128, 8)])
def test_device_int4_pack_matches_host(rows, cols, rb):
    """moe_pack_int4 writes the same bytes as the host packer: scales,
    ties to even (w / s exactly k + 1/2), groups of zeros and the clamp."""
    rng = np.random.default_rng(rows + cols)
    w = synth.round_bf16(rng.standard_normal((rows, cols)).astype(np.float32) * 0.05)
    w[0, :128] = 0.0                                    # s = 0: every code 0
    w[1, :128] = np.float32(0.25) * np.resize(np.arange(-7.0, 7.5, 0.5), 128).astype(np.float32)
    w[1, 0] = np.float32(1.75)                          # max 1.75: s = 0.25, w / s hits every half step
    q, s = synth.quantize_int4(w)
    want = synth.pack_int4_tiles(q, s, rb)
    got = moe.moe_pack_int4(torch.from_numpy(w).to(gu.DEV).to(torch.bfloat16), rb)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), want)


@pytest.mark.parametrize("mode,k0", [(TOPK, 2), (OEA, 1)])
def test_bad_slot_is_flagged(mode, k0):
    """An out-of-range slot of an activated expert raises MOE_FLAG_BAD_INDEX.
    A router bias far above the score spread puts expert 5 first for every
    token, so the bad slot is always read."""
    w = synth.Workload("t_mixed_bad", N=16, k=2, d=256, F=256, B=8, seed=3)
    L = synth.make_layer(w, 0, 8)
    L["bias"] = np.zeros(16, np.float32)
    L["bias"][5] = 30.0
    hot_w, mixed, _ = build_mixed(w, L, range(8))
    mixed.slot[5] = 100          # out of range
    D = gu.device_inputs(L, True)
    prm = gu.params_for(w, 8, mode, k0)
    r = moe.Routing(prm, gu.DEV)
    ws = moe.alloc_workspace(prm, w.F, gu.DEV)
    out = torch.empty(8, w.d, dtype=torch.bfloat16, device=gu.DEV)
    moe.moe_route(D["x"], D["w_router"], D["bias"], prm, r, ws)
    moe.moe_expert_ffn_mixed(D["x"], hot_w["w_gate"], hot_w["w_up"], hot_w["w_down"], mixed, w.F, prm, r, out, ws)
    flags = moe.moe_device_status(ws)
    assert int((r.expert_idx[:, 0] == 5).sum().item()) == 8
    assert flags & moe.FLAG_BAD_INDEX


@pytest.mark.parametrize("mode,k0,p,B", [(OEA, 2, 0.7, 12), (TOPK, 4, 1.0, 20), (OEA, 0, 1.0, 37)])
def test_mixed_layer_one_call(mode, k0, p, B):
    """moe_decode_layer_mixed (routing and mixed experts in one call) against
    the oracle, and bit for bit against the two-call sequence."""
    w = synth.Workload("t_mixed_one", N=32, k=4, d=512, F=256, B=B, seed=43, zipf=True)
    L = synth.make_layer(w, 0, B)
    hot = [0, 2, 6, 7, 12, 19, 22, 30]
    hot_w, mixed, eff = build_mixed(w, L, hot)
    D = gu.device_inputs(L, True)
    prm = gu.params_for(w, B, mode, k0, p)
    r = moe.Routing(prm, gu.DEV, with_logits=True)
    ws = moe.alloc_workspace(prm, w.F, gu.DEV)
    out = torch.full((B, w.d), float("nan"), dtype=torch.bfloat16, device=gu.DEV)
    for _ in range(2):
        moe.moe_decode_layer_mixed(D["x"], D["w_router"], D["bias"], hot_w["w_gate"], hot_w["w_up"],
                                   hot_w["w_down"], mixed, w.F, prm, r, out, ws)
        assert moe.moe_device_status(ws) == 0
        g = gu.to_np(r)
        gu.check_routing(g, prm, B)
        ref = oracle.moe_experts(L["x"], eff["w_gate"], eff["w_up"], eff["w_down"], g["expert_idx"],
                                 g["weights"].astype(np.float64))
        gu.check_output(out, ref, True)
    r2, out2 = run_mixed(w, L, D, hot_w, mixed, prm)
    assert torch.equal(out, out2) and torch.equal(r.expert_idx, r2.expert_idx)


def test_full_size_mixed_every_token(pool):
    """The 30B mixed workload (B=32): hot set from a 200-step EMA trace,
    every cold expert packed to INT4 from its real weights, the whole layer
    in one call (moe_decode_layer_mixed); routing and every output element
    of every token against the oracle on the same packed bytes.  The hot
    experts are generated on the device (the generator is bit-identical to
    the host's)."""
    w = synth.WORKLOADS["qwen3_30b_a3b_mixed_int4_b32"]
    B, N, d = w.B, w.N, w.d
    dev = gu.DEV
    bf = torch.bfloat16
    x = synth.make_tensor(w, 0, synth.T_X, B)
    L = {"x": x, "w_router": synth.make_tensor(w, 0, synth.T_ROUTER), "bias": synth.make_bias(w, 0)}
    D = gu.device_inputs(L, True)
    # hotness trace: vanilla top-8 on fresh seeded batches; the oracle routes the same scores
    prm_t = moe.RouteParams(B=32, d=d, N=N, k=w.k)
    rt = moe.Routing(prm_t, dev, with_logits=True)
    wst = moe.alloc_workspace(prm_t, 0, dev)
    xt = torch.empty(32, d, dtype=bf, device=dev)
    counts = []
    for step in range(200):
        moe.moe_synth_normal(xt, synth.trace_seed(w, 0, step), float(synth.scale_f32(1.0)))
        moe.moe_route(xt, D["w_router"], D["bias"], prm_t, rt, wst)
        c = rt.counts.cpu().numpy()
        if step % 50 == 0:
            ref = oracle.route(rt.logits.cpu().numpy(), oracle.TOPK, w.k)
            assert np.array_equal(c, ref["counts"])
        counts.append(c)
    hot = [int(e) for e in moe.ema_hot_set(np.array(counts), w.hot_n)]
    cold = [e for e in range(N) if e not in hot]
    slot = np.empty(N, np.int32)
    for i, e in enumerate(hot):
        slot[e] = i
    for i, e in enumerate(cold):
        slot[e] = -1 - i
    hot_w = {}
    for name, tid in (("w_gate", synth.T_GATE), ("w_up", synth.T_UP), ("w_down", synth.T_DOWN)):
        t = torch.empty((len(hot),) + synth.tensor_shape(w, tid)[1:], dtype=bf, device=dev)
        per = t[0].numel()
        for i, e in enumerate(hot):
            moe.moe_synth_normal(t[i], synth.tensor_seed(w.seed, 0, tid),
                                 float(synth.scale_f32(synth.tensor_std(w, tid))), start=e * per)
        hot_w[name] = t
    packed = pool.pack_cold(w, 0, cold)
    q = [torch.from_numpy(np.stack([pk[m] for pk in packed])).to(dev) for m in range(3)]
    mixed = moe.MixedExperts(torch.from_numpy(slot).to(dev), q[0], q[1], q[2], len(hot), len(cold))
    res = []
    for mode, k0, p in ((OEA, 5, 1.0), (TOPK, 8, 1.0)):
        prm = gu.params_for(w, B, mode, k0, p)
        r = moe.Routing(prm, dev, with_logits=True)
        ws = moe.alloc_workspace(prm, w.F, dev)
        out = torch.full((B, d), float("nan"), dtype=bf, device=dev)
        moe.moe_decode_layer_mixed(D["x"], D["w_router"], D["bias"], hot_w["w_gate"], hot_w["w_up"],
                                   hot_w["w_down"], mixed, w.F, prm, r, out, ws)
        assert moe.moe_device_status(ws) == 0
        g = gu.to_np(r)
        gu.check_routing(g, prm, B)
        res.append((g, out))
    assert any(slot[e] < 0 for g, _ in res for e in g["active"][:g["T"]])   # INT4 experts are activated
    refs = pool.layer_outputs(w, 0, x, [(g["expert_idx"], g["weights"].astype(np.float64)) for g, _ in res],
                              cold=frozenset(cold))
    for (g, out), ref in zip(res, refs):
        gu.check_output(out, ref, True)
