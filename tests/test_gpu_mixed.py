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


def build_mixed(w, L, hot, active=None):
    """Device buffers of a mixed layer and the oracle's effective weights.
    Cold experts outside `active` (if given) get zero images (never read)."""
    N, d, F = w.N, w.d, w.F
    hot = list(hot)
    cold = [e for e in range(N) if e not in hot]
    slot = np.empty(N, np.int32)
    for i, e in enumerate(hot):
        slot[e] = i
    for i, e in enumerate(cold):
        slot[e] = -1 - i
    eff = {k: L[k].copy() for k in ("w_gate", "w_up", "w_down")}
    na, nd = F * d // 2 + F * (d // 64) * 2, d * F // 2 + d * (F // 64) * 2   # codes + a scale per 64-column chunk
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


@pytest.mark.parametrize("mode,k0,p,B", [(TOPK, 4, 1.0, 20), (OEA, 2, 0.7, 20), (OEA, 3, 1.0, 37)])
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


def test_bad_slot_is_flagged():
    w = synth.Workload("t_mixed_bad", N=16, k=2, d=256, F=256, B=8, seed=3)
    L = synth.make_layer(w, 0, 8)
    hot_w, mixed, _ = build_mixed(w, L, range(8))
    mixed.slot[5] = 100          # out of range
    D = gu.device_inputs(L, True)
    prm = gu.params_for(w, 8, TOPK)
    r = moe.Routing(prm, gu.DEV)
    ws = moe.alloc_workspace(prm, w.F, gu.DEV)
    out = torch.empty(8, w.d, dtype=torch.bfloat16, device=gu.DEV)
    moe.moe_route(D["x"], D["w_router"], D["bias"], prm, r, ws)
    moe.moe_expert_ffn_mixed(D["x"], hot_w["w_gate"], hot_w["w_up"], hot_w["w_down"], mixed, w.F, prm, r, out, ws)
    flags = moe.moe_device_status(ws)
    if int((r.expert_idx == 5).sum().item()) > 0:
        assert flags & moe.FLAG_BAD_INDEX


def test_full_size_mixed_sampled():
    """The 30B mixed workload (B=32): hot set from a 200-step EMA trace, cold
    experts INT4; sampled tokens against the oracle.  The hot experts are
    generated on the device (the generator is bit-identical to the host's);
    the host packs the cold experts of the sampled tokens (other cold slots
    hold zero images and contribute nothing to the checked tokens)."""
    w = synth.WORKLOADS["qwen3_30b_a3b_mixed_int4_b32"]
    B, N, d, F = w.B, w.N, w.d, w.F
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
    # hot pool on the device
    hot_w = {}
    for name, tid in (("w_gate", synth.T_GATE), ("w_up", synth.T_UP), ("w_down", synth.T_DOWN)):
        t = torch.empty((len(hot),) + synth.tensor_shape(w, tid)[1:], dtype=bf, device=dev)
        per = t[0].numel()
        for i, e in enumerate(hot):
            moe.moe_synth_normal(t[i], synth.tensor_seed(w.seed, 0, tid),
                                 float(synth.scale_f32(synth.tensor_std(w, tid))), start=e * per)
        hot_w[name] = t
    # routing of the layer, then the cold experts the sampled tokens use
    prm = gu.params_for(w, B, OEA, 5, 1.0)
    r0 = moe.Routing(prm, dev)
    ws0 = moe.alloc_workspace(prm, 0, dev)
    moe.moe_route(D["x"], D["w_router"], D["bias"], prm, r0, ws0)
    idx0 = r0.expert_idx.cpu().numpy()
    sample = (0, 13, B - 1)
    used = {int(e) for i in sample for e in idx0[i] if e >= 0}
    na, nd = F * d // 2 + F * (d // 64) * 2, d * F // 2 + d * (F // 64) * 2   # codes + a scale per 64-column chunk
    qg = np.zeros((len(cold), na), np.uint8)
    qu = np.zeros((len(cold), na), np.uint8)
    qd = np.zeros((len(cold), nd), np.uint8)
    eff = {}
    for e in used:
        g, u, dn = synth.make_expert(w, 0, e)
        if e in hot:
            eff[e] = (g, u, dn)
        else:
            (pg, pu, pd), _ = synth.pack_int4_expert(g, u, dn)
            i = cold.index(e)
            qg[i], qu[i], qd[i] = pg, pu, pd
            eff[e] = (oracle.dequant_int4(pg, F, d, synth.INT4_RB_GATE_UP), oracle.dequant_int4(pu, F, d, synth.INT4_RB_GATE_UP),
                      oracle.dequant_int4(pd, d, F, synth.INT4_RB_DOWN))
    mixed = moe.MixedExperts(torch.from_numpy(slot).to(dev), torch.from_numpy(qg).to(dev),
                             torch.from_numpy(qu).to(dev), torch.from_numpy(qd).to(dev), len(hot), len(cold))
    r, out = run_mixed(w, L, D, hot_w, mixed, prm)
    g = gu.to_np(r)
    gu.check_routing(g, prm, B)
    got = out.float().cpu().numpy()
    for i in sample:
        ref = np.zeros(d)
        for j, e in enumerate(g["expert_idx"][i]):
            if e >= 0:
                ref += float(g["weights"][i, j]) * oracle.expert_ffn(x[i], *eff[int(e)])
        assert np.abs(got[i] - ref).max() <= gu.TOL_BF16 * np.abs(ref).max()
