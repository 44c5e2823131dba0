"""Expert residency while the layer runs (DynaExq page, sections 2.2-2.5
and 3.2-3.5), on the GPU through the C ABI: every call's routing and output
against the oracle with the version (bf16 or INT4) each expert's handle held
for that call, the bf16 pool holding exactly the expert its handle names,
and the bf16 set following the oracle's hotness update and selection with
hysteresis."""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("aware_expert_routing_gb300")
import gpu_util as gu  # noqa: E402

OEA = 1


@pytest.fixture(scope="module", autouse=True)
def built():
    from aware_expert_routing_gb300 import build as b
    b.build()
    oracle.build()
    moe.load()


def setup_layer(w, L, initial_hot):
    dev, bf = gu.DEV, torch.bfloat16
    host = {k: torch.from_numpy(L[k]).to(bf).contiguous().pin_memory() for k in ("w_gate", "w_up", "w_down")}
    hot = {k: host[k][initial_hot].to(dev).contiguous() for k in host}
    packed = [synth.pack_int4_expert(L["w_gate"][e], L["w_up"][e], L["w_down"][e])[0] for e in range(w.N)]
    q = {k: torch.from_numpy(np.stack([p[m] for p in packed])).to(dev) for m, k in enumerate(("w_gate", "w_up", "w_down"))}
    int4 = {}
    for e in range(w.N):
        pg, pu, pd = packed[e]
        int4[e] = (oracle.dequant_int4(pg, w.F, w.d, synth.INT4_RB_GATE_UP),
                   oracle.dequant_int4(pu, w.F, w.d, synth.INT4_RB_GATE_UP),
                   oracle.dequant_int4(pd, w.d, w.F, synth.INT4_RB_DOWN))
    return host, hot, q, int4


def effective_weights(w, L, int4, table):
    eff = {k: L[k].copy() for k in ("w_gate", "w_up", "w_down")}
    for e in range(w.N):
        if table[e] < 0:
            assert table[e] == -1 - e          # every expert's own INT4 image
            eff["w_gate"][e], eff["w_up"][e], eff["w_down"][e] = int4[e]
    return eff


@pytest.mark.parametrize("max_inflight", [1, 4])
def test_residency_follows_the_routing(max_inflight):
    w = synth.Workload("t_res", N=32, k=4, d=256, F=256, B=16, seed=51)
    L = synth.make_layer(w, 0, w.B)
    initial = list(range(8))
    host, hot, q, int4 = setup_layer(w, L, initial)
    alpha, margin, U = 0.5, 0.5, 2
    res = moe.Residency(w.N, w.d, w.F, initial, hot, q, host, alpha=alpha, margin=margin, update_every=U,
                        max_inflight=max_inflight)
    D = gu.device_inputs({"w_router": L["w_router"]}, True)
    prm = gu.params_for(w, w.B, OEA, 2, 1.0)
    r = moe.Routing(prm, gu.DEV, with_logits=True)
    ws = moe.alloc_workspace(prm, w.F, gu.DEV)
    out = torch.empty(w.B, w.d, dtype=torch.bfloat16, device=gu.DEV)
    # routing drifts: experts 16-23 favoured first, then 0-7 again
    bias_a = np.zeros(w.N, np.float32)
    bias_a[16:24] = 4.0
    bias_b = np.zeros(w.N, np.float32)
    bias_b[0:8] = 4.0
    # oracle replay of the policy (the issue queue as the library runs it)
    S = np.zeros(w.N)
    members = np.zeros(w.N, bool)
    members[initial] = True
    queue, inflight, counts_log = [], 0, []
    for t in range(16):
        bias = bias_a if t < 8 else bias_b
        x = synth.make_tensor(w, 0, synth.T_X, w.B, step=t)
        xd = torch.from_numpy(x).to(gu.DEV).to(torch.bfloat16)
        bd = torch.from_numpy(bias).to(gu.DEV)
        torch.cuda.synchronize()
        table = res.slot.cpu().numpy()
        for e in range(w.N):   # a handle on the bf16 pool names a slot holding exactly that expert
            s = int(table[e])
            if s >= 0:
                for k in ("w_gate", "w_up", "w_down"):
                    assert torch.equal(hot[k][s].cpu(), host[k][e]), (t, e, s, k)
        moe.moe_decode_layer_mixed(xd, D["w_router"], bd, hot["w_gate"], hot["w_up"], hot["w_down"], res.mixed(),
                                   w.F, prm, r, out, ws)
        assert moe.moe_device_status(ws) == 0
        g = gu.to_np(r)
        ref = gu.check_routing(g, prm, w.B)
        eff = effective_weights(w, L, int4, table)
        o = oracle.moe_experts(x, eff["w_gate"], eff["w_up"], eff["w_down"], g["expert_idx"],
                               g["weights"].astype(np.float64))
        gu.check_output(out, o, True)
        res.observe(r.counts)
        torch.cuda.synchronize()
        # the library's steps at this call: publish, score update (from the
        # snapshot of the previous interval), selection if nothing pending,
        # then issue
        counts_log.append(ref["counts"].astype(np.float64))
        inflight = 0
        c = t + 1
        if c - 1 >= U and (c - 1) % U == 0:
            S = oracle.ema_update(S, np.sum(counts_log[c - 1 - U:c - 1], axis=0), alpha)
            if not queue:
                members_sel, pro, dem = oracle.hot_select(S, members, margin)
                queue = list(zip(pro, dem))
        while queue and inflight < max_inflight:
            o_, i_ = queue.pop(0)
            members[o_], members[i_] = True, False
            inflight += 1
        state, scores, stats = res.query()
        assert np.allclose(scores, S, rtol=0, atol=1e-9), t
        assert np.array_equal(state != moe.MOE_RESIDENT_LO, members), (t, np.nonzero(state)[0], np.nonzero(members)[0])
    res.flush()
    torch.cuda.synchronize()
    state, _, stats = res.query()
    assert stats["promotions"] > 0 and stats["promotions"] == stats["demotions"] and stats["pending"] == 0
    assert (state != moe.MOE_PROMOTING).all() and (state == moe.MOE_RESIDENT_HI).sum() == len(initial)
    table = res.slot.cpu().numpy()
    assert sorted(int(table[e]) for e in np.nonzero(table >= 0)[0]) == list(range(len(initial)))
    res.close()
