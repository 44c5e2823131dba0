"""moe_decode_layer_static: the decode layer for callers that cannot allocate
device memory (no workspace; the scratch is a fixed array in the library's
own device memory).  Collected last so that a failure here leaves every
other test already run; it passes alone in a fresh process as well."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("aware_expert_routing_gb300")
import gpu_util as gu  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    from aware_expert_routing_gb300 import build as b
    b.build()
    assert torch.cuda.is_available()
    moe.load()


@pytest.mark.parametrize("mode,k0,p,B", [(1, 3, 0.7, 24), (0, 8, 1.0, 16), (1, 5, 1.0, 40)])
def test_static_scratch_matches_workspace_call(mode, k0, p, B):
    w = synth.Workload("t_static", N=128, k=8, d=512, F=256, B=B, seed=77, zipf=True)
    D = gu.device_inputs(synth.make_layer(w, 0, B), True)
    prm = gu.params_for(w, B, mode, k0, p)
    r_ref, out_ref, _, flags = gu.run_layer(w, D, prm)
    assert flags == 0
    ref = out_ref.float().cpu().numpy().astype(np.float64)
    for _ in range(2):   # two calls in a row: the shared array keeps the last contents
        r = moe.Routing(prm, gu.DEV, with_logits=True)
        out = torch.full((B, w.d), float("nan"), dtype=torch.bfloat16, device=gu.DEV)
        moe.moe_decode_layer_static(D["x"], D["w_router"], D["bias"], D["w_gate"], D["w_up"], D["w_down"],
                                    w.F, prm, r, out)
        torch.cuda.synchronize()
        assert torch.equal(r.expert_idx, r_ref.expert_idx) and int(r.T.item()) == int(r_ref.T.item())
        got = out.float().cpu().numpy().astype(np.float64)
        assert np.abs(got - ref).max() <= gu.TOL_BF16 * np.abs(ref).max()


def test_static_scratch_rejects_oversized_batch():
    # B=256 with d=4096, d_ff=1536 needs more scratch than the fixed array
    prm = moe.RouteParams(B=256, d=4096, N=128, k=8)
    assert moe.moe_workspace_bytes(prm, 1536) > moe.STATIC_SCRATCH_BYTES
    r = moe.Routing(prm, gu.DEV)
    t = torch.empty(8, dtype=torch.bfloat16, device=gu.DEV)
    with pytest.raises(moe.MoeError) as ei:
        moe.load().moe_decode_layer_static  # symbol present
        out = torch.empty(256, 4096, dtype=torch.bfloat16, device=gu.DEV)
        x = torch.empty(256, 4096, dtype=torch.bfloat16, device=gu.DEV)
        moe.moe_decode_layer_static(x, t, None, t, t, t, 1536, prm, r, out)
    assert ei.value.status == moe.MOE_ERR_WORKSPACE
