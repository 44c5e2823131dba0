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


def static_call(w, D, prm):
    r = moe.Routing(prm, gu.DEV, with_logits=True)
    out = torch.full((prm.B, w.d), float("nan"), dtype=torch.bfloat16, device=gu.DEV)
    moe.moe_decode_layer_static(D["x"], D["w_router"], D["bias"], D["w_gate"], D["w_up"], D["w_down"],
                                w.F, prm, r, out)
    return r, out


@pytest.mark.parametrize("mode,k0,p,B", [(1, 3, 0.7, 8), (1, 5, 1.0, 16), (1, 3, 0.7, 24), (0, 8, 1.0, 16),
                                         (1, 5, 1.0, 40)])
def test_static_scratch_matches_workspace_call(mode, k0, p, B):
    """Two calls in a row give the workspace call's bits (routing and
    output), with a call of another batch shape in between, so a union,
    epoch or counter left in the shared array by a different call would be
    caught.  OEA batches of up to 16 tokens take the early start, which
    reads the union words the routing kernel publishes in the array."""
    w = synth.Workload("t_static", N=128, k=8, d=512, F=256, B=B, seed=77, zipf=True)
    D = gu.device_inputs(synth.make_layer(w, 0, B), True)
    prm = gu.params_for(w, B, mode, k0, p)
    r_ref, out_ref, _, flags = gu.run_layer(w, D, prm)
    assert flags == 0
    wo = synth.Workload("t_static_other", N=128, k=8, d=512, F=256, B=40, seed=78, zipf=True)
    Do = gu.device_inputs(synth.make_layer(wo, 0, 40), True)
    prm_o = gu.params_for(wo, 40, 1, 5, 1.0)
    assert moe.moe_device_status_static() == 0
    for call in range(2):
        r, out = static_call(w, D, prm)
        assert moe.moe_device_status_static() == 0
        for name in ("expert_idx", "weights", "T", "active", "counts", "offsets", "perm", "n_base", "logits"):
            assert torch.equal(getattr(r, name), getattr(r_ref, name)), name
        assert torch.equal(out, out_ref)
        if call == 0:   # another batch shape in between
            static_call(wo, Do, prm_o)
            assert moe.moe_device_status_static() == 0


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
