"""Helpers for the GPU parity tests: run the library on seeded synthetic
inputs and compare with the oracle.  Imported only by tests marked gpu."""
from __future__ import annotations

import numpy as np
import torch

import aware_expert_routing_gb300 as moe
import oracle
import synth

DEV = torch.device("cuda:0")

# Tolerances: bf16 weights -> max|d| <= 1e-2 max|ref|; fp32 -> 1e-5 relative.
TOL_BF16 = 1e-2
TOL_F32 = 1e-5
TOL_W = 1e-5          # routing weights (fp32 on the GPU, fp64 in the oracle)
NEAR_TIE_P = 1e-4     # top-p prefixes this close to p are decided by rounding


def device_inputs(L: dict, bf16: bool) -> dict:
    dt = torch.bfloat16 if bf16 else torch.float32
    out = {}
    for k, v in L.items():
        if v is None:
            out[k] = None
        elif k == "bias":
            out[k] = torch.from_numpy(v).to(DEV)
        else:
            out[k] = torch.from_numpy(v).to(DEV).to(dt).contiguous()
    return out


def params_for(w: synth.Workload, B: int, mode: int, k0=None, p=1.0, maxP=0, kmax=0, B_valid=-1):
    """k0 None: k; k0 <= 0 (OEA): the library's batch-size policy."""
    return moe.RouteParams(B=B, d=w.d, N=w.N, k=w.k, mode=mode, k0=w.k if k0 is None else k0, p=p, maxP=maxP,
                           kmax=kmax, B_valid=B_valid,
                           dtype=moe.DTYPE_BF16 if w.bf16 else moe.DTYPE_F32)


def resolved_k0_p(prm: moe.RouteParams, B_valid: int):
    """(k0, p) the routing runs with: the oracle's batch-size policy when
    prm.k0 <= 0 in OEA mode."""
    if prm.mode == moe.MODE_OEA and prm.k0 <= 0:
        return oracle.policy_k0(B_valid, prm.k, prm.p)
    return prm.k0, prm.p


def run_layer(w: synth.Workload, D: dict, prm: moe.RouteParams, ws=None, stream=None):
    r = moe.Routing(prm, DEV, with_logits=True)
    if ws is None:
        ws = moe.alloc_workspace(prm, w.F, DEV)
    out = torch.full((prm.B, w.d), float("nan"), dtype=prm.torch_dtype, device=DEV)
    moe.moe_decode_layer(D["x"], D["w_router"], D["bias"], D["w_gate"], D["w_up"], D["w_down"], w.F, prm,
                         r, out, ws, stream)
    flags = moe.moe_device_status(ws, stream)
    return r, out, ws, flags


def to_np(r: moe.Routing) -> dict:
    g = {k: getattr(r, k).cpu().numpy() for k in
         ("expert_idx", "weights", "T", "active", "counts", "offsets", "perm", "n_base", "logits")}
    g["T"] = int(g["T"][0])
    return g


def near_tie_choices(logits: np.ndarray, p: float, k0: int, B_valid: int) -> dict:
    """Tokens whose top-p prefix (fp64) at one of the first k0 ranks lies
    within NEAR_TIE_P of p, where fp32 rounding order decides t_i, each with
    the baseline sizes that decision can give: stopping at that rank, or
    one rank later (capped at k0)."""
    if p >= 1:
        return {}
    out = {}
    for i in range(min(B_valid, logits.shape[0])):
        l = logits[i].astype(np.float64)
        P = np.exp(l - l.max())
        P /= P.sum()
        c = np.cumsum(np.sort(P)[::-1])[:k0]
        near = np.nonzero(np.abs(c - p) < NEAR_TIE_P)[0]
        if len(near):
            out[i] = {int(t) + 1 for t in near} | {min(int(t) + 2, k0) for t in near}
    return out


def near_tie_tokens(logits: np.ndarray, p: float, k0: int, B_valid: int) -> set:
    return set(near_tie_choices(logits, p, k0, B_valid))


def check_routing(g: dict, prm: moe.RouteParams, B_valid: int):
    """The GPU routing equals the oracle's routing of the GPU's own scores,
    for the whole batch: bit-exact for n_i, T, indices, counts, offsets,
    active list and grouping; weights within TOL_W.  A token whose top-p
    prefix lies within NEAR_TIE_P of p (a near-tie: fp32 rounding order
    decides its t_i) may take either baseline size that rounding can give;
    every other token's n_i must be the oracle's, and the oracle is then
    rerun with the GPU's n_i so that the rest of the batch is compared
    exactly.  Returns the oracle result and the near-tie count."""
    mode = oracle.OEA if prm.mode == moe.MODE_OEA else oracle.TOPK
    kmax = prm.kmax if prm.kmax > 0 else prm.k
    maxP = prm.maxP if 0 < prm.maxP < prm.N else prm.N
    k0, p = resolved_k0_p(prm, B_valid)
    ref = oracle.route(g["logits"], mode, prm.k, prm.k0, prm.p, maxP, kmax, B_valid)
    ties = near_tie_choices(g["logits"], p, k0, B_valid) if mode == oracle.OEA else {}
    if ties:
        nb = g["n_base"][:prm.B].astype(np.int32)
        for i in range(B_valid):
            if i in ties:
                assert nb[i] in ties[i] | {int(ref["nbase"][i])}, (i, nb[i], ties[i])
            else:
                assert nb[i] == ref["nbase"][i], (i, nb[i], ref["nbase"][i])
        ref = oracle.route(g["logits"], mode, prm.k, prm.k0, prm.p, maxP, kmax, B_valid, nbase=nb)
    assert g["T"] == ref["T"]
    assert np.array_equal(g["n_base"][:prm.B], ref["nbase"])
    assert np.array_equal(g["expert_idx"], ref["idx"])
    assert np.abs(g["weights"].astype(np.float64) - ref["w"]).max(initial=0.0) <= TOL_W
    assert np.array_equal(g["counts"], ref["counts"])
    assert np.array_equal(g["offsets"], ref["offsets"])
    assert np.array_equal(g["active"][:g["T"]], ref["active"])
    assert (g["active"][g["T"]:] == -1).all()
    n = int(ref["offsets"][-1])
    assert np.array_equal(g["perm"][:n], ref["perm"])
    ref["near_ties"] = len(ties)
    return ref


def check_output(out_gpu: torch.Tensor, ref: np.ndarray, bf16: bool):
    got = out_gpu.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    scale = np.abs(ref).max()
    err = np.abs(got - ref).max()
    tol = (TOL_BF16 if bf16 else TOL_F32) * max(scale, 1e-30)
    assert err <= tol, f"max|d|={err:.3e} > {tol:.3e} (max|ref|={scale:.3e})"
    return err / max(scale, 1e-30)
