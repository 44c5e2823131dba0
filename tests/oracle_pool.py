"""The oracle's expert outputs for whole full-size batches, in parallel.

Each task is one expert of one layer: the worker regenerates that expert's
weights from the seeded generator (``synth``), packs them to INT4 and
decodes the packed bytes with the oracle when the expert is cold in a
mixed-precision layer, and runs the oracle's SwiGLU expert on every token
routed to it.  Workers start with the ``spawn`` method, so nothing of the
parent's CUDA state is inherited.  Test infrastructure only: it imports the
oracle and the input generator, never the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np

import oracle
import synth


def _expert_task(wname: str, layer: int, e: int, cold: bool, xrows: np.ndarray):
    """(packed images or None, y [rows][d] fp64) of expert e on the given
    hidden-state rows."""
    w = synth.WORKLOADS[wname]
    g, u, dn = synth.make_expert(w, layer, e)
    packed = None
    if cold:
        packed, _ = synth.pack_int4_expert(g, u, dn)
        pg, pu, pd = packed
        g = oracle.dequant_int4(pg, w.F, w.d, synth.INT4_RB_GATE_UP)
        u = oracle.dequant_int4(pu, w.F, w.d, synth.INT4_RB_GATE_UP)
        dn = oracle.dequant_int4(pd, w.d, w.F, synth.INT4_RB_DOWN)
    ys = np.stack([oracle.expert_ffn(xr, g, u, dn) for xr in xrows]) if len(xrows) else \
        np.zeros((0, w.d), np.float64)
    return packed, ys


def _pack_task(wname: str, layer: int, e: int):
    w = synth.WORKLOADS[wname]
    packed, _ = synth.pack_int4_expert(*synth.make_expert(w, layer, e))
    return packed


class OraclePool:
    def __init__(self, workers: int | None = None):
        n = workers or max(1, min(16, (os.cpu_count() or 1)))
        self.ex = cf.ProcessPoolExecutor(max_workers=n, mp_context=mp.get_context("spawn"))

    def close(self):
        self.ex.shutdown(wait=True, cancel_futures=True)

    def pack_cold(self, w: synth.Workload, layer: int, cold: list) -> list:
        """Packed (gate, up, down) images of the cold experts, in order."""
        futs = [self.ex.submit(_pack_task, w.name, layer, int(e)) for e in cold]
        return [f.result() for f in futs]

    def layer_outputs(self, w: synth.Workload, layer: int, x: np.ndarray, runs: list, cold=frozenset()):
        """Oracle outputs out[i] = sum_j w_ij y_{e_ij}(x_i), in slot order,
        for each routing in `runs` (a list of (idx [B][kslots], weights
        [B][kslots])) of the same batch x.  Each expert is generated once
        for all runs; experts in `cold` use their INT4 images."""
        need = {}   # expert -> sorted tokens
        for idx, _ in runs:
            for i, row in enumerate(idx):
                for e in row:
                    if e >= 0:
                        need.setdefault(int(e), set()).add(i)
        futs = {}
        for e, toks in need.items():
            toks = sorted(toks)
            futs[e] = (toks, self.ex.submit(_expert_task, w.name, layer, e, e in cold,
                                            np.ascontiguousarray(x[toks], np.float32)))
        y = {}
        for e, (toks, f) in futs.items():
            _, ys = f.result()
            for t, row in zip(toks, ys):
                y[(t, e)] = row
        outs = []
        for idx, wts in runs:
            out = np.zeros((x.shape[0], w.d), np.float64)
            for i, row in enumerate(idx):
                for j, e in enumerate(row):   # slot order
                    if e >= 0:
                        out[i] += float(wts[i, j]) * y[(i, int(e))]
            outs.append(out)
        return outs
