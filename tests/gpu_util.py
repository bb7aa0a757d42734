"""Helpers of the GPU parity tests: run the CUDA path through the C ABI and the oracle on the same
seeded inputs, and compare them with the acceptance rules of the scoring path."""
from __future__ import annotations

import numpy as np

import oracle
import synth
from synth.harness import DeviceWorkload, make_scorer

# pCVR acceptance: |gpu - oracle| <= ATOL + RTOL * |oracle| (bf16 dense compute vs fp64)
ATOL, RTOL = 2e-3, 1e-2


class GpuRun:
    def __init__(self, wl, w, graph=True, debug=True, tables=None, **cfg):
        import torch
        import cvr_ranking_model_gb300 as cvr
        self.wl, self.w = wl, w
        self.dw = DeviceWorkload(wl, tables=tables)
        self.sc = make_scorer(self.dw, w, **cfg)
        self.sc.set_option(cvr.OPT_CUDA_GRAPH, int(graph))
        n_bags = wl.n_req * 8 + wl.n_cand * 8
        self.pooled = torch.full((n_bags, 32), float("nan"), dtype=torch.float32, device="cuda:0") if debug else None
        self.rows = torch.full((max(len(wl.bag_ids), 1),), -7, dtype=torch.int64, device="cuda:0") if debug else None
        self.debug = debug

    def run(self, check=True):
        r, b, o, s, out = self.dw.ptrs()
        wl = self.wl
        if self.debug:
            st = self.sc.score_debug(wl.n_req, wl.n_cand, r, b, o, s, out, self.pooled.data_ptr(), self.rows.data_ptr(),
                                     check=check)
        else:
            st = self.sc.score(wl.n_req, wl.n_cand, r, b, o, s, out, check=check)
        return st

    def out(self):
        return self.dw.out.cpu().numpy().astype(np.float64)

    def stage(self, stage, shape, dtype):
        import torch
        t = torch.empty(shape, dtype=dtype, device="cuda:0")
        self.sc.debug_stage(stage, t.data_ptr(), t.numel() * t.element_size())
        return t.float().cpu().numpy().astype(np.float64)


def assert_pcvr_close(gpu, ref, what=""):
    ok = np.isfinite(ref).all(axis=1)
    g, r = gpu[ok], ref[ok]
    err = np.abs(g - r)
    bound = ATOL + RTOL * np.abs(r)
    worst = int(np.argmax(err - bound))
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    assert np.all(err <= bound), (f"{what}: {int((err > bound).sum())} of {err.size} pCVR values out of tolerance; "
                                 f"worst |d|={err.flat[worst]:.3e} at {worst} (ref {r.flat[worst]:.4f}); max |d|={err.max():.3e}")
    return float(err.max())


def rel_close(a, b, rtol, what=""):
    """Stage comparison relative to the stage's RMS (bf16 intermediates vs fp64)."""
    scale = np.sqrt(np.mean(b ** 2)) + 1e-30
    e = np.abs(a - b).max() / scale
    assert e <= rtol, f"{what}: max |d| / rms = {e:.3e} > {rtol}"
    return e
