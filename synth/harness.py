"""Places a synthetic workload on the GPU and builds a scorer over it (tests, smoke check, benchmark).

Tables are filled on the device by the seeded generator; the sparse inputs are uploaded as torch
tensors; the scorer is created through the C ABI binding. No model arithmetic happens here.
"""
from __future__ import annotations

from typing import Dict, List, Optional

import numpy as np

import synth


class DeviceWorkload:
    def __init__(self, wl: "synth.Workload", device: str = "cuda:0", tables: Optional[List] = None):
        import torch
        self.wl = wl
        self.device = device
        E = synth.DIMS["emb_dim"]
        if tables is None:
            tables = []
            stream = torch.cuda.current_stream(device).cuda_stream
            for t in list(range(16)) + [synth.SEQ_TABLE]:
                buf = torch.empty((wl.table_rows(t), E), dtype=torch.float32, device=device)
                synth.fill_device_table(buf.data_ptr(), wl, t, stream)
                tables.append(buf)
            torch.cuda.synchronize(device)
        self.tables = tables
        self.req_ids = torch.from_numpy(np.ascontiguousarray(wl.req_ids)).to(device)
        self.bag_ids = torch.from_numpy(wl.bag_ids).to(device)
        self.bag_offsets = torch.from_numpy(wl.bag_offsets).to(device)
        self.seq_ids = torch.from_numpy(np.ascontiguousarray(wl.seq_ids)).to(device)
        self.out = torch.empty((wl.n_cand, synth.DIMS["n_tasks"]), dtype=torch.float32, device=device)

    def ptrs(self):
        return (self.req_ids.data_ptr(), self.bag_ids.data_ptr(), self.bag_offsets.data_ptr(),
                self.seq_ids.data_ptr(), self.out.data_ptr())


def make_scorer(dw: DeviceWorkload, weights: Dict[str, np.ndarray], stream: int = 0, **cfg_over):
    import cvr_ranking_model_gb300 as cvr
    wl = dw.wl
    d = synth.DIMS
    cfg = cvr.make_config(seq_len=wl.seq_len, n_layers=wl.n_layers, user_rows=[wl.user_rows] * 8,
                          item_rows=[wl.item_rows] * 8, seq_rows=wl.seq_rows,
                          tau=cfg_over.get("tau", d["tau"]), clamp=cfg_over.get("clamp", d["clamp"]),
                          rms_eps=cfg_over.get("rms_eps", d["rms_eps"]))
    w, keep = cvr.make_weights([t.data_ptr() for t in dw.tables], weights, wl.n_layers)
    sc = cvr.Scorer(cfg, w, stream)
    sc._keep = keep
    return sc


def score(sc, dw: DeviceWorkload, check: bool = True) -> int:
    wl = dw.wl
    r, b, o, s, out = dw.ptrs()
    return sc.score(wl.n_req, wl.n_cand, r, b, o, s, out, check=check)
