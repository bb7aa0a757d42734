"""Seeded synthetic workloads for the CVR scoring path (inputs only, no model arithmetic).

The five workloads are the ones the scoring path is specified on: a tiny CPU-sized
case, the production shape, a long-sequence variant, an embedding-heavy variant and
a two-layer interaction stack. Every table entry, id and weight is a pure function
of (seed, stream, index) implemented in ``cvr_synth.c`` / ``cvr_synth.h``; this file
only sizes the arrays, calls that library through ctypes and names the dense weights.

Both the CUDA scoring path and the CPU oracle take their inputs from here and from
nowhere else.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
_HOST_LIB = os.path.join(HERE, "libcvr_synth.so")
_FILL_LIB = os.path.join(HERE, "libcvr_synth_fill.so")

# Model dimensions fixed by the workload definitions (HyFormer-style CVR model).
DIMS = dict(
    n_user_fields=8, n_item_fields=8, emb_dim=32, n_tokens=13, token_dim=128, n_groups=3,
    seq_cols=4, ffn_hidden=256, heads=4, n_experts=3, expert_dim=256, n_tasks=2, head_hidden=128,
    tau=2.0, clamp=10.0, rms_eps=1e-6,
)

# Workloads: requests R x candidates C, per-group sequence lengths, table sizes, id law.
CONFIGS: Dict[str, dict] = {
    "tiny": dict(index=0, n_req=2, n_cand=4, seq_len=(16, 16, 16), user_rows=1000, item_rows=1000,
                 seq_rows=10_000, bag_min=1, bag_max=4, zipf_s=1.1, n_layers=1),
    "prod": dict(index=1, n_req=8, n_cand=512, seq_len=(50, 100, 200), user_rows=100_000, item_rows=100_000,
                 seq_rows=1_000_000, bag_min=1, bag_max=8, zipf_s=1.1, n_layers=1),
    "longseq": dict(index=2, n_req=16, n_cand=256, seq_len=(1000, 1000, 2000), user_rows=100_000,
                    item_rows=100_000, seq_rows=1_000_000, bag_min=1, bag_max=8, zipf_s=1.1, n_layers=1),
    "embheavy": dict(index=3, n_req=64, n_cand=500, seq_len=(50, 100, 200), user_rows=100_000,
                     item_rows=5_000_000, seq_rows=100_000_000, bag_min=1, bag_max=8, zipf_s=1.05, n_layers=1),
    "deep": dict(index=4, n_req=32, n_cand=512, seq_len=(200, 200, 500), user_rows=100_000, item_rows=100_000,
                 seq_rows=1_000_000, bag_min=1, bag_max=8, zipf_s=1.1, n_layers=2),
}
TABLE_SCALE = 0.05  # tables ~ U(-0.05, 0.05)
SEQ_TABLE = 16      # table index of the shared sequence table (0..15 are the per-field tables)


# ----------------------------------------------------------------------------------------------
# build + load
def build(verbose: bool = False) -> None:
    """Compile the host generator (gcc) and the device table fill (nvcc, sm_103a)."""
    src = os.path.join(HERE, "cvr_synth.c")
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-o", _HOST_LIB, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=not verbose)
    fill = os.path.join(HERE, "synth_fill.cu")
    cmd = ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-Xcompiler", "-fPIC",
           "-shared", "-fmad=false", "-o", _FILL_LIB, fill]
    subprocess.run(cmd, check=True, capture_output=not verbose)


_lib = None
_fill = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(_HOST_LIB):
            build()
        L = ctypes.CDLL(_HOST_LIB)
        u64, u32, i64, i32, dbl = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
        P = ctypes.c_void_p
        L.synth_table_rows.argtypes = [u64, u32, u64, u64, u32, dbl, P]
        L.synth_uniform_bf16.argtypes = [u64, u32, i64, dbl, P]
        L.synth_zipf_rank.argtypes = [u64, u32, u64, i64, dbl]
        L.synth_zipf_rank.restype = i64
        L.synth_rank_to_row.argtypes = [u64, u32, i64, i64]
        L.synth_rank_to_row.restype = i64
        L.synth_bags.argtypes = [u64, i64, P, P, i32, i32, dbl, P, P]
        L.synth_seq_ids.argtypes = [u64, i64, i64, i32, i64, dbl, P]
        L.synth_seq_lens.argtypes = [u64, i64, i32, P, i32, P]
        _lib = L
    return _lib


def fill_lib() -> ctypes.CDLL:
    global _fill
    if _fill is None:
        if not os.path.exists(_FILL_LIB):
            build()
        L = ctypes.CDLL(_FILL_LIB)
        L.synth_fill_table_device.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64,
                                              ctypes.c_uint32, ctypes.c_double, ctypes.c_void_p]
        L.synth_fill_table_device.restype = ctypes.c_int
        _fill = L
    return _fill


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ----------------------------------------------------------------------------------------------
# workloads
@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    n_req: int
    n_cand: int
    seq_len: Tuple[int, int, int]
    n_layers: int
    user_rows: int
    item_rows: int
    seq_rows: int
    zipf_s: float
    table_scale: float
    cand_per_req: np.ndarray      # [n_req] int64
    req_ids: np.ndarray           # [n_cand] int32, non-decreasing request index of each candidate
    bag_offsets: np.ndarray       # [n_req*Fu + n_cand*Fi + 1] int64 CSR (user bags by (r,f), then item bags by (c,f))
    bag_ids: np.ndarray           # [nnz] int64 field-local row ids
    seq_ids: np.ndarray           # [n_req][sum_len][4] int64 row ids of the shared sequence table

    @property
    def sum_len(self) -> int:
        return int(sum(self.seq_len))

    def table_rows(self, t: int) -> int:
        if t == SEQ_TABLE:
            return self.seq_rows
        return self.user_rows if t < DIMS["n_user_fields"] else self.item_rows

    def host_table(self, t: int, row0: int = 0, nrows: Optional[int] = None) -> np.ndarray:
        """Rows [row0, row0+nrows) of table t as fp32 [nrows][32] (evaluated on demand)."""
        if nrows is None:
            nrows = self.table_rows(t) - row0
        out = np.empty((nrows, DIMS["emb_dim"]), dtype=np.float32)
        lib().synth_table_rows(self.seed, t, row0, nrows, DIMS["emb_dim"], self.table_scale, _ptr(out))
        return out


def default_seed(name: str) -> int:
    """Seed of a named workload's inputs and weights."""
    return 0xC0FFEE + CONFIGS[name]["index"]


def make_workload(name: str, n_req: Optional[int] = None, n_cand: Optional[int] = None,
                  cand_per_req: Optional[Sequence[int]] = None, seq_len: Optional[Sequence[int]] = None,
                  seed: Optional[int] = None, table_scale: float = TABLE_SCALE, **over) -> Workload:
    """Draws the sparse inputs of a workload. ``n_cand`` is candidates per request, or pass
    ``cand_per_req`` for a ragged mix. Table contents are not drawn here (see host_table / fill_device)."""
    c = dict(CONFIGS[name])
    c.update(over)
    R = int(n_req if n_req is not None else c["n_req"])
    if cand_per_req is None:
        C = int(n_cand if n_cand is not None else c["n_cand"])
        cand_per_req = [C] * R
    cpr = np.asarray(cand_per_req, dtype=np.int64)
    assert len(cpr) == R
    B = int(cpr.sum())
    L = tuple(int(x) for x in (seq_len if seq_len is not None else c["seq_len"]))
    sd = int(seed if seed is not None else default_seed(name))
    Fu, Fi = DIMS["n_user_fields"], DIMS["n_item_fields"]
    n_bags = R * Fu + B * Fi
    field = np.empty(n_bags, dtype=np.int32)
    field[: R * Fu] = np.tile(np.arange(Fu, dtype=np.int32), R)
    field[R * Fu:] = np.tile(np.arange(Fu, Fu + Fi, dtype=np.int32), B)
    rows = np.array([c["user_rows"]] * Fu + [c["item_rows"]] * Fi, dtype=np.int64)
    assert 0 <= c["bag_min"] <= c["bag_max"] <= 64  # bag_min = 0 draws empty bags
    offsets = np.empty(n_bags + 1, dtype=np.int64)
    lib().synth_bags(sd, n_bags, _ptr(field), _ptr(rows), c["bag_min"], c["bag_max"], c["zipf_s"], _ptr(offsets), None)
    ids = np.empty(int(offsets[-1]), dtype=np.int64)
    lib().synth_bags(sd, n_bags, _ptr(field), _ptr(rows), c["bag_min"], c["bag_max"], c["zipf_s"], _ptr(offsets),
                     _ptr(ids))
    SL = sum(L)
    seq = np.empty((R, SL, DIMS["seq_cols"]), dtype=np.int64)
    lib().synth_seq_ids(sd, R, SL, DIMS["seq_cols"], c["seq_rows"], c["zipf_s"], _ptr(seq))
    req_ids = np.repeat(np.arange(R, dtype=np.int32), cpr)
    return Workload(name=name, seed=sd, n_req=R, n_cand=B, seq_len=L, n_layers=int(c["n_layers"]),
                    user_rows=int(c["user_rows"]), item_rows=int(c["item_rows"]), seq_rows=int(c["seq_rows"]),
                    zipf_s=float(c["zipf_s"]), table_scale=float(table_scale), cand_per_req=cpr, req_ids=req_ids,
                    bag_offsets=offsets, bag_ids=ids, seq_ids=seq)


def make_seq_lens(wl: Workload, min_len: int = 0, seed: Optional[int] = None) -> np.ndarray:
    """Variable sequence lengths [n_req][3] int32: the events each request really has in each group,
    uniform in [min_len, seq_len[g]]."""
    L = np.ascontiguousarray(wl.seq_len, dtype=np.int32)
    out = np.empty((wl.n_req, DIMS["n_groups"]), dtype=np.int32)
    lib().synth_seq_lens(int(seed if seed is not None else wl.seed), wl.n_req, DIMS["n_groups"], _ptr(L), int(min_len),
                         _ptr(out))
    return out


def pad_seq_ids(wl: Workload, lens: np.ndarray, fill: int) -> np.ndarray:
    """seq_ids with every padding slot (past a request's length) set to ``fill``."""
    ids = wl.seq_ids.copy()
    base = 0
    for g, L in enumerate(wl.seq_len):
        for r in range(wl.n_req):
            ids[r, base + int(lens[r, g]): base + L, :] = fill
        base += L
    return ids


# ----------------------------------------------------------------------------------------------
# dense weights: (name, shape, kind); kind 'w' = Glorot-uniform, 'b' = bias, 'g' = RMSNorm gain.
def weight_specs(n_layers: int) -> List[Tuple[str, Tuple[int, ...], str]]:
    D, H, T = DIMS["token_dim"], DIMS["ffn_hidden"], DIMS["n_tokens"]
    IN = (DIMS["n_user_fields"] + DIMS["n_item_fields"]) * DIMS["emb_dim"]
    X = T * D
    specs: List[Tuple[str, Tuple[int, ...], str]] = [("tok_w", (X, IN), "w"), ("tok_b", (X,), "b")]
    for g in range(DIMS["n_groups"]):
        specs += [(f"seq{g}_w1", (H, D), "w"), (f"seq{g}_b1", (H,), "b"), (f"seq{g}_w3", (H, D), "w"),
                  (f"seq{g}_b3", (H,), "b"), (f"seq{g}_w2", (D, H), "w"), (f"seq{g}_b2", (D,), "b")]
    for l in range(n_layers):
        for g in range(DIMS["n_groups"]):
            specs += [(f"l{l}_q{g}_w", (D, X + D), "w"), (f"l{l}_q{g}_b", (D,), "b")]
        specs += [(f"l{l}_tm_w1", (H, D), "w"), (f"l{l}_tm_b1", (H,), "b"), (f"l{l}_tm_w3", (H, D), "w"),
                  (f"l{l}_tm_b3", (H,), "b"), (f"l{l}_tm_w2", (D, H), "w"), (f"l{l}_tm_b2", (D,), "b"),
                  (f"l{l}_tm_gain", (D,), "g")]
    YD = (T + DIMS["n_groups"]) * D
    for k in range(DIMS["n_experts"]):
        specs += [(f"ple{k}_w", (DIMS["expert_dim"], YD), "w"), (f"ple{k}_b", (DIMS["expert_dim"],), "b")]
    for t in range(DIMS["n_tasks"]):
        specs += [(f"gate{t}_w", (DIMS["n_experts"], YD), "w"), (f"gate{t}_b", (DIMS["n_experts"],), "b")]
    for t in range(DIMS["n_tasks"]):
        specs += [(f"head{t}_w1", (DIMS["head_hidden"], DIMS["expert_dim"]), "w"),
                  (f"head{t}_b1", (DIMS["head_hidden"],), "b"),
                  (f"head{t}_w2", (1, DIMS["head_hidden"]), "w"), (f"head{t}_b2", (1,), "b")]
    return specs


def make_weights(n_layers: int, seed: int, bias_scale: float = 0.0, gain_jitter: float = 0.0,
                 weight_scale: float = 1.0) -> Dict[str, np.ndarray]:
    """Dense weights as bf16-valued fp32 arrays in [out][in] layout.

    Matrices are Glorot-uniform U(+-sqrt(6/(fan_in+fan_out))) (times ``weight_scale``), biases are
    zero unless ``bias_scale`` > 0 (then U(+-bias_scale)), RMSNorm gains are 1 (+ U(+-gain_jitter))."""
    out: Dict[str, np.ndarray] = {}
    for i, (name, shape, kind) in enumerate(weight_specs(n_layers)):
        n = int(np.prod(shape))
        a = np.zeros(n, dtype=np.float32)
        stream = 0x1000 + i
        if kind == "w":
            bound = math.sqrt(6.0 / (shape[0] + shape[1])) * weight_scale
            lib().synth_uniform_bf16(seed, stream, n, bound, _ptr(a))
        elif kind == "b":
            if bias_scale > 0:
                lib().synth_uniform_bf16(seed, stream, n, bias_scale, _ptr(a))
        else:
            if gain_jitter > 0:
                lib().synth_uniform_bf16(seed, stream, n, gain_jitter, _ptr(a))
            a = (a + np.float32(1.0)).astype(np.float32)
            # 1 + jitter is rounded once more to bf16 so that the gain stays bf16-valued
            u = a.view(np.uint32).astype(np.uint64)
            u = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
            a = u.view(np.float32)
        out[name] = a.reshape(shape)
    return out


def fill_device_table(ptr: int, wl: Workload, t: int, stream_handle: int = 0) -> None:
    """Writes table t of the workload into device memory at ``ptr`` ([rows][32] fp32)."""
    rc = fill_lib().synth_fill_table_device(ptr, wl.seed, t, wl.table_rows(t), DIMS["emb_dim"], wl.table_scale,
                                            stream_handle)
    if rc != 0:
        raise RuntimeError(f"synth_fill_table_device failed with CUDA error {rc}")
