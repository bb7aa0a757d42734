"""CPU oracle of the CVR scoring forward pass -- TEST INFRASTRUCTURE.

A plain fp64 loop-nest restatement of the model (``cvr_oracle.c``), loaded through ctypes.
Only the tests, the smoke check and the benchmark's CPU-baseline leg may use it; the scoring
library never loads it and shares no code with it. See ``cvr_oracle.h`` for the sources of
each step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Dict, Optional, Sequence

import numpy as np

import synth

HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = os.path.join(HERE, "liboracle.so")

MAX_GROUPS, MAX_LAYERS, MAX_EXPERTS, MAX_TASKS = 3, 4, 8, 4
E_ARG, E_ID_RANGE = 1, 3

_P = ctypes.POINTER(ctypes.c_float)


class Model(ctypes.Structure):
    _fields_ = [("n_user_fields", ctypes.c_int32), ("n_item_fields", ctypes.c_int32), ("emb_dim", ctypes.c_int32),
                ("n_tokens", ctypes.c_int32), ("token_dim", ctypes.c_int32), ("n_groups", ctypes.c_int32),
                ("seq_len", ctypes.c_int32 * MAX_GROUPS), ("seq_cols", ctypes.c_int32),
                ("ffn_hidden", ctypes.c_int32), ("heads", ctypes.c_int32), ("n_layers", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("expert_dim", ctypes.c_int32), ("n_tasks", ctypes.c_int32),
                ("head_hidden", ctypes.c_int32), ("tau", ctypes.c_double), ("clamp", ctypes.c_double),
                ("rms_eps", ctypes.c_double)]


class Table(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("rows", ctypes.c_int64), ("seed", ctypes.c_uint64),
                ("index", ctypes.c_uint32), ("scale", ctypes.c_double)]


class Weights(ctypes.Structure):
    _fields_ = [("tok_w", _P), ("tok_b", _P)] + \
        [(n, _P * MAX_GROUPS) for n in ("seq_w1", "seq_b1", "seq_w3", "seq_b3", "seq_w2", "seq_b2")] + \
        [("q_w", (_P * MAX_GROUPS) * MAX_LAYERS), ("q_b", (_P * MAX_GROUPS) * MAX_LAYERS)] + \
        [(n, _P * MAX_LAYERS) for n in ("tm_w1", "tm_b1", "tm_w3", "tm_b3", "tm_w2", "tm_b2", "tm_gain")] + \
        [("ple_w", _P * MAX_EXPERTS), ("ple_b", _P * MAX_EXPERTS)] + \
        [(n, _P * MAX_TASKS) for n in ("gate_w", "gate_b", "head_w1", "head_b1", "head_w2", "head_b2")]


class Dumps(ctypes.Structure):
    _fields_ = [("pooled", ctypes.c_void_p), ("rows", ctypes.c_void_p), ("H", ctypes.c_void_p),
                ("Q", ctypes.c_void_p), ("Z", ctypes.c_void_p), ("Y", ctypes.c_void_p), ("R", ctypes.c_void_p)]


def build(verbose: bool = False) -> None:
    """Compile the oracle (plain C, fp64, OpenMP) together with the seeded generator it reads tables from."""
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off", "-o", _LIB,
           os.path.join(HERE, "cvr_oracle.c"), os.path.join(synth.HERE, "cvr_synth.c"), "-lm"]
    subprocess.run(cmd, check=True, capture_output=not verbose)


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB):
            build()
        L = ctypes.CDLL(_LIB)
        V, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        L.oracle_score.argtypes = [V, V, V, i32, i32, V, V, V, V, V, i32, V, V, i32]
        L.oracle_score.restype = ctypes.c_int
        L.oracle_score_lens.argtypes = [V, V, V, i32, i32, V, V, V, V, V, V, i32, V, V, i32]
        L.oracle_score_lens.restype = ctypes.c_int
        L.oracle_pool_bag.argtypes = [V, V, i64, i32, dbl, V, V]
        L.oracle_pool_bag.restype = ctypes.c_int
        L.oracle_bf16.argtypes = [ctypes.c_float]
        L.oracle_bf16.restype = dbl
        L.oracle_swiglu.argtypes = [V, i32, i32, i32, V, V, V, V, V, V, V]
        L.oracle_tokenize.argtypes = [V, i32, V, i32, V, V, i32, i32, V]
        L.oracle_query.argtypes = [V, i32, i32, V, V, V, V]
        L.oracle_cross_attention.argtypes = [V, V, i32, i32, i32, dbl, V, V]
        L.oracle_mix.argtypes = [V, i32, i32, V]
        L.oracle_revert.argtypes = [V, i32, i32, V]
        L.oracle_rmsnorm.argtypes = [V, i32, V, dbl, V]
        L.oracle_token_mixer.argtypes = [V, i32, i32, i32, V, V, V, V, V, V, V, dbl, V]
        L.oracle_ple.argtypes = [V, i32, i32, i32, i32, V, V, V, V, V, V]
        L.oracle_head.argtypes = [V, i32, i32, V, V, V, V]
        L.oracle_head.restype = dbl
        L.oracle_threads.argtypes = [i32]
        L.oracle_threads.restype = i32
        _lib = L
    return _lib


def _p(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _fp(a: Optional[np.ndarray]):
    return ctypes.cast(a.ctypes.data, _P) if a is not None else _P()


def f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def model_struct(wl: "synth.Workload", **over) -> Model:
    d = synth.DIMS
    m = Model()
    for k in ("n_user_fields", "n_item_fields", "emb_dim", "n_tokens", "token_dim", "n_groups", "seq_cols",
              "ffn_hidden", "heads", "n_experts", "expert_dim", "n_tasks", "head_hidden"):
        setattr(m, k, d[k])
    for g in range(d["n_groups"]):
        m.seq_len[g] = wl.seq_len[g]
    m.n_layers = wl.n_layers
    m.tau, m.clamp, m.rms_eps = d["tau"], d["clamp"], d["rms_eps"]
    for k, v in over.items():
        setattr(m, k, v)
    return m


def weights_struct(w: Dict[str, np.ndarray], n_layers: int) -> Weights:
    """Fills the oracle's weight struct; the arrays in ``w`` must stay alive while it is used."""
    s = Weights()
    s.tok_w, s.tok_b = _fp(w["tok_w"]), _fp(w["tok_b"])
    for g in range(synth.DIMS["n_groups"]):
        for n in ("w1", "b1", "w3", "b3", "w2", "b2"):
            getattr(s, "seq_" + n)[g] = _fp(w[f"seq{g}_{n}"])
    for l in range(n_layers):
        for g in range(synth.DIMS["n_groups"]):
            s.q_w[l][g] = _fp(w[f"l{l}_q{g}_w"])
            s.q_b[l][g] = _fp(w[f"l{l}_q{g}_b"])
        for n in ("w1", "b1", "w3", "b3", "w2", "b2", "gain"):
            getattr(s, "tm_" + n)[l] = _fp(w[f"l{l}_tm_{n}"])
    for k in range(synth.DIMS["n_experts"]):
        s.ple_w[k], s.ple_b[k] = _fp(w[f"ple{k}_w"]), _fp(w[f"ple{k}_b"])
    for t in range(synth.DIMS["n_tasks"]):
        s.gate_w[t], s.gate_b[t] = _fp(w[f"gate{t}_w"]), _fp(w[f"gate{t}_b"])
        for n in ("w1", "b1", "w2", "b2"):
            getattr(s, "head_" + n)[t] = _fp(w[f"head{t}_{n}"])
    return s


def tables_array(wl: "synth.Workload", host_tables: Optional[Dict[int, np.ndarray]] = None):
    """Table descriptors for the oracle: materialised where given, else generated on demand."""
    n = synth.DIMS["n_user_fields"] + synth.DIMS["n_item_fields"] + 1
    arr = (Table * n)()
    for t in range(n):
        tab = synth.SEQ_TABLE if t == n - 1 else t
        data = host_tables.get(tab) if host_tables else None
        arr[t].data = _p(data) if data is not None else None
        arr[t].rows = wl.table_rows(tab)
        arr[t].seed, arr[t].index, arr[t].scale = wl.seed, tab, wl.table_scale
    return arr


class Result:
    def __init__(self, out, status, dumps):
        self.out = out
        self.status = status
        self.dumps = dumps


def score(wl: "synth.Workload", w: Dict[str, np.ndarray], requests: Optional[Sequence[int]] = None,
          dumps: bool = False, threads: int = 0, host_tables: Optional[Dict[int, np.ndarray]] = None,
          seq_lens: Optional[np.ndarray] = None, **model_over) -> Result:
    """Runs the oracle over ``requests`` (default: all). ``out`` is [n_cand][n_tasks] fp64 (NaN for the
    candidates of requests not scored). ``seq_lens`` [n_req][3]: events each request really has per group
    (variable-length sequences; None = every slot). ``model_over`` overrides tau, clamp or rms_eps."""
    d = synth.DIMS
    m = model_struct(wl, **model_over)
    ws = weights_struct(w, wl.n_layers)
    tabs = tables_array(wl, host_tables)
    B, R, SL, D = wl.n_cand, wl.n_req, wl.sum_len, d["token_dim"]
    T = d["n_tokens"] + d["n_groups"]
    out = np.full((B, d["n_tasks"]), np.nan, dtype=np.float64)
    dm = None
    dstruct = None
    if dumps:
        nb = R * d["n_user_fields"] + B * d["n_item_fields"]
        dm = dict(pooled=np.full((nb, d["emb_dim"]), np.nan, np.float32),
                  rows=np.full(len(wl.bag_ids), -1, np.int64),
                  H=np.full((R, SL, D), np.nan), Q=np.full((wl.n_layers, B, d["n_groups"], D), np.nan),
                  Z=np.full((wl.n_layers, B, T, D), np.nan), Y=np.full((wl.n_layers, B, T, D), np.nan),
                  R=np.full((B, d["n_tasks"], d["expert_dim"]), np.nan))
        dstruct = Dumps(*[_p(dm[k]) for k in ("pooled", "rows", "H", "Q", "Z", "Y", "R")])
    sub = None if requests is None else np.ascontiguousarray(requests, dtype=np.int32)
    req_ids = np.ascontiguousarray(wl.req_ids, dtype=np.int32)
    lens = None if seq_lens is None else np.ascontiguousarray(seq_lens, dtype=np.int32)
    st = lib().oracle_score_lens(ctypes.byref(m), ctypes.addressof(tabs), ctypes.byref(ws), R, B, _p(req_ids),
                                 _p(wl.bag_offsets), _p(wl.bag_ids), _p(wl.seq_ids), _p(lens), _p(sub),
                                 0 if sub is None else len(sub), _p(out),
                                 ctypes.byref(dstruct) if dstruct is not None else None, threads)
    return Result(out, st, dm)


def threads_used(threads: int = 0) -> int:
    return int(lib().oracle_threads(threads))


# ---- single stages (for the pins) ----
def pool_bag(table: np.ndarray, ids, clamp: float = 10.0):
    table = f32(table)
    ids = np.ascontiguousarray(ids, dtype=np.int64)
    t = Table(_p(table), table.shape[0], 0, 0, 0.0)
    out = np.empty(table.shape[1], np.float32)
    rows = np.empty(max(len(ids), 1), np.int64)
    st = lib().oracle_pool_bag(ctypes.byref(t), _p(ids), len(ids), table.shape[1], clamp, _p(out), _p(rows))
    return out, rows[: len(ids)], st


def bf16(x: float) -> float:
    return float(lib().oracle_bf16(x))


def swiglu(x, w1, b1, w3, b3, w2, b2) -> np.ndarray:
    x, w1, b1, w3, b3, w2, b2 = f64(x), f32(w1), f32(b1), f32(w3), f32(b3), f32(w2), f32(b2)
    y = np.empty(w2.shape[0])
    lib().oracle_swiglu(_p(x), x.size, w1.shape[0], w2.shape[0], _p(w1), _p(b1), _p(w3), _p(b3), _p(w2), _p(b2),
                        _p(y))
    return y


def tokenize(u, it, w, b, n_tokens, token_dim) -> np.ndarray:
    u, it, w, b = f64(u), f64(it), f32(w), f32(b)
    x = np.empty((n_tokens, token_dim))
    lib().oracle_tokenize(_p(u), u.size, _p(it), it.size, _p(w), _p(b), n_tokens, token_dim, _p(x))
    return x


def query(x, m_g, w, b) -> np.ndarray:
    x, m_g, w, b = f64(x), f64(m_g), f32(w), f32(b)
    q = np.empty(w.shape[0])
    lib().oracle_query(_p(x), x.shape[0], x.shape[1], _p(m_g), _p(w), _p(b), _p(q))
    return q


def cross_attention(q, H, heads, tau):
    q, H = f64(q), f64(H)
    L, D = H.shape
    d = np.empty(D)
    probs = np.empty((heads, max(L, 1)))
    lib().oracle_cross_attention(_p(q), _p(H), L, D, heads, tau, _p(d), _p(probs))
    return d, probs[:, :L]


def mix(z) -> np.ndarray:
    z = f64(z)
    out = np.empty_like(z)
    lib().oracle_mix(_p(z), z.shape[0], z.shape[1], _p(out))
    return out


def revert(m) -> np.ndarray:
    m = f64(m)
    out = np.empty_like(m)
    lib().oracle_revert(_p(m), m.shape[0], m.shape[1], _p(out))
    return out


def rmsnorm(x, gain, eps) -> np.ndarray:
    x, gain = f64(x), f32(gain)
    y = np.empty_like(x)
    lib().oracle_rmsnorm(_p(x), x.size, _p(gain), eps, _p(y))
    return y


def token_mixer(z, w1, b1, w3, b3, w2, b2, gain, eps) -> np.ndarray:
    z = f64(z)
    args = [f32(a) for a in (w1, b1, w3, b3, w2, b2, gain)]
    y = np.empty_like(z)
    lib().oracle_token_mixer(_p(z), z.shape[0], z.shape[1], args[0].shape[0], *[_p(a) for a in args], eps, _p(y))
    return y


def ple(y, we, be, wg, bg):
    y = f64(y)
    we, be, wg, bg = [f32(a) for a in we], [f32(a) for a in be], [f32(a) for a in wg], [f32(a) for a in bg]
    nE, nT, de = len(we), len(wg), we[0].shape[0]
    keep = [(ctypes.c_void_p * len(L))(*[_p(a) for a in L]) for L in (we, be, wg, bg)]
    r = np.empty((nT, de))
    gates = np.empty((nT, nE))
    lib().oracle_ple(_p(y), y.size, nE, de, nT, *[ctypes.addressof(k) for k in keep], _p(r), _p(gates))
    return r, gates


def head(r, w1, b1, w2, b2) -> float:
    r, w1, b1, w2, b2 = f64(r), f32(w1), f32(b1), f32(w2), f32(b2)
    return float(lib().oracle_head(_p(r), r.size, w1.shape[0], _p(w1), _p(b1), _p(w2), _p(b2)))
