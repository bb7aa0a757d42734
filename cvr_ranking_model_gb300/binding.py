"""Thin ctypes binding of the C ABI in include/cvr.h (argument marshalling only).

Every step of the scoring path runs in the CUDA kernels of libcvr.so; this module only lays out
the configuration and weight structs, passes device pointers (e.g. ``tensor.data_ptr()``) and
turns status codes into exceptions. It fails loudly when the library is missing.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Mapping, Optional, Sequence, Tuple

import numpy as np

from . import _build

MAX_LAYERS, N_USER_FIELDS, N_ITEM_FIELDS, N_GROUPS, N_EXPERTS, N_TASKS = 4, 8, 8, 3, 3, 2
STAGE_H, STAGE_Z, STAGE_Q, STAGE_Y, STAGE_EXPERTS, STAGE_GATES = range(6)
OPT_PROFILE, OPT_CUDA_GRAPH, OPT_PDL, OPT_ATTENTION_TC, OPT_PLE_INT8, OPT_KEEP_STAGES = 0, 1, 2, 3, 4, 5
NOALLOC_MAX_CAND = 1024  # CVR_NOALLOC_MAX_CAND
TIMELINE_RECORDS = 10 * 8192 * 3  # CVR_TIMELINE_RECORDS
TIMELINE_KERNELS = ["sparse", "seq_mlp", "seq_colsum", "tokenizer", "query", "attention", "token_mixer", "ple_heads",
                    "attention_tc"]

STATUS = {0: "CVR_OK", 1: "CVR_E_ARG", 2: "CVR_E_SHAPE", 3: "CVR_E_ID_RANGE", 4: "CVR_E_OOM", 5: "CVR_E_CUDA",
          6: "CVR_E_INPUT", 7: "CVR_E_TIMEOUT"}

_F = ctypes.POINTER(ctypes.c_float)


class Config(ctypes.Structure):
    _fields_ = [("n_user_fields", ctypes.c_int32), ("n_item_fields", ctypes.c_int32), ("emb_dim", ctypes.c_int32),
                ("n_tokens", ctypes.c_int32), ("token_dim", ctypes.c_int32), ("n_groups", ctypes.c_int32),
                ("seq_len", ctypes.c_int32 * 3), ("seq_cols", ctypes.c_int32), ("ffn_hidden", ctypes.c_int32),
                ("heads", ctypes.c_int32), ("n_layers", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("expert_dim", ctypes.c_int32), ("n_tasks", ctypes.c_int32), ("head_hidden", ctypes.c_int32),
                ("tau", ctypes.c_float), ("clamp", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("user_rows", ctypes.c_int64 * 8), ("item_rows", ctypes.c_int64 * 8), ("seq_rows", ctypes.c_int64)]


class Weights(ctypes.Structure):
    _fields_ = [("user_tables", _F * 8), ("item_tables", _F * 8), ("seq_table", _F), ("tok_w", _F), ("tok_b", _F)] + \
        [(n, _F * 3) for n in ("seq_w1", "seq_b1", "seq_w3", "seq_b3", "seq_w2", "seq_b2")] + \
        [("q_w", (_F * 3) * MAX_LAYERS), ("q_b", (_F * 3) * MAX_LAYERS)] + \
        [(n, _F * MAX_LAYERS) for n in ("tm_w1", "tm_b1", "tm_w3", "tm_b3", "tm_w2", "tm_b2", "tm_gain")] + \
        [("ple_w", _F * 3), ("ple_b", _F * 3)] + \
        [(n, _F * 2) for n in ("gate_w", "gate_b", "head_w1", "head_b1", "head_w2", "head_b2")]


class CvrError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{STATUS.get(status, status)}: {detail}")
        self.status = status


_lib = None


def lib() -> ctypes.CDLL:
    """Loads libcvr.so (building it in-tree first if it is absent)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            _build.build(timeline=_build.LIB == _build.LIB_TIMELINE)
        L = ctypes.CDLL(_build.LIB)
        V, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        L.cvr_create.argtypes = [V, V, V, ctypes.POINTER(V)]
        L.cvr_create.restype = ctypes.c_int
        L.cvr_score.argtypes = [V, i32, i32, V, V, V, V, V]
        L.cvr_score.restype = ctypes.c_int
        L.cvr_score_async.argtypes = [V, i32, i32, V, V, V, V, V]
        L.cvr_score_async.restype = ctypes.c_int
        L.cvr_sync.argtypes = [V]
        L.cvr_sync.restype = ctypes.c_int
        L.cvr_score_debug.argtypes = [V, i32, i32, V, V, V, V, V, V, V]
        L.cvr_score_debug.restype = ctypes.c_int
        L.cvr_score_host.argtypes = [V, i32, i32, V, V, i64, V, V, V]
        L.cvr_score_host.restype = ctypes.c_int
        L.cvr_debug_stage.argtypes = [V, i32, V, i64]
        L.cvr_debug_stage.restype = ctypes.c_int
        L.cvr_set_option.argtypes = [V, i32, i64]
        L.cvr_set_option.restype = ctypes.c_int
        L.cvr_stage_times.argtypes = [V, ctypes.POINTER(f32), ctypes.POINTER(ctypes.c_char_p), i32,
                                      ctypes.POINTER(i32)]
        L.cvr_stage_times.restype = ctypes.c_int
        L.cvr_last_launch_count.argtypes = [V]
        L.cvr_last_launch_count.restype = i32
        L.cvr_last_error.argtypes = [V]
        L.cvr_last_error.restype = ctypes.c_char_p
        L.cvr_status_string.argtypes = [ctypes.c_int]
        L.cvr_status_string.restype = ctypes.c_char_p
        L.cvr_score_varlen.argtypes = [V, i32, i32, V, V, V, V, V, V]
        L.cvr_score_varlen.restype = ctypes.c_int
        L.cvr_score_varlen_async.argtypes = [V, i32, i32, V, V, V, V, V, V]
        L.cvr_score_varlen_async.restype = ctypes.c_int
        L.cvr_selftest_wait_timeout.argtypes = [V]
        L.cvr_selftest_wait_timeout.restype = ctypes.c_int
        L.cvr_timeline.argtypes = [V, V, i64, i32]
        L.cvr_timeline.restype = ctypes.c_int
        L.cvr_predict_noalloc.argtypes = [V, i32, V, V]
        L.cvr_predict_noalloc.restype = ctypes.c_int
        L.cvr_cache_enable.argtypes = [V, i32, i64]
        L.cvr_cache_enable.restype = ctypes.c_int
        L.cvr_cache_stats.argtypes = [V, ctypes.POINTER(i64), ctypes.POINTER(i64)]
        L.cvr_cache_stats.restype = ctypes.c_int
        L.cvr_destroy.argtypes = [V]
        L.cvr_destroy.restype = None
        _lib = L
    return _lib


def make_config(seq_len: Sequence[int], n_layers: int, user_rows: Sequence[int], item_rows: Sequence[int],
                seq_rows: int, tau: float = 2.0, clamp: float = 10.0, rms_eps: float = 1e-6) -> Config:
    c = Config(n_user_fields=8, n_item_fields=8, emb_dim=32, n_tokens=13, token_dim=128, n_groups=3, seq_cols=4,
               ffn_hidden=256, heads=4, n_layers=n_layers, n_experts=3, expert_dim=256, n_tasks=2, head_hidden=128,
               tau=tau, clamp=clamp, rms_eps=rms_eps, seq_rows=seq_rows)
    for g in range(3):
        c.seq_len[g] = int(seq_len[g])
    for f in range(8):
        c.user_rows[f] = int(user_rows[f])
        c.item_rows[f] = int(item_rows[f])
    return c


def _fp(a: np.ndarray):
    return ctypes.cast(a.ctypes.data, _F)


def make_weights(tables: Sequence[int], dense: Mapping[str, np.ndarray], n_layers: int):
    """tables: 17 device pointers (8 user fields, 8 item fields, the shared sequence table).
    dense: host fp32 arrays named tok_w, tok_b, seq{g}_{w1,b1,w3,b3,w2,b2}, l{l}_q{g}_{w,b},
    l{l}_tm_{w1,b1,w3,b3,w2,b2,gain}, ple{k}_{w,b}, gate{t}_{w,b}, head{t}_{w1,b1,w2,b2}.
    Returns (struct, keep-alive list)."""
    keep = []

    def arr(name):
        a = np.ascontiguousarray(dense[name], dtype=np.float32)
        keep.append(a)
        return _fp(a)

    w = Weights()
    for f in range(8):
        w.user_tables[f] = ctypes.cast(ctypes.c_void_p(int(tables[f])), _F)
        w.item_tables[f] = ctypes.cast(ctypes.c_void_p(int(tables[8 + f])), _F)
    w.seq_table = ctypes.cast(ctypes.c_void_p(int(tables[16])), _F)
    w.tok_w, w.tok_b = arr("tok_w"), arr("tok_b")
    for g in range(3):
        for n in ("w1", "b1", "w3", "b3", "w2", "b2"):
            getattr(w, "seq_" + n)[g] = arr(f"seq{g}_{n}")
    for l in range(n_layers):
        for g in range(3):
            w.q_w[l][g] = arr(f"l{l}_q{g}_w")
            w.q_b[l][g] = arr(f"l{l}_q{g}_b")
        for n in ("w1", "b1", "w3", "b3", "w2", "b2", "gain"):
            getattr(w, "tm_" + n)[l] = arr(f"l{l}_tm_{n}")
    for k in range(3):
        w.ple_w[k], w.ple_b[k] = arr(f"ple{k}_w"), arr(f"ple{k}_b")
    for t in range(2):
        w.gate_w[t], w.gate_b[t] = arr(f"gate{t}_w"), arr(f"gate{t}_b")
        for n in ("w1", "b1", "w2", "b2"):
            getattr(w, "head_" + n)[t] = arr(f"head{t}_{n}")
    return w, keep


class Scorer:
    """One cvr_handle. Inputs of score() are device pointers (ints), e.g. torch tensors' data_ptr()."""

    def __init__(self, config: Config, weights: Weights, stream: int = 0):
        self._lib = lib()
        h = ctypes.c_void_p()
        st = self._lib.cvr_create(ctypes.byref(weights), ctypes.byref(config), ctypes.c_void_p(stream), ctypes.byref(h))
        if st != 0:
            raise CvrError(st, "cvr_create failed (see stderr)")
        self._h = h
        self.config = config

    def _check(self, st: int):
        if st != 0:
            raise CvrError(st, self._lib.cvr_last_error(self._h).decode())

    def score(self, n_req: int, n_cand: int, req_ids: int, bag_ids: int, bag_offsets: int, seq_ids: int, out: int,
              check: bool = True) -> int:
        st = self._lib.cvr_score(self._h, n_req, n_cand, req_ids, bag_ids, bag_offsets, seq_ids, out)
        if check:
            self._check(st)
        return st

    def score_varlen(self, n_req: int, n_cand: int, req_ids: int, bag_ids: int, bag_offsets: int, seq_ids: int,
                     seq_lens: int, out: int, check: bool = True) -> int:
        """cvr_score_varlen: seq_lens is a device int32 [n_req][3] of real sequence lengths."""
        st = self._lib.cvr_score_varlen(self._h, n_req, n_cand, req_ids, bag_ids, bag_offsets, seq_ids, seq_lens, out)
        if check:
            self._check(st)
        return st

    def score_varlen_async(self, n_req: int, n_cand: int, req_ids: int, bag_ids: int, bag_offsets: int,
                           seq_ids: int, seq_lens: int, out: int) -> None:
        self._check(self._lib.cvr_score_varlen_async(self._h, n_req, n_cand, req_ids, bag_ids, bag_offsets, seq_ids,
                                                     seq_lens, out))

    def score_async(self, n_req: int, n_cand: int, req_ids: int, bag_ids: int, bag_offsets: int, seq_ids: int,
                    out: int) -> None:
        self._check(self._lib.cvr_score_async(self._h, n_req, n_cand, req_ids, bag_ids, bag_offsets, seq_ids, out))

    def sync(self, check: bool = True) -> int:
        st = self._lib.cvr_sync(self._h)
        if check:
            self._check(st)
        return st

    def score_debug(self, n_req, n_cand, req_ids, bag_ids, bag_offsets, seq_ids, out, pooled: Optional[int],
                    rows: Optional[int], check: bool = True) -> int:
        st = self._lib.cvr_score_debug(self._h, n_req, n_cand, req_ids, bag_ids, bag_offsets, seq_ids, out, pooled,
                                       rows)
        if check:
            self._check(st)
        return st

    def score_host(self, n_req: int, n_cand: int, req_ids: np.ndarray, bag_ids: np.ndarray,
                   bag_offsets: np.ndarray, seq_ids: np.ndarray, out: np.ndarray, check: bool = True) -> int:
        """Host arrays (numpy, or pinned torch CPU tensors' data via numpy views)."""
        for a, dt in ((req_ids, np.int32), (bag_ids, np.int64), (bag_offsets, np.int64), (seq_ids, np.int64),
                      (out, np.float32)):
            assert a.dtype == dt and a.flags["C_CONTIGUOUS"], "host arrays must be C-contiguous with the C ABI dtypes"
        st = self._lib.cvr_score_host(self._h, n_req, n_cand, req_ids.ctypes.data, bag_ids.ctypes.data,
                                      bag_ids.size, bag_offsets.ctypes.data, seq_ids.ctypes.data, out.ctypes.data)
        if check:
            self._check(st)
        return st

    def selftest_wait_timeout(self) -> int:
        """cvr_selftest_wait_timeout: a wait that nothing ends; returns the status (7 = CVR_E_TIMEOUT)."""
        return int(self._lib.cvr_selftest_wait_timeout(self._h))

    def timeline(self, clear: bool = True) -> np.ndarray:
        """cvr_timeline: uint64 [10 kernels][8192 CTAs][3] (entry, dependency wait returned, exit; ns, 0 = none)
        of a library built with -DCVR_TIMELINE."""
        rec = np.zeros(TIMELINE_RECORDS, dtype=np.uint64)
        self._check(self._lib.cvr_timeline(self._h, rec.ctypes.data, rec.size, int(clear)))
        return rec.reshape(10, 8192, 3)

    def predict_noalloc(self, n_cand: int, y: int, out: int, check: bool = True) -> int:
        """cvr_predict_noalloc: PLE + heads on a device bf16 [n_cand][16][128] Token Mixer output, with
        no device allocation (n_cand <= NOALLOC_MAX_CAND)."""
        st = self._lib.cvr_predict_noalloc(self._h, n_cand, y, out)
        if check:
            self._check(st)
        return st

    def cache_enable(self, table: int, slots: int, check: bool = True) -> int:
        """cvr_cache_enable: a hot-row cache of `slots` rows (power of two, 0 = none) in front of table
        0..7 (user), 8..15 (item) or 16 (sequence)."""
        st = self._lib.cvr_cache_enable(self._h, table, slots)
        if check:
            self._check(st)
        return st

    def cache_stats(self) -> Tuple[int, int]:
        """cvr_cache_stats: (hits, misses) since the last read."""
        hits, misses = ctypes.c_int64(0), ctypes.c_int64(0)
        self._check(self._lib.cvr_cache_stats(self._h, ctypes.byref(hits), ctypes.byref(misses)))
        return int(hits.value), int(misses.value)

    def debug_stage(self, stage: int, dst: int, nbytes: int) -> None:
        self._check(self._lib.cvr_debug_stage(self._h, stage, dst, nbytes))

    def set_option(self, option: int, value: int) -> None:
        self._check(self._lib.cvr_set_option(self._h, option, value))

    def stage_times(self) -> Dict[str, float]:
        cap = 64
        ms = (ctypes.c_float * cap)()
        names = (ctypes.c_char_p * cap)()
        n = ctypes.c_int32()
        self._check(self._lib.cvr_stage_times(self._h, ms, names, cap, ctypes.byref(n)))
        out: Dict[str, float] = {}
        for i in range(n.value):
            k = names[i].decode()
            out[k] = out.get(k, 0.0) + ms[i]
        return out

    def stage_list(self):
        cap = 64
        ms = (ctypes.c_float * cap)()
        names = (ctypes.c_char_p * cap)()
        n = ctypes.c_int32()
        self._check(self._lib.cvr_stage_times(self._h, ms, names, cap, ctypes.byref(n)))
        return [(names[i].decode(), ms[i]) for i in range(n.value)]

    def last_launch_count(self) -> int:
        return int(self._lib.cvr_last_launch_count(self._h))

    def last_error(self) -> str:
        return self._lib.cvr_last_error(self._h).decode()

    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.cvr_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


EXPORTED = ["cvr_create", "cvr_score", "cvr_score_async", "cvr_sync", "cvr_score_debug", "cvr_score_host", "cvr_debug_stage", "cvr_set_option",
            "cvr_stage_times", "cvr_last_launch_count", "cvr_last_error", "cvr_status_string", "cvr_destroy"]
