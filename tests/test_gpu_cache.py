"""Hot-row cache in HBM in front of embedding tables kept in host memory (cvr_cache_enable).

The item tables and the shared sequence table are moved to pinned host memory, which the GPU reads
directly; caches of a few thousand slots sit in front of them. Cached rows are exact copies, so every
call must give the same bits as the all-HBM path -- pooled fp32 values, resolved rows and pCVR -- whatever
hits or misses; repeated and varying batches exercise admission and eviction, and the hit counts show the
cache warming up.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import GpuRun, assert_pcvr_close

pytestmark = pytest.mark.gpu

HOST_TABLES = list(range(8, 16)) + [16]  # item fields and the sequence table


def _host_tables(dw):
    import torch
    tables = []
    for t, buf in enumerate(dw.tables):
        if t in HOST_TABLES:
            h = torch.empty(buf.shape, dtype=buf.dtype, pin_memory=True)
            h.copy_(buf)
            tables.append(h)
        else:
            tables.append(buf)
    return tables


def _run(g):
    g.run()
    return g.pooled.cpu().numpy().copy(), g.rows.cpu().numpy().copy(), g.dw.out.cpu().numpy().copy()


def _assert_same(a, b, what):
    for x, y, name in zip(a, b, ("pooled", "rows", "pCVR")):
        assert np.array_equal(x, y, equal_nan=True), f"{what}: {name} differs from the all-HBM path"


def _assert_oracle(got, wl, w, what, requests=None):
    """The cached call against the CPU oracle itself: pooled fp32 bits and resolved rows of the scored
    requests' bags, and pCVR within the acceptance tolerance."""
    pooled, rows, out = got
    ref = oracle.score(wl, w, dumps=True, requests=requests)
    assert ref.status == 0
    sel = np.ones(wl.n_cand, bool) if requests is None else np.isin(wl.req_ids, requests)
    reqs = range(wl.n_req) if requests is None else requests
    bags = np.concatenate([np.arange(r * 8, r * 8 + 8) for r in reqs] +
                          [wl.n_req * 8 + np.arange(c * 8, c * 8 + 8) for c in np.nonzero(sel)[0]])
    assert np.array_equal(pooled[bags].view(np.uint32), ref.dumps["pooled"][bags].view(np.uint32)), \
        f"{what}: pooled fp32 not bit-exact with the oracle"
    for bag in bags:
        lo, hi = wl.bag_offsets[bag], wl.bag_offsets[bag + 1]
        assert np.array_equal(rows[lo:hi], ref.dumps["rows"][lo:hi]), f"{what}: rows of bag {bag} differ"
    assert_pcvr_close(out.astype(np.float64)[sel], ref.out[sel], what)


def _workload(seed=None, n_req=2):
    return synth.make_workload("prod", n_req=n_req, seed=seed)


def test_cached_host_tables_give_identical_bits_and_warm_up():
    import torch
    wl = _workload()
    w = synth.make_weights(wl.n_layers, wl.seed)
    base = GpuRun(wl, w)
    ref = _run(base)
    torch.cuda.synchronize()
    g = GpuRun(wl, w, tables=_host_tables(base.dw))
    for t in HOST_TABLES:
        g.sc.cache_enable(t, 1 << 14)
    hit_rates = []
    for call in range(3):
        got = _run(g)
        _assert_same(got, ref, f"call {call}")
        if call == 1:  # a warm call, served mostly from the caches
            _assert_oracle(got, wl, w, "warm cached call")
        hits, misses = g.sc.cache_stats()
        assert hits + misses > 0
        hit_rates.append(hits / (hits + misses))
    assert hit_rates[0] == 0.0, "the first call starts from empty caches"
    assert hit_rates[1] > 0.5 and hit_rates[2] >= hit_rates[1], f"hit rates {hit_rates}"


def test_varying_batches_evict_and_stay_exact():
    # four batches (different ids, the same tables) through one scorer with small caches: rows of one batch
    # evict those of another; each call matches the all-HBM path on the same tables
    import torch
    from synth.harness import DeviceWorkload
    w = synth.make_weights(1, synth.default_seed("prod"))
    g = dev = None
    for i, seed in enumerate([11, 12, 13, 11]):
        wl = _workload(seed=seed)
        if g is None:
            first = GpuRun(wl, w)
            dev = first.dw.tables
            g = GpuRun(wl, w, tables=_host_tables(first.dw))
            for t in HOST_TABLES:
                g.sc.cache_enable(t, 1024)
        else:
            g.wl, g.dw = wl, DeviceWorkload(wl, tables=g.dw.tables)
            g.pooled = torch.full((wl.n_req * 8 + wl.n_cand * 8, 32), float("nan"), dtype=torch.float32,
                                  device="cuda:0")
            g.rows = torch.full((max(len(wl.bag_ids), 1),), -7, dtype=torch.int64, device="cuda:0")
        ref = _run(GpuRun(wl, w, tables=dev))
        got = _run(g)
        _assert_same(got, ref, f"batch {i} (seed {seed})")
        if i == 3:  # a batch seen before, after three others evicted part of its rows
            _assert_oracle(got, wl, w, f"batch {i} (seed {seed})", requests=[0])
    hits, misses = g.sc.cache_stats()
    assert hits > 0 and misses > 0


def test_cache_on_device_tables_and_removal():
    # a cache in front of HBM tables is legal too (same bits); slots 0 removes it
    wl = _workload(n_req=1)
    w = synth.make_weights(wl.n_layers, wl.seed)
    g = GpuRun(wl, w)
    ref = _run(g)
    g.sc.cache_enable(16, 1 << 12)
    g.sc.cache_enable(3, 1 << 10)
    _assert_same(_run(g), ref, "cached")
    _assert_same(_run(g), ref, "cached, warm")
    assert sum(g.sc.cache_stats()) > 0
    g.sc.cache_enable(16, 0)
    g.sc.cache_enable(3, 0)
    _assert_same(_run(g), ref, "cache removed")


def test_cache_argument_errors_and_id_range():
    import torch
    wl = synth.make_workload("tiny")
    w = synth.make_weights(wl.n_layers, wl.seed)
    g = GpuRun(wl, w)
    assert g.sc.cache_enable(17, 1024, check=False) == 1   # CVR_E_ARG: no such table
    assert g.sc.cache_enable(0, 1000, check=False) == 1    # not a power of two
    assert g.sc.cache_enable(0, 512, check=False) == 1     # below the minimum
    assert g.sc.cache_enable(0, 1024, check=False) == 0
    # an id outside its table is still reported (row 0 is read, never logged as a cache row of that id)
    bad = g.dw.bag_ids.clone()
    bad[0] = wl.user_rows + 5
    g.dw.bag_ids = bad
    assert g.run(check=False) == 3  # CVR_E_ID_RANGE
    g.dw.bag_ids = torch.from_numpy(wl.bag_ids).to("cuda:0")
    assert g.run(check=False) == 0
