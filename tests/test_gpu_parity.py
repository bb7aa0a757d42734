"""Parity of the CUDA scoring path (through the C ABI) with the CPU oracle.

Bit-exact: the pooled fp32 embedding means and the rows each id read. Within abs 2e-3 / rel 1e-2:
every pCVR. Small workloads are compared on every candidate and every stage; the full-size
workloads, in the launch configuration the benchmark times, on the candidates of sampled requests
(requests are independent, so a sampled request is scored exactly as in the full batch).
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import GpuRun, assert_pcvr_close, rel_close

pytestmark = pytest.mark.gpu


def _check_full(wl, w, graph=True, stages=False, **cfg):
    g = GpuRun(wl, w, graph=graph, **cfg)
    g.run()
    ref = oracle.score(wl, w, dumps=True, **cfg)
    assert ref.status == 0
    pooled = g.pooled.cpu().numpy()
    assert np.array_equal(pooled.view(np.uint32), ref.dumps["pooled"].view(np.uint32)), "pooled fp32 not bit-exact"
    assert np.array_equal(g.rows.cpu().numpy()[: len(wl.bag_ids)], ref.dumps["rows"]), "gather rows differ"
    if stages:
        import torch
        import cvr_ranking_model_gb300 as cvr
        B, R, SL = wl.n_cand, wl.n_req, wl.sum_len
        L = wl.seq_len
        Hg = g.stage(cvr.STAGE_H, (R * SL, 128), torch.bfloat16)
        # GPU layout: group-major [g][r][l]; oracle: [r][sum_len]
        off = 0
        parts = []
        for gi in range(3):
            parts.append(Hg[off: off + R * L[gi]].reshape(R, L[gi], 128))
            off += R * L[gi]
        H = np.concatenate(parts, axis=1)
        rel_close(H, ref.dumps["H"], 0.03, "H")
        last = wl.n_layers - 1
        Z = g.stage(cvr.STAGE_Z, (B, 16, 128), torch.bfloat16)
        rel_close(Z[:, :13], ref.dumps["Z"][last][:, :13], 0.03, "tokens x")
        Q = g.stage(cvr.STAGE_Q, (B, 3, 128), torch.bfloat16)
        rel_close(Q, ref.dumps["Q"][last], 0.03, "queries")
        for gi in range(3):
            rel_close(Z[:, 13 + gi], ref.dumps["Z"][last][:, 13 + gi], 0.05, f"decoded token {gi}")
        Y = g.stage(cvr.STAGE_Y, (B, 16, 128), torch.bfloat16)
        rel_close(Y, ref.dumps["Y"][last], 0.03, "token mixer output")
    return assert_pcvr_close(g.out(), ref.out, wl.name)


def test_tiny_every_candidate_and_stage():
    wl = synth.make_workload("tiny")
    w = synth.make_weights(wl.n_layers, wl.seed)
    _check_full(wl, w, stages=True)


def test_expert_and_gate_stages_when_kept():
    """CVR_OPT_KEEP_STAGES: the PLE also writes its expert outputs and task gates, which match the PLE of
    iQIYI CVR 3.2.4 recomputed in fp64 from the oracle's last Token Mixer output; the scores are the same
    bits with and without the option, and without it the two stages are refused."""
    import torch
    import cvr_ranking_model_gb300 as cvr
    wl = synth.make_workload("tiny", n_req=3, cand_per_req=[100, 1, 60])
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.05)
    g = GpuRun(wl, w, debug=False)
    g.run()
    plain = g.out()
    with pytest.raises(cvr.CvrError):
        g.stage(cvr.STAGE_EXPERTS, (wl.n_cand, 768), torch.bfloat16)
    g.sc.set_option(cvr.OPT_KEEP_STAGES, 1)
    g.run()
    assert np.array_equal(g.out(), plain)
    ref = oracle.score(wl, w, dumps=True)
    y = ref.dumps["Y"][-1].reshape(wl.n_cand, -1)
    e = np.maximum(0.0, y @ np.concatenate([w[f"ple{k}_w"] for k in range(3)]).T +
                   np.concatenate([w[f"ple{k}_b"] for k in range(3)]))
    rel_close(g.stage(cvr.STAGE_EXPERTS, (wl.n_cand, 768), torch.bfloat16), e, 0.03, "expert outputs")
    gates = g.stage(cvr.STAGE_GATES, (wl.n_cand, 8), torch.float32)
    for t in range(2):
        gl = y @ w[f"gate{t}_w"].T + w[f"gate{t}_b"]
        p = np.exp(gl - gl.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        assert np.max(np.abs(gates[:, 3 * t:3 * t + 3] - p)) < 0.02, t
    assert not gates[:, 6:].any()


def test_tiny_with_biases_and_gains():
    wl = synth.make_workload("tiny")
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.05, gain_jitter=0.1)
    _check_full(wl, w, stages=True)


def test_clamp_binds():
    # tables ~ U(-20, 20): the [-10, 10] clamp binds on pooled means and on sequence rows; small dense
    # weights keep the rest of the network in its ordinary range
    wl = synth.make_workload("tiny", table_scale=20.0)
    w = synth.make_weights(wl.n_layers, wl.seed, weight_scale=0.1, bias_scale=0.05)
    ref = oracle.score(wl, w, dumps=True)
    assert np.mean(np.abs(ref.dumps["pooled"]) == 10.0) > 0.2
    _check_full(wl, w, stages=True)


def test_peaked_attention():
    # tables ~ U(-1, 1) and tau = 0.05: the softmax puts 15-60% of its mass on one position (uniform: 6%)
    wl = synth.make_workload("tiny", table_scale=1.0)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.05)
    ref = oracle.score(wl, w, dumps=True, tau=0.05)
    H, Q = ref.dumps["H"], ref.dumps["Q"][0]
    pmax = [oracle.cross_attention(Q[b, 2], H[wl.req_ids[b], 32:48], 4, 0.05)[1].max() for b in range(wl.n_cand)]
    assert np.median(pmax) > 0.15
    _check_full(wl, w, stages=True, tau=0.05)


def test_ragged_requests_and_odd_lengths():
    # candidates per request 1..70, 130-row tiles crossing requests, sequence lengths off the 64-chunk
    wl = synth.make_workload("tiny", n_req=5, cand_per_req=[1, 70, 3, 64, 9], seq_len=(3, 70, 129),
                             user_rows=5000, item_rows=3000)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.02, gain_jitter=0.05)
    _check_full(wl, w, stages=True)


@pytest.mark.parametrize("n_req", [32, 33, 150])
def test_request_counts_around_the_tokeniser_user_paths(n_req):
    # up to 32 requests each tokeniser CTA computes the user half of its own column tile for every request;
    # above that the user rows are row-tiles of the launch that the item tiles wait for (150 requests: two)
    cand = [1 + (r * 7) % 5 for r in range(n_req)]
    wl = synth.make_workload("tiny", n_req=n_req, cand_per_req=cand, seq_len=(5, 9, 17), user_rows=5000,
                             item_rows=5000)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.02)
    _check_full(wl, w, stages=True)


def test_sequence_lengths_on_chunk_boundaries():
    # every group's length a multiple of the attention's 64-position chunk (1, 2 and 3 chunks): no chunk has keys
    # to mask
    wl = synth.make_workload("tiny", n_req=3, cand_per_req=[40, 7, 25], seq_len=(64, 128, 192), user_rows=3000,
                             item_rows=3000)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.02)
    _check_full(wl, w, stages=True)


def test_two_layers_small():
    wl = synth.make_workload("deep", n_req=3, n_cand=40, seq_len=(17, 33, 65), user_rows=1000, item_rows=1000,
                             seq_rows=10_000)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.02, gain_jitter=0.05)
    _check_full(wl, w, stages=True)


@pytest.mark.parametrize("bag_min,bag_max", [(0, 3), (9, 17), (0, 64)])
def test_empty_and_long_bags(bag_min, bag_max):
    # empty bags (pool to 0) on the user and the item side, and bags longer than the 8 ids a bag's lanes hold
    # at once (the second and later passes of the gather's id loop: 9, 16, 17 and 64 ids), bit for bit
    wl = synth.make_workload("tiny", n_req=3, n_cand=37, bag_min=bag_min, bag_max=bag_max, user_rows=5000,
                             item_rows=5000)
    sizes = np.diff(wl.bag_offsets)
    nu = wl.n_req * 8
    if bag_min == 0:
        assert (sizes[:nu] == 0).any() and (sizes[nu:] == 0).any(), "the workload has empty user and item bags"
    for n in (9, 16, 17, 64):
        if bag_min <= n <= bag_max:
            assert (sizes == n).any(), f"the workload has a bag of {n} ids"
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.02)
    _check_full(wl, w, stages=True)


def test_single_request_single_candidate():
    wl = synth.make_workload("tiny", n_req=1, n_cand=1, seq_len=(1, 1, 1))
    w = synth.make_weights(wl.n_layers, wl.seed)
    _check_full(wl, w)


def test_eager_and_graph_agree_and_repeat():
    wl = synth.make_workload("tiny", n_req=3, n_cand=50)
    w = synth.make_weights(wl.n_layers, wl.seed)
    g = GpuRun(wl, w, graph=False)
    g.run()
    a = g.out()
    import cvr_ranking_model_gb300 as cvr
    g.sc.set_option(cvr.OPT_CUDA_GRAPH, 1)
    g.run()
    b = g.out()
    g.run()
    c = g.out()
    assert np.array_equal(a, b) and np.array_equal(b, c)


def test_host_entry_point_matches_device_entry_point():
    # pageable arrays are staged by copies; pinned ones are read (and out written) in place over the C2C
    # link; every mix gives the device entry point's bits
    import torch
    wl = synth.make_workload("tiny", n_req=2, n_cand=33)
    w = synth.make_weights(wl.n_layers, wl.seed)
    g = GpuRun(wl, w)
    g.run()
    dev = g.out()
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory().numpy()
    arrays = [wl.req_ids, wl.bag_ids, wl.bag_offsets, np.ascontiguousarray(wl.seq_ids)]
    ref = oracle.score(wl, w).out
    for mask in (0b00000, 0b11111, 0b01010, 0b10101):
        ins = [pin(a) if mask >> i & 1 else np.ascontiguousarray(a) for i, a in enumerate(arrays)]
        out = pin(np.zeros((wl.n_cand, 2), np.float32)) if mask >> 4 & 1 else np.zeros((wl.n_cand, 2), np.float32)
        g.sc.score_host(wl.n_req, wl.n_cand, *ins, out)
        assert np.array_equal(out.astype(np.float64), dev), f"pinned mask {mask:05b}"
        assert_pcvr_close(out.astype(np.float64), ref, f"host entry point, pinned mask {mask:05b}")


def test_host_entry_point_prod_matches_oracle():
    # the host-buffer entry point on the production shape (pinned inputs read in place, as the benchmark's
    # end-to-end leg calls it), every candidate against the oracle
    import torch
    wl = synth.make_workload("prod")
    w = synth.make_weights(wl.n_layers, wl.seed)
    g = GpuRun(wl, w, debug=False)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory().numpy()
    ins = [pin(a) for a in (wl.req_ids, wl.bag_ids, wl.bag_offsets, np.ascontiguousarray(wl.seq_ids))]
    out = pin(np.zeros((wl.n_cand, 2), np.float32))
    g.sc.score_host(wl.n_req, wl.n_cand, *ins, out)
    assert_pcvr_close(out.astype(np.float64), oracle.score(wl, w).out, "prod through the host entry point")


# ------------------------------------------------------------------ error reporting (no fault)
def test_out_of_range_id_is_reported_not_read():
    import cvr_ranking_model_gb300 as cvr
    wl = synth.make_workload("tiny")
    wl.bag_ids = wl.bag_ids.copy()
    wl.bag_ids[5] = 10 ** 12
    wl.seq_ids = wl.seq_ids.copy()
    wl.seq_ids[0, 3, 1] = -4
    w = synth.make_weights(wl.n_layers, wl.seed)
    g = GpuRun(wl, w)
    st = g.run(check=False)
    assert st == 3, cvr.binding.STATUS.get(st)
    assert g.rows.cpu().numpy()[5] == 0


def test_bad_offsets_and_request_ids_are_reported():
    wl = synth.make_workload("tiny")
    w = synth.make_weights(wl.n_layers, wl.seed)
    wl2 = synth.make_workload("tiny")
    wl2.bag_offsets = wl2.bag_offsets.copy()
    wl2.bag_offsets[7] = wl2.bag_offsets[9] + 1   # bag 6 ends after bag 7 starts... offsets decrease at 8
    g = GpuRun(wl2, w)
    assert g.run(check=False) == 6
    wl3 = synth.make_workload("tiny")
    wl3.req_ids = wl3.req_ids.copy()
    wl3.req_ids[0] = 1                             # decreasing sequence 1, 0, ...
    g = GpuRun(wl3, w)
    assert g.run(check=False) == 6
    wl4 = synth.make_workload("tiny")
    wl4.req_ids = wl4.req_ids.copy()
    wl4.req_ids[-1] = 99                           # out of range
    g = GpuRun(wl4, w)
    assert g.run(check=False) == 6


def test_negative_offsets_are_reported_not_read():
    # a negative first offset (and a negative offset in the middle) would point before bag_ids: the bag is read
    # as empty and the call reports CVR_E_INPUT; the handle keeps working
    wl = synth.make_workload("tiny")
    w = synth.make_weights(wl.n_layers, wl.seed)
    for pos, val in ((0, -3), (5, -1)):
        bad = synth.make_workload("tiny")
        bad.bag_offsets = bad.bag_offsets.copy()
        bad.bag_offsets[pos] = val
        g = GpuRun(bad, w)
        assert g.run(check=False) == 6
        assert np.all(g.pooled.cpu().numpy()[pos] == 0.0), "the malformed bag pools to zero"
    g = GpuRun(wl, w)
    assert g.run(check=False) == 0


def test_shape_errors_on_the_host():
    wl = synth.make_workload("tiny")
    w = synth.make_weights(wl.n_layers, wl.seed)
    g = GpuRun(wl, w, debug=False)
    r, b, o, s, out = g.dw.ptrs()
    assert g.sc.score(0, 4, r, b, o, s, out, check=False) == 2
    assert g.sc.score(2, 0, r, b, o, s, out, check=False) == 2
    assert g.sc.score(2, 8, 0, b, o, s, out, check=False) == 1
    assert g.sc.score(2, 8, r, b, o, s, out, check=False) == 0   # the handle still works


# ------------------------------------------------------------------ full-size workloads (sampled)
_TABLES = {}


def _full(name, requests, n_cand=None, n_req=None):
    wl = synth.make_workload(name, n_cand=n_cand) if n_req is None else synth.make_workload(name, n_cand=n_cand,
                                                                                            n_req=n_req)
    w = synth.make_weights(wl.n_layers, wl.seed)
    g = GpuRun(wl, w, graph=True)
    g.run()
    ref = oracle.score(wl, w, requests=requests, dumps=True)
    assert ref.status == 0
    sel = np.isin(wl.req_ids, requests)
    assert_pcvr_close(g.out()[sel], ref.out[sel], name)
    # pooled sums of the sampled requests' bags, bit for bit
    pooled = g.pooled.cpu().numpy()
    nb_user = wl.n_req * 8
    user_bags = np.concatenate([np.arange(r * 8, r * 8 + 8) for r in requests])
    item_bags = nb_user + np.concatenate([np.arange(c * 8, c * 8 + 8) for c in np.nonzero(sel)[0]])
    bags = np.concatenate([user_bags, item_bags])
    assert np.array_equal(pooled[bags].view(np.uint32), ref.dumps["pooled"][bags].view(np.uint32))
    rows = g.rows.cpu().numpy()
    for bag in bags[:: max(1, len(bags) // 2000)]:
        lo, hi = wl.bag_offsets[bag], wl.bag_offsets[bag + 1]
        assert np.array_equal(rows[lo:hi], ref.dumps["rows"][lo:hi])
    return g


def test_prod_full_batch():
    _full("prod", requests=list(range(8)))


def test_longseq_sampled():
    _full("longseq", requests=[0, 15])


def test_embheavy_sampled():
    _full("embheavy", requests=[0, 37, 63])


@pytest.mark.parametrize("c", [64, 512, 2048])
def test_deep_sampled(c):
    _full("deep", requests=[0, 31] if c < 2048 else [5], n_cand=c)


def test_deep_wide_query_tiles_with_a_ragged_row_tile():
    # 24 x 500 = 12,000 candidates: the stacked layer's query GEMM takes its 128-column tiles (2 rounds of tiles
    # over the grid instead of 3) and its last row tile holds 96 candidates
    _full("deep", requests=[0, 23], n_cand=500, n_req=24)


def test_async_calls_match_sync_and_report_errors():
    wl = synth.make_workload("tiny", n_req=3, n_cand=20)
    w = synth.make_weights(wl.n_layers, wl.seed)
    g = GpuRun(wl, w, debug=False)
    g.run()
    ref = g.out()
    r, b, o, s, out = g.dw.ptrs()
    g.dw.out.zero_()
    for _ in range(3):
        g.sc.score_async(wl.n_req, wl.n_cand, r, b, o, s, out)
    assert g.sc.sync(check=False) == 0
    assert np.array_equal(g.out(), ref)
    # a bad id in one of several in-flight calls is reported by the next sync, then cleared
    import torch
    bad = g.dw.bag_ids.clone()
    bad[3] = 10 ** 10
    g.sc.score_async(wl.n_req, wl.n_cand, r, bad.data_ptr(), o, s, out)
    g.sc.score_async(wl.n_req, wl.n_cand, r, b, o, s, out)
    assert g.sc.sync(check=False) == 3
    g.sc.score_async(wl.n_req, wl.n_cand, r, b, o, s, out)
    assert g.sc.sync(check=False) == 0
    torch.cuda.synchronize()
