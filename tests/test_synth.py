"""The seeded input generator: determinism, ranges and the id law of the workload definitions."""
import numpy as np

import synth


def test_workload_shapes_and_ranges():
    wl = synth.make_workload("prod")
    R, B = wl.n_req, wl.n_cand
    assert (R, B) == (8, 8 * 512) and wl.seq_len == (50, 100, 200)
    sizes = np.diff(wl.bag_offsets)
    assert len(sizes) == R * 8 + B * 8 and sizes.min() >= 1 and sizes.max() <= 8
    assert abs(sizes.mean() - 4.5) < 0.05
    assert wl.bag_ids.min() >= 0 and wl.bag_ids.max() < 100_000
    assert wl.seq_ids.shape == (R, 350, 4) and wl.seq_ids.max() < 1_000_000
    assert np.all(np.diff(wl.req_ids) >= 0) and wl.req_ids[-1] == R - 1


def test_generator_is_deterministic_and_seeded():
    a = synth.make_workload("tiny")
    b = synth.make_workload("tiny")
    c = synth.make_workload("tiny", seed=7)
    assert np.array_equal(a.bag_ids, b.bag_ids) and np.array_equal(a.seq_ids, b.seq_ids)
    assert not np.array_equal(a.seq_ids, c.seq_ids)
    t1 = a.host_table(3, 10, 5)
    t2 = a.host_table(3)[10:15]
    assert np.array_equal(t1, t2) and np.abs(t1).max() <= 0.05


def test_zipf_ranks_follow_the_power_law():
    lib = synth.lib()
    n, s = 100_000, 1.1
    ranks = np.array([lib.synth_zipf_rank(99, 0x3000, i, n, s) for i in range(200_000)])
    assert ranks.min() >= 1 and ranks.max() <= n
    c = np.bincount(ranks, minlength=10)
    # P(1)/P(2) = 2^s, P(1)/P(4) = 4^s (binomial noise ~2-4%)
    assert abs(c[1] / c[2] - 2 ** s) < 0.12 and abs(c[1] / c[4] - 4 ** s) < 0.3


def test_rank_to_row_is_a_bijection():
    lib = synth.lib()
    rows = 1000
    got = {lib.synth_rank_to_row(5, 3, r, rows) for r in range(1, rows + 1)}
    assert got == set(range(rows))


def test_weights_are_bf16_valued_glorot():
    w = synth.make_weights(1, 123)
    for k, a in w.items():
        u = a.view(np.uint32)
        assert np.all((u & 0xFFFF) == 0), k
    bound = np.sqrt(6.0 / (1664 + 512))
    assert np.abs(w["tok_w"]).max() <= bound * (1 + 2 ** -8)
    assert np.all(w["tok_b"] == 0) and np.all(w["l0_tm_gain"] == 1)
    wb = synth.make_weights(1, 123, bias_scale=0.05, gain_jitter=0.1)
    assert np.abs(wb["tok_b"]).max() > 0 and np.abs(wb["l0_tm_gain"] - 1).max() > 0


def test_bag_sizes_span_empty_and_long_bags():
    # bag_min = 0 draws empty bags, bag_max up to 64 long ones; sizes are uniform over [bag_min, bag_max]
    wl = synth.make_workload("tiny", n_req=4, n_cand=60, bag_min=0, bag_max=64)
    sizes = np.diff(wl.bag_offsets)
    assert sizes.min() == 0 and sizes.max() == 64
    assert abs(sizes.mean() - 32) < 2.5
    assert len(wl.bag_ids) == wl.bag_offsets[-1]
    # and repeatable
    a = synth.make_workload("tiny", n_req=4, n_cand=60, bag_min=0, bag_max=64)
    assert np.array_equal(a.bag_ids, wl.bag_ids)
