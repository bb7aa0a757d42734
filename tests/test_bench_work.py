"""The algorithmic work behind the bench's roofline fractions, against the counting rule it follows: the
user side, the sequence encoders, K/V and the mean-pooled term once per request (the pages' lazy repeat),
every Linear's FLOPs at 2 per multiply-add, zero biases counted; bytes = gathered fp32 rows of 128 B, 8-byte
ids and offsets, 4-byte request ids, the bf16 weights once, 8 bytes of output per candidate."""
import pytest

import bench
import synth

D, HID = 128, 256
SWIGLU_ROW = 2 * (D * 2 * HID + HID * D)   # up (W1, W3) and down projections of one row


def rule_flops(wl):
    R, B, NL, SL = wl.n_req, wl.n_cand, wl.n_layers, wl.sum_len
    per_request = SL * SWIGLU_ROW + 2 * 256 * 1664 + NL * 2 * 3 * D * D
    per_candidate = (2 * 256 * 1664 + NL * (2 * 1664 * 384 + 4 * D * SL + 16 * SWIGLU_ROW)
                     + 2 * (2048 * 768 + 2048 * 6) + 2 * 2 * (256 * 128 + 128))
    return R * per_request + B * per_candidate


def rule_weight_bytes(n_layers):
    tokeniser = 1664 * 512
    seq = 3 * (512 * 128 + 128 * 256)
    per_layer = 3 * 128 * 1792 + 512 * 128 + 128 * 256   # query FFNs, Token Mixer SwiGLU
    ple = 774 * 2048                                     # 3 experts of 256 and 2 x 3 gates
    heads = 2 * 128 * 256
    return 2 * (tokeniser + seq + n_layers * per_layer + ple + heads)


@pytest.mark.parametrize("name", ["prod", "longseq", "deep"])
def test_flops_follow_the_counting_rule(name):
    wl = synth.make_workload(name, n_req=2)
    flops, _, _ = bench.algorithmic_work(wl, len(wl.bag_ids))
    assert sum(flops.values()) == rule_flops(wl)


def test_weight_bytes_one_and_two_layers():
    assert rule_weight_bytes(1) == 7_168_000      # 7.17 MB
    assert rule_weight_bytes(2) == 8_740_864      # 8.74 MB


@pytest.mark.parametrize("name", ["prod", "deep"])
def test_bytes_follow_the_counting_rule(name):
    wl = synth.make_workload(name, n_req=2)
    R, B, SL, nnz = wl.n_req, wl.n_cand, wl.sum_len, len(wl.bag_ids)
    _, total, _ = bench.algorithmic_work(wl, nnz)
    gathered = (nnz + 4 * R * SL) * 128
    ids = (nnz + 4 * R * SL) * 8 + (R * 8 + B * 8 + 1) * 8 + B * 4
    assert total == gathered + ids + rule_weight_bytes(wl.n_layers) + B * 8


def test_prod_batch_is_36_gflop():
    # the prod batch under this rule: 36.4 GFLOP (the FLOPs do not depend on the bag sizes)
    wl = synth.make_workload("prod")
    flops, _, _ = bench.algorithmic_work(wl, len(wl.bag_ids))
    assert abs(sum(flops.values()) / 1e9 - 36.4) < 0.05
