"""Pins of the CPU oracle against facts fixed by the model description and by mathematics.

Each test targets a mistake that could plausibly sit in the oracle (a dropped term, a wrong sign
or index, a transposed operand, the wrong reduction order) and would fail if it were there.
Sources: the iQIYI ad-CVR article (sections 3.1, 3.2.1-3.2.4, 3.4.5) and the GPU CTR
inference article (section 三: clamp to [-10, 10] after the lookup, then half precision).
"""
import math
import os

import numpy as np
import pytest

import oracle
import synth

HERE = os.path.dirname(os.path.abspath(__file__))
rng = np.random.default_rng(1234)
SIG1 = 0.7310585786300049  # logistic(1), a textbook constant


# ---------------------------------------------------------------- pooling, clamp, cast
def test_pool_identical_ids_give_the_row():
    tab = rng.uniform(-0.05, 0.05, size=(50, 32)).astype(np.float32)
    for n in (1, 2):
        out, rows, st = oracle.pool_bag(tab, [17] * n)
        assert st == 0 and np.array_equal(out, tab[17]) and list(rows) == [17] * n


def test_pool_identical_ids_exact_for_short_mantissas():
    tab = (rng.integers(-50, 50, size=(10, 32)) / 1024.0).astype(np.float32)
    out, _, _ = oracle.pool_bag(tab, [3] * 7)
    assert np.array_equal(out, tab[3])


def test_pool_is_mean_not_sum():
    tab = np.zeros((4, 32), np.float32)
    tab[1] = 2.0
    tab[2] = 4.0
    out, _, _ = oracle.pool_bag(tab, [1, 2])
    assert np.all(out == 3.0)


def test_pool_sums_in_fp32_in_bag_order():
    # 1e8 + 1 is absorbed in fp32, so the sequential fp32 sum of (1e8, 1, -1e8) is exactly 0;
    # fp64 or reordered sums give 1/3.
    tab = np.zeros((3, 32), np.float32)
    tab[0], tab[1], tab[2] = 1e8, 1.0, -1e8
    out, _, _ = oracle.pool_bag(tab, [0, 1, 2], clamp=1e9)
    assert np.all(out == 0.0)
    out, _, _ = oracle.pool_bag(tab, [0, 2, 1], clamp=1e9)
    assert np.all(out == np.float32(1.0) / np.float32(3.0))


def test_pool_division_is_one_ieee_division():
    tab = np.zeros((3, 32), np.float32)
    tab[0] = 1.0
    out, _, _ = oracle.pool_bag(tab, [0, 1, 2])
    assert np.all(out == np.float32(1.0) / np.float32(3.0))


def test_clamp_bounds():
    tab = np.zeros((3, 32), np.float32)
    tab[0], tab[1], tab[2] = 25.0, -25.0, 9.5
    assert np.all(oracle.pool_bag(tab, [0])[0] == 10.0)
    assert np.all(oracle.pool_bag(tab, [1])[0] == -10.0)
    assert np.all(oracle.pool_bag(tab, [2])[0] == 9.5)
    assert np.all(oracle.pool_bag(tab, [0, 2])[0] == 10.0)  # the clamp applies to the mean (17.25)


def test_empty_bag_pools_to_zero():
    tab = np.ones((3, 32), np.float32)
    out, rows, st = oracle.pool_bag(tab, [])
    assert st == 0 and np.all(out == 0.0) and len(rows) == 0


def test_out_of_range_id_reads_row_zero_and_reports():
    tab = rng.normal(size=(5, 32)).astype(np.float32)
    out, rows, st = oracle.pool_bag(tab, [7, -1, 2])
    assert st == oracle.E_ID_RANGE and list(rows) == [0, 0, 2]


def test_bf16_round_to_nearest_even():
    assert oracle.bf16(1.0 + 2.0 ** -8) == 1.0                      # tie -> even (mantissa 0)
    assert oracle.bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6      # tie -> even (mantissa 2)
    assert oracle.bf16(1.0 + 2.0 ** -8 + 2.0 ** -20) == 1.0 + 2.0 ** -7
    assert oracle.bf16(-3.0) == -3.0
    assert oracle.bf16(0.1) == 0.10009765625


# ---------------------------------------------------------------- SwiGLU
def _unit_swiglu(a_coef, g_coef, w_out, b1=0.0, b3=0.0, b2=0.0):
    w1 = np.array([[a_coef, 0.0]], np.float32)
    w3 = np.array([[0.0, g_coef]], np.float32)
    w2 = np.array([[w_out]], np.float32)
    return oracle.swiglu([1.0, 1.0], w1, [b1], w3, [b3], w2, [b2])[0]


def test_swiglu_zero_output_weights_give_bias():
    x = rng.normal(size=128)
    w1, w3 = rng.normal(size=(256, 128)), rng.normal(size=(256, 128))
    b2 = rng.normal(size=128).astype(np.float32)
    y = oracle.swiglu(x, w1, np.zeros(256), w3, np.zeros(256), np.zeros((128, 256)), b2)
    assert np.allclose(y, b2, atol=0, rtol=0)


def test_swiglu_gate_is_silu_of_w1_times_w3():
    # silu(1) * 2 = 2 * logistic(1)
    assert abs(_unit_swiglu(1.0, 2.0, 1.0) - 2 * SIG1) < 1e-15
    # silu on the W3 path instead would give silu(2) * 1 = 2 * logistic(2)
    assert abs(_unit_swiglu(2.0, 1.0, 1.0) - 2 * 0.8807970779778823) < 1e-15
    # a very negative W1 branch switches the unit off whatever the W3 branch is
    assert abs(_unit_swiglu(-40.0, 1.0, 1.0, b2=0.25) - 0.25) < 1e-14
    # biases enter inside: silu(1 - 1) = 0
    assert _unit_swiglu(1.0, 5.0, 1.0, b1=-1.0) == 0.0
    assert abs(_unit_swiglu(1.0, 1.0, 3.0, b3=1.0) - 3 * 2 * SIG1) < 1e-14


# ---------------------------------------------------------------- tokenisation, query
def test_tokenize_one_hot_selects_a_weight_column_in_token_order():
    w = rng.normal(size=(13 * 128, 512)).astype(np.float32)
    b = rng.normal(size=13 * 128).astype(np.float32)
    for k in (0, 200, 256, 511):          # user half then item half
        e = np.zeros(512)
        e[k] = 1.0
        x = oracle.tokenize(e[:256], e[256:], w, b, 13, 128)
        assert x.shape == (13, 128)
        assert np.allclose(x[5, 7], float(w[5 * 128 + 7, k]) + float(b[5 * 128 + 7]), rtol=0, atol=1e-12)
        assert np.allclose(x.reshape(-1), w[:, k].astype(np.float64) + b, rtol=0, atol=1e-12)


def test_query_one_hot_tokens_and_mean_pool():
    w = rng.normal(size=(128, 13 * 128 + 128)).astype(np.float32)
    b = rng.normal(size=128).astype(np.float32)
    x = np.zeros((13, 128))
    m = np.zeros(128)
    x[12, 3] = 1.0
    assert np.allclose(oracle.query(x, m, w, b), w[:, 12 * 128 + 3].astype(np.float64) + b, atol=1e-12)
    x[:] = 0
    m[9] = 2.0
    assert np.allclose(oracle.query(x, m, w, b), 2 * w[:, 13 * 128 + 9].astype(np.float64) + b, atol=1e-12)


# ---------------------------------------------------------------- cross-attention
def test_attention_identical_keys_returns_mean_of_values():
    h = rng.normal(size=128)
    H = np.tile(h, (37, 1))
    d, p = oracle.cross_attention(rng.normal(size=128) * 5, H, 4, 2.0)
    assert np.allclose(d, h, atol=1e-12)
    assert np.allclose(p.sum(axis=1), 1.0, atol=1e-12)


def test_attention_zero_query_is_mean_over_the_sequence():
    H = rng.normal(size=(21, 128))
    d, p = oracle.cross_attention(np.zeros(128), H, 4, 2.0)
    assert np.allclose(d, H.mean(axis=0), atol=1e-12)
    assert np.allclose(p, 1.0 / 21, atol=1e-15)


def test_attention_temperature_and_head_scale_closed_form():
    # two keys, k0 = 0 and k1 = e_0 (head 0); q_0 = tau * sqrt(32) * ln 3 * e_0
    # -> logits 0 and ln 3 -> weights 1/4, 3/4 on head 0; other heads see q = 0 -> uniform.
    tau = 2.0
    H = np.zeros((2, 128))
    H[1, 0] = 1.0
    H[1, 40] = 6.0     # head 1 value, weight 1/2 there
    q = np.zeros(128)
    q[0] = tau * math.sqrt(32.0) * math.log(3.0)
    d, p = oracle.cross_attention(q, H, 4, tau)
    assert np.allclose(p[0], [0.25, 0.75], atol=1e-14)
    assert np.allclose(p[1:], 0.5, atol=1e-15)
    assert abs(d[0] - 0.75) < 1e-14 and abs(d[40] - 3.0) < 1e-14
    assert np.all(d[1:32] == 0)


def test_attention_large_logit_selects_that_row_per_head():
    H = rng.normal(size=(9, 128))
    q = np.zeros(128)
    q[96:128] = H[4, 96:128] * 400.0   # head 3 only, strongly aligned with row 4
    d, _ = oracle.cross_attention(q, H, 4, 2.0)
    assert np.allclose(d[96:], H[4, 96:], atol=1e-9)
    assert np.allclose(d[:96], H[:, :96].mean(axis=0), atol=1e-12)


def test_attention_single_position():
    H = rng.normal(size=(1, 128))
    d, p = oracle.cross_attention(rng.normal(size=128), H, 4, 2.0)
    assert np.array_equal(d, H[0]) and np.all(p == 1.0)


# ---------------------------------------------------------------- token mixer
def test_mix_worked_example():
    z = 1000.0 * np.arange(16)[:, None] + np.arange(128)[None, :]
    m = oracle.mix(z)
    rows = np.loadtxt(os.path.join(HERE, "golden", "mix_example.txt"), dtype=np.int64)
    for j, pos, expected in rows:
        assert m[j, pos] == expected, (j, pos)


def test_revert_inverts_mix_and_mix_is_not_identity():
    z = rng.normal(size=(16, 128))
    assert np.array_equal(oracle.revert(oracle.mix(z)), z)
    assert np.array_equal(oracle.mix(oracle.revert(z)), z)
    assert not np.allclose(oracle.mix(z), z)


def test_rmsnorm_closed_forms():
    g = np.ones(128, np.float32)
    # constant row c with c^2 = eps: y = c / sqrt(2 c^2) = 1/sqrt(2) (eps inside the root, added to the mean square)
    y = oracle.rmsnorm(np.full(128, 1e-3), g, 1e-6)
    assert np.allclose(y, 1 / math.sqrt(2), atol=1e-12)
    x = rng.normal(size=128)
    y = oracle.rmsnorm(x, g, 1e-6)
    assert abs((y ** 2).mean() - 1.0 / (1.0 + 1e-6 / (x ** 2).mean())) < 1e-12
    y2 = oracle.rmsnorm(x, np.full(128, 2.0, np.float32), 1e-6)
    assert np.allclose(y2, 2 * y, atol=1e-14)
    assert np.allclose(oracle.rmsnorm(-x, g, 1e-6), -y, atol=1e-15)


def _tm(z, w1, b1, w3, b3, w2, b2, gain):
    return oracle.token_mixer(z, w1, b1, w3, b3, w2, b2, gain, 1e-6)


def test_token_mixer_zero_ffn_is_rmsnorm_of_input():
    z = rng.normal(size=(16, 128))
    zero = np.zeros
    y = _tm(z, rng.normal(size=(256, 128)), zero(256), rng.normal(size=(256, 128)), zero(256), zero((128, 256)),
            zero(128), np.ones(128))
    ref = z / np.sqrt((z ** 2).mean(axis=1, keepdims=True) + 1e-6)
    assert np.allclose(y, ref, atol=1e-12)


def test_token_mixer_revert_sends_slot_t_back_to_token_t():
    # F(mixed_j) = beta for every j: the reverted output token t holds beta[8t:8t+8] in every head
    beta = rng.normal(size=128).astype(np.float32)
    z = np.zeros((16, 128))
    zero = np.zeros
    y = _tm(z, zero((256, 128)), zero(256), zero((256, 128)), zero(256), zero((128, 256)), beta, np.ones(128))
    rev = np.stack([np.tile(beta[8 * t:8 * t + 8], 16) for t in range(16)]).astype(np.float64)
    ref = rev / np.sqrt((rev ** 2).mean(axis=1, keepdims=True) + 1e-6)
    assert np.allclose(y, ref, atol=1e-12)


def test_token_mixer_residual_adds_input():
    beta = np.full(128, 0.5, np.float32)
    z = np.full((16, 128), 1.5)
    zero = np.zeros
    y = _tm(z, zero((256, 128)), zero(256), zero((256, 128)), zero(256), zero((128, 256)), beta, np.full(128, 3.0))
    assert np.allclose(y, 3.0 * 2.0 / math.sqrt(4.0 + 1e-6), atol=1e-12)


# ---------------------------------------------------------------- PLE + heads
def _experts(n=3, de=256, dy=2048):
    return ([rng.normal(size=(de, dy)).astype(np.float32) * 0.03 for _ in range(n)],
            [rng.normal(size=de).astype(np.float32) for _ in range(n)])


def test_ple_identical_experts_ignore_the_gates():
    we, be = _experts()
    we = [we[0]] * 3
    be = [be[0]] * 3
    y = rng.normal(size=2048)
    wg = [rng.normal(size=(3, 2048)).astype(np.float32) for _ in range(2)]
    bg = [rng.normal(size=3).astype(np.float32) for _ in range(2)]
    r, gates = oracle.ple(y, we, be, wg, bg)
    e = np.maximum(we[0].astype(np.float64) @ y + be[0], 0)
    assert np.allclose(r[0], e, atol=1e-12) and np.allclose(r[1], e, atol=1e-12)
    assert np.allclose(gates.sum(axis=1), 1.0, atol=1e-14)


def test_ple_gate_bias_selects_an_expert_per_task():
    we, be = _experts()
    y = rng.normal(size=2048)
    wg = [np.zeros((3, 2048), np.float32) for _ in range(2)]
    bg = [np.array([0, 0, 60], np.float32), np.array([60, 0, 0], np.float32)]
    r, gates = oracle.ple(y, we, be, wg, bg)
    e = [np.maximum(we[k].astype(np.float64) @ y + be[k], 0) for k in range(3)]
    assert np.allclose(r[0], e[2], atol=1e-20 + 1e-12) and np.allclose(r[1], e[0], atol=1e-12)
    assert np.all(e[0] >= 0) and np.any(we[0].astype(np.float64) @ y + be[0] < 0)   # ReLU active


def test_ple_zero_gates_average_the_experts():
    we, be = _experts()
    y = rng.normal(size=2048)
    z = [np.zeros((3, 2048), np.float32)] * 2
    r, gates = oracle.ple(y, we, be, z, [np.zeros(3, np.float32)] * 2)
    e = [np.maximum(we[k].astype(np.float64) @ y + be[k], 0) for k in range(3)]
    assert np.allclose(gates, 1 / 3, atol=1e-15)
    assert np.allclose(r[0], (e[0] + e[1] + e[2]) / 3, atol=1e-12)


def test_head_closed_forms():
    r = rng.normal(size=256)
    z = np.zeros
    assert oracle.head(r, z((128, 256)), z(128), z((1, 128)), [0.0]) == 0.5
    # b2 = ln 3 stored in fp32 (rel. error <= 2^-24): sigma(ln 3) = 3/4 to within 1e-7
    assert abs(oracle.head(r, z((128, 256)), z(128), z((1, 128)), [math.log(3.0)]) - 0.75) < 1e-7
    w1 = z((128, 256))
    w1[5, 17] = 1.0
    w2 = z((1, 128))
    w2[0, 5] = 1.0
    r = z(256)
    r[17] = math.log(3.0)
    assert abs(oracle.head(r, w1, z(128), w2, [0.0]) - 0.75) < 1e-15
    r[17] = -5.0                                           # ReLU cuts the hidden unit
    assert oracle.head(r, w1, z(128), w2, [0.0]) == 0.5
    # b1 = 1 lifts the pre-activation to -4, still cut; logit = b2 = -1 -> 1 - logistic(1)
    assert abs(oracle.head(r, w1, np.full(128, 1.0), w2, [-1.0]) - (1 - SIG1)) < 1e-15


# ---------------------------------------------------------------- whole model
def _host_tables(wl):
    return {t: wl.host_table(t) for t in list(range(16)) + [synth.SEQ_TABLE]}


@pytest.mark.parametrize("variant", [
    dict(name="tiny"),
    dict(name="tiny", bias_scale=0.05, gain_jitter=0.1),
    dict(name="deep", n_req=2, n_cand=3, seq_len=(5, 9, 2), bias_scale=0.05, gain_jitter=0.1),
    dict(name="tiny", cand_per_req=[1, 5, 2], n_req=3, seq_len=(1, 3, 7), table_scale=20.0, weight_scale=3.0),
])
def test_oracle_agrees_with_matrix_formulation(variant):
    import np_model
    v = dict(variant)
    bias, gain, ws = v.pop("bias_scale", 0.0), v.pop("gain_jitter", 0.0), v.pop("weight_scale", 1.0)
    name = v.pop("name")
    wl = synth.make_workload(name, user_rows=1000, item_rows=1000, seq_rows=10_000, **v)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=bias, gain_jitter=gain, weight_scale=ws)
    tabs = _host_tables(wl)
    res = oracle.score(wl, w)
    ref = np_model.forward(wl, w, tabs)
    assert res.status == 0
    assert np.allclose(res.out, ref, atol=1e-10, rtol=0), np.abs(res.out - ref).max()


def test_oracle_on_demand_tables_equal_materialised_tables():
    wl = synth.make_workload("tiny")
    w = synth.make_weights(wl.n_layers, wl.seed)
    a = oracle.score(wl, w)
    b = oracle.score(wl, w, host_tables=_host_tables(wl))
    assert np.array_equal(a.out, b.out)


def test_oracle_subset_and_threads_are_consistent():
    wl = synth.make_workload("tiny", n_req=3, n_cand=3)
    w = synth.make_weights(wl.n_layers, wl.seed)
    full = oracle.score(wl, w, threads=3).out
    one = oracle.score(wl, w, threads=1).out
    sub = oracle.score(wl, w, requests=[2]).out
    assert np.array_equal(full, one)
    assert np.array_equal(sub[6:9], full[6:9]) and np.all(np.isnan(sub[:6]))


def test_candidates_are_scored_independently():
    # reversing the candidates of a request (with their item bags) reverses the scores
    wl = synth.make_workload("tiny", n_req=1, n_cand=5)
    w = synth.make_weights(wl.n_layers, wl.seed)
    base = oracle.score(wl, w).out
    Fu, Fi = 8, 8
    off, ids = wl.bag_offsets, wl.bag_ids
    bags = [ids[off[i]:off[i + 1]] for i in range(len(off) - 1)]
    user, items = bags[:Fu], bags[Fu:]
    per_c = [items[c * Fi:(c + 1) * Fi] for c in range(5)][::-1]
    new = user + [b for c in per_c for b in c]
    wl.bag_offsets = np.concatenate([[0], np.cumsum([len(b) for b in new])]).astype(np.int64)
    wl.bag_ids = np.concatenate(new).astype(np.int64)
    rev = oracle.score(wl, w).out
    assert np.array_equal(rev, base[::-1])


def test_oracle_dumps_pooled_and_rows():
    wl = synth.make_workload("tiny")
    w = synth.make_weights(wl.n_layers, wl.seed)
    res = oracle.score(wl, w, dumps=True)
    assert np.array_equal(res.dumps["rows"], wl.bag_ids)
    t0 = wl.host_table(0)
    b0 = wl.bag_ids[wl.bag_offsets[0]:wl.bag_offsets[1]]
    out, _, _ = oracle.pool_bag(t0, b0)
    assert np.array_equal(res.dumps["pooled"][0], out)


def test_oracle_reports_out_of_range_ids():
    wl = synth.make_workload("tiny")
    w = synth.make_weights(wl.n_layers, wl.seed)
    wl.bag_ids = wl.bag_ids.copy()
    wl.bag_ids[3] = 10 ** 9
    assert oracle.score(wl, w).status == oracle.E_ID_RANGE
