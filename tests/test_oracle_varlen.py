"""Pins of the oracle's variable-length sequences (sequence lengths are a dynamic input, iQIYI ad-CVR
article 3.3; sequences are padded, 3.4.2): each request with lengths l_g must score exactly as the
fixed-length model run on that request alone with its sequences cut to l_g events -- an independent
formulation -- and the padding must never be read."""
import dataclasses

import numpy as np

import oracle
import synth


def _wl(**kw):
    return synth.make_workload("tiny", n_req=4, cand_per_req=[3, 1, 5, 2], seq_len=(17, 33, 65),
                               user_rows=3000, item_rows=3000, **kw)


def _alone(wl, r, lens_r):
    """The fixed-length workload of request r alone, its sequences cut to lens_r events per group."""
    Fu, Fi = 8, 8
    cands = np.nonzero(wl.req_ids == r)[0]
    bags = list(range(r * Fu, r * Fu + Fu)) + [wl.n_req * Fu + b * Fi + f for b in cands for f in range(Fi)]
    offs, ids = [0], []
    for bag in bags:
        seg = wl.bag_ids[wl.bag_offsets[bag]: wl.bag_offsets[bag + 1]]
        ids.extend(seg.tolist())
        offs.append(len(ids))
    parts, base = [], 0
    for g, L in enumerate(wl.seq_len):
        parts.append(wl.seq_ids[r, base: base + int(lens_r[g])])
        base += L
    seq = np.ascontiguousarray(np.concatenate(parts)[None], dtype=np.int64)
    return dataclasses.replace(wl, n_req=1, n_cand=len(cands), seq_len=tuple(int(x) for x in lens_r),
                               cand_per_req=np.array([len(cands)], np.int64),
                               req_ids=np.zeros(len(cands), np.int32),
                               bag_offsets=np.array(offs, np.int64), bag_ids=np.array(ids, np.int64), seq_ids=seq), cands


def test_full_lengths_equal_the_fixed_length_model():
    wl = _wl()
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.05)
    full = np.tile(np.array(wl.seq_len, np.int32), (wl.n_req, 1))
    a = oracle.score(wl, w)
    b = oracle.score(wl, w, seq_lens=full)
    assert a.status == b.status == 0
    assert np.array_equal(a.out, b.out)


def test_each_request_scores_as_its_truncated_fixed_length_model():
    wl = _wl()
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.05, gain_jitter=0.1)
    lens = synth.make_seq_lens(wl, min_len=1)
    assert (lens < np.array(wl.seq_len)).any()
    var = oracle.score(wl, w, seq_lens=lens)
    assert var.status == 0
    for r in range(wl.n_req):
        one, cands = _alone(wl, r, lens[r])
        ref = oracle.score(one, w)
        assert ref.status == 0
        np.testing.assert_allclose(var.out[cands], ref.out, rtol=0, atol=1e-12)


def test_two_layers_truncated():
    wl = synth.make_workload("deep", n_req=3, n_cand=4, seq_len=(9, 20, 33), user_rows=2000, item_rows=2000,
                             seq_rows=5000)
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.05)
    lens = synth.make_seq_lens(wl, min_len=1, seed=7)
    var = oracle.score(wl, w, seq_lens=lens)
    for r in range(wl.n_req):
        one, cands = _alone(wl, r, lens[r])
        np.testing.assert_allclose(var.out[cands], oracle.score(one, w).out, rtol=0, atol=1e-12)


def test_padding_is_never_read():
    wl = _wl()
    w = synth.make_weights(wl.n_layers, wl.seed)
    lens = synth.make_seq_lens(wl, min_len=0, seed=3)
    clean = oracle.score(wl, w, seq_lens=lens)
    bad = dataclasses.replace(wl, seq_ids=synth.pad_seq_ids(wl, lens, wl.seq_rows + 12345))
    dirty = oracle.score(bad, w, seq_lens=lens)
    assert clean.status == 0 and dirty.status == 0   # an out-of-range id in the padding is no error
    assert np.array_equal(clean.out, dirty.out)


def test_empty_group_decodes_to_zero_and_single_event_to_its_row():
    wl = _wl()
    w = synth.make_weights(wl.n_layers, wl.seed, bias_scale=0.05)
    lens = np.tile(np.array(wl.seq_len, np.int32), (wl.n_req, 1))
    lens[0] = [5, 0, 1]    # request 0: group 1 empty, group 2 a single event
    res = oracle.score(wl, w, seq_lens=lens, dumps=True)
    assert res.status == 0
    Z, H = res.dumps["Z"][0], res.dumps["H"]
    for b in np.nonzero(wl.req_ids == 0)[0]:
        assert np.all(Z[b, 13 + 1] == 0.0)
        # one key: softmax weight exactly 1, so the decoded token is that event's encoded row
        assert np.array_equal(Z[b, 13 + 2], H[0, wl.seq_len[0] + wl.seq_len[1]])


def test_lengths_out_of_range_are_rejected():
    wl = _wl()
    w = synth.make_weights(wl.n_layers, wl.seed)
    lens = np.tile(np.array(wl.seq_len, np.int32), (wl.n_req, 1))
    lens[2, 1] = wl.seq_len[1] + 1
    assert oracle.score(wl, w, seq_lens=lens).status == 1
    lens[2, 1] = -1
    assert oracle.score(wl, w, seq_lens=lens).status == 1
