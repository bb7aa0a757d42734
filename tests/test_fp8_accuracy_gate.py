"""Accuracy gate for 8-bit dense operands in the PLE and tokeniser GEMMs (the INT8 / mixed-precision
direction of the iQIYI article's outlook section; the GPU CTR inference article, section 三, reports an
AUC loss from INT8 embeddings).

Each scheme rounds a GEMM's operands the way a kernel consuming them would, and everything else is
computed in fp64 by the oracle's own stage functions, so the score difference is that GEMM's
quantisation alone. The schemes, weights W [out][K] and activations A [rows][K], blocks along K:

- ``bf16``: both operands bf16 (what the library does);
- ``e4m3-row-w``: e4m3 weights with one fp32 scale per output row, bf16 activations;
- ``e4m3-row-wa``: the same weights, activations cast to e4m3 without a scale;
- ``mxfp8``: OCP MX FP8, both operands e4m3 with one power-of-two (ue8m0) scale per 32 K-elements,
  the operand layout ``tcgen05.mma`` block-scaled kinds consume;
- ``int8-b32``: symmetric INT8, both operands, one fp32 scale per 32 K-elements;
- ``int8-b32-w``: the same INT8 weights, dequantised to bf16 (q x scale, rounded) for a bf16 MMA;
- ``int8-row-w``: INT8 weights with one fp32 scale per output row, bf16 activations. The scale is constant
  along K, so it comes out of the dot product: a bf16 MMA on the exact integers, scaled after the sum.
  The PLE kernel's INT8 mode (CVR_OPT_PLE_INT8) computes exactly this;
- ``int8-row-wa``: INT8 weights and activations, one scale per row of each (the tcgen05 kind::i8 form).

A candidate fails when its pCVR or pCTR leaves abs 2e-3 + rel 1e-2 of the oracle. The gate runs on one
request of the production shape and of the two-layer shape. Measured: every FP8 scheme puts 23-76% of
candidates outside the tolerance (e4m3 keeps 3 mantissa bits whatever the scaling); the INT8
weight-only schemes and bf16 stay inside it on both GEMMs; INT8 activations break the PLE's tolerance.
Which scheme passes where is asserted below, so a change in any of them shows up as a failing test.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")

ATOL, RTOL = 2e-3, 1e-2
D = synth.DIMS


def _cast(x, dtype):
    return torch.from_numpy(np.asarray(x, np.float64)).float().to(dtype).double().numpy()


def _ident(x):
    return np.asarray(x, np.float64)


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).double().numpy()


def _e4m3(x):
    """Round to e4m3 with saturation at its largest finite value (448)."""
    return _cast(np.clip(x, -448.0, 448.0), torch.float8_e4m3fn)


def _e4m3_rows(W):
    s = np.abs(W).max(axis=-1, keepdims=True) / 448.0
    s[s == 0] = 1.0
    return _e4m3(W / s) * s


def _blocks(x, blk=32):
    x = np.asarray(x, np.float64)
    assert x.shape[-1] % blk == 0
    return x.reshape(x.shape[:-1] + (x.shape[-1] // blk, blk))


def _mx_e4m3(x, blk=32):
    """OCP MX: shared scale 2^(floor(log2(amax)) - 8) per block (8 = e4m3's largest exponent), each
    element the e4m3 rounding of x / scale, saturated at 448."""
    b = _blocks(x, blk)
    amax = np.abs(b).max(axis=-1, keepdims=True)
    e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 8.0, 0.0)
    s = np.exp2(e)
    return (_e4m3(b / s) * s).reshape(np.shape(x))


def _int8_blocks(x, blk=32):
    """Symmetric INT8, scale amax/127 per block, round half to even, clipped to [-127, 127]."""
    b = _blocks(x, blk)
    s = np.abs(b).max(axis=-1, keepdims=True) / 127.0
    s[s == 0] = 1.0
    return (np.clip(np.rint(b / s), -127, 127) * s).reshape(np.shape(x))


SCHEMES = {  # name: (weight quantiser, activation quantiser)
    "bf16": (_bf16, _bf16),
    "e4m3-row-w": (_e4m3_rows, _bf16),
    "e4m3-row-wa": (_e4m3_rows, _e4m3),
    "mxfp8": (_mx_e4m3, _mx_e4m3),
    "int8-b32": (_int8_blocks, _int8_blocks),
    "int8-b32-w": (lambda W: _bf16(_int8_blocks(W)), _bf16),
    "int8-row-w": (lambda W: _int8_blocks(W, W.shape[-1]), _bf16),
    "int8-row-wa": (lambda W: _int8_blocks(W, W.shape[-1]), lambda A: _int8_blocks(A, A.shape[-1])),
}


def _ple_heads(y, w, qw=_ident, qa=_ident, round_e=True):
    """Progressive layered extraction and the task towers (iQIYI CVR 3.2.4), fp64, with the expert and
    gate weights rounded by ``qw`` and the flattened Token Mixer output by ``qa``. ``round_e`` keeps the
    expert outputs in bf16, as the kernel stores them."""
    We = qw(np.concatenate([w[f"ple{k}_w"] for k in range(3)]))
    be = np.concatenate([w[f"ple{k}_b"] for k in range(3)])
    Wg = qw(np.concatenate([w[f"gate{t}_w"] for t in range(2)]))
    ya = qa(y)
    e = np.maximum(0.0, ya @ We.T + be)
    if round_e:
        e = _bf16(e)
    out = []
    for t in range(2):
        gl = ya @ Wg[3 * t:3 * t + 3].T + w[f"gate{t}_b"]
        g = np.exp(gl - gl.max(axis=1, keepdims=True))
        g /= g.sum(axis=1, keepdims=True)
        r = sum(g[:, k:k + 1] * e[:, 256 * k:256 * (k + 1)] for k in range(3))
        h = np.maximum(0.0, r @ w[f"head{t}_w1"].T + w[f"head{t}_b1"])
        out.append(1.0 / (1.0 + np.exp(-(h @ w[f"head{t}_w2"].T + w[f"head{t}_b2"])[:, 0])))
    return np.stack(out, 1)


def _tokeniser_inputs(wl, ref):
    """The concatenated bf16 user and item field vectors of every candidate of request 0, [B][512]."""
    Fu, Fi, E = D["n_user_fields"], D["n_item_fields"], D["emb_dim"]
    pooled = ref.dumps["pooled"].astype(np.float64)
    u = _bf16(pooled[:Fu].reshape(-1))
    it = _bf16(pooled[wl.n_req * Fu:].reshape(wl.n_cand, Fi * E))
    return np.concatenate([np.broadcast_to(u, (wl.n_cand, u.size)), it], axis=1)


def _score_from_tokens(wl, w, ref, x_in, tok_w):
    """Scores request 0 from its tokeniser inputs through the oracle's stage functions (tokeniser, query,
    cross-attention, Token Mixer, PLE, towers), in the order the oracle's scorer calls them."""
    N, Dm, G, L = D["n_tokens"], D["token_dim"], D["n_groups"], wl.seq_len
    H = ref.dumps["H"][0]
    base = np.concatenate([[0], np.cumsum(L)])
    mg = [H[base[g]:base[g + 1]].mean(axis=0) for g in range(G)]
    du = D["n_user_fields"] * D["emb_dim"]
    tw = np.asarray(tok_w, np.float32)

    def one(b):
        z = np.zeros((N + G, Dm))
        z[:N] = oracle.tokenize(x_in[b, :du], x_in[b, du:], tw, w["tok_b"], N, Dm)
        for layer in range(wl.n_layers):
            if layer > 0:
                z[:N] = y[:N]
            for g in range(G):
                q = oracle.query(z[:N], mg[g], w[f"l{layer}_q{g}_w"], w[f"l{layer}_q{g}_b"])
                z[N + g] = oracle.cross_attention(q, H[base[g]:base[g + 1]], D["heads"], D["tau"])[0]
            y = oracle.token_mixer(z, *[w[f"l{layer}_tm_{n}"] for n in ("w1", "b1", "w3", "b3", "w2", "b2", "gain")],
                                   D["rms_eps"])
        r, _ = oracle.ple(y.reshape(-1), [w[f"ple{k}_w"] for k in range(3)], [w[f"ple{k}_b"] for k in range(3)],
                          [w[f"gate{t}_w"] for t in range(2)], [w[f"gate{t}_b"] for t in range(2)])
        return [oracle.head(r[t], w[f"head{t}_w1"], w[f"head{t}_b1"], w[f"head{t}_w2"], w[f"head{t}_b2"])
                for t in range(2)]

    with ThreadPoolExecutor(8) as ex:
        return np.array(list(ex.map(one, range(wl.n_cand))))


def _share_out(p, ref_out):
    bound = ATOL + RTOL * np.abs(ref_out)
    err = np.abs(p - ref_out)
    return float(np.mean(np.any(err > bound, axis=1))), float(np.max(err / bound))


@pytest.fixture(scope="module", params=["prod", "deep"])
def one_request(request):
    wl = synth.make_workload(request.param, n_req=1)
    w = synth.make_weights(wl.n_layers, wl.seed)
    ref = oracle.score(wl, w, dumps=True)
    return request.param, wl, w, ref


def ple_shares(wl, w, ref):
    y = ref.dumps["Y"][-1].reshape(wl.n_cand, -1)
    return {s: _share_out(_ple_heads(y, w, qw, qa), ref.out) for s, (qw, qa) in SCHEMES.items()}


def tokeniser_shares(wl, w, ref, schemes=tuple(SCHEMES)):
    x = _tokeniser_inputs(wl, ref)
    return {s: _share_out(_score_from_tokens(wl, w, ref, SCHEMES[s][1](x), SCHEMES[s][0](w["tok_w"])), ref.out)
            for s in schemes}


# the schemes that keep every candidate inside the tolerance, per GEMM and workload
PASSING = {
    ("ple", "prod"): {"bf16", "int8-b32-w", "int8-row-w"},
    ("ple", "deep"): {"bf16", "int8-b32-w", "int8-row-w", "int8-b32"},
    ("tok", "prod"): {"bf16", "int8-b32", "int8-b32-w", "int8-row-w", "int8-row-wa"},
    ("tok", "deep"): {"bf16", "int8-b32", "int8-b32-w", "int8-row-w", "int8-row-wa"},
}


def test_ple_restatement_matches_the_oracle(one_request):
    _, wl, w, ref = one_request
    y = ref.dumps["Y"][-1].reshape(wl.n_cand, -1)
    assert np.max(np.abs(_ple_heads(y, w, round_e=False) - ref.out)) < 1e-9


def test_token_pipeline_reproduces_the_oracle(one_request):
    """Unrounded tokeniser inputs through the stage functions give the scorer's own output exactly."""
    _, wl, w, ref = one_request
    p = _score_from_tokens(wl, w, ref, _tokeniser_inputs(wl, ref), w["tok_w"])
    assert np.array_equal(p, ref.out)


def test_quantisers():
    """Each quantiser against values it must reproduce: e4m3 and MX grids, INT8 block grids."""
    x = np.array([[0.0, 1.0, -448.0, 500.0, 0.0625, 1.0625, 0.001953125, 3.0]])
    assert np.array_equal(_e4m3(x), [[0.0, 1.0, -448.0, 448.0, 0.0625, 1.0, 0.001953125, 3.0]])
    b = np.zeros((1, 32))
    b[0, :4] = [1000.0, 3.0, -1.0, 2.0 ** -20]  # amax 1000: scale 2^(9-8) = 2
    q = _mx_e4m3(b)
    assert np.array_equal(q[0, :4], [448.0 * 2, 3.0, -1.0, 0.0]) and not q[0, 4:].any()
    b = np.zeros((1, 64))
    b[0, :2] = [127.0, 0.5]  # scale 1: 0.5 rounds to the even 0
    b[0, 32:35] = [-7.9375, 0.09375, 0.15625]  # scale 1/16: 1.5 and 2.5 steps both round to 2
    q = _int8_blocks(b)
    assert np.array_equal(q[0, :2], [127.0, 0.0]) and np.array_equal(q[0, 32:35], [-7.9375, 0.125, 0.125])


@pytest.mark.parametrize("scheme", list(SCHEMES))
def test_ple_scheme(one_request, scheme):
    name, wl, w, ref = one_request
    y = ref.dumps["Y"][-1].reshape(wl.n_cand, -1)
    qw, qa = SCHEMES[scheme]
    share, worst = _share_out(_ple_heads(y, w, qw, qa), ref.out)
    if scheme in PASSING["ple", name]:
        assert share == 0.0 and worst < 1.0, (name, scheme, share, worst)
    else:  # FP8 fails on 20% or more of the candidates
        assert share > (0.15 if "e4m3" in scheme or "mx" in scheme else 0.0) and worst > 1.0, (name, scheme, share, worst)


@pytest.mark.parametrize("scheme", list(SCHEMES))
def test_tokeniser_scheme(one_request, scheme):
    name, wl, w, ref = one_request
    share, worst = tokeniser_shares(wl, w, ref, (scheme,))[scheme]
    if scheme in PASSING["tok", name]:
        assert share == 0.0 and worst < 1.0, (name, scheme, share, worst)
    else:
        assert share > 0.15 and worst > 1.0, (name, scheme, share, worst)
