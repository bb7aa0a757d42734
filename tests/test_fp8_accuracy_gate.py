"""Accuracy gate for FP8 dense operands in the PLE GEMM (the FP8/INT8 direction of the iQIYI article's
outlook section; the GPU CTR inference article, section 三, reports an AUC loss from INT8 embeddings).

The PLE and the task towers are recomputed in fp64 from the oracle's own last Token Mixer output, with
the operands rounded the way a kernel would round them: bf16 (what the library does), FP8 e4m3 weights
with per-output-channel scales, and FP8 e4m3 weights and activations. bf16 stays well inside the pCVR
tolerance; both FP8 forms put a large share of candidates outside it, which is why the library keeps
the PLE and tokeniser GEMMs in bf16.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")

ATOL, RTOL = 2e-3, 1e-2


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).double().numpy()


def _e4m3(x):
    return torch.from_numpy(np.asarray(x, np.float64)).float().to(torch.float8_e4m3fn).double().numpy()


def _e4m3_rows(W):
    s = np.abs(W).max(axis=1, keepdims=True) / 448.0  # e4m3's largest finite value
    s[s == 0] = 1.0
    return _e4m3(W / s) * s


def _ple_heads(y, w, mode):
    We = np.concatenate([w[f"ple{k}_w"] for k in range(3)])
    be = np.concatenate([w[f"ple{k}_b"] for k in range(3)])
    Wg = np.concatenate([w[f"gate{t}_w"] for t in range(2)])
    ya = y
    if mode in ("w8", "w8a8"):
        We, Wg = _e4m3_rows(We), _e4m3_rows(Wg)
    if mode == "w8a8":
        ya = _e4m3(y)
    e = _bf16(np.maximum(0.0, ya @ We.T + be))  # expert outputs are kept in bf16
    out = []
    for t in range(2):
        gl = ya @ Wg[3 * t:3 * t + 3].T + w[f"gate{t}_b"]
        g = np.exp(gl - gl.max(axis=1, keepdims=True))
        g /= g.sum(axis=1, keepdims=True)
        r = sum(g[:, k:k + 1] * e[:, 256 * k:256 * (k + 1)] for k in range(3))
        h = np.maximum(0.0, r @ w[f"head{t}_w1"].T + w[f"head{t}_b1"])
        out.append(1.0 / (1.0 + np.exp(-(h @ w[f"head{t}_w2"].T + w[f"head{t}_b2"])[:, 0])))
    return np.stack(out, 1)


@pytest.fixture(scope="module")
def prod_one_request():
    wl = synth.make_workload("prod", n_req=1)
    w = synth.make_weights(wl.n_layers, wl.seed)
    ref = oracle.score(wl, w, dumps=True)
    return wl, w, ref


def _share_out(p, ref):
    err = np.abs(p - ref)
    return float(np.mean(err > ATOL + RTOL * np.abs(ref))), float(np.max(err / (ATOL + RTOL * np.abs(ref))))


def test_bf16_operands_stay_inside_the_tolerance(prod_one_request):
    wl, w, ref = prod_one_request
    y = _bf16(ref.dumps["Y"][-1].reshape(wl.n_cand, -1))
    share, worst = _share_out(_ple_heads(y, w, "bf16"), ref.out)
    assert share == 0.0 and worst < 0.5, (share, worst)


@pytest.mark.parametrize("mode", ["w8", "w8a8"])
def test_fp8_operands_break_the_tolerance(prod_one_request, mode):
    wl, w, ref = prod_one_request
    y = _bf16(ref.dumps["Y"][-1].reshape(wl.n_cand, -1))
    share, worst = _share_out(_ple_heads(y, w, mode), ref.out)
    assert share > 0.05 and worst > 2.0, (mode, share, worst)
