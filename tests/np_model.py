"""Second, independently written fp64 formulation of the CVR forward pass, in matrix form.

The oracle (oracle/cvr_oracle.c) is a per-candidate loop nest; this module computes the same
model for a whole batch with NumPy matrix products, reshapes and fancy indexing. The two share
nothing but the inputs, so agreement on small workloads pins the oracle's index arithmetic
(concatenation orders, reshapes, head splits, the mix/revert transpose) against a different
way of writing the same definitions.
"""
from __future__ import annotations

import numpy as np

import synth


def _bf16(a: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return u.view(np.float32).astype(np.float64)


def _pool(table: np.ndarray, ids: np.ndarray, offsets: np.ndarray, bags: np.ndarray, clamp: float) -> np.ndarray:
    """fp32 mean of each bag, summed position by position in bag order (vectorised over bags)."""
    start, end = offsets[bags], offsets[bags + 1]
    n = end - start
    acc = np.zeros((len(bags), table.shape[1]), np.float32)
    for p in range(int(n.max(initial=0))):
        live = p < n
        rows = table[ids[start[live] + p]]
        acc[live] = acc[live] + rows
    with np.errstate(invalid="ignore", divide="ignore"):
        mean = np.where(n[:, None] > 0, acc / n[:, None].astype(np.float32), np.float32(0))
    return np.clip(mean.astype(np.float32), np.float32(-clamp), np.float32(clamp))


def _silu(a):
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def forward(wl: "synth.Workload", w, tables) -> np.ndarray:
    d = synth.DIMS
    Fu, Fi, E, D, N, G = d["n_user_fields"], d["n_item_fields"], d["emb_dim"], d["token_dim"], d["n_tokens"], d["n_groups"]
    T, heads, clamp = N + G, d["heads"], d["clamp"]
    R, B = wl.n_req, wl.n_cand
    f64 = lambda k: w[k].astype(np.float64)

    # user / item embeddings: [R, Fu*E], [B, Fi*E]
    U = np.concatenate([_bf16(_pool(tables[f], wl.bag_ids, wl.bag_offsets, np.arange(R) * Fu + f, clamp))
                        for f in range(Fu)], axis=1)
    I = np.concatenate([_bf16(_pool(tables[Fu + f], wl.bag_ids, wl.bag_offsets, R * Fu + np.arange(B) * Fi + f, clamp))
                        for f in range(Fi)], axis=1)
    emb = np.concatenate([U[wl.req_ids], I], axis=1)                      # [B, 512]
    X = (emb @ f64("tok_w").T + f64("tok_b")).reshape(B, N, D)            # [B, N, D]

    # sequences: [R, SL, cols] ids -> [R, SL, cols*E] rows -> per-group SwiGLU
    seq_rows = np.clip(tables[synth.SEQ_TABLE][wl.seq_ids], -clamp, clamp)  # [R, SL, cols, E] fp32
    S = _bf16(seq_rows).reshape(R, wl.sum_len, -1)
    Hs, Ms = [], []
    off = 0
    for g, L in enumerate(wl.seq_len):
        x = S[:, off:off + L]
        a = x @ f64(f"seq{g}_w1").T + f64(f"seq{g}_b1")
        c = x @ f64(f"seq{g}_w3").T + f64(f"seq{g}_b3")
        h = (_silu(a) * c) @ f64(f"seq{g}_w2").T + f64(f"seq{g}_b2")        # [R, L, D]
        Hs.append(h)
        Ms.append(h.mean(axis=1))                                           # [R, D]
        off += L

    hd = D // heads
    Z = np.zeros((B, T, D))
    Z[:, :N] = X
    for l in range(wl.n_layers):
        if l > 0:
            Z = Y.copy()
        for g in range(G):
            qin = np.concatenate([Z[:, :N].reshape(B, N * D), Ms[g][wl.req_ids]], axis=1)
            q = qin @ f64(f"l{l}_q{g}_w").T + f64(f"l{l}_q{g}_b")            # [B, D]
            K = Hs[g][wl.req_ids]                                            # [B, L, D]
            qh = q.reshape(B, heads, hd)
            Kh = K.reshape(B, K.shape[1], heads, hd)
            s = np.einsum("bhi,blhi->bhl", qh, Kh) / (d["tau"] * np.sqrt(hd))
            p = np.exp(s - s.max(axis=2, keepdims=True))
            p /= p.sum(axis=2, keepdims=True)
            Z[:, N + g] = np.einsum("bhl,blhi->bhi", p, Kh).reshape(B, D)
        # token mixer: [B, T(token), T(head), hd] -> swap token/head axes
        mh = D // T  # token-mixer head width
        mixed = Z.reshape(B, T, T, mh).transpose(0, 2, 1, 3).reshape(B, T, D)
        a = mixed @ f64(f"l{l}_tm_w1").T + f64(f"l{l}_tm_b1")
        c = mixed @ f64(f"l{l}_tm_w3").T + f64(f"l{l}_tm_b3")
        F = (_silu(a) * c) @ f64(f"l{l}_tm_w2").T + f64(f"l{l}_tm_b2")
        rev = F.reshape(B, T, T, mh).transpose(0, 2, 1, 3).reshape(B, T, D)
        res = Z + rev
        Y = res / np.sqrt((res ** 2).mean(axis=2, keepdims=True) + d["rms_eps"]) * f64(f"l{l}_tm_gain")
    y = Y.reshape(B, T * D)
    ex = np.stack([np.maximum(y @ f64(f"ple{k}_w").T + f64(f"ple{k}_b"), 0.0) for k in range(d["n_experts"])], 1)
    out = np.zeros((B, d["n_tasks"]))
    for t in range(d["n_tasks"]):
        gl = y @ f64(f"gate{t}_w").T + f64(f"gate{t}_b")
        gt = np.exp(gl - gl.max(axis=1, keepdims=True))
        gt /= gt.sum(axis=1, keepdims=True)
        r = np.einsum("bk,bki->bi", gt, ex)
        h = np.maximum(r @ f64(f"head{t}_w1").T + f64(f"head{t}_b1"), 0.0)
        logit = h @ f64(f"head{t}_w2").T[:, 0] + f64(f"head{t}_b2")[0]
        out[:, t] = 1.0 / (1.0 + np.exp(-logit))
    return out
