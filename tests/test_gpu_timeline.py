"""The per-CTA timeline diagnostic (cvr_timeline): the normal build refuses it; the diagnostic build records,
for every kernel of a call, entry <= dependency wait <= exit on the device clock, and the kernels start in the
order the call's dependencies allow."""
import os
import subprocess
import sys

import numpy as np
import pytest

import synth
from gpu_util import GpuRun

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_normal_build_refuses_the_timeline():
    import cvr_ranking_model_gb300 as cvr
    wl = synth.make_workload("tiny")
    g = GpuRun(wl, synth.make_weights(wl.n_layers, wl.seed), debug=False)
    g.run()
    with pytest.raises(cvr.binding.CvrError):
        g.sc.timeline()


def test_timeline_build_orders_the_kernels():
    # a process of its own: the diagnostic library is built and loaded instead of the normal one
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--timeline", "--config", "prod",
                          "--warmup", "3"], capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    rows = {}
    for line in out.stdout.splitlines():
        parts = line.split()
        if len(parts) == 8 and parts[0] in ("sparse", "seq_mlp", "seq_colsum", "tokenizer", "attention",
                                            "token_mixer", "ple_heads"):
            rows[parts[0]] = [float(x) for x in parts[1:]]
    assert set(rows) == {"sparse", "seq_mlp", "seq_colsum", "tokenizer", "attention", "token_mixer", "ple_heads"}
    for name, (ctas, s_min, s_med, s_max, w_med, e_med, e_max) in rows.items():
        assert ctas >= 1 and s_min <= s_med <= s_max and s_min <= e_med <= e_max, name
        assert np.isnan(w_med) or s_min <= w_med <= e_max, name
    # each kernel's data dependency: its wait returns after its producer's last CTA has finished
    for prod, cons in (("sparse", "seq_mlp"), ("sparse", "tokenizer"), ("seq_mlp", "seq_colsum"),
                       ("seq_colsum", "attention"), ("tokenizer", "attention")):
        assert rows[cons][4] >= rows[prod][6] - 0.05, (prod, cons)
    # the Token Mixer's tiles wait for the attention blocks of their own candidates (the attention counts each
    # block as its groups are written), so its first tile starts after attention CTAs have run, not after all
    assert rows["token_mixer"][4] >= rows["attention"][1] - 0.05
    assert rows["token_mixer"][6] >= rows["attention"][6] - 0.05
