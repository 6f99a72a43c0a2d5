"""Seeded random shapes through every plan family, against the fp64 oracle.

Each case draws M, N and K (ragged against the 16-token, 128-row and 64-wide
K tiles), the weight layout, bias and output type from one seeded generator,
and a planner option that steers it into one plan family: the planner's own
choice, stream-K only (no clusters), a forced cluster split, several clusters
per tile, one k-block a stage, CTA pairs wherever the tile allows, half
tiles.  Every output element is compared with the oracle, and a rerun must
give the same bits.  A plan the device cannot hold (a forced cluster shape
that does not fit) falls back inside proj_create; the test then checks the
fallback just the same.
"""
import numpy as np
import pytest

import gpu_util as gu
import oracle
import synth

pytestmark = pytest.mark.gpu

OPTIONS = [
    {},
    {"PROJ_MAX_CLUSTER": "0"},
    {"PROJ_FORCE_CLUSTER": "3", "PROJ_CLUSTER_FILL_PCT": "1"},
    {"PROJ_FORCE_CLUSTER": "2", "PROJ_CLUSTER_GROUPS": "3", "PROJ_CLUSTER_FILL_PCT": "1"},
    {"PROJ_KPB": "1"},
    {"PROJ_CTA_PAIR": "2"},
    {"PROJ_HALF_TILES": "2"},
]


def _cases(n=28, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        M = int(rng.choice([1, 3, 16, 17, 40, 64, 100, 130, 257]))
        N = int(rng.integers(1, 24)) * 64 + int(rng.choice([0, 0, 8, 40]))
        K = int(rng.integers(1, 40)) * 64 + int(rng.choice([0, 0, 8, 24]))
        layout = int(rng.choice([synth.W_NK, synth.W_KN]))
        bias = bool(rng.integers(0, 2))
        yd = str(rng.choice(["bf16", "f32"]))
        opt = OPTIONS[i % len(OPTIONS)]
        out.append((M, N, K, layout, bias, yd, opt))
    return out


@pytest.mark.parametrize("M,N,K,layout,bias,yd,opt", _cases(),
                         ids=lambda v: str(v) if not isinstance(v, dict) else "-".join(
                             f"{k[5:]}={x}" for k, x in v.items()) or "default")
def test_random_shape(M, N, K, layout, bias, yd, opt, monkeypatch):
    import torch
    import dense_linear_projection_gb300 as dlp
    monkeypatch.setenv("PROJ_TM_CLUSTER", "0")
    for k, v in opt.items():
        monkeypatch.setenv(k, v)
    w = synth.Workload("t", M, N, K, layout, bias, yd, seed=M * 7 + N * 3 + K)
    inp = synth.make_inputs(w)
    proj, Y, (X, W, b) = gu.run(w, inp)
    again = proj(X, W, b).clone()
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    r = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
    gu.assert_within_tol(gu.y_to_f64(Y), r, f"M={M} N={N} K={K} plan={proj.plan}")
    iv = torch.int16 if yd == "bf16" else torch.int32
    assert torch.equal(again.view(iv), Y.view(iv)), "rerun differs"
