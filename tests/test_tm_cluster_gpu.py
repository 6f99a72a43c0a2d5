"""GPU parity of token-major cluster splits (at most 32 tokens).

The tokens take the MMA's M side (128 rows, zero beyond M) and 256 weight rows
its N side; each tile's K range is split over the S CTAs of a cluster, and
rank c mod S adds 16-column chunk c of the partial sums, which the other
ranks store into its shared memory.  It is an option: PROJ_TM_CLUSTER=1 lets
proj_create prefer it to a swapped cluster split, 2 forces it on any shape of
at most 32 tokens with few enough tiles.  Cases: every cluster size, ragged N and K,
[K,N] weights as stored and packed, fp32 output, bias, the fused epilogue and
SwiGLU; each against the fp64 oracle, rerun bit for bit.
"""
import numpy as np
import pytest

import gpu_util as gu
import oracle
import synth

pytestmark = pytest.mark.gpu


def _run(w, inp, packed=False):
    import torch
    import dense_linear_projection_gb300 as dlp
    proj = dlp.Projection(w.M, w.N, w.K, w.w_layout,
                          dlp.PROJ_F32 if w.y_dtype == "f32" else dlp.PROJ_BF16, has_bias=w.has_bias)
    X, W = gu.to_dev(inp["X"]), gu.to_dev(inp["W"])
    b = gu.to_dev(inp["bias"]) if w.has_bias else None
    Wr = proj.pack(W) if packed else W
    Y = proj(X, Wr, b, packed=packed)
    again = proj(X, Wr, b, packed=packed)
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    iv = torch.int16 if w.y_dtype == "bf16" else torch.int32
    assert torch.equal(again.view(iv), Y.view(iv)), "rerun differs"
    return proj, Y


FORCE = {"PROJ_TM_CLUSTER": "2"}
TM_CASES = [
    (16, 2048, 8192, synth.W_NK, False, "f32", {"PROJ_TM_CLUSTER": "1"}),  # the 2048-row decode weight
    (16, 2048, 8192, synth.W_NK, True, "bf16", FORCE),
    (9, 1000, 1032, synth.W_NK, True, "bf16", FORCE),      # ragged N (4 tiles, the last 232 rows), 17 k-blocks
    (16, 2048, 4104, synth.W_KN, True, "bf16", FORCE),     # [K,N] as stored (64-column boxes), ragged K
    (32, 3000, 520, synth.W_NK, False, "f32", FORCE),      # 32 tokens, ragged
    (1, 256, 8192, synth.W_NK, True, "bf16", FORCE),       # one token, one tile
]


@pytest.mark.parametrize("case", TM_CASES, ids=lambda c: "M{}_N{}_K{}_{}_{}_{}".format(
    c[0], c[1], c[2], "KN" if c[3] else "NK", c[5], "TM" + c[6]["PROJ_TM_CLUSTER"]))
@pytest.mark.parametrize("packed", [False, True], ids=["stored", "packed"])
def test_tm_cluster_parity(case, packed, monkeypatch):
    M, N, K, layout, bias, yd, env = case
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    w = synth.Workload("t", M, N, K, layout, bias, yd, seed=121)
    inp = synth.make_inputs(w)
    proj, Y = _run(w, inp, packed)
    p = proj.plan
    assert p["swap_ab"] == 0 and p["block_n"] == 256 and p["cluster_split"] >= 2
    assert p["grid"] == p["tiles_sk"] * p["cluster_split"]
    r = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
    gu.assert_within_tol(gu.y_to_f64(Y), r, f"tm cluster {case[:6]} packed={packed}")


@pytest.mark.parametrize("S", [2, 3, 5, 7, 8, 11, 16])
def test_tm_every_cluster_size(S, monkeypatch):
    # Cluster sizes that do and do not divide the 16 chunks of a tile.
    monkeypatch.setenv("PROJ_TM_CLUSTER", "2")
    monkeypatch.setenv("PROJ_MAX_CLUSTER", str(S))
    monkeypatch.setenv("PROJ_CLUSTER_FILL_PCT", "1")
    w = synth.Workload("t", 12, 600, 1032, synth.W_NK, True, "bf16", seed=130 + S)
    inp = synth.make_inputs(w)
    proj, Y = _run(w, inp)
    assert proj.plan["swap_ab"] == 0 and proj.plan["cluster_split"] == S
    r = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
    gu.assert_within_tol(gu.y_to_f64(Y), r, f"tm S={S}")


def test_tm_cluster_small_integers_bit_exact(monkeypatch):
    import torch
    import dense_linear_projection_gb300 as dlp
    monkeypatch.setenv("PROJ_TM_CLUSTER", "2")
    M, N, K = 16, 2048, 8192
    rng = np.random.default_rng(13)
    X = rng.integers(-3, 4, size=(M, K)).astype(np.float64)
    Wnk = rng.integers(-3, 4, size=(N, K)).astype(np.float64)
    proj = dlp.Projection(M, N, K, dlp.PROJ_W_NK, dlp.PROJ_F32)
    assert proj.plan["swap_ab"] == 0 and proj.plan["cluster_split"] >= 2
    Y = proj(gu.to_dev(synth.to_bf16_bits(X)), gu.to_dev(synth.to_bf16_bits(Wnk)), None)
    torch.cuda.synchronize()
    assert np.array_equal(gu.y_to_f64(Y), X @ Wnk.T)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_tm_cluster_fused_epilogue(act, monkeypatch):
    import torch
    import dense_linear_projection_gb300 as dlp
    monkeypatch.setenv("PROJ_TM_CLUSTER", "2")
    M, N, K = 16, 2 * 1100, 2056
    has_bias = act == "gelu"
    w = synth.Workload("t", M, N, K, synth.W_NK, has_bias, "bf16", seed=122)
    inp = synth.make_inputs(w)
    proj = dlp.Projection(M, N, K, synth.W_NK, dlp.PROJ_BF16, has_bias=has_bias)
    assert proj.plan["swap_ab"] == 0 and proj.plan["cluster_split"] >= 2
    X, W = gu.to_dev(inp["X"]), gu.to_dev(inp["W"])
    b = gu.to_dev(inp["bias"]) if has_bias else None
    F = N // 2 if act == "swiglu" else N
    R = synth.normal_bf16(123, 7, M * F, 1.0).reshape(M, F)
    R64 = oracle.bf16_to_double(R)
    if act == "gelu":
        proj.set_activation(dlp.PROJ_ACT_GELU)
        Y = proj(X, W, b, residual=gu.to_dev(R))
        ref = oracle.project_fused(inp["X"], inp["W"], synth.W_NK, inp["bias"], oracle.ACT_GELU, R64)
    else:
        proj.set_activation(dlp.PROJ_ACT_SWIGLU)
        Y = proj(X, proj.pack(W), None, packed=True, residual=gu.to_dev(R))
        ref = oracle.project_swiglu(inp["X"], inp["W"], synth.W_NK, R64)
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    gu.assert_within_tol(gu.y_to_f64(Y), ref, f"tm cluster fused {act}")
