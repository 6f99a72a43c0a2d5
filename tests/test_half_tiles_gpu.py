"""GPU parity of half tiles: swapped tiles of 64 weight rows.

The tensor-core MMA keeps M = 128; a half tile's stage loads 64 weight rows
into the 128-row A region, and accumulator rows 64-127 (from the region's
other half) are never read: the epilogue warps of those rows only release the
accumulator.  They are an option (PROJ_HALF_TILES=2) for any swapped plan of
at most 64 tokens: cluster splits, stream-K, whole tiles, [K,N] weights, the
fused epilogue and SwiGLU.  Each case is compared with the fp64
oracle and must rerun bit for bit.
"""
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


FORCE = {"PROJ_HALF_TILES": "2"}
SK = {"PROJ_HALF_TILES": "2", "PROJ_MAX_CLUSTER": "0"}
# (M, N, K, layout, bias, y_dtype, environment, expected split kind)
HALF_CASES = [
    (16, 2048, 8192, synth.W_NK, False, "f32", FORCE, "cluster"),     # the 2048-row decode weight
    (16, 2048, 8192, synth.W_NK, True, "bf16", FORCE, "cluster"),
    (9, 1000, 1032, synth.W_NK, True, "bf16", FORCE, "cluster"),     # ragged N, 17 k-blocks
    (16, 2048, 8192, synth.W_NK, False, "f32", SK, "stream-K"),       # split tiles through scratch
    (9, 2504, 1032, synth.W_KN, True, "bf16", SK, "stream-K"),        # [K,N] as stored, ragged
    (16, 20000, 256, synth.W_NK, True, "bf16", FORCE, "stream-K"),    # whole tiles + split tail
    (40, 3000, 520, synth.W_KN, False, "f32", FORCE, None),
]


@pytest.mark.parametrize("case", HALF_CASES, ids=lambda c: "M{}_N{}_K{}_{}_{}_{}".format(
    c[0], c[1], c[2], "KN" if c[3] else "NK", c[5], "_".join(f"{k[5:]}{v}" for k, v in c[6].items()) or "auto"))
@pytest.mark.parametrize("packed", [False, True], ids=["stored", "packed"])
def test_half_tile_parity(case, packed, monkeypatch):
    M, N, K, layout, bias, yd, env, kind = case
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    w = synth.Workload("t", M, N, K, layout, bias, yd, seed=111)
    inp = synth.make_inputs(w)
    proj, Y = _run(w, inp, packed)
    p = proj.plan
    assert p["swap_ab"] == 1 and p["block_n"] == 64
    if kind == "cluster":
        assert p["cluster_split"] >= 2
    elif kind == "stream-K":
        assert p["cluster_split"] == 0 and p["tiles_sk"] > 0
    r = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
    gu.assert_within_tol(gu.y_to_f64(Y), r, f"half tiles {case[:6]} packed={packed}")


def test_half_tile_small_integers_bit_exact(monkeypatch):
    # Integer operands keep every partial sum exact: the half-tile cluster
    # split must give exactly X·Wᵀ.
    import numpy as np
    import torch
    import dense_linear_projection_gb300 as dlp
    monkeypatch.setenv("PROJ_HALF_TILES", "2")
    M, N, K = 16, 2048, 8192
    rng = np.random.default_rng(12)
    X = rng.integers(-3, 4, size=(M, K)).astype(np.float64)
    Wnk = rng.integers(-3, 4, size=(N, K)).astype(np.float64)
    proj = dlp.Projection(M, N, K, dlp.PROJ_W_NK, dlp.PROJ_F32)
    assert proj.plan["block_n"] == 64 and proj.plan["cluster_split"] >= 2
    Y = proj(gu.to_dev(synth.to_bf16_bits(X)), gu.to_dev(synth.to_bf16_bits(Wnk)), None)
    torch.cuda.synchronize()
    assert np.array_equal(gu.y_to_f64(Y), X @ Wnk.T)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_half_tile_fused_epilogue(act, monkeypatch):
    import torch
    import dense_linear_projection_gb300 as dlp
    monkeypatch.setenv("PROJ_HALF_TILES", "2")
    M, N, K = 16, 2 * 1100, 2056
    has_bias = act == "gelu"
    w = synth.Workload("t", M, N, K, synth.W_NK, has_bias, "bf16", seed=112)
    inp = synth.make_inputs(w)
    proj = dlp.Projection(M, N, K, synth.W_NK, dlp.PROJ_BF16, has_bias=has_bias)
    assert proj.plan["block_n"] == 64
    X, W = gu.to_dev(inp["X"]), gu.to_dev(inp["W"])
    b = gu.to_dev(inp["bias"]) if has_bias else None
    F = N // 2 if act == "swiglu" else N
    R = synth.normal_bf16(113, 7, M * F, 1.0).reshape(M, F)
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
    gu.assert_within_tol(gu.y_to_f64(Y), ref, f"half tiles fused {act}")
