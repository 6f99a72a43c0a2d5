"""GPU parity of CTA-pair plans: each tile computed by the two CTAs of a
cluster with one 256-row tcgen05 MMA (cta_group::2), each CTA staging half of
the tile's weight rows and half of its token rows.

Planner-chosen pairs (swapped 256-token tiles) and pairs forced on other
tiles (PROJ_CTA_PAIR=2): token-major tiles (the QKV shape among them),
narrower token tiles, several tiles per pair with both accumulator buffers in
turn, ragged M, N and K, [K,N] weights loaded as stored and packed, fp32
output, the fused epilogue and SwiGLU.  Each is compared with the fp64
oracle, must rerun bit for bit and must leave the device status clear (both
CTAs of a pair see the same tensor memory).
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


# (M, N, K, layout, bias, y_dtype, environment, expected (swap, block_t, block_n, tmem_cols))
PAIR = {"PROJ_CTA_PAIR": "2"}
PAIR_CASES = [
    # Planner-chosen swapped pairs: 256 weight rows x 256 tokens, 2.1 waves.
    (512, 20480, 256, synth.W_NK, True, "bf16", {}, (1, 256, 256, 512)),
    (700, 9000, 1032, synth.W_NK, False, "f32", {}, (1, 256, 256, 512)),  # ragged M, N, K
    # Forced token-major pairs.
    (600, 1000, 1032, synth.W_NK, False, "bf16", PAIR, (0, 256, 64, 128)),
    (1024, 4096, 1024, synth.W_NK, True, "bf16", PAIR, None),
    (1024, 4096, 1024, synth.W_NK, True, "f32", PAIR, None),
    (300, 2600, 520, synth.W_NK, True, "bf16", PAIR, None),           # ragged M (44 rows), N, 9 k-blocks
    # Forced: 256-column accumulators, several tiles per pair (2 waves).
    (1024, 8192, 512, synth.W_NK, True, "bf16", {"PROJ_CTA_PAIR": "2", "PROJ_FORCE_BLOCK_N": "256"},
     (0, 256, 256, 512)),
    # Forced swapped pairs: 256 weight rows x 64 tokens, two accumulators.
    (100, 2600, 1032, synth.W_NK, True, "bf16", {"PROJ_CTA_PAIR": "2", "PROJ_FORCE_BLOCK_T": "64"},
     (1, 64, 256, 128)),
    (100, 2600, 1032, synth.W_KN, False, "f32", {"PROJ_CTA_PAIR": "2", "PROJ_FORCE_BLOCK_T": "64"},
     (1, 64, 256, 128)),
    # Forced swapped pairs with two accumulators and 4-5 tiles per pair.
    (100, 40000, 264, synth.W_NK, True, "bf16", {"PROJ_CTA_PAIR": "2", "PROJ_FORCE_BLOCK_T": "64"},
     (1, 64, 256, 128)),
    # Forced swapped pairs of 256 tokens, many tiles per pair.
    (1000, 6000, 520, synth.W_NK, True, "bf16", {"PROJ_CTA_PAIR": "2", "PROJ_FORCE_BLOCK_T": "256"},
     (1, 256, 256, 512)),
    # [K,N] weights as stored with whole 64-column halves (128-row tiles).
    (512, 3000, 1032, synth.W_KN, True, "bf16", {"PROJ_CTA_PAIR": "2", "PROJ_FORCE_BLOCK_N": "128"},
     (0, 256, 128, 256)),
]


def _ids(c):
    env = "_".join(f"{k[5:]}{v}" for k, v in c[6].items())
    return "M{}_N{}_K{}_{}_{}_{}".format(c[0], c[1], c[2], "KN" if c[3] else "NK", c[5], env or "auto")


@pytest.mark.parametrize("case", PAIR_CASES, ids=_ids)
@pytest.mark.parametrize("packed", [False, True], ids=["stored", "packed"])
def test_pair_parity(case, packed, monkeypatch):
    M, N, K, layout, bias, yd, env, expect = case
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    w = synth.Workload("t", M, N, K, layout, bias, yd, seed=91)
    inp = synth.make_inputs(w)
    proj, Y = _run(w, inp, packed)
    p = proj.plan
    assert p["cta_pair"] == 1 and p["grid"] % 2 == 0
    if expect is not None:
        assert (p["swap_ab"], p["block_t"], p["block_n"], p["tmem_cols"]) == expect
    r = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
    gu.assert_within_tol(gu.y_to_f64(Y), r, f"pair {case[:6]} packed={packed}")


# Stream-K over CTA pairs (PROJ_PAIR_SK=1): token-major pair tiles of 256
# weight columns whose last partial wave and one full wave are shared along K
# by all pairs; each CTA of a pair writes and reads its own 128 rows of a
# split tile's partial slots and counts its own row quarters.
PAIR_SK_CASES = [
    (256, 12288, 4096, synth.W_KN, True, "bf16"),   # the QKV shape: 48 tiles on 76 pairs, all split
    (384, 5000, 2056, synth.W_NK, True, "f32"),     # 2 x 20 tiles, ragged N and K
    (300, 30000, 520, synth.W_KN, False, "bf16"),   # 2 x 118 tiles: whole waves plus a split tail
    (256, 2000, 8192, synth.W_NK, True, "bf16"),    # 8 tiles on 76 pairs: many contributors a tile
]


@pytest.mark.parametrize("case", PAIR_SK_CASES, ids=lambda c: "M{}_N{}_K{}_{}_{}".format(
    c[0], c[1], c[2], "KN" if c[3] else "NK", c[5]))
@pytest.mark.parametrize("packed", [False, True], ids=["stored", "packed"])
def test_pair_stream_k_parity(case, packed, monkeypatch):
    M, N, K, layout, bias, yd = case
    monkeypatch.setenv("PROJ_PAIR_SK", "1")
    monkeypatch.setenv("PROJ_CTA_PAIR", "2")  # pairs also where the planner would not take them
    monkeypatch.setenv("PROJ_FORCE_BLOCK_N", "256")  # token-major tiles of 256 weight columns
    w = synth.Workload("t", M, N, K, layout, bias, yd, seed=93)
    inp = synth.make_inputs(w)
    proj, Y = _run(w, inp, packed)  # also checks a bit-identical rerun
    p = proj.plan
    assert p["cta_pair"] == 1 and p["swap_ab"] == 0 and p["block_n"] == 256 and p["tiles_sk"] > 0
    r = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
    gu.assert_within_tol(gu.y_to_f64(Y), r, f"pair stream-K {case} packed={packed}")


@pytest.mark.parametrize("M,N,K", [(1024, 4096, 1024), (768, 20480, 512)])
def test_pair_agrees_with_single_ctas(M, N, K, monkeypatch):
    # The same problem on pairs (PROJ_CTA_PAIR=2) and on single CTAs (0),
    # each against the oracle.  (Each output is rounded to bf16 on its own,
    # so the two may differ by one unit in the last place where the fp32 sums
    # differ in their last bits: they are not compared with each other.)
    w = synth.Workload("t", M, N, K, synth.W_NK, True, "bf16", seed=92)
    inp = synth.make_inputs(w)
    monkeypatch.setenv("PROJ_CTA_PAIR", "2")
    proj, Y = _run(w, inp)
    assert proj.plan["cta_pair"] == 1
    monkeypatch.setenv("PROJ_CTA_PAIR", "0")
    single, Ys = _run(w, inp)
    assert single.plan["cta_pair"] == 0
    r = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
    gu.assert_within_tol(gu.y_to_f64(Y), r, "pairs")
    gu.assert_within_tol(gu.y_to_f64(Ys), r, "single CTAs")


def test_qkv_shape_pairs_sampled(monkeypatch):
    # The QKV shape (256 x 12288 x 4096, [K,N] weights, bias) on pairs:
    # packed weights run on 70 pair tiles of 176 weight rows; weights as
    # stored (halves of 88 columns are not whole boxes) on the handle's
    # single-CTA plan.  Sampled cells against the oracle, and both runs
    # against each other.
    import torch
    import dense_linear_projection_gb300 as dlp
    monkeypatch.setenv("PROJ_CTA_PAIR", "2")
    w = synth.WORKLOADS["qkv_kn_bias"]
    inp = synth.make_inputs(w)
    proj = dlp.Projection(w.M, w.N, w.K, w.w_layout, dlp.PROJ_BF16, has_bias=True)
    assert proj.plan["cta_pair"] == 1 and proj.plan["block_n"] == 176 and proj.plan["grid"] == 140
    X, W, b = gu.to_dev(inp["X"]), gu.to_dev(inp["W"]), gu.to_dev(inp["bias"])
    Yp = proj(X, proj.pack(W), b, packed=True)
    Ys = proj(X, W, b)
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    ms, ns = gu.sample_cells(w.M, w.N, 512, seed=5, tile_n=176)
    ref = oracle.project_cells(inp["X"], inp["W"], w.w_layout, inp["bias"], ms, ns)
    yp, ys = gu.y_to_f64(Yp), gu.y_to_f64(Ys)
    gu.assert_within_tol(yp[ms, ns], ref, "qkv pairs (packed)")
    gu.assert_within_tol(ys[ms, ns], ref, "qkv single CTAs (stored)")
    # Everywhere: the two runs within twice the tolerance of each other (each
    # is within the tolerance of the exact value).
    assert (np.abs(yp - ys) <= 2 * (gu.TOL_ABS + gu.TOL_REL * np.abs(ys))).all()


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_pair_fused_epilogue(act, monkeypatch):
    # The fused instance of the pair kernel: GELU + residual on a
    # planner-chosen pair plan; SwiGLU on forced swapped pairs (16 gate and
    # 16 up rows per 32-row quarter of each CTA's 128 rows).
    import torch
    import dense_linear_projection_gb300 as dlp
    if act == "gelu":
        M, N, K, env = 512, 20480, 256, {}
    else:
        M, N, K, env = 100, 2 * 1300, 1032, {"PROJ_CTA_PAIR": "2", "PROJ_FORCE_BLOCK_T": "64"}
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    has_bias = act == "gelu"
    w = synth.Workload("t", M, N, K, synth.W_NK, has_bias, "bf16", seed=93)
    inp = synth.make_inputs(w)
    proj = dlp.Projection(M, N, K, synth.W_NK, dlp.PROJ_BF16, has_bias=has_bias)
    assert proj.plan["cta_pair"] == 1
    X, W = gu.to_dev(inp["X"]), gu.to_dev(inp["W"])
    b = gu.to_dev(inp["bias"]) if has_bias else None
    F = N // 2 if act == "swiglu" else N
    R = synth.normal_bf16(94, 7, M * F, 1.0).reshape(M, F)
    R64 = oracle.bf16_to_double(R)
    Rd = gu.to_dev(R)
    if act == "gelu":
        proj.set_activation(dlp.PROJ_ACT_GELU)
        Y = proj(X, W, b, residual=Rd)
        ref = oracle.project_fused(inp["X"], inp["W"], synth.W_NK, inp["bias"], oracle.ACT_GELU, R64)
    else:
        proj.set_activation(dlp.PROJ_ACT_SWIGLU)
        Y = proj(X, proj.pack(W), None, packed=True, residual=Rd)
        ref = oracle.project_swiglu(inp["X"], inp["W"], synth.W_NK, R64)
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    gu.assert_within_tol(gu.y_to_f64(Y), ref, f"pair fused {act}")


def test_pair_graph_replay_follows_fresh_inputs():
    import torch
    import dense_linear_projection_gb300 as dlp
    w = synth.Workload("t", 512, 20480, 256, synth.W_NK, True, "bf16", 95)
    inp = synth.make_inputs(w)
    proj, Y, (X, W, b) = gu.run(w, inp)
    assert proj.plan["cta_pair"] == 1
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        proj(X, W, b, out=Y, stream=s)
    for seed in (96, 97):
        x = synth.normal_bf16(seed, synth.STREAM_X, w.M * w.K, 1.0).reshape(w.M, w.K)
        X.copy_(gu.to_dev(x))
        Y.zero_()
        g.replay()
        torch.cuda.synchronize()
        gu.assert_within_tol(gu.y_to_f64(Y), oracle.project(x, inp["W"], w.w_layout, inp["bias"]),
                             f"pair replay seed {seed}")
    assert proj.status() == dlp.PROJ_OK
