"""Two 64-wide k-blocks a pipeline stage (plan block_k = 128).

The weight-streaming swapped plans (at most 64 tokens, K a multiple of 64)
load a stage's two k-blocks of W and of X with one TMA op each (3-D tensor
maps).  These cases cover what that adds: an odd number of k-blocks (the last
stage's second k-block lies past K and reads as zeros), every cluster-split
size, stream-K, half tiles, [K,N] weights as stored (one box per k-block),
packed weights (whole stages of zero-padded blocks), fp32 router weights whose
[H | L] halves are an even number of k-blocks, and the fused epilogues.  Each
is checked against the fp64 oracle, and against the same shape with one
k-block a stage (PROJ_KPB=1).
"""
import numpy as np
import pytest

import gpu_util as gu
import oracle
import synth

pytestmark = pytest.mark.gpu


def run(w, inp, packed, env, monkeypatch):
    import torch
    import dense_linear_projection_gb300 as dlp
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    proj = dlp.Projection(w.M, w.N, w.K, w.w_layout, dlp.PROJ_F32 if w.y_dtype == "f32" else dlp.PROJ_BF16,
                          has_bias=w.has_bias)
    for k in env:
        monkeypatch.delenv(k)
    X, W = gu.to_dev(inp["X"]), gu.to_dev(inp["W"])
    b = gu.to_dev(inp["bias"]) if w.has_bias else None
    Wr = proj.pack(W) if packed else W
    Y = proj(X, Wr, b, packed=packed)
    again = proj(X, Wr, b, packed=packed).clone()
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    plan = proj.plan
    proj.close()
    iv = torch.int16 if w.y_dtype == "bf16" else torch.int32
    assert torch.equal(again.view(iv), Y.view(iv)), "reruns differ"
    return plan, gu.y_to_f64(Y)


CASES = [  # (M, N, K, layout, bias, y_dtype, env)
    (16, 512, 1088, synth.W_NK, True, "bf16", {}),                           # 17 k-blocks: cluster split
    (16, 512, 1088, synth.W_NK, False, "f32", {"PROJ_MAX_CLUSTER": "0"}),    # stream-K, odd k-blocks
    (9, 2500, 2112, synth.W_NK, True, "bf16", {}),                           # ragged M and N, 33 k-blocks
    (16, 28672, 1024, synth.W_NK, False, "bf16", {}),                        # 224 tiles: stream-K pairs
    (64, 1024, 4160, synth.W_NK, True, "bf16", {}),                          # 64 tokens, 65 k-blocks
    (16, 1024, 1088, synth.W_KN, True, "bf16", {}),                          # [K,N] weights, swapped
    (33, 520, 576, synth.W_KN, False, "f32", {"PROJ_MAX_CLUSTER": "0"}),     # [K,N], ragged N, 9 k-blocks
    (16, 2048, 8192, synth.W_NK, False, "f32", {"PROJ_HALF_TILES": "2"}),    # half tiles
] + [
    (16, 384, 1088, synth.W_NK, True, "bf16", {"PROJ_MAX_CLUSTER": str(S), "PROJ_CLUSTER_FILL_PCT": "1"})
    for S in (2, 3, 4, 5, 6, 7, 8, 9)                                        # 3 tiles, 9 stages of K
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "M{}_N{}_K{}_{}_{}{}".format(
    c[0], c[1], c[2], "KN" if c[3] else "NK", c[5], "".join(f"_{k[5:]}{v}" for k, v in c[6].items())))
@pytest.mark.parametrize("packed", [False, True], ids=["stored", "packed"])
def test_two_kblocks_a_stage(case, packed, monkeypatch):
    M, N, K, layout, bias, yd, env = case
    w = synth.Workload("t", M, N, K, layout, bias, yd, seed=131)
    inp = synth.make_inputs(w)
    r = oracle.project(inp["X"], inp["W"], layout, inp["bias"])
    plan, u = run(w, inp, packed, env, monkeypatch)
    assert plan["block_k"] == 128 and plan["k_blocks"] == -(-K // 128), plan
    if "PROJ_MAX_CLUSTER" in env and env["PROJ_MAX_CLUSTER"] != "0":
        assert 2 <= plan["cluster_split"] <= int(env["PROJ_MAX_CLUSTER"])
    gu.assert_within_tol(u, r, f"block_k 128 {case} packed={packed}")
    # The same shape with one k-block a stage.
    plan1, u1 = run(w, inp, packed, dict(env, PROJ_KPB="1"), monkeypatch)
    assert plan1["block_k"] == 64
    gu.assert_within_tol(u1, r, f"block_k 64 {case} packed={packed}")


@pytest.mark.parametrize("K", [1024, 1088])
def test_router_even_and_odd_kblocks(K):
    # fp32 router weights: [H | L] along K.  With an even number of k-blocks
    # in K (1024: 16) a stage holds two of them and never straddles the
    # halves; with an odd number (1088: 17) the plan keeps one a stage.
    import torch
    import dense_linear_projection_gb300 as dlp
    M, N = 16, 256
    w = synth.Workload("t", M, N, K, synth.W_NK, False, "f32", seed=132, w_dtype="f32")
    inp = synth.make_inputs(w)
    proj = dlp.Projection(M, N, K, synth.W_NK, dlp.PROJ_F32, w_dtype=dlp.PROJ_F32)
    kt = K // 64
    assert proj.plan["block_k"] == (128 if kt % 2 == 0 else 64)
    assert proj.plan["k_blocks"] * proj.plan["block_k"] == 2 * kt * 64
    P = proj.pack(torch.from_numpy(inp["W"]).cuda())
    Y = proj(gu.to_dev(inp["X"]), P, None, packed=True)
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    exact = oracle.project_f32w(inp["X"], inp["W"], synth.W_NK, None)
    u = gu.y_to_f64(Y)
    assert np.linalg.norm(u - exact) / np.linalg.norm(exact) <= 1e-4  # the router's 0.01 % rule


def test_fused_gelu_residual_two_kblocks():
    import torch
    import dense_linear_projection_gb300 as dlp
    M, N, K = 16, 1024, 1088
    w = synth.Workload("t", M, N, K, synth.W_NK, True, "bf16", seed=133)
    inp = synth.make_inputs(w)
    proj = dlp.Projection(M, N, K, synth.W_NK, dlp.PROJ_BF16, has_bias=True)
    assert proj.plan["block_k"] == 128
    proj.set_activation(dlp.PROJ_ACT_GELU)
    Rb = synth.normal_bf16(134, 7, M * N, 1.0).reshape(M, N)
    P = proj.pack(gu.to_dev(inp["W"]))
    Y = proj(gu.to_dev(inp["X"]), P, gu.to_dev(inp["bias"]), packed=True, residual=gu.to_dev(Rb))
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    r = oracle.gelu(oracle.project(inp["X"], inp["W"], synth.W_NK, inp["bias"])) + oracle.bf16_to_double(Rb)
    gu.assert_within_tol(gu.y_to_f64(Y), r, "fused gelu + residual, block_k 128")
