"""The allocation-free entry point, proj_run_noalloc.

It exists for callers that cannot call cudaMalloc (a serving loop where an
allocation may stall every stream, a plug-in whose host owns all device
memory).  It must give the same results as the handle-based proj_run, call
after call: its fixed device scratch keeps the previous call's contents, so
two calls in a row check that nothing stale leaks into the second.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test; it passes alone in a fresh process
as well as after the rest.
"""
import numpy as np
import pytest

import gpu_util as gu
import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K,layout,bias,yd", [
    (16, 8192, 8192, synth.W_NK, True, "bf16"),   # decode shape: stream-K over every SM
    (16, 2048, 8192, synth.W_NK, False, "f32"),   # 16 tiles split over clusters
    (16, 28672, 1024, synth.W_NK, True, "bf16"),  # 224 tiles: split-K through the scratch
    (3, 520, 1032, synth.W_KN, True, "bf16"),     # [K,N] weights, ragged edges
    (256, 19456, 256, synth.W_NK, False, "bf16"), # 76 whole tiles on CTA pairs, one wave: no split scratch
])
def test_noalloc_matches_proj_run_twice(M, N, K, layout, bias, yd):
    import torch
    import dense_linear_projection_gb300 as dlp
    y_dtype = dlp.PROJ_F32 if yd == "f32" else dlp.PROJ_BF16
    tdt = torch.float32 if yd == "f32" else torch.bfloat16
    w = synth.Workload("t", M, N, K, layout, bias, yd, seed=41)
    first = synth.make_inputs(w)
    second = dict(first, X=synth.normal_bf16(42, synth.STREAM_X, M * K, 1.0).reshape(M, K))
    proj = dlp.Projection(M, N, K, layout, y_dtype, has_bias=bias)
    for inp in (first, second):  # two calls in a row
        X, W = gu.to_dev(inp["X"]), gu.to_dev(inp["W"])
        b = gu.to_dev(inp["bias"]) if bias else None
        ref = proj(X, W, b)
        out = torch.full((M, N), float("nan"), dtype=tdt, device="cuda")
        dlp.proj_run_noalloc(M, N, K, layout, y_dtype, X, W, b, out,
                             torch.cuda.current_stream())
        torch.cuda.synchronize()
        gu.assert_within_tol(gu.y_to_f64(out), gu.y_to_f64(ref), f"noalloc M={M} N={N} K={K}")


def test_noalloc_refuses_plans_beyond_its_scratch():
    import torch
    import dense_linear_projection_gb300 as dlp
    M, N, K = 64, 20000, 512  # split tiles of 64 tokens: about 9.5 MiB of scratch
    assert dlp.proj_plan_compute(M, N, K)["scratch_bytes"] > 8 << 20
    X = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dlp.ProjError) as e:
        dlp.proj_run_noalloc(M, N, K, dlp.PROJ_W_NK, dlp.PROJ_BF16, X, W, None, Y)
    assert e.value.status == dlp.PROJ_ERR_UNSUPPORTED
