"""The allocation-free entry point, proj_run_noalloc, and its status readback.

It exists for callers that cannot call cudaMalloc (a serving loop where an
allocation may stall every stream, a plug-in whose host owns all device
memory).  It runs the same kernel with the same plan as the handle-based
proj_run, so its output must be the same bits, call after call: its fixed
device scratch keeps the previous call's contents, so two calls in a row
check that nothing stale leaks into the second.  One shape is also checked
against the fp64 oracle directly, and the status word the kernel writes is
read back through proj_noalloc_device_status.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test; it passes alone in a fresh process
as well as after the rest.
"""
import numpy as np
import pytest

import gpu_util as gu
import oracle
import synth

pytestmark = pytest.mark.gpu


def _bits(t):
    import torch
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


@pytest.mark.parametrize("M,N,K,layout,bias,yd", [
    (16, 8192, 8192, synth.W_NK, True, "bf16"),   # decode shape: clusters of 2
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
    assert dlp.proj_noalloc_device_status() == dlp.PROJ_OK
    for inp in (first, second):  # two calls in a row
        X, W = gu.to_dev(inp["X"]), gu.to_dev(inp["W"])
        b = gu.to_dev(inp["bias"]) if bias else None
        ref = proj(X, W, b)
        out = torch.full((M, N), float("nan"), dtype=tdt, device="cuda")
        dlp.proj_run_noalloc(M, N, K, layout, y_dtype, X, W, b, out,
                             torch.cuda.current_stream())
        torch.cuda.synchronize()
        # Same kernel, same plan, same inputs: the same bits.
        assert torch.equal(_bits(out), _bits(ref)), f"noalloc M={M} N={N} K={K} differs from proj_run"
        assert dlp.proj_noalloc_device_status() == dlp.PROJ_OK
    proj.close()


def test_noalloc_against_the_oracle():
    # The decode shape with a bias, straight against the fp64 oracle (the
    # whole output, both calls of a pair with different activations).
    import torch
    import dense_linear_projection_gb300 as dlp
    M, N, K = 16, 8192, 8192
    w = synth.Workload("t", M, N, K, synth.W_NK, True, "bf16", seed=43)
    inp = synth.make_inputs(w)
    W, b = gu.to_dev(inp["W"]), gu.to_dev(inp["bias"])
    for seed in (44, 45):
        Xh = synth.normal_bf16(seed, synth.STREAM_X, M * K, 1.0).reshape(M, K)
        out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        dlp.proj_run_noalloc(M, N, K, synth.W_NK, dlp.PROJ_BF16, gu.to_dev(Xh), W, b, out)
        torch.cuda.synchronize()
        assert dlp.proj_noalloc_device_status() == dlp.PROJ_OK
        r = oracle.project(Xh, inp["W"], oracle.W_NK, inp["bias"])
        gu.assert_within_tol(gu.y_to_f64(out), r, f"noalloc vs oracle (X seed {seed})")


def test_noalloc_status_reports_a_timed_out_wait():
    # A bounded wait that nothing completes gives up, records the timeout in
    # the fixed array's status word, and the readback reports it once.
    import torch
    import dense_linear_projection_gb300 as dlp
    assert dlp.proj_noalloc_device_status() == dlp.PROJ_OK
    dlp.proj_noalloc_selftest_wait_timeout(100_000)
    assert dlp.proj_noalloc_device_status() == dlp.PROJ_ERR_DEVICE_TIMEOUT
    assert dlp.proj_noalloc_device_status() == dlp.PROJ_OK  # read clears the word
    # The path still works afterwards.
    M, N, K = 16, 1024, 512
    w = synth.Workload("t", M, N, K, synth.W_NK, False, "f32", seed=46)
    inp = synth.make_inputs(w)
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    dlp.proj_run_noalloc(M, N, K, synth.W_NK, dlp.PROJ_F32, gu.to_dev(inp["X"]), gu.to_dev(inp["W"]),
                         None, out)
    assert dlp.proj_noalloc_device_status() == dlp.PROJ_OK
    gu.assert_within_tol(gu.y_to_f64(out), oracle.project(inp["X"], inp["W"], oracle.W_NK, None),
                         "noalloc after a timed-out wait")
    with pytest.raises(dlp.ProjError) as e:
        dlp.proj_noalloc_selftest_wait_timeout(10)  # below the 1 µs minimum
    assert e.value.status == dlp.PROJ_ERR_INVALID_ARG


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
