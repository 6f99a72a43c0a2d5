"""GPU parity of the fused epilogue Y = act(X·Wᵀ + bias) + residual.

The worklog's second page writes the FFN intermediate once by fusing GELU
into the projection's epilogue, and fuses the residual add of an output
projection; GELU is taken from its definition x·Φ(x).  Every plan kind
(cluster split, stream-K, whole tiles, token-major tiles, [K,N] weights,
packed weights) is compared with the fp64 oracle's project_fused, with and
without GELU, with a separate residual and with the residual being Y itself.
"""
import numpy as np
import pytest

import gpu_util as gu
import oracle
import synth

pytestmark = pytest.mark.gpu

SHAPES = [
    (16, 2048, 8192, synth.W_NK, True, "bf16"),    # cluster split
    (16, 8192, 2048, synth.W_NK, False, "f32"),    # stream-K pairs
    (9, 1000, 1032, synth.W_NK, True, "bf16"),     # ragged N and K
    (256, 12288, 1024, synth.W_KN, True, "bf16"),  # token-major, [K,N]
    (300, 1000, 2056, synth.W_KN, False, "f32"),   # token-major, ragged
    (600, 1000, 1032, synth.W_NK, True, "bf16"),   # several token tiles
]


def _residual(w, seed, tdt):
    import torch
    R = synth.normal_bf16(seed, 7, w.M * w.N, 1.0).reshape(w.M, w.N)
    t = gu.to_dev(R)
    return (t.float() if tdt == torch.float32 else t), oracle.bf16_to_double(R)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "M{}_N{}_K{}_{}_{}".format(
    s[0], s[1], s[2], "KN" if s[3] else "NK", s[5]))
@pytest.mark.parametrize("act", [0, 1], ids=["noact", "gelu"])
@pytest.mark.parametrize("res", ["none", "separate", "in_place"])
def test_fused_epilogue_parity(shape, act, res):
    import torch
    import dense_linear_projection_gb300 as dlp
    M, N, K, layout, bias, yd = shape
    w = synth.Workload("t", M, N, K, layout, bias, yd, seed=101)
    inp = synth.make_inputs(w)
    proj = dlp.Projection(M, N, K, layout, dlp.PROJ_F32 if yd == "f32" else dlp.PROJ_BF16,
                          has_bias=bias)
    proj.set_activation(act)
    X, W = gu.to_dev(inp["X"]), gu.to_dev(inp["W"])
    b = gu.to_dev(inp["bias"]) if bias else None
    tdt = torch.float32 if yd == "f32" else torch.bfloat16
    R, R64 = (None, None) if res == "none" else _residual(w, 102, tdt)
    if res == "in_place":
        Y = R.clone()
        proj(X, W, b, out=Y, residual=Y)
    else:
        Y = proj(X, W, b, residual=R)
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    r = oracle.project_fused(inp["X"], inp["W"], layout, inp["bias"], act, R64)
    gu.assert_within_tol(gu.y_to_f64(Y), r, f"{shape} act={act} res={res}")


def test_fused_with_packed_weights_matches_stored():
    import torch
    import dense_linear_projection_gb300 as dlp
    w = synth.Workload("t", 16, 28672, 1024, synth.W_NK, False, "bf16", 103)  # the FFN up shape, short K
    inp = synth.make_inputs(w)
    proj = dlp.Projection(w.M, w.N, w.K, w.w_layout, dlp.PROJ_BF16)
    proj.set_activation(dlp.PROJ_ACT_GELU)
    X, W = gu.to_dev(inp["X"]), gu.to_dev(inp["W"])
    P = proj.pack(W)
    R, R64 = _residual(w, 104, torch.bfloat16)
    Y1 = proj(X, W, None, residual=R)
    Y2 = proj(X, P, None, residual=R, packed=True)
    torch.cuda.synchronize()
    assert torch.equal(Y1.view(torch.int16), Y2.view(torch.int16))
    gu.assert_within_tol(gu.y_to_f64(Y2), oracle.project_fused(inp["X"], inp["W"], 0, None, 1, R64),
                         "packed fused")


def test_fused_empty_sum_fill():
    # K = 0: Y = act(bias) + residual.
    import torch
    import dense_linear_projection_gb300 as dlp
    M, N = 5, 40
    proj = dlp.Projection(M, N, 0, dlp.PROJ_W_NK, dlp.PROJ_F32, has_bias=True)
    proj.set_activation(dlp.PROJ_ACT_GELU)
    bb = synth.to_bf16_bits(np.linspace(-3, 3, N))
    b = gu.to_dev(bb)
    R = torch.arange(M * N, dtype=torch.float32, device="cuda").reshape(M, N) / 8
    X = torch.zeros((M, 0), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((N, 0), dtype=torch.bfloat16, device="cuda")
    Y = proj(X, W, b, residual=R)
    torch.cuda.synchronize()
    want = oracle.gelu(np.broadcast_to(oracle.bf16_to_double(bb), (M, N))) + R.cpu().numpy()
    gu.assert_within_tol(Y.cpu().numpy().astype(np.float64), want, "fill")


def test_fused_bad_arguments():
    import torch
    import dense_linear_projection_gb300 as dlp
    L = dlp.lib()
    proj = dlp.Projection(16, 256, 512, dlp.PROJ_W_NK, dlp.PROJ_BF16)
    assert L.proj_set_activation(proj.handle, 5) == dlp.PROJ_ERR_INVALID_ARG
    assert L.proj_set_activation(None, 0) == dlp.PROJ_ERR_INVALID_ARG
    X = torch.zeros((16, 512), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((256, 512), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((16, 256), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert L.proj_run_fused(proj.handle, X.data_ptr(), W.data_ptr(), 0, None, Y.data_ptr() + 1,
                            Y.data_ptr(), s) == dlp.PROJ_ERR_MISALIGNED
    assert L.proj_run_fused(proj.handle, X.data_ptr(), W.data_ptr(), 2, None, None,
                            Y.data_ptr(), s) == dlp.PROJ_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
