"""GPU parity of the fused SwiGLU epilogue (Shazeer, "GLU Variants Improve
Transformer"): W stacks the gate rows then the up rows, packing interleaves
them inside each tile, and Y = SiLU(X·W_gateᵀ) · (X·W_upᵀ) (+ residual).

Every plan kind (cluster split, stream-K, token-major tiles, [K,N] weights,
ragged feature counts) is compared with the oracle's project_swiglu.
"""
import numpy as np
import pytest

import gpu_util as gu
import oracle
import synth

pytestmark = pytest.mark.gpu

SHAPES = [  # (M, F, K, layout, y_dtype, residual)
    (16, 1024, 8192, synth.W_NK, "bf16", False),   # 16 tiles: cluster split
    (16, 14336, 1024, synth.W_NK, "bf16", True),   # the FFN gate+up shape, short K: stream-K
    (9, 1000, 1032, synth.W_NK, "f32", False),     # ragged features and K
    (256, 2048, 1024, synth.W_NK, "bf16", True),   # token-major tiles
    (300, 520, 2056, synth.W_KN, "f32", True),     # token-major, [K,N], ragged
    (600, 512, 1032, synth.W_NK, "bf16", False),   # several token tiles
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "M{}_F{}_K{}_{}_{}{}".format(
    s[0], s[1], s[2], "KN" if s[3] else "NK", s[4], "_res" if s[5] else ""))
def test_swiglu_parity(shape):
    import torch
    import dense_linear_projection_gb300 as dlp
    M, F, K, layout, yd, res = shape
    w = synth.Workload("t", M, 2 * F, K, layout, False, yd, seed=111)
    inp = synth.make_inputs(w)
    proj = dlp.Projection(M, 2 * F, K, layout, dlp.PROJ_F32 if yd == "f32" else dlp.PROJ_BF16)
    proj.set_activation(dlp.PROJ_ACT_SWIGLU)
    X, W = gu.to_dev(inp["X"]), gu.to_dev(inp["W"])
    P = proj.pack(W)
    R, R64 = None, None
    if res:
        Rb = synth.normal_bf16(112, 7, M * F, 1.0).reshape(M, F)
        R = gu.to_dev(Rb)
        if yd == "f32":
            R = R.float()
        R64 = oracle.bf16_to_double(Rb)
    Y = proj(X, P, None, packed=True, residual=R)
    again = proj(X, P, None, packed=True, residual=R).clone()
    torch.cuda.synchronize()
    assert Y.shape == (M, F)
    assert proj.status() == dlp.PROJ_OK
    r = oracle.project_swiglu(inp["X"], inp["W"], layout, R64)
    gu.assert_within_tol(gu.y_to_f64(Y), r, f"swiglu {shape}")
    iv = torch.int16 if yd == "bf16" else torch.int32
    assert torch.equal(again.view(iv), Y.view(iv))


def test_swiglu_refusals():
    import torch
    import dense_linear_projection_gb300 as dlp
    L = dlp.lib()
    with_bias = dlp.Projection(16, 256, 512, dlp.PROJ_W_NK, dlp.PROJ_BF16, has_bias=True)
    assert L.proj_set_activation(with_bias.handle, dlp.PROJ_ACT_SWIGLU) == dlp.PROJ_ERR_UNSUPPORTED
    odd = dlp.Projection(16, 255, 512, dlp.PROJ_W_NK, dlp.PROJ_BF16)
    assert L.proj_set_activation(odd.handle, dlp.PROJ_ACT_SWIGLU) == dlp.PROJ_ERR_UNSUPPORTED
    fp32w = dlp.Projection(16, 256, 512, dlp.PROJ_W_NK, dlp.PROJ_F32, w_dtype=dlp.PROJ_F32)
    assert L.proj_set_activation(fp32w.handle, dlp.PROJ_ACT_SWIGLU) == dlp.PROJ_ERR_UNSUPPORTED
    proj = dlp.Projection(16, 256, 512, dlp.PROJ_W_NK, dlp.PROJ_BF16)
    proj.set_activation(dlp.PROJ_ACT_SWIGLU)
    X = torch.zeros((16, 512), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((256, 512), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((16, 128), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    # The interleaved layout exists only packed.
    assert L.proj_run(proj.handle, X.data_ptr(), W.data_ptr(), None, Y.data_ptr(), s) == dlp.PROJ_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
