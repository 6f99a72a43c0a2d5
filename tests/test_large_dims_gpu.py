"""Large dimensions, one at a time, against the fp64 oracle.

Index arithmetic that is exact at the benchmark shapes can still overflow
when one dimension grows: TMA coordinates and packed-plane indices are 32-bit,
output offsets must be 64-bit.  Each case stretches one dimension well past
the benchmark's (N: 131072 weight rows, 1 GiB of weights; M: 65536 tokens;
K: 262144, 2 GiB of weights) and compares the whole output with the oracle,
for the weights as stored and packed (which must give the same bits).
"""
import numpy as np
import pytest

import gpu_util as gu
import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K,layout,bias,yd", [
    (16, 131072, 4096, synth.W_NK, True, "bf16"),   # 1024 weight tiles, stream-K over every SM
    (65536, 512, 512, synth.W_NK, False, "bf16"),   # 256 token tiles, 64 MiB of output
    (4, 4096, 262144, synth.W_NK, False, "f32"),    # 4096 k-blocks, a 512 KiB activation row
], ids=["N131072", "M65536", "K262144"])
def test_large_dimension(M, N, K, layout, bias, yd):
    import torch
    import dense_linear_projection_gb300 as dlp
    w = synth.Workload("t", M, N, K, layout, bias, yd, seed=101)
    inp = synth.make_inputs(w)
    proj, Y, (X, W, b) = gu.run(w, inp)
    Yp = proj(X, proj.pack(W), b, packed=True)
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    r = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
    gu.assert_within_tol(gu.y_to_f64(Y), r, f"M={M} N={N} K={K} plan={proj.plan}")
    iv = torch.int16 if yd == "bf16" else torch.int32
    assert torch.equal(Yp.view(iv), Y.view(iv)), "packed weights differ from the weights as stored"
