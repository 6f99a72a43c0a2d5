"""GPU parity of pre-packed weights (proj_pack_weights + proj_run_packed).

The packed layout is the preparation step of "How I made Muse's GPU
projections 1.32× faster in the Open Kernel Challenge", section "Sometimes
moving the same numbers around was enough": each weight tile's values stored
next to each other.  The tests rebuild the layout from its definition with
numpy (not with the library) and compare it bit for bit.  They run packed
weights through every kind of plan against the fp64 oracle, and require the
same bits as the unpacked run for [N,K] weights (the same loads reach shared
memory in the same order).
"""
import numpy as np
import pytest

import gpu_util as gu
import oracle
import synth

pytestmark = pytest.mark.gpu


def expected_packed(W_bits, layout, N, K, block_n, k_blocks, tiles_n):
    """The packed layout from its definition: block (t, b) = rows t·block_n + r,
    K positions b·64 + c, K contiguous; zero outside the matrix."""
    Wnk = W_bits if layout == synth.W_NK else np.ascontiguousarray(W_bits.T)
    full = np.zeros((tiles_n * block_n, k_blocks * 64), dtype=np.uint16)
    full[:N, :K] = Wnk.reshape(N, K)
    blocks = full.reshape(tiles_n, block_n, k_blocks, 64).transpose(0, 2, 1, 3)
    return np.ascontiguousarray(blocks).reshape(-1)


# (M, N, K, layout, bias, y_dtype): cluster split, stream-K, whole tiles,
# token-major tiles, [K,N] weights, ragged N and K.
PACKED_SHAPES = [
    (16, 8192, 8192, synth.W_NK, True, "bf16"),    # decode: clusters of 2
    (16, 2048, 8192, synth.W_NK, False, "f32"),    # decode, fp32 out
    (16, 28672, 1024, synth.W_NK, False, "bf16"),  # 224 tiles: stream-K pairs
    (9, 2500, 1032, synth.W_NK, True, "bf16"),     # ragged N, ragged last K block
    (256, 12288, 4096, synth.W_KN, True, "bf16"),  # the qkv shape: token-major, [K,N]
    (300, 1000, 2056, synth.W_KN, True, "f32"),    # token-major, ragged everything
    (600, 1000, 1032, synth.W_NK, False, "bf16"),  # several token tiles
    (512, 20480, 256, synth.W_NK, True, "bf16"),   # data-parallel waves + split tail
]


def _ids(s):
    return "M{}_N{}_K{}_{}".format(s[0], s[1], s[2], "KN" if s[3] else "NK")


@pytest.mark.parametrize("shape", PACKED_SHAPES, ids=_ids)
def test_packed_run_parity(shape):
    import torch
    import dense_linear_projection_gb300 as dlp
    M, N, K, layout, bias, yd = shape
    w = synth.Workload("t", M, N, K, layout, bias, yd, seed=81)
    inp = synth.make_inputs(w)
    proj, Y, (X, W, b) = gu.run(w, inp)
    P = proj.pack(W)
    Yp = proj(X, P, b, packed=True)
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    r = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
    gu.assert_within_tol(gu.y_to_f64(Yp), r, f"packed {shape}")
    if layout == synth.W_NK:
        iv = torch.int16 if yd == "bf16" else torch.int32
        assert torch.equal(Yp.view(iv), Y.view(iv))


@pytest.mark.parametrize("M,N,K,layout", [(16, 300, 1032, synth.W_NK), (9, 2500, 1032, synth.W_NK),
                                          (300, 1000, 2056, synth.W_KN), (40, 136, 520, synth.W_KN)])
def test_pack_layout_matches_definition(M, N, K, layout):
    import torch
    import dense_linear_projection_gb300 as dlp
    w = synth.Workload("t", M, N, K, layout, False, "bf16", seed=82)
    inp = synth.make_inputs(w)
    proj = dlp.Projection(M, N, K, layout, dlp.PROJ_BF16)
    p = proj.plan
    nbytes = dlp.proj_packed_weight_bytes(proj.handle)
    kblk = p["k_blocks"] * (p["block_k"] // 64)  # 64-wide k-blocks per weight tile, whole stages
    assert nbytes == p["tiles_n"] * kblk * p["block_n"] * 128
    W = gu.to_dev(inp["W"])
    # Pre-fill the destination so that unwritten or non-zero padding shows.
    P = torch.full((nbytes // 2,), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    dlp.proj_pack_weights(proj.handle, W, P, torch.cuda.current_stream())
    torch.cuda.synchronize()
    got = P.view(torch.int16).cpu().numpy().view(np.uint16)
    want = expected_packed(inp["W"], layout, N, K, p["block_n"], kblk, p["tiles_n"])
    assert np.array_equal(got, want)


def test_packed_graph_replay_follows_fresh_inputs():
    import torch
    import dense_linear_projection_gb300 as dlp
    w = synth.Workload("t", 16, 8192, 8192, synth.W_NK, True, "bf16", 83)
    inp = synth.make_inputs(w)
    proj, Y, (X, W, b) = gu.run(w, inp)
    P = proj.pack(W)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        proj(X, P, b, out=Y, stream=s, packed=True)
    for seed in (84, 85):
        x = synth.normal_bf16(seed, synth.STREAM_X, w.M * w.K, 1.0).reshape(w.M, w.K)
        X.copy_(gu.to_dev(x))
        Y.zero_()
        g.replay()
        torch.cuda.synchronize()
        gu.assert_within_tol(gu.y_to_f64(Y), oracle.project(x, inp["W"], w.w_layout, inp["bias"]),
                             f"packed replay seed {seed}")
    assert proj.status() == dlp.PROJ_OK


def test_packed_bad_arguments():
    import torch
    import dense_linear_projection_gb300 as dlp
    L = dlp.lib()
    proj = dlp.Projection(16, 256, 512, dlp.PROJ_W_NK, dlp.PROJ_BF16)
    W = torch.zeros((256, 512), dtype=torch.bfloat16, device="cuda")
    P = proj.pack(W)
    s = torch.cuda.current_stream().cuda_stream
    assert L.proj_pack_weights(None, W.data_ptr(), P.data_ptr(), s) == dlp.PROJ_ERR_INVALID_ARG
    assert L.proj_pack_weights(proj.handle, None, P.data_ptr(), s) == dlp.PROJ_ERR_INVALID_ARG
    assert L.proj_pack_weights(proj.handle, W.data_ptr() + 2, P.data_ptr(), s) == dlp.PROJ_ERR_MISALIGNED
    X = torch.zeros((16, 512), dtype=torch.bfloat16, device="cuda")
    Y = torch.empty((16, 256), dtype=torch.bfloat16, device="cuda")
    assert L.proj_run_packed(proj.handle, X.data_ptr(), P.data_ptr() + 2, None, Y.data_ptr(),
                             s) == dlp.PROJ_ERR_MISALIGNED
    assert L.proj_packed_weight_bytes(None, None) == dlp.PROJ_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK


def test_packed_host_run_matches_device_run():
    import torch
    import dense_linear_projection_gb300 as dlp
    w = synth.Workload("t", 16, 1024, 2048, synth.W_NK, True, "bf16", 86)
    inp = synth.make_inputs(w)
    proj, Y, (X, W, b) = gu.run(w, inp)
    P = proj.pack(W)
    Xh = torch.from_numpy(inp["X"].view(np.int16)).view(torch.bfloat16).pin_memory()
    Yh = torch.empty((w.M, w.N), dtype=torch.bfloat16).pin_memory()
    s = torch.cuda.current_stream()
    dlp.proj_run_host_packed(proj.handle, Xh, P, b, Yh, s)
    s.synchronize()
    assert torch.equal(Yh.view(torch.int16), Y.cpu().view(torch.int16))
