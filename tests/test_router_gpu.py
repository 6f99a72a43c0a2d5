"""GPU parity of fp32 router weights through the high/low bf16 split.

"How I made Muse's GPU projections 1.32× faster in the Open Kernel
Challenge", section "Why the high-plus-low router scheme helped": H =
roundBF16(W), L = roundBF16(W − FP32(H)), Y = X·Hᵀ + X·Lᵀ in fp32.  The
output is compared with the exact fp32-weight product under the router contract
of section "The actual error rule, including what L2 means" (values in
tests/golden/router_hilo.txt): whole-output relative L2 within 0.01 %; each
row within five times that, with its denominator its own norm or one tenth of
the mean row norm if larger; sparse probe rows (one power of two in a row of
zeros) within 0.1 %.  It must also match the method itself (oracle
project_hilo) to fp32 accumulation, and the packed H/L blocks must equal the
oracle's split bit for bit.
"""
import numpy as np
import pytest

import golden_io
import gpu_util as gu
import oracle
import synth

pytestmark = pytest.mark.gpu


def _tolerances():
    g = golden_io.load("router_hilo.txt")
    return dict((k, float(v)) for k, v in g["extra"]["tolerance"])


def _inputs(M, N, K, layout, seed, bias):
    """Router inputs with sparse probe rows: about one row in eight (at least
    one when M >= 8) is zero except one feature holding a power of two."""
    w = synth.Workload("router", M, N, K, layout, bias, "f32", seed, w_dtype="f32")
    inp = synth.make_inputs(w)
    X = inp["X"].copy()
    rng = np.random.default_rng(seed)
    probes = sorted(set(rng.choice(M, size=max(1 if M >= 8 else 0, M // 8), replace=False).tolist())) if M else []
    for m in probes:
        X[m] = 0
        X[m, rng.integers(0, K)] = synth.to_bf16_bits(np.array([2.0 ** int(rng.integers(-3, 4))]))[0]
    inp["X"] = X
    return w, inp, probes


def _check_contract(u, r, probes, what):
    tol = _tolerances()
    assert np.isfinite(u).all(), f"{what}: non-finite output"
    e = u - r
    rel = np.linalg.norm(e) / max(np.linalg.norm(r), 1e-300)
    assert rel <= tol["rel_l2"], f"{what}: relative L2 {rel:.3e}"
    rn = np.linalg.norm(r, axis=1)
    den = np.maximum(rn, tol["row_floor_fraction"] * rn.mean())
    den = np.maximum(den, 1e-30)
    row = np.linalg.norm(e, axis=1) / den
    assert row.max() <= tol["row_factor"] * tol["rel_l2"], f"{what}: row error {row.max():.3e}"
    for m in probes:
        pe = np.linalg.norm(e[m]) / max(rn[m], 1e-30)
        assert pe <= tol["probe_rel"], f"{what}: probe row {m} error {pe:.3e}"
    return rel


@pytest.mark.parametrize("M,N,K,layout,bias", [
    (1, 256, 8192, synth.W_NK, False),
    (16, 256, 8192, synth.W_NK, False),    # the router workload
    (64, 256, 8192, synth.W_NK, True),
    (200, 256, 8192, synth.W_NK, False),   # token-major tiles
    (16, 300, 1032, synth.W_NK, False),    # ragged N and last K block
    (24, 256, 2048, synth.W_KN, True),     # fp32 weights stored [K,N]
], ids=lambda v: str(v))
def test_router_contract(M, N, K, layout, bias):
    import torch
    import dense_linear_projection_gb300 as dlp
    w, inp, probes = _inputs(M, N, K, layout, 91 + M, bias)
    proj = dlp.Projection(M, N, K, layout, dlp.PROJ_F32, has_bias=bias, w_dtype=dlp.PROJ_F32)
    X = gu.to_dev(inp["X"])
    W = torch.from_numpy(inp["W"]).cuda()
    b = gu.to_dev(inp["bias"]) if bias else None
    P = proj.pack(W)
    Y = proj(X, P, b, packed=True)
    again = proj(X, P, b, packed=True).clone()
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    u = gu.y_to_f64(Y)
    exact = oracle.project_f32w(inp["X"], inp["W"], layout, inp["bias"])
    _check_contract(u, exact, probes, f"router M={M} N={N} K={K}")
    method = oracle.project_hilo(inp["X"], inp["W"], layout, inp["bias"])
    rel_m = np.linalg.norm(u - method) / np.linalg.norm(method)
    assert rel_m <= 1e-5, f"vs the method: {rel_m:.3e}"
    assert torch.equal(again.view(torch.int32), Y.view(torch.int32))


@pytest.mark.parametrize("layout", [synth.W_NK, synth.W_KN])
def test_router_packed_blocks_are_the_split(layout):
    import torch
    import dense_linear_projection_gb300 as dlp
    M, N, K = 16, 300, 1032
    w, inp, _ = _inputs(M, N, K, layout, 97, False)
    proj = dlp.Projection(M, N, K, layout, dlp.PROJ_F32, w_dtype=dlp.PROJ_F32)
    p = proj.plan
    kt = -(-K // 64)
    assert p["k_blocks"] == 2 * kt
    P = proj.pack(torch.from_numpy(inp["W"]).cuda())
    torch.cuda.synchronize()
    got = P.view(torch.int16).cpu().numpy().view(np.uint16)
    H, L = oracle.split_hilo(inp["W"])
    if layout == synth.W_KN:
        H, L = np.ascontiguousarray(H.T), np.ascontiguousarray(L.T)
    tn, bn = p["tiles_n"], p["block_n"]

    def blocks(part):
        full = np.zeros((tn * bn, kt * 64), dtype=np.uint16)
        full[:N, :K] = part
        return full.reshape(tn, bn, kt, 64).transpose(0, 2, 1, 3)

    want = np.concatenate([blocks(H), blocks(L)], axis=1).reshape(-1)
    assert got.size == want.size and np.array_equal(got, want)


def test_router_handle_runs_only_packed():
    import torch
    import dense_linear_projection_gb300 as dlp
    proj = dlp.Projection(16, 256, 512, dlp.PROJ_W_NK, dlp.PROJ_F32, w_dtype=dlp.PROJ_F32)
    X = torch.zeros((16, 512), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((256, 512), dtype=torch.float32, device="cuda")
    Y = torch.empty((16, 256), dtype=torch.float32, device="cuda")
    st = dlp.lib().proj_run(proj.handle, X.data_ptr(), W.data_ptr(), None, Y.data_ptr(),
                            torch.cuda.current_stream().cuda_stream)
    assert st == dlp.PROJ_ERR_UNSUPPORTED
    assert proj.status() == dlp.PROJ_OK
