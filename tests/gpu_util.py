"""Helpers for the GPU parity tests: move bf16 bit patterns to the device, run
the projection through the C ABI, and compare against the fp64 oracle with the
elementwise rule |u - r| <= 1e-3 + 5e-3·|r|."""
import numpy as np

TOL_ABS, TOL_REL = 1e-3, 5e-3


def to_dev(bits: np.ndarray):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to("cuda").view(torch.bfloat16)


def y_to_f64(Y) -> np.ndarray:
    return Y.float().cpu().numpy().astype(np.float64)


def run(w, inp, stream=None):
    """Run workload ``w`` on inputs ``inp`` (uint16 arrays) and return Y (torch)."""
    import dense_linear_projection_gb300 as dlp
    proj = dlp.Projection(w.M, w.N, w.K, w.w_layout,
                          dlp.PROJ_F32 if w.y_dtype == "f32" else dlp.PROJ_BF16,
                          has_bias=w.has_bias)
    X, W = to_dev(inp["X"]), to_dev(inp["W"])
    b = to_dev(inp["bias"]) if w.has_bias else None
    Y = proj(X, W, b, stream=stream)
    return proj, Y, (X, W, b)


def assert_within_tol(u: np.ndarray, r: np.ndarray, what: str = ""):
    assert u.shape == r.shape, (u.shape, r.shape)
    assert np.isfinite(u).all(), f"{what}: non-finite output"
    err = np.abs(u - r)
    lim = TOL_ABS + TOL_REL * np.abs(r)
    bad = err > lim
    if bad.any():
        idx = np.argwhere(bad)
        i = tuple(idx[0])
        raise AssertionError(f"{what}: {len(idx)} of {u.size} elements out of tolerance; first "
                             f"at {i}: gpu {u[i]!r} oracle {r[i]!r} (|diff| {err[i]:.3e} > "
                             f"{lim[i]:.3e})")
    return float(err.max()) if err.size else 0.0


def sample_cells(M: int, N: int, count: int, seed: int = 0, tile_n: int = 128):
    """Random cells plus the corners and tile edges of the output."""
    rng = np.random.default_rng(seed)
    ms = list(rng.integers(0, M, size=count))
    ns = list(rng.integers(0, N, size=count))
    edge_m = sorted({0, M - 1, min(M - 1, 15), min(M - 1, 16), min(M - 1, 255), min(M - 1, 256)})
    edge_n = sorted({0, N - 1, min(N - 1, tile_n - 1), min(N - 1, tile_n), (N - 1) // 2})
    for m in edge_m:
        for n in edge_n:
            ms.append(m)
            ns.append(n)
    return np.array(ms, dtype=np.int64), np.array(ns, dtype=np.int64)
