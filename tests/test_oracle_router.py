"""Pins of the oracle's fp32 router-weight functions: the high/low bf16 split
(f32_to_bf16, split_hilo) and the exact fp32-weight product (project_f32w).

Pinned against the page's worked example (tests/golden/router_hilo.txt),
closed-form bounds, the bf16 rounding pins shared with the decode fixture,
small-integer brute force and an independent numpy restatement of
round-to-nearest-even.
"""
import numpy as np

import golden_io
import oracle


def test_split_worked_example():
    g = golden_io.load("router_hilo.txt")
    (w, h, l), = g["extra"]["split"]
    H, L = oracle.split_hilo(np.array([float(w)], dtype=np.float32))
    assert H[0] == int(h, 16) and L[0] == int(l, 16)
    back = oracle.bf16_to_double(H) + oracle.bf16_to_double(L)
    assert back[0] == float(w)


def test_rounding_matches_decode_fixture():
    g = golden_io.load("bf16_values.txt")
    for value, bits in g["extra"]["round"]:
        assert oracle.f32_to_bf16(np.float32(float(value))) == int(bits, 16)


def _rne_numpy(x):
    """Independent restatement: the nearest bf16 neighbour of each fp32 value,
    ties to the even one, found by comparing distances in fp64."""
    x = np.asarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lo = (u >> 16) << 16                      # truncated toward zero
    hi = lo + (1 << 16)
    f = lambda b: b.astype(np.uint32).view(np.float32).astype(np.float64)
    d_lo = np.abs(x.astype(np.float64) - f(lo))
    d_hi = np.abs(f(hi) - x.astype(np.float64))
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (((lo >> 16) & 1) == 1))
    return np.where(pick_hi, hi >> 16, lo >> 16).astype(np.uint16)


def test_rounding_matches_independent_restatement():
    rng = np.random.default_rng(5)
    vals = np.concatenate([rng.standard_normal(20000).astype(np.float32),
                           (rng.standard_normal(5000) * 1e-20).astype(np.float32),
                           (rng.standard_normal(5000) * 1e20).astype(np.float32),
                           np.array([1.00390625, 1.01171875, -1.00390625, 0.0, -0.0, 3.0],
                                    dtype=np.float32)])
    assert np.array_equal(oracle.f32_to_bf16(vals), _rne_numpy(vals))


def test_split_error_bound():
    # H holds 8 significant bits of W, so |R| <= 2^-8·|W|; R = W − H is exact
    # in fp32; L holds 8 bits of R, so |W − (H + L)| = |R − L| <= 2^-8·|R|
    # <= 2^-16·|W| (normal values).
    rng = np.random.default_rng(6)
    W = (rng.standard_normal(50000) / np.sqrt(8192)).astype(np.float32)
    H, L = oracle.split_hilo(W)
    h, l = oracle.bf16_to_double(H), oracle.bf16_to_double(L)
    w = W.astype(np.float64)
    assert np.all(np.abs(w - h) <= 2.0 ** -8 * np.abs(w))
    assert np.all(np.abs(w - (h + l)) <= 2.0 ** -16 * np.abs(w))
    # The high part alone is the plain bf16 rounding; the low part is not zero
    # in general (it carries the next 8 bits).
    assert np.array_equal(H, _rne_numpy(W))
    assert np.count_nonzero(L) > 0.9 * L.size


def test_split_exact_for_two_bf16_terms():
    # Values that are a bf16 value plus a small bf16 value below its half-ulp
    # come back exactly: e.g. 1 + 2^-9, 3 − 2^-12, -0.75 + 2^-14.
    W = np.array([1 + 2 ** -9, 3 - 2 ** -12, -0.75 + 2 ** -14, 2 ** -20 + 2 ** -30],
                 dtype=np.float32)
    H, L = oracle.split_hilo(W)
    assert np.array_equal(oracle.bf16_to_double(H) + oracle.bf16_to_double(L),
                          W.astype(np.float64))


def test_project_f32w_small_integers_brute_force():
    rng = np.random.default_rng(7)
    for (M, N, K) in [(1, 1, 1), (2, 3, 5), (4, 7, 9), (3, 5, 64)]:
        X = rng.integers(-4, 5, size=(M, K)).astype(np.float64)
        W = rng.integers(-6, 7, size=(N, K)).astype(np.float32) * np.float32(0.25)
        b = rng.integers(-3, 4, size=N).astype(np.float64)
        xb = oracle.f32_to_bf16(X.astype(np.float32))
        bb = oracle.f32_to_bf16(b.astype(np.float32))
        want = X @ W.astype(np.float64).T + b
        assert np.array_equal(oracle.project_f32w(xb, W, 0, bb), want)
        assert np.array_equal(oracle.project_f32w(xb, np.ascontiguousarray(W.T), 1, bb), want)


def test_project_f32w_keeps_fp32_detail():
    # A weight that bf16 cannot hold (1 + 2^-20) must reach the product intact:
    # 3·(1 + 2^-20) exactly, not 3.
    X = oracle.f32_to_bf16(np.array([[3.0]], dtype=np.float32))
    W = np.array([[1 + 2 ** -20]], dtype=np.float32)
    assert oracle.project_f32w(X, W)[0, 0] == 3 * (1 + 2 ** -20)


def test_method_error_within_closed_form_bound():
    # |X·(H+L)ᵀ − X·Wᵀ| <= Σ_k |x_k|·|w_k − h_k − l_k| <= 2^-16·Σ_k |x_k·w_k|.
    rng = np.random.default_rng(8)
    M, N, K = 5, 7, 512
    X = oracle.f32_to_bf16(rng.standard_normal((M, K)).astype(np.float32))
    W = (rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32)
    exact = oracle.project_f32w(X, W)
    approx = oracle.project_hilo(X, W)
    xd = oracle.bf16_to_double(X)
    bound = 2.0 ** -16 * (np.abs(xd) @ np.abs(W.astype(np.float64)).T)
    assert np.all(np.abs(approx - exact) <= bound + 1e-300)
    # And the method is far inside the router's 0.01 % relative L2 contract.
    g = golden_io.load("router_hilo.txt")
    tol = dict((k, float(v)) for k, v in g["extra"]["tolerance"])
    rel = np.linalg.norm(approx - exact) / np.linalg.norm(exact)
    assert rel < tol["rel_l2"] / 10
