"""Pins of the oracle's fused-epilogue functions: GELU and act(X·Wᵀ + b) + R.

GELU is taken from its definition x·Φ(x) (the pages fuse "GELU" into the FFN
projection's epilogue without writing it out).  It is pinned against the
standard normal CDF of an independent library routine (scipy.special.ndtr),
against the Maclaurin series of erf summed here term by term, the identity
GELU(x) − GELU(−x) = x (from Φ(x) + Φ(−x) = 1), and its limits.  SiLU is
pinned against scipy's logistic function and against the tanh form of the
logistic, σ(x) = (1 + tanh(x/2)) / 2.  scipy is required: a missing scipy
fails these tests rather than skipping them.
"""
import math

import numpy as np
import scipy.special as scipy_special

import oracle
import synth


def erf_series(z: float) -> float:
    """erf(z) = 2/√π · Σ (−1)^n z^(2n+1) / (n! (2n+1)), summed until the terms
    vanish (|z| ≤ 3 keeps the cancellation below 1e-13)."""
    t, total, n = z, z, 0
    while True:
        n += 1
        t *= -z * z / n
        term = t / (2 * n + 1)
        total += term
        if abs(term) < 1e-18:
            return 2.0 / math.sqrt(math.pi) * total


def test_gelu_against_the_erf_series():
    # For x < 0, 1 + erf(x/√2) cancels: about 1e-14 absolute error at most
    # over this range, hence the absolute tolerance.
    xs = np.linspace(-4.0, 4.0, 161)
    want = np.array([0.5 * x * (1.0 + erf_series(x / math.sqrt(2.0))) for x in xs])
    assert np.allclose(oracle.gelu(xs), want, rtol=1e-12, atol=1e-13)
    # The series itself against two printed values: erf(1) = 0.8427007929497149,
    # erf(0.5) = 0.5204998778130465.
    assert abs(erf_series(1.0) - 0.8427007929497149) < 1e-15
    assert abs(erf_series(0.5) - 0.5204998778130465) < 1e-15


def test_silu_against_the_tanh_form():
    # 1 + tanh(x/2) cancels for x << 0: the range stops at −8, where the
    # relative error of the tanh form stays near 1e-13.
    xs = np.linspace(-8.0, 30.0, 381)
    want = np.array([x * 0.5 * (1.0 + math.tanh(x / 2.0)) for x in xs])
    assert np.allclose(oracle.silu(xs), want, rtol=1e-11, atol=1e-15)


def test_gelu_definition_against_normal_cdf():
    rng = np.random.default_rng(21)
    x = np.concatenate([rng.standard_normal(2000) * 3.0, [0.0, 1.0, -1.0, np.sqrt(2.0), 0.5]])
    want = x * scipy_special.ndtr(x)
    got = oracle.gelu(x)
    assert np.allclose(got, want, rtol=1e-13, atol=1e-15)
    assert oracle.gelu([0.0])[0] == 0.0


def test_gelu_odd_part_identity_and_limits():
    x = np.linspace(-6.0, 6.0, 1201)
    g_pos, g_neg = oracle.gelu(x), oracle.gelu(-x)
    assert np.allclose(g_pos - g_neg, x, rtol=0, atol=1e-14)
    assert abs(oracle.gelu([12.0])[0] - 12.0) < 1e-12
    assert abs(oracle.gelu([-12.0])[0]) < 1e-12
    # Monotone on [−0.75, ∞) (its minimum is near x = −0.7518).
    g = oracle.gelu(np.linspace(-0.75, 6.0, 500))
    assert np.all(np.diff(g) > 0)


def _bits(a):
    return synth.to_bf16_bits(np.asarray(a, dtype=np.float64))


def test_fused_epilogue_order_and_residual():
    # W = 0: Y = act(bias) + residual, whatever X is.
    M, N, K = 3, 5, 8
    X = _bits(np.ones((M, K)))
    W = _bits(np.zeros((N, K)))
    b = _bits([-2.0, -1.0, 0.0, 1.0, 2.0])
    R = np.arange(M * N, dtype=np.float64).reshape(M, N) / 4.0
    bd = oracle.bf16_to_double(b)
    got = oracle.project_fused(X, W, oracle.W_NK, b, oracle.ACT_GELU, R)
    assert np.array_equal(got, oracle.gelu(np.broadcast_to(bd, (M, N))) + R)
    # The activation applies to the projection plus bias, before the residual:
    # X·Wᵀ = 2 in every cell, bias 0.5: GELU(2.5) + R.
    X2 = _bits(np.full((M, K), 0.25))
    Wn = _bits(np.ones((N, K)))
    got2 = oracle.project_fused(X2, Wn, oracle.W_NK, _bits(np.full(N, 0.5)), oracle.ACT_GELU, R)
    assert np.allclose(got2, 2.5 * scipy_special.ndtr(2.5) + R, rtol=1e-14, atol=0)
    # No activation, no residual: the plain projection.
    assert np.array_equal(oracle.project_fused(X2, Wn, oracle.W_NK, None),
                          oracle.project(X2, Wn, oracle.W_NK, None))


def test_silu_definition_against_logistic():
    rng = np.random.default_rng(22)
    x = np.concatenate([rng.standard_normal(2000) * 4.0, [0.0, 1.0, -1.0, 20.0, -20.0]])
    assert np.allclose(oracle.silu(x), x * scipy_special.expit(x), rtol=1e-13, atol=1e-300)
    # σ(x) + σ(−x) = 1, so SiLU(x) − SiLU(−x) = x.
    assert np.allclose(oracle.silu(x) - oracle.silu(-x), x, rtol=0, atol=1e-12)
    assert oracle.silu([0.0])[0] == 0.0


def test_swiglu_gates_the_up_projection():
    # W = [W_gate; W_up]: Y = SiLU(X·W_gateᵀ) · (X·W_upᵀ).
    rng = np.random.default_rng(23)
    M, F, K = 3, 5, 16
    Xf = rng.integers(-2, 3, size=(M, K)).astype(np.float64)
    Wg = rng.integers(-2, 3, size=(F, K)).astype(np.float64)
    Wu = rng.integers(-2, 3, size=(F, K)).astype(np.float64)
    X, W = _bits(Xf), _bits(np.vstack([Wg, Wu]))
    G, U = Xf @ Wg.T, Xf @ Wu.T
    want = G * scipy_special.expit(G) * U
    got = oracle.project_swiglu(X, W)
    assert np.allclose(got, want, rtol=1e-13, atol=1e-13)
    # The gate, not the up half, goes through the nonlinearity: swapping the
    # halves changes the result.
    assert not np.allclose(oracle.project_swiglu(X, _bits(np.vstack([Wu, Wg]))), want)
    # [K,2F] storage gives the same result; a residual is added last.
    R = np.arange(M * F, dtype=np.float64).reshape(M, F)
    assert np.allclose(oracle.project_swiglu(X, np.ascontiguousarray(W.T), oracle.W_KN, R),
                       want + R, rtol=1e-13, atol=1e-13)
    # A zero up projection gives zero; a zero gate gives zero (SiLU(0) = 0).
    assert not oracle.project_swiglu(X, _bits(np.vstack([Wg, 0 * Wu]))).any()
    assert not oracle.project_swiglu(X, _bits(np.vstack([0 * Wg, Wu]))).any()
