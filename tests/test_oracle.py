"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Worked examples printed on "How I made Muse's GPU projections 1.32× faster in
the Open Kernel Challenge" (fixtures in tests/golden/, each citing its section),
closed forms, exact integer brute force, invariants (linearity, the swapped
product, layout equivalence) and an fp64 BLAS cross-check.  Each is chosen so a
plausible oracle mistake fails at least one: a dropped or doubled k term, a
sign error, transposed operands or a mixed-up W layout, fp32 accumulation, a
bias added twice or not at all.
"""
import itertools

import numpy as np
import pytest

import golden_io
import oracle
import synth

rng = np.random.default_rng(12345)


def bits(a):
    """bf16 bit patterns of values that bf16 holds exactly (small integers here)."""
    a = np.asarray(a, dtype=np.float64)
    b = synth.to_bf16_bits(a)
    back = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(back, a), "fixture value not exactly representable in bf16"
    return b


def as_storage(Wnk, layout):
    return Wnk if layout == oracle.W_NK else np.ascontiguousarray(Wnk.T)


# ---------------------------------------------------------------- worked examples
@pytest.mark.parametrize("name", golden_io.names())
def test_worked_examples(name):
    g = golden_io.load(name)
    b = bits(g["bias"]) if "bias" in g else None
    Y = oracle.project(bits(g["X"]), bits(g["W"]), g["layout"], b)
    assert np.array_equal(Y, g["Y"]), (name, Y, g["Y"])


def test_split_sum_partials():
    # 70 = 17 + 53: each half of K, then the whole (section "A reduction, worked
    # out with small numbers").  Every k term is used exactly once.
    g = golden_io.load("split_sum.txt")
    X, W = bits(g["X"]), bits(g["W"])
    p0 = oracle.project(X[:, :2], W[:, :2])[0, 0]
    p1 = oracle.project(X[:, 2:], W[:, 2:])[0, 0]
    assert [p0, p1] == list(g["partials"])
    assert p0 + p1 == oracle.project(X, W)[0, 0] == g["Y"][0, 0]


def test_rounding_order_needs_fp64():
    # Section "Algebraic rearrangements can change rounding": an fp32 running
    # sum loses the 1; the oracle must not.
    g = golden_io.load("rounding_order.txt")
    Y = oracle.project(bits(g["X"]), bits(g["W"]))
    assert Y[0, 0] == 1.0
    acc = np.float32(0)
    for x, w in zip(g["X"][0], g["W"][0]):
        acc = np.float32(acc + np.float32(x) * np.float32(w))
    assert float(acc) == float(g["extra"]["fp32_left_to_right"][0][0]) == 0.0


# ---------------------------------------------------------------- bf16 decoding
def test_bf16_decode_fixture():
    g = golden_io.load("bf16_values.txt")
    for hexbits, val in g["extra"]["decode"]:
        got = oracle.bf16_to_double(np.array([int(hexbits, 16)], dtype=np.uint16))[0]
        assert got == float(val), (hexbits, got, val)


def test_bf16_decode_specials():
    d = oracle.bf16_to_double(np.array([0x7F80, 0xFF80, 0x7FC0, 0x8000, 0x0001, 0x7F7F],
                                       dtype=np.uint16))
    assert d[0] == np.inf and d[1] == -np.inf and np.isnan(d[2])
    assert d[3] == 0.0 and np.signbit(d[3])
    assert d[4] == 2.0 ** -133                     # smallest subnormal
    assert d[5] == (2 - 2.0 ** -7) * 2.0 ** 127    # largest finite


def test_bf16_decode_all_patterns_against_fp32_view():
    # Every finite pattern: the oracle's decoder agrees with numpy's fp32 view.
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = (allb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    sample = allb[::97]
    got = oracle.bf16_to_double(sample)
    r = ref[::97]
    ok = np.isnan(r) & np.isnan(got) | (got == r)
    assert ok.all()


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("layout", [oracle.W_NK, oracle.W_KN])
def test_zero_input_gives_bias(layout):
    M, N, K = 3, 5, 7
    Wnk = rng.integers(-4, 5, size=(N, K))
    bias = rng.integers(-4, 5, size=N)
    Y = oracle.project(bits(np.zeros((M, K))), bits(as_storage(Wnk, layout)), layout)
    assert np.array_equal(Y, np.zeros((M, N)))
    Yb = oracle.project(bits(np.zeros((M, K))), bits(as_storage(Wnk, layout)), layout,
                        bits(bias))
    assert np.array_equal(Yb, np.broadcast_to(bias, (M, N)))


@pytest.mark.parametrize("layout", [oracle.W_NK, oracle.W_KN])
def test_identity_weight_returns_input(layout):
    M, K = 4, 9
    X = rng.integers(-16, 17, size=(M, K))
    Y = oracle.project(bits(X), bits(np.eye(K)), layout)
    assert np.array_equal(Y, X)


@pytest.mark.parametrize("layout", [oracle.W_NK, oracle.W_KN])
def test_identity_input_returns_weight_transpose(layout):
    N, K = 6, 5
    Wnk = rng.integers(-16, 17, size=(N, K))
    Y = oracle.project(bits(np.eye(K)), bits(as_storage(Wnk, layout)), layout)
    assert np.array_equal(Y, Wnk.T)


def test_sparse_probe_isolates_a_column():
    # One power-of-two entry per row isolates a scaled column of Wᵀ (section
    # "What a useful correctness check has to catch").
    N, K = 11, 13
    Wnk = rng.integers(-64, 65, size=(N, K))
    X = np.zeros((K, K))
    for j in range(K):
        X[j, j] = 2.0 ** (j % 5 - 2)
    Y = oracle.project(bits(X), bits(Wnk))
    for j in range(K):
        assert np.array_equal(Y[j], X[j, j] * Wnk[:, j])


# ---------------------------------------------------------------- brute force
def exact_projection(X, Wnk, bias):
    """Exact integer arithmetic in Python ints: an independent statement."""
    M, K = len(X), len(X[0])
    N = len(Wnk)
    out = []
    for m in range(M):
        row = []
        for n in range(N):
            s = sum(int(X[m][k]) * int(Wnk[n][k]) for k in range(K))
            row.append(s + (int(bias[n]) if bias is not None else 0))
        out.append(row)
    return np.array(out, dtype=np.float64)


@pytest.mark.parametrize("layout", [oracle.W_NK, oracle.W_KN])
def test_brute_force_tiny_shapes(layout):
    shapes = list(itertools.product(range(1, 10), repeat=3))
    for (M, N, K) in [shapes[i] for i in rng.choice(len(shapes), 60, replace=False)]:
        X = rng.integers(-8, 9, size=(M, K))
        Wnk = rng.integers(-8, 9, size=(N, K))
        bias = rng.integers(-8, 9, size=N) if rng.random() < 0.5 else None
        Y = oracle.project(bits(X), bits(as_storage(Wnk, layout)), layout,
                           None if bias is None else bits(bias))
        assert np.array_equal(Y, exact_projection(X, Wnk, bias)), (M, N, K, layout)


def test_long_k_integer_exact():
    # The real K = 8192: small integers keep every partial sum exact, so any
    # dropped, repeated or misindexed k term shows.
    M, N, K = 2, 3, 8192
    X = rng.integers(-3, 4, size=(M, K))
    Wnk = rng.integers(-3, 4, size=(N, K))
    Y = oracle.project(bits(X), bits(Wnk))
    assert np.array_equal(Y, exact_projection(X, Wnk, None))


# ---------------------------------------------------------------- invariants
def test_linearity_exact():
    # Y(a·X1 + X2) = a·Y(X1) + Y(X2) (section "What makes it linear?"), exact
    # with small integers and a power-of-two a.
    M, N, K = 5, 7, 33
    X1 = rng.integers(-8, 9, size=(M, K))
    X2 = rng.integers(-8, 9, size=(M, K))
    Wnk = rng.integers(-8, 9, size=(N, K))
    a = 4
    lhs = oracle.project(bits(a * X1 + X2), bits(Wnk))
    rhs = a * oracle.project(bits(X1), bits(Wnk)) + oracle.project(bits(X2), bits(Wnk))
    assert np.array_equal(lhs, rhs)


def test_swapped_product():
    # Yᵀ = W·Xᵀ (section "Prove the swapped product before worrying about its
    # speed"): exchanging the operands transposes the result term by term.
    M, N, K = 6, 10, 40
    X = synth.normal_bf16(7, 1, M * K, 1.0).reshape(M, K)
    W = synth.normal_bf16(7, 2, N * K, 0.1).reshape(N, K)
    Y = oracle.project(X, W)
    Yt = oracle.project(W, X)
    assert np.array_equal(Yt.T, Y)


def test_layouts_agree_on_random_values():
    M, N, K = 3, 17, 29
    X = synth.normal_bf16(8, 1, M * K, 1.0).reshape(M, K)
    W = synth.normal_bf16(8, 2, N * K, 0.2).reshape(N, K)
    b = synth.normal_bf16(8, 3, N, 0.02)
    assert np.array_equal(oracle.project(X, W, oracle.W_NK, b),
                          oracle.project(X, np.ascontiguousarray(W.T), oracle.W_KN, b))


def test_bias_added_once_after_the_sum():
    M, N, K = 4, 6, 12
    X = rng.integers(-8, 9, size=(M, K))
    Wnk = rng.integers(-8, 9, size=(N, K))
    bias = rng.integers(-8, 9, size=N)
    d = oracle.project(bits(X), bits(Wnk), 0, bits(bias)) - oracle.project(bits(X), bits(Wnk))
    assert np.array_equal(d, np.broadcast_to(bias, (M, N)))


def test_cells_match_full():
    M, N, K = 9, 31, 70
    X = synth.normal_bf16(9, 1, M * K, 1.0).reshape(M, K)
    W = synth.normal_bf16(9, 2, N * K, 0.1).reshape(K, N)
    b = synth.normal_bf16(9, 3, N, 0.02)
    full = oracle.project(X, W, oracle.W_KN, b)
    ms = rng.integers(0, M, size=50)
    ns = rng.integers(0, N, size=50)
    assert np.array_equal(oracle.project_cells(X, W, oracle.W_KN, b, ms, ns), full[ms, ns])


def test_random_values_against_blas_fp64():
    # An fp64 BLAS product of the decoded inputs agrees to fp64 rounding.
    M, N, K = 7, 33, 257
    X = synth.normal_bf16(10, 1, M * K, 1.0).reshape(M, K)
    W = synth.normal_bf16(10, 2, N * K, 1 / np.sqrt(K)).reshape(N, K)
    dec = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = dec(X) @ dec(W).T
    Y = oracle.project(X, W)
    scale = np.abs(dec(X)) @ np.abs(dec(W)).T
    assert np.all(np.abs(Y - ref) <= 1e-13 * scale)


def test_unit_variance_reading():
    # X ~ N(0,1), W ~ N(0, 1/K) (variance 1/K): each output is ~N(0,1), the
    # scale the elementwise tolerance 1e-3 + 5e-3·|r| is meant for.
    w = synth.workload("decode_bias")
    M, N, K = 16, 512, w.K
    X = synth.normal_bf16(w.seed, synth.STREAM_X, M * K, 1.0).reshape(M, K)
    W = synth.normal_bf16(w.seed, synth.STREAM_W, N * K, w.w_std).reshape(N, K)
    Y = oracle.project(X, W)
    assert abs(Y.std() - 1.0) < 0.05 and abs(Y.mean()) < 0.05


def test_rejects_bad_arguments():
    X = np.zeros((2, 3), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.project(X, np.zeros((4, 5), dtype=np.uint16))
    with pytest.raises(TypeError):
        oracle.project(X.astype(np.float32), np.zeros((4, 3), dtype=np.uint16))
    with pytest.raises(IndexError):
        oracle.project_cells(X, np.zeros((4, 3), dtype=np.uint16), 0, None, [2], [0])
