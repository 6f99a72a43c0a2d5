"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small and mid-size problems are compared element by element on the whole
output; shapes span several tiles, ragged tails in M, N and K, the
data-parallel + split-K hybrid and both weight layouts.  Exact cases (small
integers, sparse probes, identity and zero) must match bit for bit.
"""
import numpy as np
import pytest

import gpu_util as gu
import oracle
import synth

pytestmark = pytest.mark.gpu

# (M, N, K, layout, bias, y_dtype): the planner's regimes and ragged edges.
SHAPES = [
    (1, 256, 64, synth.W_NK, False, "f32"),       # one k-block, two weight tiles
    (3, 130, 72, synth.W_NK, True, "bf16"),       # ragged N (130) and K (72 = 64 + 8)
    (16, 1000, 1024, synth.W_NK, True, "bf16"),   # decode-like, split-K, ragged N
    (17, 384, 2048, synth.W_NK, False, "f32"),    # M just past one 16-row MMA step
    (33, 520, 4104, synth.W_NK, True, "bf16"),    # ragged K block at the end
    (64, 1024, 8192, synth.W_NK, False, "f32"),   # the real K
    (100, 264, 520, synth.W_KN, True, "bf16"),    # [K,N] weights, ragged everything
    (256, 384, 1024, synth.W_KN, True, "bf16"),   # the largest single token tile
    (257, 300, 256, synth.W_NK, False, "bf16"),   # two token tiles, 1-row tail
    (512, 20480, 256, synth.W_NK, True, "bf16"),  # 320 tiles: two data-parallel waves + split-K
    (600, 1000, 1032, synth.W_KN, False, "f32"),  # [K,N] with several token tiles
    (200, 1024, 512, synth.W_NK, True, "bf16"),   # token tile halved to 64: many-way split
    (130, 3000, 2048, synth.W_KN, True, "f32"),   # [K,N], two-contributor split tiles
    (16, 28672, 1024, synth.W_NK, False, "bf16"), # 224 tiles, all split in pairs
]


@pytest.mark.parametrize("block_t", [16, 64, 128, 256])
def test_forced_token_tiles(block_t, monkeypatch):
    # The same problem under every token tile: data-parallel, pair and
    # many-way split paths all agree with the oracle.
    monkeypatch.setenv("PROJ_FORCE_BLOCK_T", str(block_t))
    w = _workload(256, 1536, 2048, synth.W_KN, True, "bf16", seed=21)
    inp = synth.make_inputs(w)
    proj, Y, _ = gu.run(w, inp)
    assert proj.plan["block_t"] == block_t
    r = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
    gu.assert_within_tol(gu.y_to_f64(Y), r, f"block_t={block_t}")


@pytest.mark.parametrize("layout,block_n", [(synth.W_NK, 64), (synth.W_NK, 80), (synth.W_NK, 176),
                                            (synth.W_NK, 256), (synth.W_KN, 64), (synth.W_KN, 192),
                                            (synth.W_KN, 256)])
def test_forced_weight_tiles(layout, block_n, monkeypatch):
    # Token rows on the MMA's M side with every kind of weight tile: widths
    # that are and are not multiples of 64, ragged last tiles, both layouts,
    # data-parallel and split plans.
    monkeypatch.setenv("PROJ_FORCE_BLOCK_N", str(block_n))
    w = _workload(300, 1000, 2056, layout, True, "bf16", seed=22)
    inp = synth.make_inputs(w)
    proj, Y, _ = gu.run(w, inp)
    assert proj.plan["swap_ab"] == 0 and proj.plan["block_n"] == block_n
    r = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
    gu.assert_within_tol(gu.y_to_f64(Y), r, f"block_n={block_n}")


@pytest.mark.parametrize("env", [{"PROJ_FORCE_BLOCK_N": "192", "PROJ_FORCE_STAGES": "3"},
                                 {"PROJ_FORCE_BLOCK_N": "176", "PROJ_FORCE_STAGES": "2"},
                                 {"PROJ_FORCE_BLOCK_T": "64", "PROJ_FORCE_STAGES": "2"}])
def test_forced_pipeline_depth(env, monkeypatch):
    # A shallower ring than planned, in both orientations: the launch's shared
    # memory must follow the B operand of the orientation in use.
    import dense_linear_projection_gb300 as dlp
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    layout = synth.W_KN if env.get("PROJ_FORCE_BLOCK_N") == "192" else synth.W_NK
    w = _workload(256, 1536, 8192, layout, True, "bf16", seed=23)  # planned depth 4-6
    inp = synth.make_inputs(w)
    proj, Y, _ = gu.run(w, inp)
    assert proj.plan["stages"] == int(env["PROJ_FORCE_STAGES"])
    import torch
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    r = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
    gu.assert_within_tol(gu.y_to_f64(Y), r, str(env))


def _workload(M, N, K, layout, bias, yd, seed=5):
    return synth.Workload("t", M, N, K, layout, bias, yd, seed)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "M{}_N{}_K{}_{}{}_{}".format(
    s[0], s[1], s[2], "KN" if s[3] else "NK", "_bias" if s[4] else "", s[5]))
def test_full_output_parity(shape):
    w = _workload(*shape)
    inp = synth.make_inputs(w)
    proj, Y, _ = gu.run(w, inp)
    import torch
    torch.cuda.synchronize()
    assert proj.status() == 0
    r = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
    gu.assert_within_tol(gu.y_to_f64(Y), r, str(shape))


def _int_inputs(M, N, K, layout, bias, lo=-4, hi=4, seed=3):
    rng = np.random.default_rng(seed)
    X = rng.integers(lo, hi + 1, size=(M, K)).astype(np.float64)
    Wnk = rng.integers(lo, hi + 1, size=(N, K)).astype(np.float64)
    Ws = Wnk if layout == synth.W_NK else np.ascontiguousarray(Wnk.T)
    b = rng.integers(lo, hi + 1, size=N).astype(np.float64) if bias else None
    bits = synth.to_bf16_bits
    return {"X": bits(X), "W": bits(Ws), "bias": None if b is None else bits(b)}


@pytest.mark.parametrize("M,N,K,layout,bias", [
    (1, 1, 8, synth.W_NK, False), (2, 3, 8, synth.W_NK, True), (9, 7, 16, synth.W_NK, False),
    (16, 300, 1024, synth.W_NK, True), (40, 136, 2048, synth.W_KN, True),
    (16, 2048, 8192, synth.W_NK, False),
])
def test_small_integers_bit_exact(M, N, K, layout, bias):
    # Small integers keep every fp32 partial and total exact, so the GPU result
    # (fp32 output) must equal the oracle exactly, split-K included.
    w = _workload(M, N, K, layout, bias, "f32")
    inp = _int_inputs(M, N, K, layout, bias)
    proj, Y, _ = gu.run(w, inp)
    r = oracle.project(inp["X"], inp["W"], layout, inp["bias"])
    assert np.array_equal(gu.y_to_f64(Y), r)


def test_sparse_probe_rows_bit_exact():
    # One power-of-two entry per row isolates a scaled weight column (section
    # "What a useful correctness check has to catch"): bit-exact in bf16.
    M, N, K = 16, 640, 4096
    w = _workload(M, N, K, synth.W_NK, False, "bf16")
    inp = synth.make_inputs(w)
    X = np.zeros((M, K))
    rng = np.random.default_rng(1)
    cols = rng.integers(0, K, size=M)
    for m in range(M):
        X[m, cols[m]] = 2.0 ** int(rng.integers(-3, 4))
    inp["X"] = synth.to_bf16_bits(X)
    proj, Y, _ = gu.run(w, inp)
    r = oracle.project(inp["X"], inp["W"], synth.W_NK, None)
    assert np.array_equal(gu.y_to_f64(Y), r)


@pytest.mark.parametrize("layout", [synth.W_NK, synth.W_KN])
def test_identity_weight_and_zero_input(layout):
    import torch
    M, K = 24, 256
    w = _workload(M, K, K, layout, True, "bf16")
    inp = synth.make_inputs(w)
    inp["W"] = synth.to_bf16_bits(np.eye(K))
    inp["bias"] = synth.to_bf16_bits(np.zeros(K))
    proj, Y, _ = gu.run(w, inp)
    assert np.array_equal(gu.y_to_f64(Y), oracle.bf16_to_double(inp["X"]))
    # Zero input: Y is the bias exactly.
    inp2 = synth.make_inputs(w)
    b = inp2["bias"]
    X0 = gu.to_dev(np.zeros((M, K), dtype=np.uint16))
    Y0 = proj(X0, gu.to_dev(inp2["W"]), gu.to_dev(b))
    torch.cuda.synchronize()
    assert np.array_equal(gu.y_to_f64(Y0), np.broadcast_to(oracle.bf16_to_double(b), (M, K)))


def test_repeat_runs_bit_identical():
    import torch
    w = synth.Workload("t", 16, 4096, 8192, synth.W_NK, True, "bf16", 1)
    inp = synth.make_inputs(w)
    proj, Y, (X, W, b) = gu.run(w, inp)
    outs = [Y.clone()]
    for _ in range(4):
        outs.append(proj(X, W, b).clone())
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


def test_graph_replay_follows_fresh_inputs():
    # A captured graph must not keep an old answer (section "Fresh graph replay
    # is a correctness test too"): [2,3] -> [5,8,5], then [3,1] -> [11,5,-3].
    import torch
    import dense_linear_projection_gb300 as dlp
    K = 64
    Wnk = np.zeros((3, K))
    Wnk[:, :2] = [[4, -1], [1, 2], [-2, 3]]
    x1 = np.zeros((1, K)); x1[0, :2] = [2, 3]
    x2 = np.zeros((1, K)); x2[0, :2] = [3, 1]
    proj = dlp.Projection(1, 3, K, dlp.PROJ_W_NK, dlp.PROJ_F32)
    X = gu.to_dev(synth.to_bf16_bits(x1))
    W = gu.to_dev(synth.to_bf16_bits(Wnk))
    Y = torch.empty((1, 3), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        proj(X, W, None, out=Y, stream=s)  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        proj(X, W, None, out=Y, stream=s)
    Y.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert Y.cpu().tolist() == [[5.0, 8.0, 5.0]]
    X.copy_(gu.to_dev(synth.to_bf16_bits(x2)))
    g.replay()
    torch.cuda.synchronize()
    assert Y.cpu().tolist() == [[11.0, 5.0, -3.0]]


def test_graph_replay_split_k_counters_reset():
    # Many replays of a split-K plan: counters must return to zero every time.
    import torch
    w = synth.Workload("t", 16, 1000, 4096, synth.W_NK, True, "bf16", 7)
    inp = synth.make_inputs(w)
    proj, Y, (X, W, b) = gu.run(w, inp)
    assert proj.plan["tiles_sk"] > 0
    torch.cuda.synchronize()
    ref = Y.clone()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(5):
            proj(X, W, b, out=Y, stream=s)
    for _ in range(20):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(Y.view(torch.int16), ref.view(torch.int16))
    assert proj.status() == 0


def test_two_handles_interleaved_on_one_stream():
    import torch
    wa = synth.Workload("a", 16, 2048, 8192, synth.W_NK, False, "f32", 11)
    wb = synth.Workload("b", 40, 520, 1024, synth.W_KN, True, "bf16", 12)
    ia, ib = synth.make_inputs(wa), synth.make_inputs(wb)
    pa, Ya, ta = gu.run(wa, ia)
    pb, Yb, tb = gu.run(wb, ib)
    for _ in range(3):
        pa(*ta, out=Ya)
        pb(*tb, out=Yb)
    torch.cuda.synchronize()
    gu.assert_within_tol(gu.y_to_f64(Ya), oracle.project(ia["X"], ia["W"], 0, None), "a")
    gu.assert_within_tol(gu.y_to_f64(Yb), oracle.project(ib["X"], ib["W"], 1, ib["bias"]), "b")


def test_run_host_matches_device_run():
    import torch
    import dense_linear_projection_gb300 as dlp
    w = synth.Workload("t", 16, 1024, 2048, synth.W_NK, True, "bf16", 13)
    inp = synth.make_inputs(w)
    proj, Y, (X, W, b) = gu.run(w, inp)
    Xh = torch.from_numpy(inp["X"].view(np.int16)).view(torch.bfloat16).pin_memory()
    Yh = torch.empty((w.M, w.N), dtype=torch.bfloat16).pin_memory()
    s = torch.cuda.current_stream()
    dlp.proj_run_host(proj.handle, Xh, W, b, Yh, s)
    s.synchronize()
    assert torch.equal(Yh.view(torch.int16), Y.cpu().view(torch.int16))


def test_empty_and_degenerate_shapes():
    import torch
    import dense_linear_projection_gb300 as dlp
    # M == 0 / N == 0: nothing to do, nothing launched.
    for M, N in [(0, 64), (4, 0)]:
        p = dlp.Projection(M, N, 64)
        assert p.plan["kernel"] == "none"
        p(torch.empty((M, 64), dtype=torch.bfloat16, device="cuda"),
          torch.empty((N, 64), dtype=torch.bfloat16, device="cuda"))
    # K == 0: empty sums, Y = bias (or 0).
    b = gu.to_dev(synth.normal_bf16(1, 3, 70, 0.5))
    p = dlp.Projection(5, 70, 0, has_bias=True)
    assert p.plan["kernel"] == "fill"
    Xe = torch.empty((5, 0), dtype=torch.bfloat16, device="cuda")
    We = torch.empty((70, 0), dtype=torch.bfloat16, device="cuda")
    Y = p(Xe, We, b)
    torch.cuda.synchronize()
    assert torch.equal(Y, b.unsqueeze(0).expand(5, 70))
    p0 = dlp.Projection(3, 9, 0, y_dtype=dlp.PROJ_F32)
    Y0 = p0(torch.empty((3, 0), dtype=torch.bfloat16, device="cuda"),
            torch.empty((9, 0), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert torch.count_nonzero(Y0).item() == 0


def test_boundary_rejects_bad_arguments():
    import torch
    import dense_linear_projection_gb300 as dlp
    with pytest.raises(dlp.ProjError) as e:
        dlp.Projection(4, 64, 12)                           # K % 8 != 0
    assert e.value.status == dlp.PROJ_ERR_MISALIGNED
    with pytest.raises(dlp.ProjError) as e:
        dlp.Projection(4, 60, 64, w_layout=dlp.PROJ_W_KN)   # [K,N] needs N % 8 == 0
    assert e.value.status == dlp.PROJ_ERR_MISALIGNED
    with pytest.raises(dlp.ProjError) as e:
        dlp.proj_create(4, 64, 64, x_dtype=dlp.PROJ_F32)
    assert e.value.status == dlp.PROJ_ERR_UNSUPPORTED
    with pytest.raises(dlp.ProjError) as e:
        dlp.proj_create(-1, 64, 64)
    assert e.value.status == dlp.PROJ_ERR_INVALID_ARG
    p = dlp.Projection(4, 64, 64, has_bias=True)
    X = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dlp.ProjError) as e:
        p(X, W, None)                                       # bias required
    assert e.value.status == dlp.PROJ_ERR_INVALID_ARG
    big = torch.zeros(4 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dlp.ProjError) as e:
        p(big[1:1 + 4 * 64].view(4, 64), W, b)              # X not 16-byte aligned
    assert e.value.status == dlp.PROJ_ERR_MISALIGNED
    with pytest.raises(dlp.ProjError) as e:
        dlp.proj_run(p.handle, X, W, b, None)
    assert e.value.status == dlp.PROJ_ERR_INVALID_ARG
    Y = p(X, W, b)                                          # still usable
    torch.cuda.synchronize()
    assert torch.count_nonzero(Y).item() == 0


def test_bounded_wait_gives_up_without_fault():
    # A device wait on a barrier nothing arrives on returns a status instead of
    # hanging; the context stays usable afterwards.
    import torch
    import dense_linear_projection_gb300 as dlp
    assert dlp.proj_selftest_wait_timeout(2_000_000) == dlp.PROJ_ERR_DEVICE_TIMEOUT
    w = synth.Workload("t", 16, 256, 512, synth.W_NK, True, "bf16", 2)
    inp = synth.make_inputs(w)
    proj, Y, _ = gu.run(w, inp)
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    gu.assert_within_tol(gu.y_to_f64(Y), oracle.project(inp["X"], inp["W"], 0, inp["bias"]))


@pytest.mark.parametrize("mode", [0, 1, 2], ids=["none", "prologue", "weights"])
def test_overlap_modes_see_inputs_written_just_before(mode):
    # Programmatic dependent launch: X written by the kernel right before each
    # run (inside one captured graph) must be the X the run uses, and
    # back-to-back split-K runs must not disturb each other's scratch.
    import torch
    import dense_linear_projection_gb300 as dlp
    w = synth.Workload("t", 16, 1000, 2048, synth.W_NK, True, "bf16", 31)
    inp = synth.make_inputs(w)
    X2 = synth.normal_bf16(32, synth.STREAM_X, w.M * w.K, 1.0).reshape(w.M, w.K)
    proj = dlp.Projection(w.M, w.N, w.K, w.w_layout, dlp.PROJ_BF16, True, overlap=mode)
    assert proj.plan["tiles_sk"] > 0
    Xs = [gu.to_dev(inp["X"]), gu.to_dev(X2)]
    W, b = gu.to_dev(inp["W"]), gu.to_dev(inp["bias"])
    X = torch.empty_like(Xs[0])
    Ys = [torch.empty((w.M, w.N), dtype=torch.bfloat16, device="cuda") for _ in range(6)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        X.copy_(Xs[0])
        proj(X, W, b, out=Ys[0], stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for i in range(6):
            X.mul_(0).add_(Xs[i % 2])  # kernels that write X just before the run
            proj(X, W, b, out=Ys[i], stream=s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    refs = [oracle.project(inp["X"], inp["W"], 0, inp["bias"]),
            oracle.project(X2, inp["W"], 0, inp["bias"])]
    for i in range(6):
        gu.assert_within_tol(gu.y_to_f64(Ys[i]), refs[i % 2], f"mode {mode} run {i}")
    assert torch.equal(Ys[0].view(torch.int16), Ys[2].view(torch.int16))


def test_handles_with_different_rings_in_any_creation_order():
    # Plans differ in shared memory; creating a second handle must not break
    # launches of the first, whichever of the two needs more.
    import torch
    ws = [synth.Workload("a", 16, 8192, 8192, synth.W_NK, False, "f32", 51),
          synth.Workload("b", 40, 520, 1024, synth.W_KN, True, "bf16", 52),
          synth.Workload("c", 4096, 1024, 512, synth.W_NK, False, "bf16", 53)]
    inps = [synth.make_inputs(w) for w in ws]
    for order in ([0, 1, 2], [2, 1, 0]):
        runs = {i: gu.run(ws[i], inps[i]) for i in order}
        assert len({runs[i][0].plan["smem_bytes"] for i in order}) > 1
        for i in order:
            proj, Y, t = runs[i]
            proj(*t, out=Y)
        torch.cuda.synchronize()
        for i in order:
            w, inp, (proj, Y, _) = ws[i], inps[i], runs[i]
            r = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
            gu.assert_within_tol(gu.y_to_f64(Y), r, w.name)


@pytest.mark.parametrize("M,N,K,yd", [(16, 1024, 2048, "bf16"), (5, 1001, 520, "f32"), (3, 999, 256, "bf16")])
def test_run_host_copy_paths(M, N, K, yd):
    # A pinned X goes through the copy kernel (chained to the projection by
    # programmatic dependent launch) and a pinned Y is written by the
    # projection's epilogue through its device address; pageable or
    # unaligned buffers go through cudaMemcpyAsync and the staging buffers.
    # Mixed cases take one route for X and the other for Y.  Odd N leaves a
    # Y tail that is not a whole 16-byte chunk.  Every path gives the device
    # run's bits.
    import torch
    import dense_linear_projection_gb300 as dlp
    w = synth.Workload("t", M, N, K, synth.W_NK, True, yd, 14)
    inp = synth.make_inputs(w)
    proj, Y, (X, W, b) = gu.run(w, inp)
    torch.cuda.synchronize()
    dt = torch.float32 if yd == "f32" else torch.bfloat16
    iv = torch.int32 if yd == "f32" else torch.int16
    xh = torch.from_numpy(inp["X"].view(np.int16)).view(torch.bfloat16)
    s = torch.cuda.current_stream()
    # Pinned X and Y; pageable X and Y; pinned but unaligned (offset by one element).
    Xp, Yp = xh.pin_memory(), torch.empty((M, N), dtype=dt).pin_memory()
    Xu_buf = torch.empty(M * K + 8, dtype=torch.bfloat16).pin_memory()
    Yu_buf = torch.empty(M * N + 8, dtype=dt).pin_memory()
    Xu, Yu = Xu_buf[1:1 + M * K].view(M, K), Yu_buf[1:1 + M * N].view(M, N)
    Xu.copy_(xh)
    cases = [("pinned", Xp, Yp), ("pageable", xh.clone(), torch.empty((M, N), dtype=dt)), ("unaligned", Xu, Yu),
             ("pinned Y only", xh.clone(), Yp), ("pinned X only", Xp, torch.empty((M, N), dtype=dt))]
    for name, Xh, Yh in cases:
        Yh.zero_()
        dlp.proj_run_host(proj.handle, Xh, W, b, Yh, s)
        s.synchronize()
        assert torch.equal(Yh.view(iv), Y.cpu().view(iv)), name
    assert proj.status() == dlp.PROJ_OK


def test_run_host_back_to_back_calls_keep_their_inputs():
    # Eight host-buffer calls in a row on one stream, with no synchronisation
    # between them: each call's X reaches the shared staging buffer only after
    # the previous projection has read its own, and each call's Y lands in
    # its own pinned buffer.
    import torch
    import dense_linear_projection_gb300 as dlp
    w = synth.Workload("t", 16, 2048, 4096, synth.W_NK, True, "bf16", 15)
    inp = synth.make_inputs(w)
    proj, _, (X, W, b) = gu.run(w, inp)
    xs = [inp["X"], synth.normal_bf16(16, synth.STREAM_X, w.M * w.K, 1.0).reshape(w.M, w.K)]
    Xh = [torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in xs]
    Yh = [torch.empty((w.M, w.N), dtype=torch.bfloat16).pin_memory() for _ in range(8)]
    s = torch.cuda.current_stream()
    for i in range(8):
        dlp.proj_run_host(proj.handle, Xh[i % 2], W, b, Yh[i], s)
    s.synchronize()
    refs = [oracle.project(x, inp["W"], w.w_layout, inp["bias"]) for x in xs]
    for i in range(8):
        gu.assert_within_tol(gu.y_to_f64(Yh[i]), refs[i % 2], f"call {i}")
    assert proj.status() == dlp.PROJ_OK
