"""GPU parity of cluster-split plans: each narrow swapped tile split along K
over the S CTAs of one thread-block cluster, partial sums added in shared
memory in rank (= K) order.

The planner's own choices (S = 2 .. 16 on 152 SMs; the handle lowers S where
the device cannot hold every cluster at once) and every cluster size forced on
a few tiles: K ranges that do not divide evenly by S, ragged N and K tails,
both weight layouts and two token tiles.  Each is compared with the fp64
oracle and must rerun bit for bit; the planner's cases must also agree with
the stream-K plan of the same problem (cluster splits off).
"""
import numpy as np
import pytest

import gpu_util as gu
import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _swapped_clusters_only(monkeypatch):
    # These cases are about the swapped cluster split; the token-major one
    # (which proj_create may prefer for at most 32 tokens) has its own tests.
    monkeypatch.setenv("PROJ_TM_CLUSTER", "0")

# (M, N, K, layout, bias, y_dtype, S the planner picks on 152 SMs)
CLUSTER_SHAPES = [
    (16, 2048, 8192, synth.W_NK, False, "f32", 9),   # 16 tiles x 9 (x 6 where 16 clusters of 9 do not fit)
    (9, 2500, 1032, synth.W_NK, True, "bf16", 7),    # 20 tiles x 7, ragged N, 17 k-blocks
    (16, 3304, 1032, synth.W_KN, True, "bf16", 5),   # [K,N] weights, 26 tiles x 5
    (16, 4000, 2056, synth.W_NK, True, "bf16", 4),   # 32 tiles x 4, ragged K block
    (12, 5300, 1032, synth.W_NK, False, "f32", 3),   # 42 tiles x 3
    (16, 6144, 8192, synth.W_NK, True, "bf16", 3),   # 48 tiles x 3 (x 2 where 48 clusters of 3 do not fit)
    (100, 1024, 8192, synth.W_NK, True, "bf16", 9),  # two 64-token tiles x 8 weight tiles
    (16, 1024, 8192, synth.W_NK, False, "bf16", 16), # 8 tiles x 16: the largest clusters
]


def _ids(s):
    return "M{}_N{}_K{}_{}_S{}".format(s[0], s[1], s[2], "KN" if s[3] else "NK", s[6])


@pytest.mark.parametrize("shape", CLUSTER_SHAPES, ids=_ids)
def test_cluster_split_parity(shape, monkeypatch):
    import torch
    import dense_linear_projection_gb300 as dlp
    M, N, K, layout, bias, yd, S = shape
    planned = dlp.proj_plan_compute(M, N, K, layout)
    assert planned["cluster_split"] == S
    w = synth.Workload("t", M, N, K, layout, bias, yd, seed=61)
    inp = synth.make_inputs(w)
    proj, Y, (X, W, b) = gu.run(w, inp)
    # The device may hold fewer clusters of this size at once; then the handle
    # uses a smaller split (or stream-K), which must be just as correct.
    assert 0 <= proj.plan["cluster_split"] <= S
    again = proj(X, W, b).clone()
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    r = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
    gu.assert_within_tol(gu.y_to_f64(Y), r, f"cluster S={proj.plan['cluster_split']}")
    assert torch.equal(again.view(torch.int16 if yd == "bf16" else torch.int32),
                       Y.view(torch.int16 if yd == "bf16" else torch.int32))
    # The same problem without cluster splits (stream-K through global scratch).
    monkeypatch.setenv("PROJ_MAX_CLUSTER", "0")
    proj_sk, Y_sk, _ = gu.run(w, inp)
    assert proj_sk.plan["cluster_split"] == 0
    torch.cuda.synchronize()
    gu.assert_within_tol(gu.y_to_f64(Y_sk), r, "stream-K")


@pytest.mark.parametrize("S,M,N,K,layout,bias,yd", [
    (S, *shape) for S in (2, 3, 4, 5, 6, 7, 8, 9, 12, 16) for shape in (
        (16, 512, 1032, synth.W_NK, True, "bf16"),   # 4 tiles, 17 k-blocks
        (100, 264, 520, synth.W_KN, True, "f32"),    # 2 token x 3 weight tiles, 9 k-blocks, ragged
    ) if S <= -(-shape[2] // 64)
], ids=lambda v: str(v))
@pytest.mark.parametrize("half", ["0", "2"], ids=["full_tiles", "half_tiles"])
def test_every_cluster_size(S, M, N, K, layout, bias, yd, half, monkeypatch):
    # Full tiles take exactly S; half tiles (64 weight rows, twice the
    # clusters) take S or, where that many clusters of S do not fit at once,
    # a smaller split.
    import torch
    import dense_linear_projection_gb300 as dlp
    monkeypatch.setenv("PROJ_MAX_CLUSTER", str(S))
    monkeypatch.setenv("PROJ_CLUSTER_FILL_PCT", "1")  # a few tiles: any fill will do
    monkeypatch.setenv("PROJ_HALF_TILES", half)
    w = synth.Workload("t", M, N, K, layout, bias, yd, seed=70 + S)
    inp = synth.make_inputs(w)
    proj, Y, (X, W, b) = gu.run(w, inp)
    if half == "0":
        assert proj.plan["cluster_split"] == S and proj.plan["block_n"] == 128
    else:
        assert 2 <= proj.plan["cluster_split"] <= S and proj.plan["block_n"] == 64
    again = proj(X, W, b).clone()
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    r = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
    gu.assert_within_tol(gu.y_to_f64(Y), r, f"forced S={S}")
    iv = torch.int16 if yd == "bf16" else torch.int32
    assert torch.equal(again.view(iv), Y.view(iv))


@pytest.mark.parametrize("S,G,M,N,K,layout,bias,yd", [
    (4, 2, 16, 2048, 8192, synth.W_NK, False, "f32"),   # 16 tiles x 2 clusters of 4 (128 CTAs)
    (3, 3, 16, 2048, 8192, synth.W_NK, True, "bf16"),   # 16 tiles x 3 clusters of 3 (144 CTAs)
    (2, 3, 9, 2500, 1032, synth.W_NK, True, "bf16"),    # ragged N, 17 k-blocks in 6 parts
    (2, 2, 16, 3304, 1032, synth.W_KN, True, "f32"),    # [K,N] weights, 26 tiles
    (4, 2, 100, 1024, 8192, synth.W_NK, True, "bf16"),  # two 64-token tiles
], ids=lambda v: str(v))
def test_cluster_groups_parity(S, G, M, N, K, layout, bias, yd, monkeypatch):
    # Each tile's K range over G clusters of S CTAs: every cluster adds its
    # ranks in shared memory, the G cluster sums meet in the scratch, and the
    # cluster that completes last adds them in group order.  Oracle parity
    # and bit-identical reruns (the arrival order of the clusters varies).
    import torch
    import dense_linear_projection_gb300 as dlp
    monkeypatch.setenv("PROJ_FORCE_CLUSTER", str(S))
    monkeypatch.setenv("PROJ_CLUSTER_GROUPS", str(G))
    w = synth.Workload("t", M, N, K, layout, bias, yd, seed=90 + S * G)
    inp = synth.make_inputs(w)
    proj, Y, (X, W, b) = gu.run(w, inp)
    pl = proj.plan
    # A device that cannot hold every cluster at once falls back to one per tile.
    assert pl["cluster_split"] == S and pl["cluster_groups"] in (1, G)
    if pl["cluster_groups"] == G:
        assert pl["grid"] == pl["tiles_sk"] * S * G
    iv = torch.int16 if yd == "bf16" else torch.int32
    runs = [proj(X, W, b).clone() for _ in range(3)]
    torch.cuda.synchronize()
    assert proj.status() == dlp.PROJ_OK
    r = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
    gu.assert_within_tol(gu.y_to_f64(Y), r, f"S={S} G={pl['cluster_groups']}")
    for again in runs:
        assert torch.equal(again.view(iv), Y.view(iv))


def test_cluster_groups_on_the_decode_shape():
    # The 2048-row decode weight in 2 clusters of 4 per tile fits GB300's
    # SMs at once (32 clusters), so the grouped plan is the one that runs.
    import os
    import torch
    import dense_linear_projection_gb300 as dlp
    os.environ["PROJ_FORCE_CLUSTER"], os.environ["PROJ_CLUSTER_GROUPS"] = "4", "2"
    try:
        proj = dlp.Projection(16, 2048, 8192, dlp.PROJ_W_NK, dlp.PROJ_F32)
    finally:
        del os.environ["PROJ_FORCE_CLUSTER"], os.environ["PROJ_CLUSTER_GROUPS"]
    assert (proj.plan["cluster_split"], proj.plan["cluster_groups"], proj.plan["grid"]) == (4, 2, 128)


def test_handle_keeps_only_clusters_that_fit():
    # The 8192-row decode projection (64 tiles) runs in 64 clusters of 2 (all
    # resident at once on GB300); the 28672-row FFN weight (224 tiles) runs
    # stream-K on every SM; the 2048-row one (16 tiles) keeps a cluster split
    # whose clusters all fit at once.  Whatever split size a handle ends
    # with, its clusters fit together.
    import torch
    import dense_linear_projection_gb300 as dlp
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    proj = dlp.Projection(16, 8192, 8192, dlp.PROJ_W_NK, dlp.PROJ_BF16, has_bias=True)
    assert proj.plan["cluster_split"] == 2 and proj.plan["grid"] == 128
    proj = dlp.Projection(16, 28672, 8192, dlp.PROJ_W_NK, dlp.PROJ_BF16)
    assert proj.plan["cluster_split"] == 0 and proj.plan["grid"] == sms
    p = dlp.Projection(16, 2048, 8192, dlp.PROJ_W_NK, dlp.PROJ_F32).plan
    assert p["cluster_split"] >= 2 and p["grid"] == 16 * p["cluster_split"]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for N in (2048, 2500, 3304, 4000, 5300):
        p = dlp.Projection(16, N, 8192, dlp.PROJ_W_NK, dlp.PROJ_BF16).plan
        assert p["grid"] <= sms
        if p["cluster_split"]:
            assert p["grid"] == p["tiles_sk"] * p["cluster_split"]


def test_cluster_split_small_integers_bit_exact():
    # Integer operands keep every partial sum exact, whatever the split.
    import torch
    import dense_linear_projection_gb300 as dlp
    M, N, K = 16, 4000, 2056
    rng = np.random.default_rng(8)
    X = rng.integers(-4, 5, size=(M, K)).astype(np.float64)
    Wnk = rng.integers(-4, 5, size=(N, K)).astype(np.float64)
    proj = dlp.Projection(M, N, K, dlp.PROJ_W_NK, dlp.PROJ_F32)
    assert proj.plan["cluster_split"] >= 2
    Y = proj(gu.to_dev(synth.to_bf16_bits(X)), gu.to_dev(synth.to_bf16_bits(Wnk)), None)
    torch.cuda.synchronize()
    assert np.array_equal(gu.y_to_f64(Y), X @ Wnk.T)


def test_cluster_split_graph_replay_follows_fresh_inputs():
    # Replays of a captured cluster launch: each replay reads the X it is given.
    import torch
    import dense_linear_projection_gb300 as dlp
    w = synth.Workload("t", 16, 2048, 8192, synth.W_NK, True, "bf16", 62)
    inp = synth.make_inputs(w)
    proj, Y, (X, W, b) = gu.run(w, inp)
    assert proj.plan["cluster_split"] >= 2
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        proj(X, W, b, out=Y, stream=s)
    for seed in (63, 64):
        x = synth.normal_bf16(seed, synth.STREAM_X, w.M * w.K, 1.0).reshape(w.M, w.K)
        X.copy_(gu.to_dev(x))
        Y.zero_()
        g.replay()
        torch.cuda.synchronize()
        gu.assert_within_tol(gu.y_to_f64(Y), oracle.project(x, inp["W"], w.w_layout, inp["bias"]),
                             f"replay seed {seed}")
    assert proj.status() == dlp.PROJ_OK
