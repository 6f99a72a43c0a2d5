"""The C-ABI library on a machine without a GPU: it loads, exports what
include/proj.h declares, and its planner (pure host code, the same
decomposition code the kernel runs) cuts every problem correctly."""
import collections
import itertools
import os
import re

import numpy as np
import pytest

import dense_linear_projection_gb300 as dlp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "proj.h")
GB300 = dict(sm_count=152, smem_optin_bytes=232448)


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(proj_\w+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_function():
    names = header_functions()
    assert "proj_create" in names and "proj_run" in names and "proj_destroy" in names
    lib = dlp.lib()
    for name in names:
        assert hasattr(lib, name), f"{name} declared in proj.h but not exported"
    assert set(names) == set(dlp.EXPORTED_SYMBOLS)


def test_status_strings():
    for code, name in [(0, "PROJ_OK"), (1, "PROJ_ERR_INVALID_ARG"), (2, "PROJ_ERR_UNSUPPORTED"),
                       (3, "PROJ_ERR_MISALIGNED"), (4, "PROJ_ERR_OUT_OF_MEMORY"),
                       (5, "PROJ_ERR_CUDA"), (6, "PROJ_ERR_DEVICE_TIMEOUT")]:
        assert dlp.proj_status_string(code) == name
    assert dlp.proj_status_string(99) == "PROJ_ERR_UNKNOWN"


def test_create_without_a_gpu_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(dlp.ProjError) as e:
        dlp.proj_create(16, 256, 256)
    assert e.value.status in (dlp.PROJ_ERR_CUDA, dlp.PROJ_ERR_UNSUPPORTED)


def test_null_handle_calls_are_rejected():
    assert dlp.lib().proj_run(None, None, None, None, None, None) == dlp.PROJ_ERR_INVALID_ARG
    assert dlp.lib().proj_destroy(None) == dlp.PROJ_OK
    assert dlp.proj_device_status(None) == dlp.PROJ_ERR_INVALID_ARG
    assert dlp.lib().proj_set_trace(None, None, 0) == dlp.PROJ_ERR_INVALID_ARG


# ---------------------------------------------------------------- planner
def plan(M, N, K, layout=0, **dev):
    return dlp.proj_plan_compute(M, N, K, layout, **(dev or GB300))


def check_decomposition(p, M, N, K, sms=GB300["sm_count"]):
    G, KT = p["grid"], p["k_blocks"]
    tiles = p["tiles_m"] * p["tiles_n"]
    assert p["tiles_m"] == -(-M // p["block_t"]) and p["tiles_n"] == -(-N // p["block_n"])
    pair = p["cta_pair"]
    if pair:
        # CTA pairs: 256 rows on the MMA's M side (two CTAs of 128), the N
        # side in [64, 256] split in halves, a multiple of 32 (swapped) or 16
        # (token-major); whole tiles dealt to pairs, two CTAs each.
        a, b = ("block_n", "block_t") if p["swap_ab"] else ("block_t", "block_n")
        assert p[a] == 256 and p[b] % (32 if p["swap_ab"] else 16) == 0 and 64 <= p[b] <= 256
        assert p["cluster_split"] == 0 and p["tiles_sk"] == 0 and p["scratch_bytes"] == 256
        assert G % 2 == 0 and G == 2 * min(tiles, sms // 2)
    elif p["swap_ab"]:
        assert p["block_n"] == 128 and p["block_t"] % 16 == 0
    else:
        assert p["block_t"] == 128 and p["block_n"] % 16 == 0 and 64 <= p["block_n"] <= 256
    # Two 64-wide k-blocks a stage for the weight-streaming swapped plans (at
    # most 64 tokens) and for CTA pairs, K a multiple of 64; one otherwise.
    kpb = 2 if (K % 64 == 0 and (pair or (p["swap_ab"] and p["block_t"] <= 64))) else 1
    assert p["block_k"] == 64 * kpb
    assert KT == -(-K // p["block_k"])
    assert 1 <= G <= GB300["sm_count"]
    assert p["tiles_dp"] + p["tiles_sk"] == tiles
    S = p["cluster_split"]
    if S:
        # Cluster split: every tile its own cluster of S CTAs (S <= 16), at
        # least 10 % of the SMs busy, fewer than a third as many tiles as SMs,
        # narrow swapped tiles, partials in shared memory.
        assert 2 <= S <= 16 and S <= KT and p["swap_ab"] == 1 and p["block_t"] <= 64
        # Two k-blocks a stage: S = SMs / tiles >= 2; one: fewer than a third
        # as many tiles as SMs.
        assert p["tiles_dp"] == 0 and G == tiles * S and 10 * G >= sms
        assert (2 * tiles <= sms) if kpb == 2 else (3 * tiles < sms)
        assert p["scratch_bytes"] == 256
    if p["tiles_sk"]:
        assert p["tiles_dp"] % G == 0
    elif not pair:  # whole tiles only: the last wave is nearly full (95 % swapped, 80 % token-major)
        waves = -(-tiles // G)
        pct = 95 if p["swap_ab"] else 80
        assert tiles % G == 0 or 100 * tiles >= pct * waves * G
    assert p["units_sk"] == p["tiles_sk"] * KT
    assert p["smem_bytes"] <= GB300["smem_optin_bytes"] and p["stages"] >= 2
    assert p["block_t"] % 16 == 0 and 16 <= p["block_t"] <= 256
    b_rows = p["block_t"] if p["swap_ab"] else p["block_n"]
    if pair:
        # Two accumulator buffers (at most 512 columns a pair allocates per SM).
        assert p["tmem_cols"] <= 512 and p["tmem_cols"] >= 2 * b_rows
    else:
        assert p["tmem_cols"] >= 2 * b_rows
    # The launch's shared memory covers the ring (A 128 rows + B rows, 64 K each),
    # its barriers, the epilogue's bias and output staging, 1024-byte alignment slack,
    # and in a cluster split the peers' partial sums: S - 1 partials of 32 rows
    # for each quarter the CTA reduces (quarter q goes to rank q mod S, S <= 4,
    # or to rank q).
    red = 0
    if S:
        quarters = -(-4 // S) if S <= 4 else 1
        red = quarters * (S - 1) * 32 * b_rows * 4
    # A CTA of a pair stages half of the B rows.
    assert p["smem_bytes"] == p["stages"] * kpb * (128 + (b_rows // 2 if pair else b_rows)) * 128 + red + 25600
    cover = np.zeros((tiles, KT), dtype=np.int32)
    by_tile = collections.defaultdict(list)
    coords = {}
    slots = set()
    for c in range(0, G, 2 if pair else 1):
        if pair:  # both CTAs of a pair run the pair's tiles
            assert dlp.proj_plan_segments(p, c) == dlp.proj_plan_segments(p, c + 1)
        for (tile, tm, tn, kb0, kb1, slot, split) in dlp.proj_plan_segments(p, c):
            assert 0 <= tm < p["tiles_m"] and 0 <= tn < p["tiles_n"] and 0 <= kb0 < kb1 <= KT
            assert coords.setdefault(tile, (tm, tn)) == (tm, tn)
            cover[tile, kb0:kb1] += 1
            by_tile[tile].append((c, slot, split, kb0, kb1))
            if split and S:
                r = c % S
                assert (tile, kb0, kb1, slot) == (c // S, r * KT // S, (r + 1) * KT // S, -1)
            elif split:
                assert 0 <= slot < 2 * G and slot not in slots
                slots.add(slot)
            else:
                assert (kb0, kb1) == (0, KT) and slot == -1
    assert (cover == 1).all(), "every (tile, k-block) exactly once"
    assert len(set(coords.values())) == tiles, "tile -> (token, weight) tile is one-to-one"
    share = p["units_sk"] // G if p["units_sk"] else 0
    for tile, segs in by_tile.items():
        split = len(segs) > 1
        assert all(bool(s[2]) == split for s in segs)
        if split:
            ts = tile - p["tiles_dp"]
            assert ts >= 0
            segs.sort(key=lambda s: s[3])  # K order
            order = dlp.proj_plan_reduction_order(p, ts)
            assert order == [(s[0], s[1]) for s in segs]
            assert [s[0] for s in segs] == sorted(s[0] for s in segs)
            if share >= KT:  # the two-contributor case the kernel's pair path assumes
                (c0, s0, _, a0, b0), (c1, s1, _, a1, b1) = segs
                assert c1 == c0 + 1 and a0 == 0 and b1 == KT and b0 == a1
                assert s0 == 2 * c0 + 1 and s1 == 2 * c1


CONFIG_SHAPES = [(16, 2048, 8192, 0), (16, 8192, 8192, 0), (16, 28672, 8192, 0),
                 (256, 12288, 4096, 1), (4096, 8192, 8192, 0)] + [
    (m, 28672, 8192, 0) for m in (1, 2, 4, 8, 32, 64)]


@pytest.mark.parametrize("M,N,K,layout", CONFIG_SHAPES)
def test_plans_of_the_workloads(M, N, K, layout):
    p = plan(M, N, K, layout)
    assert p["kernel"] == dlp.PROJ_KERNEL_TC
    check_decomposition(p, M, N, K)


def test_cluster_group_decomposition():
    # Several clusters per tile: the 16 tiles of the 2048-row decode weight
    # as 2 clusters of 4 each (128 CTAs).  CTA c takes part c % 8 of tile
    # c // 8, K split into 8 integer shares; every (tile, k-block) is covered
    # once; the reduction order lists the 8 parts in K order with their
    # cluster's scratch slot (tile·2 + part // 4).
    p = dict(plan(16, 2048, 8192))
    KT = p["k_blocks"]
    S, G = 4, 2
    p.update(cluster_split=S, cluster_groups=G, grid=16 * S * G)
    cover = np.zeros((16, KT), dtype=np.int32)
    for c in range(p["grid"]):
        segs = dlp.proj_plan_segments(p, c)
        assert len(segs) == 1
        tile, tm, tn, kb0, kb1, slot, split = segs[0]
        part = c % (S * G)
        assert (tile, kb0, kb1, slot, split) == (c // (S * G), part * KT // (S * G), (part + 1) * KT // (S * G), -1, 1)
        cover[tile, kb0:kb1] += 1
    assert (cover == 1).all()
    for ts in (0, 7, 15):
        assert dlp.proj_plan_reduction_order(p, ts) == [(ts * 8 + r, ts * 2 + r // 4) for r in range(8)]
    # G = 1 (and 0) keep the one-cluster-per-tile order.
    p.update(cluster_groups=1, grid=16 * S)
    assert dlp.proj_plan_reduction_order(p, 3) == [(3 * 4 + r, -1) for r in range(4)]
    assert plan(16, 2048, 8192)["cluster_groups"] == 1


def test_pair_stream_k_decomposition():
    # Stream-K over CTA pairs (option PROJ_PAIR_SK): the QKV shape as 48
    # token-major pair tiles of 256 columns shared along K by all 76 pairs.
    # Both CTAs of a pair run the same segments; every (tile, k-block) is
    # covered once per pair; the reduction order lists pair indices in K order
    # with unique slots (2·pair for a pair's first split segment, 2·pair + 1
    # for its last).
    p = dict(dlp.proj_plan_compute(256, 12288, 4096, 1))
    KT = p["k_blocks"]
    p.update(block_n=256, tiles_n=48, grid=152, tiles_dp=0, tiles_sk=48, units_sk=48 * KT)
    cover = np.zeros((48, KT), dtype=np.int32)
    for c in range(0, 152, 2):
        segs = dlp.proj_plan_segments(p, c)
        assert segs == dlp.proj_plan_segments(p, c + 1)
        for (tile, tm, tn, kb0, kb1, slot, split) in segs:
            cover[tile, kb0:kb1] += 1
            assert split == 1 and slot in (2 * (c // 2), 2 * (c // 2) + 1)
    assert (cover == 1).all()
    for ts in range(48):
        order = dlp.proj_plan_reduction_order(p, ts)
        pairs = [c for c, _ in order]
        assert pairs == sorted(pairs) and 2 <= len(order) <= 3
        assert len({sl for _, sl in order}) == len(order)
        segs = sorted((kb0, c // 2) for c in range(0, 152, 2)
                      for (tile, _, _, kb0, _, _, _) in dlp.proj_plan_segments(p, c) if tile == ts)
        assert pairs == [q for _, q in segs]


def test_cluster_split_plans():
    # 16 tiles of the 2048-row decode weight: clusters of 9 (144 CTAs; a
    # device lowers S until all 16 clusters fit at once).
    p = plan(16, 2048, 8192)
    assert (p["cluster_split"], p["grid"], p["tiles_sk"], p["tiles_dp"]) == (9, 144, 16, 0)
    assert dlp.proj_plan_reduction_order(p, 3) == [(3 * 9 + r, -1) for r in range(9)]
    # The 2 tiles of the router weight (N = 256, [H | L]: 2·8192 K): clusters
    # of 16, the largest size.
    p = plan(16, 256, 2 * 8192)
    assert (p["cluster_split"], p["grid"]) == (16, 32)
    # 64 tiles of the 8192-row decode weight (two k-blocks a stage): clusters
    # of 2 on 128 SMs; the 224 tiles of the 28672-row FFN weight: stream-K
    # over every SM.
    p = plan(16, 8192, 8192)
    assert (p["cluster_split"], p["grid"], p["block_k"]) == (2, 128, 128)
    p = plan(16, 28672, 8192)
    assert p["cluster_split"] == 0 and p["grid"] == 152
    # Two k-blocks a stage: clusters while 2·tiles <= SMs (76 tiles: clusters
    # of 2; 77 tiles: stream-K; 50 tiles: clusters of 3).
    assert plan(16, 76 * 128, 8192)["cluster_split"] == 2
    assert plan(16, 77 * 128, 8192)["cluster_split"] == 0
    assert plan(16, 50 * 128, 8192)["cluster_split"] == 3
    # One k-block a stage (K not a multiple of 64): clusters only below a
    # third of the SMs in tiles: 50 tiles (3·50 < 152) take clusters of 3 on
    # 150 SMs; 51 tiles stream-K; 45 tiles clusters of 3.
    assert plan(16, 50 * 128, 8200)["cluster_split"] == 3
    assert plan(16, 51 * 128, 8200)["cluster_split"] == 0
    assert plan(16, 45 * 128, 8200)["cluster_split"] == 3
    assert plan(16, 51 * 128, 8200)["block_k"] == 64
    # Small devices (12 SMs, 3 tiles: clusters of 4; 8 SMs and 2 tiles:
    # clusters of 4; 5 SMs, 1 tile: clusters of 5).
    assert plan(16, 3 * 128, 8192, sm_count=12, smem_optin_bytes=232448)["cluster_split"] == 4
    assert plan(16, 2 * 128, 8192, sm_count=8, smem_optin_bytes=232448)["cluster_split"] == 4
    assert plan(16, 128, 8192, sm_count=5, smem_optin_bytes=232448)["cluster_split"] == 5
    # Fewer than 10 % of the SMs busy: 1 tile with 4 or 8 k-blocks on 152 SMs.
    assert plan(16, 128, 256)["cluster_split"] == 0
    assert plan(16, 128, 512)["cluster_split"] == 0
    # S is capped by the stages of K there are to share (5 SMs, 1 tile, K = 512
    # in 4 stages of two k-blocks).
    p = plan(16, 128, 512, sm_count=5, smem_optin_bytes=232448)
    assert p["k_blocks"] == 4 and p["block_k"] == 128 and p["cluster_split"] == 4 and p["grid"] == 4
    # Several token tiles (100 tokens in two 64-row tiles) are clustered too.
    p = plan(100, 1024, 8192)
    assert (p["block_t"], p["tiles_m"], p["cluster_split"], p["grid"]) == (64, 2, 9, 144)
    # Token-major tiles are never cluster-split.
    assert plan(256, 2048, 8192)["cluster_split"] == 0


def test_plans_of_many_shapes():
    rng = np.random.default_rng(0)
    shapes = [(1, 1, 8), (1, 128, 64), (17, 300, 72), (3, 130, 72), (257, 300, 256),
              (512, 20480, 256), (600, 1000, 1032), (9, 7, 16)]
    shapes += [(int(rng.integers(1, 700)), int(rng.integers(1, 6000)), 8 * int(rng.integers(1, 700)))
               for _ in range(40)]
    for (M, N, K) in shapes:
        for sm in (152, 148, 7, 1):
            p = plan(M, N, K, sm_count=sm, smem_optin_bytes=232448)
            assert p["grid"] <= sm
            check_decomposition(p, M, N, K, sms=sm)


def test_page_partition_42_43_43():
    # 128 K tiles shared by 3 CTAs with integer boundaries: 42, 43, 43
    # ("Why the later TMA/WGMMA kernel was a new experiment").
    p = {"kernel": dlp.PROJ_KERNEL_TC, "grid": 3, "k_blocks": 128, "tiles_m": 1, "tiles_n": 1,
         "tiles_dp": 0, "tiles_sk": 1, "units_sk": 128, "block_t": 16}
    lens = [sum(kb1 - kb0 for (_, _, _, kb0, kb1, _, _) in dlp.proj_plan_segments(p, c))
            for c in range(3)]
    assert lens == [42, 43, 43]
    assert [c for c, _ in dlp.proj_plan_reduction_order(p, 0)] == [0, 1, 2]


def test_split_k_example_every_k_covered_once():
    # Section "How splitting changes the grid" / the split-router K loop: all
    # K positions of a 8192-long sum are covered, none twice, for any split.
    for G in (2, 3, 16, 32, 152):
        p = {"kernel": dlp.PROJ_KERNEL_TC, "grid": G, "k_blocks": 128, "tiles_m": 1,
             "tiles_n": 1, "tiles_dp": 0, "tiles_sk": 1, "units_sk": 128, "block_t": 16}
        covered = []
        for c in range(G):
            for seg in dlp.proj_plan_segments(p, c):
                covered.extend(range(seg[3], seg[4]))
        assert sorted(covered) == list(range(128))


def test_degenerate_plans_and_errors():
    assert plan(0, 64, 64)["kernel"] == dlp.PROJ_KERNEL_NONE
    assert plan(4, 0, 64)["kernel"] == dlp.PROJ_KERNEL_NONE
    assert plan(4, 64, 0)["kernel"] == dlp.PROJ_KERNEL_FILL
    for bad in [(-1, 4, 8), (4, -1, 8), (4, 4, -8)]:
        with pytest.raises(dlp.ProjError) as e:
            plan(*bad)
        assert e.value.status == dlp.PROJ_ERR_INVALID_ARG
    with pytest.raises(dlp.ProjError):
        dlp.proj_plan_compute(4, 4, 8, 7)
    with pytest.raises(dlp.ProjError) as e:
        dlp.proj_plan_compute(4, 4, 8, 0, sm_count=152, smem_optin_bytes=20000)
    assert e.value.status == dlp.PROJ_ERR_UNSUPPORTED
    with pytest.raises(dlp.ProjError):
        dlp.proj_plan_segments({"kernel": 2, "grid": 4, "k_blocks": 2, "tiles_m": 1}, 4)


def test_token_tile_choice():
    assert plan(1, 8192, 8192)["block_t"] == 16
    assert plan(16, 8192, 8192)["block_t"] == 16
    assert plan(17, 8192, 8192)["block_t"] == 32
    assert plan(64, 28672, 8192)["block_t"] == 64
    assert plan(4096, 8192, 8192)["block_t"] == 256
    assert plan(256, 12288, 4096, 1)["block_t"] == 256  # token-major pairs: 256 tokens per pair
    assert plan(256, 12288, 4100, 1)["block_t"] == 128  # one k-block a stage: single CTAs, 128 tokens


def test_scratch_and_stages():
    p = plan(16, 28672, 8192)
    assert p["tiles_sk"] > 0 and p["cluster_split"] == 0
    # swapped: B holds the token rows; two k-blocks a stage
    stage = (p["block_k"] // 64) * (128 * 64 * 2 + p["block_t"] * 64 * 2)
    assert p["block_k"] == 128
    assert p["smem_bytes"] == p["stages"] * stage + 25600
    assert p["scratch_bytes"] >= 2 * p["grid"] * p["block_t"] * 128 * 4 + 4 * 4 * p["tiles_sk"]
    assert p["tmem_cols"] >= 2 * p["block_t"] and p["tmem_cols"] in (32, 64, 128, 256, 512)


def test_raster_groups():
    # Prefill: 16 token tiles of 256 rows in groups of 8 (2048 token rows);
    # within a group the token tile varies fastest, so the first wave covers
    # 8 token panels x 19 weight panels.
    # The tiles are 256 weight rows wide (CTA pairs): 76 pairs cover 8 token
    # panels x 10 weight panels.
    p = plan(4096, 8192, 8192)
    assert p["raster_group"] == 8 and p["tiles_m"] == 16 and p["cta_pair"] == 1
    first_wave = set()
    for c in range(p["grid"]):
        tile, tm, tn = dlp.proj_plan_segments(p, c)[0][:3]
        assert tile == c // 2
        first_wave.add((tm, tn))
    assert {tm for tm, _ in first_wave} == set(range(8))
    assert len({tn for _, tn in first_wave}) == 10
    assert plan(16, 8192, 8192)["raster_group"] == 1


def test_orientation_and_weight_tile_choice():
    # Fewer than 128 tokens: weight rows on the MMA's M side (swapped).
    for M in (1, 16, 64, 127):
        assert plan(M, 8192, 8192)["swap_ab"] == 1
    # From 128 tokens: tokens on the M side, weight tile sized to fill waves.
    # The QKV shape (K a multiple of 64, two k-blocks a stage): token-major CTA
    # pairs of 256 tokens x 176 weight rows, one whole wave of 70 pair tiles.
    qkv = plan(256, 12288, 4096, 1)
    assert qkv["swap_ab"] == 0 and qkv["block_t"] == 256 and qkv["cta_pair"] == 1
    assert qkv["block_n"] == 176 and qkv["tiles_m"] * qkv["tiles_n"] == 70 and qkv["grid"] == 140
    assert qkv["block_k"] == 128 and qkv["tiles_sk"] == 0
    # One k-block a stage (K not a multiple of 64): single CTAs of 128 tokens.
    qkv1 = plan(256, 12288, 4104, 1)
    assert qkv1["swap_ab"] == 0 and qkv1["block_t"] == 128 and qkv1["cta_pair"] == 0
    assert qkv1["block_n"] == 192 and qkv1["tiles_m"] * qkv1["tiles_n"] == 128
    assert qkv1["tiles_sk"] == 0  # one whole wave (84 % of the SMs) beats splitting
    # Many tiles either way (prefill): the swapped 256-token x 128-row tiles.
    # Many tiles either way (prefill): swapped 256-token tiles, on CTA pairs of
    # 2 x 128 weight rows.
    pre = plan(4096, 8192, 8192)
    assert (pre["swap_ab"], pre["block_t"], pre["block_n"], pre["tiles_sk"]) == (1, 256, 256, 0)
    assert pre["cta_pair"] == 1 and pre["tmem_cols"] == 512 and pre["grid"] == 152
    # [K,N] weights load in 64-row boxes: the weight tile of a single-CTA plan
    # is a multiple of 64.  A pair's tile is a multiple of 16 (the handle runs
    # weights as stored on a single-CTA plan when the halves are not whole
    # boxes; packed weights have no such limit).
    for N in (1000, 3000, 9000):  # few enough weight rows that swapped tiles leave SMs idle
        p = plan(300, N, 1024, 1)
        assert p["swap_ab"] == 0 and p["block_n"] % (16 if p["cta_pair"] else 64) == 0


def test_cta_pair_choice():
    # Pairs only for swapped 256-token tiles that keep half of the SMs busy.
    assert plan(16, 8192, 8192)["cta_pair"] == 0           # decode: stream-K
    assert plan(100, 1024, 8192)["cta_pair"] == 0          # two 64-token tiles: cluster split
    assert plan(64, 28672, 8192)["cta_pair"] == 0          # weight streaming
    assert plan(256, 12288, 4096, 1)["cta_pair"] == 1      # token-major, two k-blocks a stage: pairs
    assert plan(256, 12288, 4104, 1)["cta_pair"] == 0      # token-major, one k-block: single CTAs
    assert plan(1024, 4096, 4096)["cta_pair"] == 1         # token-major, 64 pair tiles
    p = plan(512, 20480, 256)
    assert (p["cta_pair"], p["swap_ab"], p["block_t"], p["block_n"]) == (1, 1, 256, 256)
    assert p["tiles_m"] * p["tiles_n"] == 160 and p["grid"] == 152
    # Stages: two k-blocks of 16 KiB of A (128 weight rows) plus half of the
    # 256 token rows.
    assert p["block_k"] == 128
    assert p["stages"] == 3 and p["smem_bytes"] == 3 * 2 * (16384 + 128 * 128) + 25600
    # A small problem: with two k-blocks a stage, token-major pairs of 64
    # weight rows (64 pair tiles on 128 SMs); with one, single CTAs.
    p = plan(256, 4096, 1024)
    assert (p["cta_pair"], p["swap_ab"], p["block_t"], p["block_n"], p["grid"]) == (1, 0, 256, 64, 128)
    assert plan(256, 4096, 1032)["cta_pair"] == 0
