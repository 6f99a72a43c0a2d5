"""The seeded input generator: published vectors, C/numpy agreement, statistics."""
import numpy as np

import golden_io
import synth


def test_splitmix64_published_vector():
    # SplitMix64 started from state 0 (Steele, Lea & Flood 2014; the widely
    # reproduced reference sequence).
    got = [int(v) for v in synth.splitmix64(np.uint64(0), np.arange(3))]
    assert got == [16294208416658607535, 7960286522194355700, 487617019471545679]


def test_c_generator_matches_numpy():
    for seed, tensor, first, n, std in [(0, 1, 0, 100_000, 1.0), (2, 2, 123_457, 50_001, 0.011),
                                        (4, 3, 7, 999, 0.02)]:
        c = synth.normal_bf16(seed, tensor, n, std, first=first)
        p = synth.normal_bf16_numpy(seed, tensor, n, std, first=first)
        assert np.array_equal(c, p)


def test_sampled_access_matches_stream():
    full = synth.normal_bf16(3, 2, 10_000, 0.5)
    idx = np.array([0, 1, 2, 3, 4097, 9999])
    assert np.array_equal(synth.sample_normal_bf16(3, 2, idx, 0.5), full[idx])


def test_normal_statistics():
    v = synth.normal_bf16(11, 1, 1 << 20, 1.0)
    f = (v.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(f.mean()) < 0.005 and abs(f.std() - 1.0) < 0.005
    assert abs(np.mean(np.abs(f) < 1.0) - 0.6827) < 0.003


def test_round_to_nearest_even_fixture():
    g = golden_io.load("bf16_values.txt")
    for val, hexbits in g["extra"]["round"]:
        assert int(synth.to_bf16_bits(np.array([float(val)]))[0]) == int(hexbits, 16)


def test_streams_are_distinct_and_w_fixed_across_m():
    a = synth.make_inputs(synth.Workload("t", 2, 8, 16, seed=5))
    b = synth.make_inputs(synth.Workload("t", 3, 8, 16, seed=5))
    assert np.array_equal(a["W"], b["W"])          # W does not depend on M
    assert np.array_equal(a["X"], b["X"][:2])      # X rows are a prefix
    assert not np.array_equal(a["X"][0], a["W"][0, :16])


def test_workload_accounting():
    # Algorithmic bytes: 2NK (W) + 2MK (X) + 2N (bias) + M·N·(2|4) (Y); FLOPs 2MNK.
    w = synth.WORKLOADS
    assert w["decode_f32out"].algorithmic_bytes == 33_947_648
    assert w["decode_bias"].algorithmic_bytes == 134_758_400
    assert w["qkv_kn_bias"].algorithmic_bytes == 109_076_480
    assert w["prefill"].algorithmic_bytes == 268_435_456
    assert w["decode_bias"].flops == 2 * 16 * 8192 * 8192
    assert w["qkv_kn_bias"].w_layout == synth.W_KN


def test_fp32_weights_share_the_bf16_stream():
    # fp32 weights are the same normals rounded to fp32 instead of bf16: their
    # bf16 rounding is the bf16 stream itself, bit for bit.
    a = synth.normal_f32(9, synth.STREAM_W, 4096, 0.01)
    b = synth.normal_bf16(9, synth.STREAM_W, 4096, 0.01)
    assert a.dtype == np.float32 and np.array_equal(synth.to_bf16_bits(a.astype(np.float64)), b)
    w = synth.WORKLOADS["router_f32w"]
    assert (w.N, w.K, w.w_dtype) == (256, 8192, "f32")
    assert w.weight_bytes == 4 * 256 * 8192
    assert w.algorithmic_bytes == 4 * 256 * 8192 + 2 * 16 * 8192 + 4 * 16 * 256
    assert synth.make_inputs(w.with_m(2))["W"].dtype == np.float32
