"""GPU parity at the five full workload sizes, in the launch configuration the
benchmark times: one handle per shape with its default plan, weights packed
once by proj_pack_weights, programmatic dependent launch (mode "prologue"),
calls back to back on one stream.

Every output element is compared with the fp64 oracle (the whole output of
every shape, the 4096 x 8192 prefill included), for the packed weights the
benchmark uses and for the weights as stored.  Reruns must give the same bits
at full size, for every shape and token count.
"""
import numpy as np
import pytest

import gpu_util as gu
import oracle
import synth

pytestmark = pytest.mark.gpu

_cache = {}
_sweep = {}


def case(name, M=None):
    """Inputs and the oracle's whole output of one workload (one at a time in
    memory).  The token-count sweep draws its weights once: the X of M token
    rows is the first M rows of the largest M's X (same seed, same stream)."""
    key = (name, M)
    if key not in _cache:
        _cache.clear()
        w = synth.workload(name, M)
        if name == "ffn_up_sweep":
            if not _sweep:
                _sweep.update(synth.make_inputs(w.with_m(max(synth.FFN_SWEEP_M))))
            inp = dict(_sweep, X=np.ascontiguousarray(_sweep["X"][:w.M]))
        else:
            _sweep.clear()
            inp = synth.make_inputs(w)
        ref = oracle.project(inp["X"], inp["W"], w.w_layout, inp["bias"])
        _cache[key] = (w, inp, ref)
    return _cache[key]


def run_bench_config(w, inp, calls=1, packed=True):
    """Y of `calls` back-to-back calls in the benchmark's configuration (the
    outputs of every call, as bf16/fp32 tensors)."""
    import torch
    import dense_linear_projection_gb300 as dlp
    proj = dlp.Projection(w.M, w.N, w.K, w.w_layout,
                          dlp.PROJ_F32 if w.y_dtype == "f32" else dlp.PROJ_BF16, w.has_bias,
                          overlap=dlp.PROJ_OVERLAP_PROLOGUE)
    X, W = gu.to_dev(inp["X"]), gu.to_dev(inp["W"])
    b = gu.to_dev(inp["bias"]) if w.has_bias else None
    Wr = proj.pack(W) if packed else W
    dt = torch.float32 if w.y_dtype == "f32" else torch.bfloat16
    outs = [torch.full((w.M, w.N), float("nan"), dtype=dt, device="cuda") for _ in range(calls)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())  # inputs, packing and the NaN fill come first
    for Y in outs:
        proj(X, Wr, b, out=Y, stream=s, packed=packed)
    torch.cuda.synchronize()
    assert proj.status(s) == dlp.PROJ_OK
    proj.close()
    return outs


def bits(t):
    import torch
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def check(name, M=None):
    import torch
    w, inp, ref = case(name, M)
    what = f"{name} M={w.M}"
    outs = run_bench_config(w, inp, calls=3)
    gu.assert_within_tol(gu.y_to_f64(outs[0]), ref, what + " (packed)")
    for Y in outs[1:]:
        assert torch.equal(bits(Y), bits(outs[0])), what + ": reruns differ"
    (stored,) = run_bench_config(w, inp, packed=False)
    gu.assert_within_tol(gu.y_to_f64(stored), ref, what + " (weights as stored)")
    if w.w_layout == synth.W_NK:
        # The same plan over the same K-major tiles: the same bits.
        assert torch.equal(bits(stored), bits(outs[0])), what + ": packed and stored differ"


def test_decode_f32out():
    check("decode_f32out")


def test_decode_bias():
    check("decode_bias")


@pytest.mark.parametrize("M", synth.FFN_SWEEP_M)
def test_ffn_up_sweep(M):
    check("ffn_up_sweep", M)


def test_qkv_kn_bias():
    check("qkv_kn_bias")


def test_prefill():
    check("prefill")
