"""mhc_boundary_run_static: the allocation-free entry point.

It serves callers that cannot allocate device memory when they need a
boundary (a caching allocator that owns the device budget, code that must
not risk the synchronisation of a cudaMalloc, threads that may not create a
handle).  Its outputs must match the handle-based entry point's on the same
inputs, within the parity tolerances, on two calls in a row (the second call
reuses the static scratch the first one left behind).  The cases cover the
tensor-core stage kernel with both weight forms, the CUDA-core stage kernel
(tp > 8, whose 64-column groups the capacity rule is written for) and the
largest accepted token count.  A stage kernel made to give up its waits (the
test hook) must come back as MHC_ERR_TIMEOUT through MHC_FLAG_CHECK_ERRORS.
The file sorts last so that a run stopping at its first failure has already
run every other test.
"""
import numpy as np
import pytest
import torch

import oracle

from gpu_harness import to_device, to_numpy
from mhc_residual_boundary_gb300 import synth
from tolerances import close_f32, layer_input_ok, ulp_diff

pytestmark = pytest.mark.gpu


def _args(capi, dev_in, outs, m):
    a = capi.mhc_run_args_t()
    a.m = m
    weight = "hc_fn_bf16" if "hc_fn_bf16" in dev_in else "hc_fn"
    for n in ("partials", "residual", "post", "comb", weight, "scale", "base", "norm_weight"):
        setattr(a, n, dev_in[n].data_ptr())
    for n, t in outs.items():
        setattr(a, n, t.data_ptr())
    return a


def _same(static, handle, inputs):
    assert np.array_equal(static["reduced_out"], handle["reduced_out"])
    assert ulp_diff(static["residual_out"], handle["residual_out"]).max() <= 2
    assert layer_input_ok(static["layer_input"], handle["layer_input"], handle["residual_out"],
                          handle["pre_out"], inputs["gamma"]).all()
    for n, atol in (("pre_out", 1e-6), ("post_out", 1e-6), ("comb_out", 1e-6), ("mixes_out", 1e-5)):
        assert close_f32(static[n], handle[n], 1e-4, atol).all(), n
    if "mxfp8_values" in handle:
        # each copy quantises its own BF16 output bit for bit; the two agree
        # wherever their BF16 blocks agree
        v, sc = oracle.mxfp8(static["layer_input"])
        assert np.array_equal(static["mxfp8_values"], v) and np.array_equal(static["mxfp8_scales"], sc)
        m, hidden = static["layer_input"].shape
        same = (static["layer_input"] == handle["layer_input"]).reshape(m, hidden // 32, 32).all(axis=2)
        sv = static["mxfp8_values"].reshape(m, hidden // 32, 32)
        hv = handle["mxfp8_values"].reshape(m, hidden // 32, 32)
        assert np.array_equal(sv[same], hv[same])


def _config(capi, hidden, tp, m, flags):
    return capi.mhc_boundary_config_t(hidden, 4, tp, m, 20, 0, 1e-6, 1e-6, 2.0, 1e-6, flags)


CASES = [
    # hidden, tp, m, mxfp8, bf16 weight
    (6144, 4, 256, True, False),      # tensor-core stage kernel, FP32 weight
    (5120, 8, 37, False, False),
    (6144, 4, 64, True, True),        # tensor-core stage kernel, BF16 [24][4H] weight
    (1024, 16, 40, False, False),     # CUDA-core stage kernel: 64-column groups
    (6144, 12, 865, False, False),    # the largest m at H = 6144, in the layout the capacity rule counts
]


@pytest.mark.parametrize("hidden,tp,m,mxfp8,bf16", CASES)
def test_static_entry_matches_handle_entry_twice(hidden, tp, m, mxfp8, bf16):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from mhc_residual_boundary_gb300 import Boundary, capi
    b = Boundary(hidden=hidden, tp=tp, max_num_tokens=m, mxfp8=mxfp8)
    flags = (capi.MHC_FLAG_MXFP8 if mxfp8 else 0) | capi.MHC_FLAG_CHECK_ERRORS
    cfg = _config(capi, hidden, tp, m, flags)
    try:
        for seed in (11, 12):                      # two calls in a row
            inputs = synth.make_inputs(hidden, tp, m, seed=seed)
            if bf16:
                inputs["hc_fn_bf16"] = synth.bf16_weight(inputs.pop("hc_fn"))
            dev_in = to_device(inputs)
            ref = b.empty_outputs(m, extras=True, mxfp8=mxfp8)
            b.run(dev_in, ref)
            b.join()
            got = b.empty_outputs(m, extras=True, mxfp8=mxfp8)
            for t in got.values():
                t.view(torch.uint8).fill_(0x5A)
            capi.mhc_boundary_run_static(cfg, _args(capi, dev_in, got, m))
            torch.cuda.synchronize()
            _same(to_numpy(got), to_numpy(ref), inputs)
    finally:
        b.close()


def test_static_entry_reports_a_wait_that_gave_up():
    # the stage kernel issues no input copies (test hook), so its bounded
    # waits run out: the call with MHC_FLAG_CHECK_ERRORS reports the timeout;
    # with the hook off the next call is correct again and reports nothing
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from mhc_residual_boundary_gb300 import Boundary, capi
    hidden, tp, m = 1024, 4, 24
    cfg = _config(capi, hidden, tp, m, capi.MHC_FLAG_CHECK_ERRORS)
    inputs = synth.make_inputs(hidden, tp, m, seed=31)
    dev_in = to_device(inputs)
    b = Boundary(hidden=hidden, tp=tp, max_num_tokens=m)
    try:
        got = b.empty_outputs(m, extras=True)
        capi.mhc_test_stall_stage_copies(True)
        try:
            with pytest.raises(capi.MhcError, match="TIMEOUT"):
                capi.mhc_boundary_run_static(cfg, _args(capi, dev_in, got, m))
        finally:
            capi.mhc_test_stall_stage_copies(False)
        capi.mhc_boundary_run_static(cfg, _args(capi, dev_in, got, m))   # word cleared, call correct
        ref = b.empty_outputs(m, extras=True)
        b.run(dev_in, ref)
        b.join()
        torch.cuda.synchronize()
        _same(to_numpy(got), to_numpy(ref), inputs)
    finally:
        b.close()


def test_static_entry_rejects_too_many_tokens():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from mhc_residual_boundary_gb300 import capi
    hidden, tp, m = 6144, 4, 866                    # one token beyond the 8 MiB scratch
    cfg = _config(capi, hidden, tp, m, 0)
    a = capi.mhc_run_args_t()
    a.m = m
    with pytest.raises(capi.MhcError, match="CAPACITY"):
        capi.mhc_boundary_run_static(cfg, a)
