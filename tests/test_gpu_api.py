"""GPU tests of the C ABI's contract: argument errors return a status before
any launch and leave every output untouched; kernels write nothing outside
their outputs (guard bands); the launch count is what the library reports."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_harness import to_device
from mhc_residual_boundary_gb300 import synth

pytestmark = pytest.mark.gpu

H, TP, M = 512, 4, 24


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from mhc_residual_boundary_gb300 import Boundary, capi
    b = Boundary(hidden=H, tp=TP, max_num_tokens=M, mxfp8=False)
    inp = to_device(synth.make_inputs(H, TP, M, seed=1))
    yield b, inp, capi
    b.close()


def _raw_args(capi, inp, outs, m=M):
    a = capi.mhc_run_args_t()
    a.m = m
    for n in ("partials", "residual", "post", "comb", "hc_fn", "scale", "base", "norm_weight"):
        setattr(a, n, inp[n].data_ptr())
    for n, t in outs.items():
        setattr(a, n, t.data_ptr())
    return a


def _sentinel_outputs(b, m=M):
    outs = b.empty_outputs(m, extras=True)
    for t in outs.values():
        t.view(torch.uint8).fill_(0x5A)
    return outs


def _untouched(outs):
    torch.cuda.synchronize()
    return all(bool((t.view(torch.uint8) == 0x5A).all()) for t in outs.values())


@pytest.mark.parametrize("case,status", [
    ("m0", "MHC_ERR_CAPACITY"), ("m_big", "MHC_ERR_CAPACITY"), ("null_residual", "MHC_ERR_INVALID_ARG"),
    ("null_partials", "MHC_ERR_INVALID_ARG"), ("misaligned_partials", "MHC_ERR_INVALID_ARG"),
    ("misaligned_layer_input", "MHC_ERR_INVALID_ARG"), ("mxfp8_without_flag", "MHC_ERR_UNSUPPORTED"),
    ("misaligned_post", "MHC_ERR_INVALID_ARG"),
    ("both_weight_forms", "MHC_ERR_INVALID_ARG"), ("no_weight", "MHC_ERR_INVALID_ARG"),
    ("misaligned_bf16_weight", "MHC_ERR_INVALID_ARG"),
])
def test_bad_arguments_launch_nothing(env, case, status):
    b, inp, capi = env
    outs = _sentinel_outputs(b)
    a = _raw_args(capi, inp, outs)
    spare = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    if case == "m0":
        a.m = 0
    elif case == "m_big":
        a.m = M + 1
    elif case == "null_residual":
        a.residual = None
    elif case == "null_partials":
        a.partials = None
    elif case == "misaligned_partials":
        a.partials = inp["partials"].data_ptr() + 2
    elif case == "misaligned_post":
        a.post = inp["post"].data_ptr() + 4
    elif case == "misaligned_layer_input":
        a.layer_input = outs["layer_input"].data_ptr() + 8
    elif case == "mxfp8_without_flag":
        a.mxfp8_values = spare.data_ptr()
        a.mxfp8_scales = spare.data_ptr()
    elif case == "both_weight_forms":
        a.hc_fn_bf16 = spare.data_ptr()
    elif case == "no_weight":
        a.hc_fn = None
    elif case == "misaligned_bf16_weight":
        a.hc_fn = None
        a.hc_fn_bf16 = spare.data_ptr() + 2
    with pytest.raises(capi.MhcError) as err:
        capi.mhc_boundary_run(b.handle, a)
    assert status in str(err.value)
    assert _untouched(outs)
    # the handle still works
    good = b.empty_outputs(M)
    b.run(inp, good)
    b.join()
    torch.cuda.synchronize()
    assert torch.isfinite(good["layer_input"].float()).all()


def test_moe_call_needs_top_k(env):
    b, inp, capi = env
    outs = _sentinel_outputs(b)
    a = capi.mhc_moe_args_t()
    a.run = _raw_args(capi, inp, outs)
    a.run.partials = None
    a.rows_per_rank = 4
    a.routed = a.shared = inp["partials"].data_ptr()
    a.idx = a.weights = inp["post"].data_ptr()
    with pytest.raises(capi.MhcError, match="UNSUPPORTED"):
        capi.mhc_boundary_finalize_moe(b.handle, a)
    assert _untouched(outs)


def test_outputs_have_clean_guard_bands(env):
    b, inp, capi = env
    guard = 4096
    bufs, outs = {}, {}
    for name, t in b.empty_outputs(M, extras=True).items():
        nbytes = t.numel() * t.element_size()
        raw = torch.full((nbytes + 2 * guard,), 0xC3, dtype=torch.uint8, device="cuda")
        bufs[name] = raw
        outs[name] = raw[guard:guard + nbytes].view(t.dtype).view(t.shape)
    b.run(inp, outs)
    b.join()
    torch.cuda.synchronize()
    for name, raw in bufs.items():
        assert bool((raw[:guard] == 0xC3).all()) and bool((raw[-guard:] == 0xC3).all()), name


def test_launch_count(env):
    # a few tokens: the one-kernel path (post / Sinkhorn inside it); a separate
    # mixes kernel adds one; beyond the one-kernel path's token range the
    # stage and finish kernels
    b, _, _ = env
    assert b.launches_per_call() == 2          # M = 24: stage and finish
    from mhc_residual_boundary_gb300 import Boundary
    few = Boundary(hidden=H, tp=TP, max_num_tokens=8)
    assert few.launches_per_call() == 1
    few.close()
    for flags in ({"side_mixes": True}, {"sync_mixes": True}):
        other = Boundary(hidden=H, tp=TP, max_num_tokens=8, **flags)
        assert other.launches_per_call() == 2
        other.close()
    many = Boundary(hidden=H, tp=TP, max_num_tokens=1000)
    assert many.launches_per_call() == 2
    many.close()
