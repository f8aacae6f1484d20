"""The PyTorch wrapper's argument checks without a GPU: a tensor in the wrong
place (host memory for a device call, or the reverse) or of the wrong shape is
refused before any pointer reaches the C library."""
import pytest
import torch

from mhc_residual_boundary_gb300 import boundary as bmod

H, TP, M = 64, 2, 3


@pytest.fixture
def b(monkeypatch):
    # a wrapper whose handle was never created: every C entry point fails the
    # test if it is reached
    def refuse(*a, **k):
        raise AssertionError("the C library was called")

    for name in ("mhc_boundary_run", "mhc_boundary_run_host", "mhc_boundary_consume",
                 "mhc_boundary_finalize_moe"):
        monkeypatch.setattr(bmod.capi, name, refuse)
    obj = object.__new__(bmod.Boundary)
    obj.hidden, obj.tp, obj.top_k, obj.capacity = H, TP, 0, 8
    obj.device = torch.device("cuda", 0)
    obj.handle = None
    return obj


def host_inputs(device="cpu"):
    out = {}
    for n in ("partials", "residual", "post", "comb", "hc_fn", "scale", "base", "norm_weight"):
        dtype, shape = bmod.INPUT_SPECS[n]
        out[n] = torch.zeros(shape(TP, M, H, 0, 0), dtype=dtype, device=device)
    return out


def host_outputs(device="cpu"):
    return {n: torch.zeros(bmod.OUTPUT_SPECS[n][1](M, H), dtype=bmod.OUTPUT_SPECS[n][0], device=device)
            for n in bmod.REQUIRED_OUTPUTS}


def test_device_call_refuses_host_tensors(b):
    with pytest.raises(ValueError, match="must be a tensor on cuda:0"):
        b.run(host_inputs(), host_outputs())


def test_host_call_refuses_device_tensors(b):
    inputs = host_inputs()
    inputs["partials"] = inputs["partials"].to("meta")
    with pytest.raises(ValueError, match="partials must be a host tensor"):
        b.run_host(inputs, host_outputs())
    outputs = host_outputs()
    outputs["layer_input"] = outputs["layer_input"].to("meta")
    with pytest.raises(ValueError, match="layer_input must be a host tensor"):
        b.run_host(host_inputs(), outputs)


def test_consumer_refuses_host_tensors(b):
    inputs = {n: t for n, t in host_inputs().items() if n in ("partials", "residual", "post", "comb")}
    outputs = {"residual_out": host_outputs()["residual_out"]}
    with pytest.raises(ValueError, match="must be a tensor on cuda:0"):
        b.consume(inputs, outputs)


def test_wrong_shape_or_dtype_is_refused(b):
    inputs = host_inputs()
    inputs["comb"] = torch.zeros(M, 4, dtype=torch.float32)
    with pytest.raises(ValueError, match="comb: expected"):
        b.run_host(inputs, host_outputs())
    inputs = host_inputs()
    inputs["post"] = inputs["post"].double()
    with pytest.raises(ValueError, match="post: expected"):
        b.run_host(inputs, host_outputs())
    outputs = host_outputs()
    outputs["residual_out"] = outputs["residual_out"].transpose(0, 1).contiguous().transpose(0, 1)
    with pytest.raises(ValueError, match="residual_out: expected contiguous"):
        b.run_host(host_inputs(), outputs)


def test_host_call_with_host_tensors_reaches_the_library(b):
    # the placement and shape checks pass: the next step is the C call
    with pytest.raises(AssertionError, match="the C library was called"):
        b.run_host(host_inputs(), host_outputs())
