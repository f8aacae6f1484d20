"""Shared helpers of the GPU tests: run the CUDA path through the C ABI on
NumPy inputs and compare every output with the oracle."""
import os

import numpy as np
import torch

import oracle
from tolerances import close_f32, floor_use, floor_use_allowed, layer_input_ok, ulp_diff

# (test id, report) of every comparison in this process; the terminal summary
# of tests/conftest.py prints how often the layer-input floor was needed
REPORTS = []

BF16_INPUTS = ("partials", "residual", "norm_weight", "routed", "shared")


def to_device(inputs: dict, device="cuda") -> dict:
    out = {}
    for name, a in inputs.items():
        key = "norm_weight" if name == "gamma" else name
        if a.dtype == np.uint16:
            t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(a))
        out[key] = t.to(device)
    return out


def to_numpy(outputs: dict) -> dict:
    res = {}
    for name, t in outputs.items():
        t = t.cpu()
        if t.dtype == torch.bfloat16:
            res[name] = t.view(torch.int16).numpy().view(np.uint16)
        else:
            res[name] = t.numpy()
    return res


def run_gpu(boundary, inputs: dict, *, moe=False, mxfp8=False, extras=True, stream=None) -> dict:
    m = inputs["residual"].shape[0]
    dev = to_device(inputs)
    outs = boundary.empty_outputs(m, extras=extras, mxfp8=mxfp8)
    if mxfp8:
        outs["mxfp8_scales"].fill_(0xAB)   # padding rows must be overwritten with 0
    if moe:
        boundary.finalize_moe(dev, outs, stream=stream)
    else:
        boundary.run(dev, outs, stream=stream)
    boundary.join(stream)
    torch.cuda.synchronize()
    return to_numpy(outs)


def oracle_outputs(problem, inputs, *, moe=False, mxfp8=False):
    return oracle.boundary(problem, inputs, moe=moe, mxfp8_out=mxfp8)


def compare(got: dict, ref: dict, inputs: dict, *, mxfp8=False) -> dict:
    """Asserts every output within its tolerance; returns a small report."""
    report = {}
    if "reduced_out" in got:
        bad = np.argwhere(got["reduced_out"].view(np.uint16) != ref["reduced"].view(np.uint16))
        assert bad.size == 0, (f"stage-1 sum is not bit-exact at {len(bad)} elements, first {bad[:4].tolist()}: "
                               f"got {[int(got['reduced_out'].view(np.uint16)[tuple(i)]) for i in bad[:4]]} "
                               f"want {[int(ref['reduced'].view(np.uint16)[tuple(i)]) for i in bad[:4]]}")
    d = ulp_diff(got["residual_out"], ref["residual_out"])
    report["residual_out_max_ulp"] = int(d.max())
    assert d.max() <= 2, f"post-mixed streams off by {d.max()} ulp"
    ok = layer_input_ok(got["layer_input"], ref["layer_input"], ref["residual_out"], ref["pre"],
                        inputs["gamma"])
    report["layer_input_max_ulp"] = int(ulp_diff(got["layer_input"], ref["layer_input"]).max())
    assert ok.all(), f"layer input outside tolerance at {np.argwhere(~ok)[:5].tolist()}"
    fu = floor_use(got["layer_input"], ref["layer_input"], ref["residual_out"], ref["pre"], inputs["gamma"])
    report.update({"layer_input_" + k: v for k, v in fu.items()})
    REPORTS.append((os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], report))
    assert floor_use_allowed(fu), f"layer input needs the cancellation floor too often: {fu}"
    for name, rname, atol in (("pre_out", "pre", 1e-6), ("post_out", "post_out", 1e-6),
                              ("comb_out", "comb_out", 1e-6), ("mixes_out", "mixes", 1e-5)):
        if name in got:
            good = close_f32(got[name], ref[rname], 1e-4, atol)
            rel = np.abs(got[name].astype(np.float64) - ref[rname]) / np.maximum(np.abs(ref[rname]), atol)
            report[name + "_max_rel"] = float(rel.max())
            assert good.all(), f"{name} outside rel 1e-4 (max rel {rel.max():.3g})"
    if mxfp8:
        # bit-identical to quantising the kernel's own BF16 output ...
        own_v, own_s = oracle.mxfp8(got["layer_input"])
        assert np.array_equal(got["mxfp8_values"], own_v), "MXFP8 values differ from quantising the output"
        assert np.array_equal(got["mxfp8_scales"], own_s), "MXFP8 scales differ from quantising the output"
        # ... and to quantising the oracle's output wherever the two agree
        m, H = got["layer_input"].shape
        same_block = (got["layer_input"] == ref["layer_input"]).reshape(m, H // 32, 32).all(axis=2)
        rv = ref["mx_values"].reshape(m, H // 32, 32)
        gv = got["mxfp8_values"].reshape(m, H // 32, 32)
        assert np.array_equal(gv[same_block], rv[same_block])
        report["mxfp8_blocks_differing_from_oracle"] = int((~same_block).sum())
    return report
