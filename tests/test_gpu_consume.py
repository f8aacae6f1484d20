"""GPU parity of the delayed-mHC consumer ([DSV] AllReduceMHC.__call__ /
finalize with a carried pre-mix, and residual_only) through the C ABI
against the oracle, plus its argument checks."""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import to_device, to_numpy
from mhc_residual_boundary_gb300 import synth
from tolerances import layer_input_ok, ulp_diff

pytestmark = pytest.mark.gpu
HC = 4


@pytest.fixture(scope="module")
def Boundary():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from mhc_residual_boundary_gb300 import Boundary as B
    return B


def run_consume(Boundary, hidden, tp, m, *, seed, moe=False, top_k=0, holes=0.0, mxfp8=False,
                residual_only=False, owner_reduce=False):
    inp = synth.make_inputs(hidden, tp, m, top_k=top_k, moe=moe, seed=seed, holes=holes)
    pre = np.random.default_rng(seed).uniform(0.05, 1.2, (m, HC)).astype(np.float32)
    p = oracle.Problem(hidden, tp, m, top_k=top_k, rows_per_rank=m * top_k if moe else 0)
    ref = oracle.consume(p, inp, pre, moe=moe, mxfp8_out=mxfp8, residual_only=residual_only)
    b = Boundary(hidden=hidden, tp=tp, max_num_tokens=m, top_k=top_k, mxfp8=mxfp8, owner_reduce=owner_reduce)
    try:
        dev = to_device(inp)
        if moe:
            dev.pop("partials", None)
        if not residual_only:
            dev["pre"] = torch.from_numpy(pre).cuda()
        else:
            dev.pop("norm_weight")
        outs = {"residual_out": torch.empty((m, HC, hidden), dtype=torch.bfloat16, device="cuda"),
                "reduced_out": torch.empty((m, hidden), dtype=torch.bfloat16, device="cuda")}
        if not residual_only:
            outs["layer_input"] = torch.empty((m, hidden), dtype=torch.bfloat16, device="cuda")
            if mxfp8:
                mx = b.empty_outputs(m, mxfp8=True)
                outs["mxfp8_values"], outs["mxfp8_scales"] = mx["mxfp8_values"], mx["mxfp8_scales"]
                outs["mxfp8_scales"].fill_(0xAB)
        b.consume(dev, outs)
        torch.cuda.synchronize()
        b.check_errors()
        return to_numpy(outs), ref, inp, pre
    finally:
        b.close()


def check(got, ref, inp, pre, *, mxfp8=False, residual_only=False):
    assert np.array_equal(got["reduced_out"], ref["reduced"]), "stage-1 sum is not bit-exact"
    assert ulp_diff(got["residual_out"], ref["residual_out"]).max() <= 2
    if residual_only:
        return
    ok = layer_input_ok(got["layer_input"], ref["layer_input"], ref["residual_out"], pre, inp["gamma"])
    assert ok.all(), f"layer input outside tolerance at {np.argwhere(~ok)[:5].tolist()}"
    if mxfp8:
        own_v, own_s = oracle.mxfp8(got["layer_input"])
        assert np.array_equal(got["mxfp8_values"], own_v)
        assert np.array_equal(got["mxfp8_scales"], own_s)


@pytest.mark.parametrize("hidden,tp,m,mxfp8", [(6144, 4, 40, False), (520, 5, 33, False), (2048, 8, 130, True),
                                               (8, 1, 3, False), (5120, 8, 256, False)])
def test_consume_matches_oracle(Boundary, hidden, tp, m, mxfp8):
    got, ref, inp, pre = run_consume(Boundary, hidden, tp, m, seed=hidden + m, mxfp8=mxfp8)
    check(got, ref, inp, pre, mxfp8=mxfp8)


@pytest.mark.parametrize("hidden,tp,m", [(6144, 4, 70), (72, 2, 9)])
def test_residual_only(Boundary, hidden, tp, m):
    got, ref, inp, pre = run_consume(Boundary, hidden, tp, m, seed=m, residual_only=True)
    check(got, ref, inp, pre, residual_only=True)


@pytest.mark.parametrize("hidden,tp,m,mxfp8", [(6144, 4, 1, False), (5120, 8, 5, True), (6144, 8, 12, True),
                                               (7168, 8, 2, False), (1032, 3, 7, False)])
def test_consume_few_tokens(Boundary, hidden, tp, m, mxfp8):
    # up to twelve tokens the consumer runs in one kernel of CTA clusters
    got, ref, inp, pre = run_consume(Boundary, hidden, tp, m, seed=hidden + tp + m, mxfp8=mxfp8)
    check(got, ref, inp, pre, mxfp8=mxfp8)


@pytest.mark.parametrize("hidden,tp,m", [(6144, 4, 1), (5120, 8, 12), (520, 5, 3)])
def test_residual_only_few_tokens(Boundary, hidden, tp, m):
    # the streams only: one kernel up to four tokens, the stage kernel above
    got, ref, inp, pre = run_consume(Boundary, hidden, tp, m, seed=7 * m + tp, residual_only=True)
    check(got, ref, inp, pre, residual_only=True)


@pytest.mark.parametrize("m,residual_only", [(6, False), (2, True)])
def test_consume_moe_few_tokens(Boundary, m, residual_only):
    got, ref, inp, pre = run_consume(Boundary, 1024, 4, m, moe=True, top_k=4, holes=0.2, seed=31 + m,
                                     residual_only=residual_only)
    check(got, ref, inp, pre, residual_only=residual_only)


def test_consume_moe(Boundary):
    got, ref, inp, pre = run_consume(Boundary, 1024, 4, 60, moe=True, top_k=4, holes=0.2, seed=23)
    check(got, ref, inp, pre)


def test_consume_argument_checks(Boundary):
    from mhc_residual_boundary_gb300 import capi
    hidden, tp, m = 256, 2, 4
    inp = to_device(synth.make_inputs(hidden, tp, m, seed=1))
    b = Boundary(hidden=hidden, tp=tp, max_num_tokens=m)
    try:
        outs = {"residual_out": torch.empty((m, HC, hidden), dtype=torch.bfloat16, device="cuda")}
        pre = torch.ones((m, HC), dtype=torch.float32, device="cuda")
        bad = dict(inp, pre=pre)
        bad.pop("norm_weight")
        with pytest.raises((capi.MhcError, KeyError)):
            b.consume(bad, outs)                    # a carried pre needs norm_weight and layer_input
        a = capi.mhc_consume_args_t()
        a.m = m
        for n in ("partials", "residual", "post", "comb"):
            setattr(a, n, inp[n].data_ptr())
        a.residual_out = outs["residual_out"].data_ptr()
        a.pre = pre.data_ptr()                       # pre without norm_weight / layer_input
        with pytest.raises(capi.MhcError, match="INVALID_ARG"):
            capi.mhc_boundary_consume(b.handle, a)
        a.pre = None
        a.mxfp8_values = a.mxfp8_scales = outs["residual_out"].data_ptr()
        with pytest.raises(capi.MhcError, match="INVALID_ARG"):   # residual only has nothing to quantize
            capi.mhc_boundary_consume(b.handle, a)
    finally:
        b.close()
