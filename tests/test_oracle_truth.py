"""The FP32 oracle against the FP64 statement of the same steps (no GPU).

Step by step (each FP64 step fed the oracle's own BF16 intermediates) the
two must agree to FP32 rounding; end to end (where a one-ulp BF16 flip early
on moves later values) within the BF16 tolerances of the parity tests.
Small sizes, H = 8 included, every tp from 1 to 8.
"""
import numpy as np
import pytest

from mhc_residual_boundary_gb300 import synth
from oracle import truth
from tolerances import f32, layer_input_ok, ulp_diff

HC, MIX = 4, 24


CASES = [(8, tp, m) for tp in range(1, 9) for m in (1, 3, 5)] + [(64, 4, 4), (520, 8, 2)]


@pytest.mark.parametrize("hidden,tp,m", CASES)
def test_steps_match_fp64(oracle_lib, hidden, tp, m):
    inp = synth.make_inputs(hidden, tp, m, seed=100 + tp * 7 + m)
    p = oracle_lib.Problem(hidden, tp, m)
    out = oracle_lib.boundary(p, inp)
    y = out["reduced"]
    assert ulp_diff(y, truth.bf16_bits(truth.stage1(inp["partials"]))).max() <= 1
    new64 = truth.post_mix(f32(y).astype(np.float64), inp["residual"], inp["post"], inp["comb"])
    assert ulp_diff(out["residual_out"], truth.bf16_bits(new64)).max() <= 1
    raw, ss = truth.prenorm(f32(out["residual_out"]).astype(np.float64), inp["hc_fn"])
    scale = inp["scale"].astype(np.float64)
    base = inp["base"].astype(np.float64)
    mixes, pre = truth.mixes_and_pre(raw, ss, scale, base, hidden, p.rms_eps, p.hc_eps)
    assert np.allclose(out["mixes"], mixes, rtol=2e-6, atol=2e-6)
    assert np.allclose(out["pre"], pre, rtol=2e-6)
    post = truth.post_from_mixes(out["mixes"].astype(np.float64), scale, base, p.post_mult)
    comb = truth.sinkhorn(out["mixes"].astype(np.float64), scale, base, p.hc_eps, p.sinkhorn_repeat)
    assert np.allclose(out["post_out"], post, rtol=2e-6)
    assert np.allclose(out["comb_out"], comb, rtol=2e-5, atol=1e-7)
    li = truth.collapse_norm(f32(out["residual_out"]).astype(np.float64),
                             out["pre"].astype(np.float64), inp["gamma"], hidden, p.norm_eps)
    assert ulp_diff(out["layer_input"], truth.bf16_bits(li)).max() <= 1


@pytest.mark.parametrize("hidden,tp,m", [(8, 1, 2), (8, 8, 5), (5120, 4, 4)])
def test_end_to_end_within_parity_tolerances(oracle_lib, hidden, tp, m):
    inp = synth.make_inputs(hidden, tp, m, seed=7)
    p = oracle_lib.Problem(hidden, tp, m)
    out = oracle_lib.boundary(p, inp)
    ref = truth.boundary(p, inp)
    assert ulp_diff(out["reduced"], truth.bf16_bits(ref["reduced"])).max() <= 1
    assert ulp_diff(out["residual_out"], truth.bf16_bits(ref["residual_out"])).max() <= 2
    # upstream one-ulp BF16 flips move pre by ~1e-5 here (not ~1e-7 as between
    # two FP32 reductions), hence the wider cancellation floor
    ok = layer_input_ok(out["layer_input"], truth.bf16_bits(ref["layer_input"]),
                        out["residual_out"], out["pre"], inp["gamma"], floor=2.0 ** -4)
    assert ok.all()
    # End to end, the few upstream BF16 flips between the FP32 and FP64 paths
    # move the mixes by up to ~2e-4 at H = 5120 (each flip shifts a mix by
    # |fn| * ulp * rstd), and softmax turns that into a like relative change
    # of comb; the step-wise test above pins these steps to FP32 rounding.
    for name in ("pre", "post_out", "comb_out"):
        assert np.allclose(out[name], ref[name], rtol=5e-4, atol=1e-6), name


@pytest.mark.parametrize("tp,k,holes", [(1, 1, 0.0), (2, 3, 0.5), (8, 8, 0.0), (8, 8, 0.3)])
def test_moe_boundary_matches_fp64(oracle_lib, tp, k, holes):
    hidden, m = 64, 3
    inp = synth.make_inputs(hidden, tp, m, top_k=k, moe=True, seed=tp + k, holes=holes)
    p = oracle_lib.Problem(hidden, tp, m, top_k=k, rows_per_rank=m * k)
    out = oracle_lib.boundary(p, inp, moe=True)
    ref = truth.bf16_bits(truth.moe_fold(inp["routed"], inp["idx"], inp["weights"], inp["shared"]))
    assert ulp_diff(out["reduced"], ref).max() <= 1


def test_boundary_rejects_bad_route_index(oracle_lib):
    inp = synth.make_inputs(16, 2, 2, top_k=2, moe=True, seed=1)
    inp["idx"][1, 0, 1] = 4                                  # rows_per_rank = 4
    p = oracle_lib.Problem(16, 2, 2, top_k=2, rows_per_rank=4)
    with pytest.raises(ValueError):
        oracle_lib.boundary(p, inp, moe=True)


def test_token_ranges_compose(oracle_lib):
    # computing tokens in two ranges gives the same bits as one range
    inp = synth.make_inputs(256, 3, 6, seed=9)
    p = oracle_lib.Problem(256, 3, 6)
    whole = oracle_lib.boundary(p, inp, mxfp8_out=False)
    parts = oracle_lib.boundary(p, inp, t0=0, t1=2)
    oracle_lib.boundary(p, inp, t0=2, t1=6, outputs=parts)
    for name in whole:
        assert np.array_equal(whole[name], parts[name]), name
