"""Pins of the oracle's delayed-mHC consumer ([DSV] AllReduceMHC.__call__ /
finalize with a carried pre-mix, and residual_only), no GPU: it is the
boundary without the GEMV, so with the boundary's own pre it reproduces the
boundary's streams and layer input bit for bit; a one-hot pre makes the
layer input the RMSNorm of one stream."""
import numpy as np
import pytest

from mhc_residual_boundary_gb300 import synth

HC = 4


def f32(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("hidden,tp,m,moe,mxfp8", [(256, 4, 5, False, False), (512, 2, 130, False, True),
                                                  (128, 3, 7, True, False)])
def test_consume_with_the_boundarys_pre_matches_the_boundary(oracle_lib, hidden, tp, m, moe, mxfp8):
    top_k = 3 if moe else 0
    inp = synth.make_inputs(hidden, tp, m, top_k=top_k, moe=moe, seed=hidden + m)
    p = oracle_lib.Problem(hidden, tp, m, top_k=top_k, rows_per_rank=m * top_k if moe else 0)
    full = oracle_lib.boundary(p, inp, moe=moe, mxfp8_out=mxfp8)
    got = oracle_lib.consume(p, inp, full["pre"], moe=moe, mxfp8_out=mxfp8)
    for name in ("residual_out", "layer_input", "reduced"):
        assert np.array_equal(got[name], full[name]), name
    if mxfp8:
        assert np.array_equal(got["mx_values"], full["mx_values"])
        assert np.array_equal(got["mx_scales"], full["mx_scales"])


def test_residual_only_writes_the_streams_alone(oracle_lib):
    hidden, tp, m = 256, 4, 9
    inp = synth.make_inputs(hidden, tp, m, seed=3)
    p = oracle_lib.Problem(hidden, tp, m)
    full = oracle_lib.boundary(p, inp)
    got = oracle_lib.consume(p, inp, np.zeros((m, HC), np.float32), residual_only=True)
    assert set(got) == {"residual_out", "reduced"}
    assert np.array_equal(got["residual_out"], full["residual_out"])


@pytest.mark.parametrize("j", range(HC))
def test_one_hot_pre_normalises_one_stream(oracle_lib, j):
    hidden, tp, m = 384, 2, 6
    inp = synth.make_inputs(hidden, tp, m, seed=20 + j)
    p = oracle_lib.Problem(hidden, tp, m, norm_eps=1e-6)
    pre = np.zeros((m, HC), np.float32)
    pre[:, j] = 1.0
    got = oracle_lib.consume(p, inp, pre)
    new = f32(got["residual_out"][:, j, :]).astype(np.float64)     # c = new_j exactly
    inv = 1.0 / np.sqrt((new * new).sum(axis=1, keepdims=True) / hidden + 1e-6)
    want = new * inv * f32(inp["gamma"]).astype(np.float64)
    out = f32(got["layer_input"]).astype(np.float64)
    # within one BF16 rounding of the FP64 value (2^-8 relative)
    assert np.all(np.abs(out - want) <= np.abs(want) * 2.0 ** -8 + 1e-30)
