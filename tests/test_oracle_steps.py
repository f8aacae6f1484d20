"""Pins of the oracle's steps against hand-worked values, closed forms,
special cases and invariants (no GPU).

Each test names the property it pins; together they are chosen so that a
dropped term, a wrong index, a transposed operand or a misplaced epsilon in
any step of the oracle fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

from conftest import golden_lines
from mhc_residual_boundary_gb300 import synth
from oracle import truth

HC, MIX = 4, 24


def bits(x):
    """BF16 patterns of FP32 values, rounded by PyTorch's own cast."""
    x = np.ascontiguousarray(x, np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f32(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def ulp_diff(a, b):
    """|a - b| in BF16 ulps (order-preserving integer map of the patterns)."""
    def key(x):
        x = np.asarray(x, np.uint16).astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7fff), 0x8000 + x)
    return np.abs(key(a) - key(b))


# ------------------------------------------------------------------ stage 1
def test_stage1_golden(oracle_lib):
    for lhs, rhs in golden_lines("stage1_rank_order.txt"):
        parts = np.array([int(h, 16) for h in lhs], np.uint16).reshape(len(lhs), 1, 1)
        y = oracle_lib.stage1(np.repeat(parts, 8, axis=2))
        assert (y == int(rhs, 16)).all(), (lhs, hex(int(y[0, 0])))


def test_stage1_tp1_is_identity_on_every_pattern(oracle_lib):
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = np.isfinite(f32(pats)) | np.isinf(f32(pats))
    pats = pats[finite & ~np.isnan(f32(pats))]
    y = oracle_lib.stage1(pats.reshape(1, 1, -1))[0]
    expect = np.where(pats == 0x8000, 0, pats)          # -0 + +0 start = +0
    assert np.array_equal(y, expect)


@pytest.mark.parametrize("tp", [2, 3, 4, 8])
def test_stage1_within_one_ulp_of_exact_sum(oracle_lib, tp):
    inp = synth.make_inputs(512, tp, 16, seed=tp)
    y = oracle_lib.stage1(inp["partials"])
    exact = f32(inp["partials"]).astype(np.float64).sum(axis=0)   # exact for these ranges
    ref = truth.bf16_bits(truth.round_bf16(exact))
    d = ulp_diff(y, ref)
    assert d.max() <= 1 and (d == 0).mean() > 0.99


def test_stage1_is_in_rank_order(oracle_lib):
    # reversing the ranks must change some results (the sum is not
    # associative in FP32); a sort or tree would hide that.
    a = np.array([[[0x4b80]], [[0x3f80]], [[0xcb80]]], np.uint16)
    assert oracle_lib.stage1(a)[0, 0] != oracle_lib.stage1(a[::-1].copy())[0, 0]


# ---------------------------------------------------------------- MoE fold
def _moe(hidden=64, tp=3, m=5, k=4, seed=0, holes=0.0):
    return synth.make_inputs(hidden, tp, m, top_k=k, moe=True, seed=seed, holes=holes)


def test_moe_all_routes_missing_gives_shared_sum(oracle_lib):
    inp = _moe()
    idx = np.full_like(inp["idx"], -1)
    y = oracle_lib.moe_fold(inp["routed"], idx, inp["weights"], inp["shared"])
    assert np.array_equal(y, oracle_lib.stage1(inp["shared"]))


def test_moe_single_unit_route_is_row_plus_shared(oracle_lib):
    inp = _moe()
    idx = np.full_like(inp["idx"], -1)
    idx[:, :, 2] = inp["idx"][:, :, 2]
    w = np.zeros_like(inp["weights"])
    w[:, 2] = 1.0
    y = oracle_lib.moe_fold(inp["routed"], idx, w, inp["shared"])
    rows = np.stack([f32(inp["routed"][r][idx[r, :, 2]]) for r in range(idx.shape[0])])
    contrib = bits(rows + f32(inp["shared"]))                 # one FP32 add, BF16 rounding
    assert np.array_equal(y, oracle_lib.stage1(contrib))


def test_moe_fma_golden(oracle_lib):
    for lhs, rhs in golden_lines("fma_reading.txt"):
        a, wa, b, wb = lhs
        fused, separate = [int(x, 16) for x in rhs.split(";")]
        routed = np.array([[[int(a, 16)] * 8, [int(b, 16)] * 8]], np.uint16)
        idx = np.array([[[0, 1]]], np.int32)
        w = np.array([[np.uint32(int(wa, 16)).view(np.float32),
                       np.uint32(int(wb, 16)).view(np.float32)]], np.float32)
        shared = np.zeros((1, 1, 8), np.uint16)
        y = oracle_lib.moe_fold(routed, idx, w, shared)
        assert (y == fused).all() and fused != separate


def test_moe_weights_are_not_shared_between_routes(oracle_lib):
    # swapping the weights of two routes changes the result (pins w[t, k]
    # against a transposed or broadcast weight index)
    inp = _moe()
    y0 = oracle_lib.moe_fold(inp["routed"], inp["idx"], inp["weights"], inp["shared"])
    w = inp["weights"][:, ::-1].copy()
    y1 = oracle_lib.moe_fold(inp["routed"], inp["idx"], w, inp["shared"])
    assert (y0 != y1).mean() > 0.5


@pytest.mark.parametrize("holes", [0.0, 0.4])
def test_moe_close_to_fp64(oracle_lib, holes):
    inp = _moe(hidden=256, tp=4, m=6, k=8, seed=3, holes=holes)
    y = oracle_lib.moe_fold(inp["routed"], inp["idx"], inp["weights"], inp["shared"])
    ref = truth.bf16_bits(truth.moe_fold(inp["routed"], inp["idx"], inp["weights"], inp["shared"]))
    d = ulp_diff(y, ref)
    assert d.max() <= 1 and (d == 0).mean() > 0.97


# ---------------------------------------------------------------- post-mix
def test_post_mix_one_hot_post_passes_y(oracle_lib):
    inp = synth.make_inputs(64, 2, 3, seed=5)
    y = oracle_lib.stage1(inp["partials"])
    for j in range(HC):
        post = np.zeros((3, HC), np.float32)
        post[:, j] = 1.0
        new = oracle_lib.post_mix(y, inp["residual"], post, np.zeros((3, HC, HC), np.float32))
        assert np.array_equal(new[:, j], y)
        others = [i for i in range(HC) if i != j]
        assert (f32(new[:, others]) == 0).all()     # +-0: 0 * y keeps the sign of y


def test_post_mix_comb_is_source_by_target(oracle_lib):
    inp = synth.make_inputs(64, 2, 3, seed=6)
    y = oracle_lib.stage1(inp["partials"])
    perm = [2, 0, 3, 1]                      # source k feeds target perm[k]
    comb = np.zeros((3, HC, HC), np.float32)
    for k, j in enumerate(perm):
        comb[:, k, j] = 1.0
    new = oracle_lib.post_mix(y, inp["residual"], np.zeros((3, HC), np.float32), comb)
    for k, j in enumerate(perm):
        assert np.array_equal(new[:, j], inp["residual"][:, k])


def test_post_mix_fma_golden(oracle_lib):
    for lhs, rhs in golden_lines("fma_reading.txt"):
        a, wa, b, wb = lhs
        fused = int(rhs.split(";")[0], 16)
        res = np.zeros((1, HC, 8), np.uint16)
        res[0, 0], res[0, 1] = int(a, 16), int(b, 16)
        comb = np.zeros((1, HC, HC), np.float32)
        comb[0, 0, 3] = np.uint32(int(wa, 16)).view(np.float32)
        comb[0, 1, 3] = np.uint32(int(wb, 16)).view(np.float32)
        new = oracle_lib.post_mix(np.zeros((1, 8), np.uint16), res, np.zeros((1, HC), np.float32), comb)
        assert (new[0, 3] == fused).all()


def test_post_mix_close_to_fp64(oracle_lib):
    inp = synth.make_inputs(512, 4, 8, seed=7)
    y = oracle_lib.stage1(inp["partials"])
    new = oracle_lib.post_mix(y, inp["residual"], inp["post"], inp["comb"])
    ref = truth.bf16_bits(truth.post_mix(f32(y).astype(np.float64), inp["residual"], inp["post"], inp["comb"]))
    d = ulp_diff(new, ref)
    assert d.max() <= 1 and (d == 0).mean() > 0.99


# ---------------------------------------------------------- GEMV and mixes
def test_gemv_one_hot_columns_pick_elements(oracle_lib):
    hidden, m = 40, 3
    inp = synth.make_inputs(hidden, 1, m, seed=8)
    streams = inp["residual"]
    for j, h, i in ((0, 0, 0), (3, 39, 23), (2, 17, 5), (1, 5, 12)):
        fn = np.zeros((HC * hidden, MIX), np.float32)
        fn[j * hidden + h, i] = 1.0
        raw, _ = oracle_lib.prenorm_gemv(streams, fn)
        assert np.array_equal(raw[:, i], f32(streams[:, j, h]))
        assert (np.delete(raw, i, axis=1) == 0).all()


def test_gemv_matches_float64_matmul(oracle_lib):
    inp = synth.make_inputs(256, 1, 7, seed=9)
    raw, ss = oracle_lib.prenorm_gemv(inp["residual"], inp["hc_fn"])
    flat = f32(inp["residual"]).reshape(7, -1).astype(np.float64)
    ref = np.matmul(flat, inp["hc_fn"].astype(np.float64))
    assert np.allclose(raw, ref, rtol=1e-6, atol=1e-6)
    assert np.allclose(ss, np.einsum("ij,ij->i", flat, flat), rtol=1e-6)


def test_gemv_bf16_weight_one_hot_pins_its_layout(oracle_lib):
    # fn is [24][4H]: a one at row i, column j*H + h selects stream j, column h
    # for output i (a transposed or stream/column-swapped read fails)
    hidden, m = 40, 3
    inp = synth.make_inputs(hidden, 1, m, seed=8)
    streams = inp["residual"]
    for j, h, i in ((0, 0, 0), (3, 39, 23), (2, 17, 5), (1, 5, 12)):
        fn = np.zeros((MIX, HC * hidden), np.uint16)
        fn[i, j * hidden + h] = 0x3F80          # BF16 1.0
        raw, _ = oracle_lib.prenorm_gemv_bf16(streams, fn)
        assert np.array_equal(raw[:, i], f32(streams[:, j, h]))
        assert (np.delete(raw, i, axis=1) == 0).all()


def test_gemv_bf16_weight_matches_float64_matmul(oracle_lib):
    inp = synth.make_inputs(256, 1, 7, seed=9)
    fn = bits(inp["hc_fn"].T)                    # [24][4H] BF16
    raw, ss = oracle_lib.prenorm_gemv_bf16(inp["residual"], fn)
    flat = f32(inp["residual"]).reshape(7, -1).astype(np.float64)
    ref = np.matmul(flat, f32(fn).astype(np.float64).T)
    assert np.allclose(raw, ref, rtol=1e-6, atol=1e-6)
    assert np.allclose(ss, np.einsum("ij,ij->i", flat, flat), rtol=1e-6)
    # the same weights widened to FP32 [4H][24] give the same bits
    raw32, ss32 = oracle_lib.prenorm_gemv(inp["residual"], np.ascontiguousarray(f32(fn).T))
    assert np.array_equal(raw, raw32) and np.array_equal(ss, ss32)


def test_mixes_rms_uses_all_four_streams(oracle_lib):
    # new = c everywhere, fn one-hot: raw = c, ss = 4H c^2, so
    # mixes = c / sqrt(c^2 + eps): +-1 up to eps, whatever H and c.
    for hidden, c in ((8, 0.5), (64, -3.0), (512, 0.03125)):
        raw = np.zeros((1, MIX), np.float32)
        raw[0, 7] = c
        ss = np.array([HC * hidden * c * c], np.float32)
        mixes, _ = oracle_lib.mixes_and_pre(raw, ss, np.ones(3, np.float32),
                                            np.zeros(MIX, np.float32), hidden)
        assert mixes[0, 7] == pytest.approx(math.copysign(1.0, c) / math.sqrt(1 + 1e-6 / c ** 2), rel=1e-6)


def test_pre_closed_form_when_fn_is_zero(oracle_lib):
    inp = synth.make_inputs(64, 1, 2, seed=10)
    raw, ss = oracle_lib.prenorm_gemv(inp["residual"], np.zeros((HC * 64, MIX), np.float32))
    assert (raw == 0).all()
    base = inp["base"]
    mixes, pre = oracle_lib.mixes_and_pre(raw, ss, inp["scale"], base, 64, hc_eps=1e-3)
    for j in range(HC):
        assert pre[0, j] == pytest.approx(1 / (1 + math.exp(-base[j])) + 1e-3, rel=1e-6)


def test_pre_uses_scale0_and_base_head(oracle_lib):
    raw = np.random.default_rng(11).standard_normal((4, MIX)).astype(np.float32)
    ss = np.full((4,), 64 * HC, np.float32)                  # rstd = 1/sqrt(1 + eps)
    base = np.arange(MIX, dtype=np.float32) / 10
    scale = np.array([0.0, 5.0, 7.0], np.float32)
    _, pre = oracle_lib.mixes_and_pre(raw, ss, scale, base, 64, hc_eps=0.0)
    assert np.allclose(pre, 1 / (1 + np.exp(-base[:HC])), rtol=1e-6)
    scale = np.array([2.0, 0.0, 0.0], np.float32)
    mixes, pre = oracle_lib.mixes_and_pre(raw, ss, scale, base, 64, hc_eps=0.0)
    assert np.allclose(pre, 1 / (1 + np.exp(-(2 * raw[:, :HC] / np.sqrt(1 + 1e-6) + base[:HC]))), rtol=2e-6)


def test_pre_and_post_ranges(oracle_lib):
    inp = synth.make_inputs(512, 4, 16, seed=12)
    p = oracle_lib.Problem(512, 4, 16, hc_eps=1e-6, post_mult=2.0)
    out = oracle_lib.boundary(p, inp)
    assert ((out["pre"] - 1e-6 > 0) & (out["pre"] - 1e-6 < 1)).all()
    assert ((out["post_out"] > 0) & (out["post_out"] < 2.0)).all()


def test_post_closed_form(oracle_lib):
    base = np.linspace(-1, 1, MIX).astype(np.float32)
    mixes = np.random.default_rng(13).standard_normal((3, MIX)).astype(np.float32)
    post = oracle_lib.post_from_mixes(mixes, np.array([1, 0, 1], np.float32), base, post_mult=3.0)
    assert np.allclose(post, 3.0 / (1 + np.exp(-base[HC:2 * HC])), rtol=1e-6)
    post = oracle_lib.post_from_mixes(mixes, np.array([0, 0.5, 0], np.float32), base, post_mult=2.0)
    assert np.allclose(post, 2.0 / (1 + np.exp(-(0.5 * mixes[:, HC:2 * HC] + base[HC:2 * HC]))), rtol=1e-6)


# ----------------------------------------------------------------- Sinkhorn
def _sk(mixes, base, eps, repeat, scale=(1, 1, 1)):
    import oracle
    return oracle.sinkhorn(np.asarray(mixes, np.float32), np.asarray(scale, np.float32),
                                         np.asarray(base, np.float32), hc_eps=eps, repeat=repeat)


@pytest.mark.parametrize("repeat", [1, 2, 3, 20])
def test_sinkhorn_uniform_logits_closed_form(oracle_lib, repeat):
    eps = 0.01
    x = 0.25 + eps                                     # softmax of equal logits, plus eps
    for it in range(repeat):
        if it > 0:
            x = x / (4 * x + eps)                      # row step from the second round on
        x = x / (4 * x + eps)                          # column step
    c = _sk(np.zeros((1, MIX)), np.zeros(MIX), eps, repeat)
    assert np.allclose(c, x, rtol=2e-7)


def test_sinkhorn_rank_one_logits_closed_form(oracle_lib):
    a = np.array([0.3, -1.2, 2.0, 0.1])
    b = np.array([-0.5, 0.7, 1.1, -2.0])
    logits = (a[:, None] + b[None, :]).reshape(-1)
    mixes = np.zeros((1, MIX))
    mixes[0, 8:] = logits
    for eps, repeat in ((0.0, 1), (0.0, 5), (0.05, 4)):
        u = np.exp(b - b.max()) / np.exp(b - b.max()).sum() + eps   # every row equals u
        for it in range(repeat):
            if it > 0:
                u = u / (u.sum() + eps)
            u = u / (4 * u + eps)
        c = _sk(mixes, np.zeros(MIX), eps, repeat)[0]
        assert np.allclose(c, np.broadcast_to(u, (4, 4)), rtol=3e-7, atol=1e-8)
        if eps == 0.0:
            assert np.allclose(c, 0.25, rtol=3e-7)


def test_sinkhorn_doubly_stochastic_on_seeded_inputs(oracle_lib):
    inp = synth.make_inputs(5120, 4, 4, seed=0)
    out = oracle_lib.boundary(oracle_lib.Problem(5120, 4, 4), inp)
    c = out["comb_out"].astype(np.float64)
    assert np.abs(c.sum(axis=1) - 1).max() < 1e-5            # columns
    assert np.abs(c.sum(axis=2) - 1).max() < 1e-5            # rows
    assert (c > 0).all()


def test_sinkhorn_equivariance_and_shift(oracle_lib):
    rng = np.random.default_rng(14)
    mixes = rng.standard_normal((1, MIX)).astype(np.float32)
    base = (rng.standard_normal(MIX) * 0.1).astype(np.float32)
    c = _sk(mixes, base, 1e-6, 20)[0]
    rp, cp = [3, 1, 0, 2], [1, 2, 3, 0]
    m2, b2 = mixes.copy(), base.copy()
    m2[0, 8:] = mixes[0, 8:].reshape(4, 4)[rp][:, cp].reshape(-1)
    b2[8:] = base[8:].reshape(4, 4)[rp][:, cp].reshape(-1)
    c2 = _sk(m2, b2, 1e-6, 20)[0]
    assert np.allclose(c2, c[rp][:, cp], rtol=2e-6)
    m3 = mixes.copy()
    m3[0, 8:12] += 3.0                                   # shift one row's logits
    assert np.allclose(_sk(m3, base, 1e-6, 20)[0], c, rtol=2e-5)
    # scale[2] = 0: logits are the comb biases alone
    assert np.allclose(_sk(mixes, base, 1e-6, 20, (1, 1, 0))[0], _sk(np.zeros_like(mixes), base, 1e-6, 20)[0])


# ------------------------------------------------------- collapse and norm
def test_collapse_single_stream_closed_form(oracle_lib):
    inp = synth.make_inputs(256, 1, 3, seed=15)
    pre = np.zeros((3, HC), np.float32)
    pre[:, 2] = 1.0
    out = oracle_lib.collapse_norm(inp["residual"], pre, inp["gamma"], norm_eps=1e-6)
    s = f32(inp["residual"][:, 2]).astype(np.float64)
    inv = 1 / np.sqrt((s * s).sum(axis=1) / 256 + 1e-6)
    ref = truth.bf16_bits(truth.round_bf16(s * inv[:, None] * f32(inp["gamma"])[None, :]))
    assert ulp_diff(out, ref).max() <= 1


def test_collapse_unit_rms_and_gamma(oracle_lib):
    inp = synth.make_inputs(1024, 1, 4, seed=16)
    out = oracle_lib.boundary(oracle_lib.Problem(1024, 1, 4), inp)
    ones = np.full(1024, 0x3F80, np.uint16)
    twos = np.full(1024, 0x4000, np.uint16)
    a = oracle_lib.collapse_norm(out["residual_out"], out["pre"], ones)
    b = oracle_lib.collapse_norm(out["residual_out"], out["pre"], twos)
    rms = np.sqrt((f32(a).astype(np.float64) ** 2).mean(axis=1))
    assert np.allclose(rms, 1.0, atol=3e-3)
    assert np.array_equal(f32(b), 2 * f32(a))


def test_collapse_equal_pre(oracle_lib):
    inp = synth.make_inputs(128, 1, 2, seed=17)
    pre = np.full((2, HC), 0.375, np.float32)
    ones = np.full(128, 0x3F80, np.uint16)
    out = oracle_lib.collapse_norm(inp["residual"], pre, ones)
    c = truth.round_bf16(0.375 * f32(inp["residual"]).astype(np.float64).sum(axis=1))
    inv = 1 / np.sqrt((c * c).sum(axis=1) / 128 + 1e-6)
    ref = truth.bf16_bits(truth.round_bf16(c * inv[:, None]))
    assert ulp_diff(out, ref).max() <= 2


# -------------------------------------------------------------------- MXFP8
def test_mxfp8_golden_blocks(oracle_lib):
    for lhs, rhs in golden_lines("mxfp8_blocks.txt"):
        first = int(lhs[0], 16)
        rest = int(lhs[1], 16) if len(lhs) > 1 else first
        expect = [int(x, 16) for x in rhs.split()]
        row = np.full((1, 128), rest, np.uint16)
        row[0, 0] = first
        values, scales = oracle_lib.mxfp8(row)
        assert scales[oracle_lib.swizzle_128x4(0, 0, 4)] == expect[0]
        assert values[0, 0] == expect[1]
        assert (values[0, 1:32] == expect[-1]).all()


def test_mxfp8_dequantises_within_e4m3_precision(oracle_lib):
    inp = synth.make_inputs(256, 2, 130, seed=18)
    x = oracle_lib.stage1(inp["partials"])
    values, scales = oracle_lib.mxfp8(x)
    deq = torch.from_numpy(values).view(torch.float8_e4m3fn).double().numpy()
    for t in (0, 1, 77, 129):
        for b in range(256 // 32):
            e = int(scales[oracle_lib.swizzle_128x4(t, b, 8)])
            got = deq[t, b * 32:(b + 1) * 32] * 2.0 ** (e - 127)
            ref = f32(x[t, b * 32:(b + 1) * 32]).astype(np.float64)
            amax = np.abs(ref).max()
            # E4M3 keeps 3 fraction bits; subnormals keep an absolute step
            assert np.all(np.abs(got - ref) <= np.maximum(np.abs(ref) * 2 ** -4, amax * 2 ** -9 / 448 * 4))


def test_mxfp8_padding_rows_are_zero_and_rest_written(oracle_lib):
    inp = synth.make_inputs(512, 1, 130, seed=19)
    values, scales = oracle_lib.mxfp8(inp["partials"][0])
    cols = 512 // 32
    written = np.zeros_like(scales, bool)
    for r in range(256):
        for c in range(cols):
            i = oracle_lib.swizzle_128x4(r, c, cols)
            written[i] = True
            if r >= 130:
                assert scales[i] == 0
    assert written.all() and (scales != 0xAB).all()
