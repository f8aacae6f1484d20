"""The seeded input generator against its stated recipe: determinism, one
stream per tensor, the BF16 storage rounding, the distributions' parameters,
and the structure of the incoming mixes and of the MoE routes."""
import numpy as np
import pytest
import torch

from mhc_residual_boundary_gb300 import synth


def f32(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def test_same_seed_same_bits_other_seed_other_bits():
    a = synth.make_inputs(256, 3, 7, seed=5)
    b = synth.make_inputs(256, 3, 7, seed=5)
    c = synth.make_inputs(256, 3, 7, seed=6)
    assert a.keys() == b.keys()
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    for k in ("partials", "residual", "post", "comb", "hc_fn", "base", "gamma"):
        assert not np.array_equal(a[k], c[k]), k


def test_a_tensor_does_not_depend_on_the_others():
    dense = synth.make_inputs(128, 2, 5, seed=1)
    moe = synth.make_inputs(128, 2, 5, seed=1, moe=True, top_k=3, holes=0.5)
    for k in ("residual", "post", "comb", "hc_fn", "base", "gamma"):
        assert np.array_equal(dense[k], moe[k]), k


def test_bf16_storage_rounds_to_nearest_even_like_torch():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(1 << 16).astype(np.float32) * np.float32(3.0)
    ties = (np.arange(1 << 12, dtype=np.uint32) << 16 | 0x8000).view(np.float32)   # exact halfway cases
    for v in (x, ties[np.isfinite(ties)]):
        want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(synth.bf16_bits(v), want)


def test_distribution_parameters():
    H, tp, m = 1024, 4, 64
    inp = synth.make_inputs(H, tp, m, seed=3)
    assert inp["partials"].dtype == np.uint16 and inp["partials"].shape == (tp, m, H)
    assert f32(inp["partials"]).std() == pytest.approx(0.05, rel=0.02)
    assert abs(f32(inp["partials"]).mean()) < 0.002
    assert f32(inp["residual"]).std() == pytest.approx(1.0, rel=0.02)
    assert inp["hc_fn"].dtype == np.float32 and inp["hc_fn"].shape == (4 * H, 24)
    assert inp["hc_fn"].std() == pytest.approx(1 / np.sqrt(4 * H), rel=0.02)
    g = f32(inp["gamma"])
    assert g.mean() == pytest.approx(1.0, abs=0.02) and g.std() == pytest.approx(0.1, rel=0.15)
    assert np.array_equal(inp["scale"], np.ones(3, np.float32))
    assert inp["base"].shape == (24,) and 0.03 < inp["base"].std() < 0.2


def test_incoming_mixes():
    inp = synth.make_inputs(64, 2, 500, seed=4, post_mult=2.0)
    post, comb = inp["post"], inp["comb"].astype(np.float64)
    assert post.shape == (500, 4) and (post > 0.04).all() and (post < 1.96).all()
    assert comb.shape == (500, 4, 4) and (comb >= 0).all()
    assert np.abs(comb.sum(axis=1) - 1).max() < 1e-6          # over sources
    assert np.abs(comb.sum(axis=2) - 1).max() < 1e-6          # over targets
    assert len({tuple(np.round(c, 6).ravel()) for c in comb}) == 500   # no two tokens alike


def test_moe_routes():
    m, k, tp = 40, 6, 3
    full = synth.make_inputs(64, tp, m, seed=8, moe=True, top_k=k)
    assert full["idx"].shape == (tp, m, k) and full["idx"].dtype == np.int32
    for r in range(tp):        # every rank holds every route exactly once
        assert np.array_equal(np.sort(full["idx"][r].ravel()), np.arange(m * k))
    assert not np.array_equal(full["idx"][0], full["idx"][1])
    w = full["weights"].astype(np.float64)
    assert (w > 0).all() and np.abs(w.sum(axis=1) - 1).max() < 1e-6
    assert full["routed"].shape == (tp, m * k, 64) and full["shared"].shape == (tp, m, 64)
    holey = synth.make_inputs(64, tp, m, seed=8, moe=True, top_k=k, holes=0.3)
    missing = holey["idx"] == -1
    assert 0.2 < missing.mean() < 0.4
    assert np.array_equal(holey["idx"][~missing], full["idx"][~missing])   # holes only remove routes
    with pytest.raises(ValueError):
        synth.make_inputs(64, tp, m, moe=True, top_k=0)


def test_bf16_weight_is_the_transposed_draw():
    inp = synth.make_inputs(64, 1, 1, seed=2)
    w = synth.bf16_weight(inp["hc_fn"])
    assert w.shape == (24, 256)
    assert np.array_equal(w, synth.bf16_bits(inp["hc_fn"].T))
    assert np.abs(f32(w) - inp["hc_fn"].T).max() <= np.abs(inp["hc_fn"]).max() * 2.0 ** -8


def test_carried_pre_of_the_consumer():
    w = synth.WORKLOADS["consume"][0]
    pre = synth.inputs_for(w)["pre"]
    assert pre.shape == (w.m, 4) and (pre >= 0.05).all() and (pre < 1.0).all()
    small = synth.Workload("residual_only", 256, 2, 3, consume=True, residual_only=True)
    assert "pre" not in synth.inputs_for(small)


def test_named_workloads():
    sizes = {name: [(w.hidden, w.tp, w.m, w.top_k, w.mxfp8) for w in ws] for name, ws in synth.WORKLOADS.items()}
    assert sizes["tiny"] == [(5120, 4, 4, 0, False)]
    assert sizes["decode"] == [(5120, 8, m, 0, False) for m in (1, 8, 32, 64)]
    assert sizes["glm"] == [(6144, 4, 1 << i, 0, False) for i in range(10)]
    assert sizes["moe"] == [(5120, 8, 256, 8, False)]
    assert sizes["large_mxfp8"] == [(6144, 8, 4096, 0, True)]
