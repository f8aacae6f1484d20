"""GPU parity: the CUDA path (through the C ABI) against the oracle on the
same seeded inputs, element by element, at every workload size and on the
edge cases (ragged slices and token tiles, tp = 1, H = 8, zero inputs,
MXFP8 padding rows, MoE routes a rank does not hold)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import compare, oracle_outputs, run_gpu, to_device, to_numpy
from mhc_residual_boundary_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Boundary():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from mhc_residual_boundary_gb300 import Boundary as B
    return B


def check(Boundary, hidden, tp, m, *, seed=0, moe=False, top_k=0, mxfp8=False, holes=0.0,
          capacity=None, mutate=None, bf16_weight=False, flags=None, **cfg):
    inp = synth.make_inputs(hidden, tp, m, top_k=top_k, moe=moe, seed=seed, holes=holes)
    if bf16_weight:
        # the GLM page's form of the weight, BF16 [24][4H], instead of hc_fn
        inp["hc_fn_bf16"] = synth.bf16_weight(inp.pop("hc_fn"))
    if mutate:
        mutate(inp)
    p = oracle.Problem(hidden, tp, m, top_k=top_k, rows_per_rank=m * top_k if moe else 0, **cfg)
    ref = oracle_outputs(p, inp, moe=moe, mxfp8=mxfp8)
    b = Boundary(hidden=hidden, tp=tp, max_num_tokens=capacity or m, top_k=top_k, mxfp8=mxfp8,
                 **(flags or {}), **cfg)
    try:
        got = run_gpu(b, inp, moe=moe, mxfp8=mxfp8)
        b.check_errors()
    finally:
        b.close()
    return compare(got, ref, inp, mxfp8=mxfp8)


def test_tiny(Boundary):
    check(Boundary, 5120, 4, 4)


@pytest.mark.parametrize("m", [1, 8, 32, 64])
def test_decode_sweep(Boundary, m):
    check(Boundary, 5120, 8, m, seed=m)


@pytest.mark.parametrize("m", [1 << i for i in range(10)])
def test_glm_style(Boundary, m):
    check(Boundary, 6144, 4, m, seed=100 + m)


def test_moe_finalize(Boundary):
    check(Boundary, 5120, 8, 256, moe=True, top_k=8)


@pytest.mark.parametrize("tp,k,holes,m", [(8, 8, 0.3, 37), (1, 1, 0.0, 5), (3, 5, 0.5, 70)])
def test_moe_routes_not_held(Boundary, tp, k, holes, m):
    check(Boundary, 512, tp, m, moe=True, top_k=k, holes=holes, seed=tp * 10 + k)


@pytest.mark.parametrize("hidden,tp,k,holes,m", [(256, 32, 3, 0.2, 9), (520, 5, 13, 0.3, 21), (128, 2, 64, 0.5, 4),
                                                 (1032, 16, 9, 0.1, 3)])
def test_moe_fold_shapes(Boundary, hidden, tp, k, holes, m):
    # the fold's layout: up to 32 ranks (four a warp), odd rank counts, route
    # counts past one batch and up to 64, and chunks of 128 fragments left
    # ragged (32, 65, 16 and 129 fragments a token row)
    check(Boundary, hidden, tp, m, moe=True, top_k=k, holes=holes, seed=hidden + tp + k)


def test_large_mxfp8(Boundary):
    rep = check(Boundary, 6144, 8, 4096, mxfp8=True, seed=4)
    print("large_mxfp8 report:", rep)


@pytest.mark.parametrize("hidden,tp,m", [(8, 1, 1), (8, 3, 9), (72, 2, 17), (520, 5, 33),
                                         (1000, 8, 300), (128, 1, 129),
                                         # more partials than one tensor-map box: CUDA-core stage kernel
                                         (1024, 12, 50),
                                         # the largest hidden size: one finish ring slot per CTA
                                         (16384, 8, 40)])
def test_ragged_shapes(Boundary, hidden, tp, m):
    check(Boundary, hidden, tp, m, seed=hidden + m)


@pytest.mark.parametrize("hidden,tp,m,mxfp8", [(6144, 4, 1, False), (6144, 4, 256, False), (5120, 8, 64, False),
                                               (520, 5, 33, False), (1000, 8, 300, False), (8, 1, 3, False),
                                               (2048, 4, 130, True)])
def test_bf16_weight(Boundary, hidden, tp, m, mxfp8):
    # the prenorm weight as BF16 [24][4H] ([GLM] fn): one BF16 term in the MMAs
    check(Boundary, hidden, tp, m, mxfp8=mxfp8, bf16_weight=True, seed=7 * m + hidden)


@pytest.mark.parametrize("hidden,tp,m,bf16", [(1032, 4, 3, False), (1032, 4, 5, True), (16384, 8, 8, False),
                                              (16384, 2, 8, True), (6144, 8, 8, False), (6144, 8, 9, False),
                                              (8, 1, 8, False), (136, 3, 7, True)])
def test_few_tokens(Boundary, hidden, tp, m, bf16):
    # up to 8 tokens, one unit a CTA: ragged last groups, both weight forms,
    # the largest width, one and nine tokens around a stage's eight
    check(Boundary, hidden, tp, m, bf16_weight=bf16, mxfp8=hidden % 128 == 0, seed=hidden + 3 * m)


@pytest.mark.parametrize("hidden,tp,m,bf16,mxfp8", [(1024, 16, 3, False, True), (512, 32, 1, False, False),
                                                   (2048, 12, 8, False, True), (4096, 9, 5, False, True),
                                                   (512, 8, 1, True, False), (776, 3, 6, False, False),
                                                   (7168, 8, 7, True, True)])
def test_one_kernel_shapes(Boundary, hidden, tp, m, bf16, mxfp8):
    # the cluster kernel for a few tokens: many partials a token (tp up to
    # 32, more than the tensor-core path takes; the BF16 weight is accepted
    # up to tp = 8), a width that is not a multiple of 32 (16-byte column
    # units), two tokens a cluster from five tokens, both weight forms
    check(Boundary, hidden, tp, m, bf16_weight=bf16, mxfp8=mxfp8, seed=hidden * 3 + tp + m)


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("m", range(1, 10))
def test_one_to_nine_tokens(Boundary, m, bf16):
    # the GLM shape in the one-kernel path's range (up to twelve tokens),
    # one to nine tokens, both weight forms
    check(Boundary, 6144, 4, m, bf16_weight=bf16, mxfp8=True, seed=31 * m + bf16)


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("hidden,tp,m", [(6144, 4, 10), (6144, 4, 12), (6144, 4, 13), (5120, 8, 11), (776, 3, 12)])
def test_ten_to_thirteen_tokens(Boundary, hidden, tp, m, bf16):
    # the top of the one-kernel path's range (two tokens a cluster, up to 12
    # tokens, an odd count leaving a cluster one token) and the stage and
    # finish kernels just beyond it
    check(Boundary, hidden, tp, m, bf16_weight=bf16, mxfp8=hidden % 128 == 0, seed=17 * m + hidden + bf16)


@pytest.mark.parametrize("hidden,tp,m,bf16", [(2048, 6, 1024, False), (2048, 3, 1024, False),
                                              (6144, 8, 512, True), (2048, 8, 1024, True),
                                              (5120, 8, 2000, False)])
def test_ring_wraps_many_times(Boundary, hidden, tp, m, bf16):
    # several units per CTA, so every ring slot is reused many times, at tp
    # values whose slot count is not a multiple of a unit's four stages; the
    # 2000-token case has more than 12 tokens an SM, where the finish kernel
    # runs two-slot CTAs, with a ragged share of tokens per CTA
    check(Boundary, hidden, tp, m, bf16_weight=bf16, seed=hidden + tp + m)


def test_bf16_weight_moe(Boundary):
    check(Boundary, 1024, 4, 60, moe=True, top_k=4, holes=0.2, bf16_weight=True, seed=17)


@pytest.mark.parametrize("m", [1, 127, 129, 300])
def test_mxfp8_padding_rows(Boundary, m):
    check(Boundary, 256, 2, m, mxfp8=True, seed=m)


def test_capacity_larger_than_call(Boundary):
    check(Boundary, 1024, 4, 40, capacity=1000)


def test_zero_and_negative_zero_inputs(Boundary):
    def zero(inp):
        inp["partials"][:] = 0x8000          # all -0: stage 1 must return +0
        inp["residual"][:, :, ::3] = 0
    check(Boundary, 256, 4, 6, mutate=zero)


def test_other_scalars(Boundary):
    check(Boundary, 640, 2, 20, sinkhorn_repeat=3, rms_eps=1e-3, hc_eps=0.01, post_mult=1.5,
          norm_eps=1e-2, seed=9)


@pytest.mark.parametrize("hidden,tp,m,bf16,moe", [(5120, 4, 4, False, False), (1024, 4, 6, True, False),
                                                  (6144, 8, 300, False, False),
                                                  (2048, 3, 1024, False, False), (6144, 4, 64, True, False),
                                                  (1024, 4, 60, False, True)])
def test_static_weight(Boundary, hidden, tp, m, bf16, moe):
    # the weight staged and split before the stage kernel waits for the
    # kernel ahead of it: same results
    check(Boundary, hidden, tp, m, bf16_weight=bf16, moe=moe, top_k=4 if moe else 0,
          mxfp8=hidden % 128 == 0, flags={"static_weight": True}, seed=hidden + m)


@pytest.mark.parametrize("m", [5, 48])
def test_static_weight_chained_calls_match(Boundary, m):
    # each call reads the previous call's residual_out, post_out and comb_out
    # on the same stream, while its kernel may start during the previous
    # call's last kernel: the chain gives the bits of the chain without the
    # early staging (5 tokens: the one-kernel path; 48: stage and finish)
    hidden, tp, calls = 2048, 4, 12
    inp = to_device(synth.make_inputs(hidden, tp, m, seed=21))
    results = {}
    for static in (False, True):
        b = Boundary(hidden=hidden, tp=tp, max_num_tokens=m, static_weight=static)
        cur, outs = dict(inp), []
        for _ in range(calls):
            o = b.empty_outputs(m, extras=True)
            b.run(cur, o)
            outs.append(o)
            cur = dict(cur)
            cur["residual"], cur["post"], cur["comb"] = o["residual_out"], o["post_out"], o["comb_out"]
        b.join()
        torch.cuda.synchronize()
        b.check_errors()
        results[static] = [to_numpy(o) for o in outs]
        b.close()
    for i, (a, c) in enumerate(zip(results[False], results[True])):
        for name in a:
            assert np.array_equal(a[name], c[name]), (i, name)


MIXES_PLACEMENTS = {"fused": {}, "side": {"side_mixes": True}, "sync": {"sync_mixes": True},
                    "static": {"static_weight": True}}


@pytest.mark.parametrize("m", [6, 50])
def test_mixes_placements_give_same_bits(Boundary, m):
    # post / Sinkhorn inside the boundary kernel (the one-kernel path at 6
    # tokens, the finish kernel at 50), in the side-stream kernel and in the
    # same kernel on the caller's stream take the same operations
    inp = synth.make_inputs(1024, 4, m, seed=3)
    outs = {}
    for name, flags in MIXES_PLACEMENTS.items():
        b = Boundary(hidden=1024, tp=4, max_num_tokens=m, **flags)
        outs[name] = run_gpu(b, inp)
        b.close()
    for name in outs["fused"]:
        for other in ("side", "sync", "static"):
            assert np.array_equal(outs["fused"][name], outs[other][name]), (name, other)


@pytest.mark.parametrize("placement", sorted(MIXES_PLACEMENTS))
def test_back_to_back_calls_chain_mixes(Boundary, placement):
    # call 2 reads call 1's post_out / comb_out on the same stream: with the
    # side-stream kernel the automatic join must order it after that kernel
    hidden, tp, m = 2048, 4, 64
    inp = synth.make_inputs(hidden, tp, m, seed=5)
    b = Boundary(hidden=hidden, tp=tp, max_num_tokens=m, **MIXES_PLACEMENTS[placement])
    dev = to_device(inp)
    o1 = b.empty_outputs(m, extras=True)
    b.run(dev, o1)
    dev2 = dict(dev)
    dev2["post"], dev2["comb"] = o1["post_out"], o1["comb_out"]
    dev2["residual"] = o1["residual_out"]
    o2 = b.empty_outputs(m, extras=True)
    b.run(dev2, o2)
    b.join()
    torch.cuda.synchronize()
    got1, got2 = to_numpy(o1), to_numpy(o2)
    b.close()
    p = oracle.Problem(hidden, tp, m)
    ref1 = oracle.boundary(p, inp)
    inp2 = dict(inp)
    inp2["post"], inp2["comb"], inp2["residual"] = got1["post_out"], got1["comb_out"], got1["residual_out"]
    ref2 = oracle.boundary(p, inp2)
    compare(got1, ref1, inp)
    compare(got2, ref2, inp2)


@pytest.mark.parametrize("m,flags", [(33, {}), (1000, {}), (2048, {"side_mixes": True}), (700, {"static_weight": True})])
def test_run_host_matches_run(Boundary, m, flags):
    # one chunk (33 tokens) and the pipelined token chunks: 1000 tokens as
    # 384 + 384 + 232, 2048 as eight 256-token chunks with the side-stream
    # mixes kernel, 700 as 384 + 316; the same bits as the device-buffer call
    hidden, tp = 1024, 4
    inp = synth.make_inputs(hidden, tp, m, seed=8)
    b = Boundary(hidden=hidden, tp=tp, max_num_tokens=max(m, 64), host_staging=True, mxfp8=True, **flags)
    dev_out = run_gpu(b, inp, mxfp8=True)
    host_in = {k: v.pin_memory() for k, v in to_device(inp, device="cpu").items()}
    host_out = b.empty_outputs(m, extras=True, mxfp8=True, device="cpu", pin_memory=True)
    b.run_host(host_in, host_out)
    b.close()
    got = to_numpy(host_out)
    for name in dev_out:
        assert np.array_equal(got[name], dev_out[name]), name


def test_bad_route_index_is_reported_and_skipped(Boundary):
    hidden, tp, m, k = 256, 2, 4, 3
    inp = synth.make_inputs(hidden, tp, m, top_k=k, moe=True, seed=2)
    bad = inp["idx"].copy()
    bad[1, 2, 0] = 10_000
    b = Boundary(hidden=hidden, tp=tp, max_num_tokens=m, top_k=k)
    got_inp = dict(inp)
    got_inp["idx"] = bad
    got = run_gpu(b, got_inp, moe=True)
    with pytest.raises(Exception, match="route index"):
        b.check_errors()
    b.check_errors()            # the flag is cleared once reported
    b.close()
    dropped = inp["idx"].copy()
    dropped[1, 2, 0] = -1
    ref_inp = dict(inp)
    ref_inp["idx"] = dropped
    ref = oracle.boundary(oracle.Problem(hidden, tp, m, top_k=k, rows_per_rank=m * k), ref_inp, moe=True)
    compare(got, ref, ref_inp)
