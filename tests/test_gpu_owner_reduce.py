"""The two-shot reduction, emulated on one GPU (MHC_FLAG_OWNER_REDUCE: an
owner-reduce kernel sums each token's partials, token t's owner being rank
t % tp, and the boundary takes the sums as its one partial; [DSV] module
text on the BT protocol), gives the same bits as the direct stage-1 sum,
on the boundary and on the delayed-mHC consumer, and matches the oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import compare, oracle_outputs, run_gpu
from mhc_residual_boundary_gb300 import synth
from test_gpu_consume import run_consume

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def Boundary():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from mhc_residual_boundary_gb300 import Boundary as B
    return B


@pytest.mark.parametrize("hidden,tp,m,mxfp8", [(6144, 4, 256, False), (5120, 8, 33, True), (520, 3, 7, False),
                                               (8, 1, 1, False), (2048, 5, 131, True),
                                               # more partials than the tensor-map kernel takes
                                               (1024, 12, 50, False), (2048, 32, 9, True)])
def test_owner_reduce_same_bits(Boundary, hidden, tp, m, mxfp8):
    inp = synth.make_inputs(hidden, tp, m, seed=hidden + tp + m)
    outs = {}
    for owner in (False, True):
        b = Boundary(hidden=hidden, tp=tp, max_num_tokens=m, mxfp8=mxfp8, owner_reduce=owner)
        try:
            outs[owner] = run_gpu(b, inp, mxfp8=mxfp8)
            b.check_errors()
            # the owner reduce adds one kernel before the boundary's one (a few
            # tokens) or two (stage and finish)
            assert b.launches_per_call() - int(owner) in (1, 2)
        finally:
            b.close()
    # the stage-1 sums and the post-mixed streams are the same bits; with at
    # most 8 partials both calls then run the same kernels on them, so every
    # output is (with more, the direct call takes the CUDA-core stage kernel,
    # whose GEMV adds in another order)
    names = list(outs[False]) if tp <= 8 else ["reduced_out", "residual_out"]
    for name in names:
        assert np.array_equal(outs[False][name], outs[True][name]), name
    compare(outs[True], oracle_outputs(oracle.Problem(hidden, tp, m), inp, mxfp8=mxfp8), inp, mxfp8=mxfp8)


@pytest.mark.parametrize("residual_only", [False, True])
def test_owner_reduce_consumer_same_bits(Boundary, residual_only):
    runs = [run_consume(Boundary, 2048, 4, 70, seed=13, residual_only=residual_only, owner_reduce=owner)[0]
            for owner in (False, True)]
    for name in runs[0]:
        assert np.array_equal(runs[0][name], runs[1][name]), name
