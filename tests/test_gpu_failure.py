"""Failure detection on the GPU without a fault: a boundary kernel whose
input copies never come gives up its bounded waits, the host reads
MHC_ERR_TIMEOUT from the error word, and the same handle and context then
compute correct results again."""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import compare, oracle_outputs, run_gpu
from mhc_residual_boundary_gb300 import capi, synth

pytestmark = pytest.mark.gpu


# 4 tokens take the one-kernel path, 200 the stage and finish kernels
@pytest.mark.parametrize("m", [4, 200])
def test_stalled_copies_report_a_timeout_and_the_handle_recovers(m):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from mhc_residual_boundary_gb300 import Boundary
    hidden, tp = 1024, 4
    inp = synth.make_inputs(hidden, tp, m, seed=77)
    ref = oracle_outputs(oracle.Problem(hidden, tp, m), inp)
    b = Boundary(hidden=hidden, tp=tp, max_num_tokens=m)
    try:
        compare(run_gpu(b, inp), ref, inp)
        b.check_errors()
        capi.mhc_test_stall_stage_copies(True)
        try:
            run_gpu(b, inp)          # the kernels give up their waits and return
        finally:
            capi.mhc_test_stall_stage_copies(False)
        with pytest.raises(capi.MhcError, match="MHC_ERR_TIMEOUT"):
            b.check_errors()
        b.check_errors()             # reported once, then cleared
        compare(run_gpu(b, inp), ref, inp)
        b.check_errors()
    finally:
        b.close()
