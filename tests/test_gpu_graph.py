"""Boundary calls recorded into a CUDA graph give the same bits as eager
calls, including post and comb (computed in the finish kernel, or by the
side-stream kernel that the capture joins back before it ends), and the graph
can be replayed."""
import numpy as np
import pytest
import torch

from gpu_harness import to_device
from mhc_residual_boundary_gb300 import synth

pytestmark = pytest.mark.gpu


def _bytes(outs):
    return {k: v.view(torch.uint8).cpu().numpy() for k, v in outs.items()}


@pytest.mark.parametrize("side_mixes,static_weight", [(False, False), (True, False), (False, True)])
def test_captured_calls_match_eager_calls(side_mixes, static_weight):
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from mhc_residual_boundary_gb300 import Boundary
    hidden, tp, m = 2048, 4, 40
    b = Boundary(hidden=hidden, tp=tp, max_num_tokens=m, mxfp8=True, side_mixes=side_mixes,
                 static_weight=static_weight)
    try:
        ins = [to_device(synth.make_inputs(hidden, tp, m, seed=s)) for s in (31, 32)]
        eager = []
        for inp in ins:
            outs = b.empty_outputs(m, extras=True, mxfp8=True)
            b.run(inp, outs)
            b.join()
            torch.cuda.synchronize()
            eager.append(_bytes(outs))
        graph_outs = [b.empty_outputs(m, extras=True, mxfp8=True) for _ in ins]
        for outs in graph_outs:
            for t in outs.values():
                t.view(torch.uint8).fill_(0x5A)
        cap = torch.cuda.Stream()
        cap.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for inp, outs in zip(ins, graph_outs):
                b.run(inp, outs, stream=cap)
            b.join(cap)
        for _ in range(2):   # replaying twice writes the same values again
            g.replay()
            torch.cuda.synchronize()
            for want, outs in zip(eager, graph_outs):
                got = _bytes(outs)
                for k in want:
                    assert np.array_equal(got[k], want[k]), k
        b.check_errors()
        # an eager call after the graph still works and orders after it
        outs = b.empty_outputs(m, extras=True, mxfp8=True)
        b.run(ins[0], outs)
        b.join()
        torch.cuda.synchronize()
        got = _bytes(outs)
        for k in eager[0]:
            assert np.array_equal(got[k], eager[0][k]), k
    finally:
        b.close()
