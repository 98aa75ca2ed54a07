"""Expert parallelism on one GPU: ``ExpertParallelLayer`` with the library's
kernels at one rank (no exchange) against the oracle and against the layer
run directly.

The forward output is bitwise the direct layer's: both send each row through
the same FC1/FC2 tiles and sum the k weighted rows in the same order. The
backward applies the probability after the expert MLP instead of before it
(the MLP's backward is linear in its upstream gradient), so dX agrees to
rounding and is checked against the oracle; dprob is the same dot product of
dOut with the saved expert output."""

import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_parity, bits_to_torch, torch_to_f64
from moe_synth import MoeShape, make_inputs

pytestmark = pytest.mark.gpu

EP_MID = MoeShape("ep_e8_h256_f384_t300_k3", E=8, H=256, F=384, T=300, k=3, routing="uniform",
                  x_std=1.0, w_std=0.05)


@pytest.fixture(scope="module")
def gg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from moe_expert_grouped_gb300 import build

    build.build()
    import moe_expert_grouped_gb300.gg as mod

    return mod


def test_expert_parallel_one_rank_matches_layer_and_oracle(gg):
    from moe_expert_grouped_gb300.ep import ExpertParallelLayer

    s = EP_MID
    inp = make_inputs(s, 4242)
    x, W1, W2, dOut = (bits_to_torch(a) for a in (inp.x, inp.W1, inp.W2, inp.dOut))
    idx = torch.from_numpy(inp.idx).cuda()
    prob = torch.from_numpy(inp.prob).cuda()

    ep = ExpertParallelLayer(s.H, s.F, s.k, s.E)
    out = ep.forward(x, idx, prob, W1, W2)
    dX, dprob = ep.backward(dOut, W1, W2)
    torch.cuda.synchronize()
    assert ep.ops._layer.status() == 0

    direct = gg.MoeLayer(s.T, s.H, s.F, s.k, s.E, 1)
    out_d = direct.forward(x, idx, prob, W1, W2)
    dX_d, dprob_d = direct.backward(dOut, W1, W2, dprob=True)
    torch.cuda.synchronize()
    assert torch.equal(out, out_d)
    torch.testing.assert_close(dprob, dprob_d, rtol=1e-5, atol=1e-6)

    fwd = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, s.E, 1)
    bwd = oracle.moe_backward(inp.dOut, fwd, inp.W1, inp.W2)
    ffw = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, s.E, 1, faithful=True)
    fbw = oracle.moe_backward(inp.dOut, ffw, inp.W1, inp.W2, faithful=True)
    assert_parity(torch_to_f64(out), fwd["out"], "out", faithful=ffw["out"])
    assert_parity(torch_to_f64(dX), bwd["dX"], "dX", faithful=fbw["dX"])
    assert_parity(dprob.cpu().numpy().astype(np.float64), bwd["dprob"], "dprob",
                  faithful=fbw["dprob"])
