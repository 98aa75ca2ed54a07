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


def _ep_faithful(inp, s):
    """BF16-faithful oracle of the expert-parallel ordering, which sizes each
    element's error floor: every routed (token, slot) row runs through the
    layer on its own (one slot, probability 1), with BF16 rounding where the
    rank-local layer stores its results, and the sending rank sums the k
    returned rows weighted by the probabilities, exactly, with one rounding.
    (The layer proper applies the probability before its BF16 stores, so its
    own faithful oracle rounds at other points.)"""
    T, k = inp.idx.shape
    rows_x = np.repeat(inp.x, k, axis=0)          # row t*k + j carries x_t
    rows_d = np.repeat(inp.dOut, k, axis=0)
    eid = inp.idx.reshape(-1, 1)
    ones = np.ones((T * k, 1), np.float32)
    f = oracle.moe_forward(rows_x, eid, ones, inp.W1, inp.W2, s.E, 1, faithful=True)
    b = oracle.moe_backward(rows_d, f, inp.W1, inp.W2, faithful=True)
    p = inp.prob.astype(np.float64)
    out = oracle.round_to_bf16(np.einsum("tj,tjh->th", p, f["out"].reshape(T, k, -1)))
    dX = oracle.round_to_bf16(np.einsum("tj,tjh->th", p, b["dX"].reshape(T, k, -1)))
    return dict(out=out, dX=dX, dprob=b["dprob"].reshape(T, k))


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
    fa = _ep_faithful(inp, s)
    assert_parity(torch_to_f64(out), fwd["out"], "out", faithful=fa["out"])
    assert_parity(torch_to_f64(dX), bwd["dX"], "dX", faithful=fa["dX"])
    assert_parity(dprob.cpu().numpy().astype(np.float64), bwd["dprob"], "dprob",
                  faithful=fa["dprob"])


def test_expert_parallel_reuses_its_layer_buffer_across_batches(gg):
    # Two forwards of different sizes on one ExpertParallelLayer run on one
    # device buffer (bound once, for the next power of two rows), each at
    # oracle parity.
    from moe_expert_grouped_gb300.ep import ExpertParallelLayer

    ep = ExpertParallelLayer(EP_MID.H, EP_MID.F, EP_MID.k, EP_MID.E)
    layers = []
    for T, seed in ((300, 4243), (171, 4244)):
        s = MoeShape(f"ep_e8_h256_f384_t{T}_k3", E=8, H=256, F=384, T=T, k=3,
                     routing="uniform", x_std=1.0, w_std=0.05)
        inp = make_inputs(s, seed)
        x, W1, W2, dOut = (bits_to_torch(a) for a in (inp.x, inp.W1, inp.W2, inp.dOut))
        out = ep.forward(x, torch.from_numpy(inp.idx).cuda(), torch.from_numpy(inp.prob).cuda(),
                         W1, W2)
        dX, dprob = ep.backward(dOut, W1, W2)
        torch.cuda.synchronize()
        assert ep.ops._layer.status() == 0
        layers.append(ep.ops._layer)
        fwd = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, s.E, 1)
        bwd = oracle.moe_backward(inp.dOut, fwd, inp.W1, inp.W2)
        fa = _ep_faithful(inp, s)
        assert_parity(torch_to_f64(out), fwd["out"], "out", faithful=fa["out"])
        assert_parity(torch_to_f64(dX), bwd["dX"], "dX", faithful=fa["dX"])
        assert_parity(dprob.cpu().numpy().astype(np.float64), bwd["dprob"], "dprob",
                      faithful=fa["dprob"])
    assert layers[0] is layers[1]
    assert layers[0].T == 1024
