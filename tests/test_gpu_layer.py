"""GPU parity of the whole expert layer (gg_moe_mlp_fwd / gg_moe_mlp_bwd).

Covers the tiny workload, a mid-size ragged case (several row and column
tiles, ragged tails, padding), the empty batch, run-to-run bitwise equality,
CUDA-graph replay, expert relabelling, replacing one expert's weights and the
1024-expert limit."""

import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_parity, bits_to_torch, torch_to_bits, torch_to_f64
from moe_synth import CONFIGS, MoeShape, make_inputs

pytestmark = pytest.mark.gpu

MID = MoeShape("mid_e8_h320_f384_t300_k2", E=8, H=320, F=384, T=300, k=2, routing="uniform",
               x_std=1.0, w_std=0.05)
MID_PAD = MoeShape("mid_e6_h256_f320_t257_k3_pad16", E=6, H=256, F=320, T=257, k=3, P=16,
                   routing="uniform", x_std=1.0, w_std=0.05)


@pytest.fixture(scope="module")
def gg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from moe_expert_grouped_gb300 import build

    build.build()
    import moe_expert_grouped_gb300.gg as mod

    return mod


def _dev(inp):
    return dict(x=bits_to_torch(inp.x), idx=torch.from_numpy(inp.idx).cuda(),
                prob=torch.from_numpy(inp.prob).cuda(), W1=bits_to_torch(inp.W1),
                W2=bits_to_torch(inp.W2), dOut=bits_to_torch(inp.dOut))


def _run(gg, shape, d, with_dprob=False, activation=0, prob_mode=0):
    layer = gg.MoeLayer(shape.T, shape.H, shape.F, shape.k, shape.E, shape.P,
                        activation=activation, prob_mode=prob_mode)
    out = layer.forward(d["x"], d["idx"], d["prob"], d["W1"], d["W2"])
    if with_dprob:
        dX, dprob = layer.backward(d["dOut"], d["W1"], d["W2"], dprob=True)
    else:
        dX = layer.backward(d["dOut"], d["W1"], d["W2"])
    torch.cuda.synchronize()
    assert layer.status() == 0
    return (layer, out, dX, dprob) if with_dprob else (layer, out, dX)


@pytest.mark.parametrize("shape,seed", [(CONFIGS[1], 1000), (MID, 77), (MID_PAD, 78)])
def test_layer_matches_oracle(gg, shape, seed):
    inp = make_inputs(shape, seed)
    d = _dev(inp)
    layer, out, dX, dprob = _run(gg, shape, d, with_dprob=True)
    fwd = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, shape.P)
    bwd = oracle.moe_backward(inp.dOut, fwd, inp.W1, inp.W2)
    ffw = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, shape.P,
                             faithful=True)
    fbw = oracle.moe_backward(inp.dOut, ffw, inp.W1, inp.W2, faithful=True)
    assert_parity(torch_to_f64(out), fwd["out"], "out", faithful=ffw["out"])
    assert_parity(torch_to_f64(dX), bwd["dX"], "dX", faithful=fbw["dX"])
    assert_parity(dprob.cpu().numpy().astype(np.float64), bwd["dprob"], "dprob",
                  faithful=fbw["dprob"])
    n = int(fwd["offsets"][-1])
    np.testing.assert_array_equal(layer.view("offsets").cpu().numpy(), fwd["offsets"])
    np.testing.assert_array_equal(layer.view("row_of_slot").cpu().numpy(), fwd["row_of_slot"])
    for name in ("H1", "A", "Yp"):
        assert_parity(torch_to_f64(layer.view(name)[:n]), fwd[name][:n], name,
                      faithful=ffw[name][:n])
    for name in ("dH", "dXp"):
        assert_parity(torch_to_f64(layer.view(name)[:n]), bwd[name][:n], name,
                      faithful=fbw[name][:n])


def test_layer_run_to_run_bitwise(gg):
    inp = make_inputs(MID, 5)
    d = _dev(inp)
    _, o1, g1, p1 = _run(gg, MID, d, with_dprob=True)
    _, o2, g2, p2 = _run(gg, MID, d, with_dprob=True)
    _, o3, g3 = _run(gg, MID, d)
    np.testing.assert_array_equal(torch_to_bits(o1), torch_to_bits(o2))
    np.testing.assert_array_equal(torch_to_bits(g1), torch_to_bits(g2))
    np.testing.assert_array_equal(p1.cpu().numpy(), p2.cpu().numpy())
    # asking for dprob leaves dX untouched
    np.testing.assert_array_equal(torch_to_bits(g1), torch_to_bits(g3))


def test_layer_empty_batch(gg):
    shape = CONFIGS[1].with_tokens(0)
    inp = make_inputs(shape, 1000)
    d = _dev(inp)
    layer, out, dX = _run(gg, shape, d)
    assert out.shape == (0, shape.H) and dX.shape == (0, shape.H)
    assert np.all(layer.view("offsets").cpu().numpy() == 0)


def test_cuda_graph_replay_matches_eager(gg):
    shape = MID
    inp = make_inputs(shape, 11)
    d = _dev(inp)
    _, out_e, dX_e = _run(gg, shape, d)
    layer = gg.MoeLayer(shape.T, shape.H, shape.F, shape.k, shape.E, shape.P)
    out = torch.empty_like(out_e)
    dX = torch.empty_like(dX_e)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up outside capture (first-use set-up)
        layer.forward(d["x"], d["idx"], d["prob"], d["W1"], d["W2"], out=out)
        layer.backward(d["dOut"], d["W1"], d["W2"], dX=dX)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    out.zero_()
    dX.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(d["x"], d["idx"], d["prob"], d["W1"], d["W2"], out=out)
        layer.backward(d["dOut"], d["W1"], d["W2"], dX=dX)
    g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(torch_to_bits(out), torch_to_bits(out_e))
    np.testing.assert_array_equal(torch_to_bits(dX), torch_to_bits(dX_e))
    # new routing written into the same input buffers is picked up by the replay
    inp2 = make_inputs(shape, 12)
    d["idx"].copy_(torch.from_numpy(inp2.idx))
    g.replay()
    torch.cuda.synchronize()
    d2 = dict(d)
    _, out_e2, dX_e2 = _run(gg, shape, d2)
    np.testing.assert_array_equal(torch_to_bits(out), torch_to_bits(out_e2))
    np.testing.assert_array_equal(torch_to_bits(dX), torch_to_bits(dX_e2))


def test_expert_relabel_is_bitwise_invariant(gg):
    shape = MID
    inp = make_inputs(shape, 21)
    d = _dev(inp)
    _, o1, g1 = _run(gg, shape, d)
    pi = np.random.default_rng(3).permutation(shape.E)
    d2 = dict(d)
    d2["idx"] = torch.from_numpy(pi[inp.idx].astype(np.int32)).cuda()
    W1p = torch.empty_like(d["W1"])
    W2p = torch.empty_like(d["W2"])
    W1p[torch.from_numpy(pi).cuda()] = d["W1"]
    W2p[torch.from_numpy(pi).cuda()] = d["W2"]
    d2["W1"], d2["W2"] = W1p, W2p
    _, o2, g2 = _run(gg, shape, d2)
    np.testing.assert_array_equal(torch_to_bits(o1), torch_to_bits(o2))
    np.testing.assert_array_equal(torch_to_bits(g1), torch_to_bits(g2))


def test_replacing_one_expert_changes_only_its_tokens(gg):
    shape = MID
    inp = make_inputs(shape, 31)
    d = _dev(inp)
    _, o1, g1 = _run(gg, shape, d)
    e = 3
    d["W1"][e].normal_(0, 0.05)
    d["W2"][e].normal_(0, 0.05)
    _, o2, g2 = _run(gg, shape, d)
    touched = np.any(inp.idx == e, axis=1)
    assert touched.any() and (~touched).any()
    b1, b2 = torch_to_bits(o1), torch_to_bits(o2)
    np.testing.assert_array_equal(b1[~touched], b2[~touched])
    assert np.all(np.any(b1[touched] != b2[touched], axis=1))
    np.testing.assert_array_equal(torch_to_bits(g1)[~touched], torch_to_bits(g2)[~touched])


ACT_NAMES = {0: "swiglu", 1: "qgeglu"}
MODE_NAMES = {0: "combine", 1: "activation", 2: "pre_fc1"}


@pytest.mark.parametrize("activation,prob_mode", [(1, 0), (0, 1), (1, 1), (0, 2), (1, 2)])
@pytest.mark.parametrize("shape,seed", [(CONFIGS[1], 1000), (MID_PAD, 79)])
def test_layer_variants_match_oracle(gg, shape, seed, activation, prob_mode):
    inp = make_inputs(shape, seed)
    d = _dev(inp)
    layer, out, dX, dprob = _run(gg, shape, d, with_dprob=True, activation=activation,
                                 prob_mode=prob_mode)
    kw = dict(activation=ACT_NAMES[activation], prob_mode=MODE_NAMES[prob_mode])
    fwd = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, shape.P, **kw)
    bwd = oracle.moe_backward(inp.dOut, fwd, inp.W1, inp.W2)
    ffw = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, shape.P,
                             faithful=True, **kw)
    fbw = oracle.moe_backward(inp.dOut, ffw, inp.W1, inp.W2, faithful=True)
    assert_parity(torch_to_f64(out), fwd["out"], "out", faithful=ffw["out"])
    assert_parity(torch_to_f64(dX), bwd["dX"], "dX", faithful=fbw["dX"])
    assert_parity(dprob.cpu().numpy().astype(np.float64), bwd["dprob"], "dprob",
                  faithful=fbw["dprob"])
    n = int(fwd["offsets"][-1])
    for name in ("Xp", "H1", "A", "Yp"):
        assert_parity(torch_to_f64(layer.view(name)[:n]), fwd[name][:n], name,
                      faithful=ffw[name][:n])


@pytest.mark.parametrize("activation,prob_mode", [(0, 0), (1, 1), (0, 2)])
def test_recompute_h1_equals_saved_h1(gg, activation, prob_mode):
    # The backward that recomputes FC1's output with a plain grouped FC1 gives
    # the same bits as the one that reads the forward's saved H1.
    shape = MID_PAD
    inp = make_inputs(shape, 81)
    d = _dev(inp)
    res = []
    for recompute in (False, True):
        layer = gg.MoeLayer(shape.T, shape.H, shape.F, shape.k, shape.E, shape.P,
                            activation=activation, prob_mode=prob_mode, recompute_h1=recompute)
        out = layer.forward(d["x"], d["idx"], d["prob"], d["W1"], d["W2"])
        torch.cuda.synchronize()
        h1_after_fwd = torch_to_bits(layer.view("H1"))
        dX, dprob = layer.backward(d["dOut"], d["W1"], d["W2"], dprob=True)
        torch.cuda.synchronize()
        assert layer.status() == 0
        n = int(layer.view("offsets")[-1].item())
        res.append((torch_to_bits(out), torch_to_bits(dX), dprob.cpu().numpy(),
                    torch_to_bits(layer.view("H1")[:n]), h1_after_fwd[:n]))
    saved, recomputed = res
    for a, b in zip(saved[:4], recomputed[:4]):
        np.testing.assert_array_equal(a, b)
    # without recompute the forward stored H1; with it the forward left the
    # (zero-initialised) region alone and the backward filled it
    np.testing.assert_array_equal(saved[4], saved[3])
    assert np.all(recomputed[4] == 0)


@pytest.mark.parametrize("activation,prob_mode,recompute", [(1, 2, True), (1, 1, False)])
def test_cuda_graph_replay_of_variants(gg, activation, prob_mode, recompute):
    # the option paths (QuickGeGLU, probability at the activation or before
    # FC1, H1 recompute) capture into a CUDA graph and replay bitwise
    shape = MID_PAD
    inp = make_inputs(shape, 83)
    d = _dev(inp)
    kw = dict(activation=activation, prob_mode=prob_mode, recompute_h1=recompute)
    eager = gg.MoeLayer(shape.T, shape.H, shape.F, shape.k, shape.E, shape.P, **kw)
    out_e = eager.forward(d["x"], d["idx"], d["prob"], d["W1"], d["W2"])
    dX_e, dp_e = eager.backward(d["dOut"], d["W1"], d["W2"], dprob=True)
    layer = gg.MoeLayer(shape.T, shape.H, shape.F, shape.k, shape.E, shape.P, **kw)
    out, dX = torch.empty_like(out_e), torch.empty_like(dX_e)
    dp = torch.empty_like(dp_e)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.forward(d["x"], d["idx"], d["prob"], d["W1"], d["W2"], out=out)
        layer.backward(d["dOut"], d["W1"], d["W2"], dX=dX, dprob=dp)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    for t in (out, dX, dp):
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(d["x"], d["idx"], d["prob"], d["W1"], d["W2"], out=out)
        layer.backward(d["dOut"], d["W1"], d["W2"], dX=dX, dprob=dp)
    g.replay()
    torch.cuda.synchronize()
    assert layer.status() == 0
    np.testing.assert_array_equal(torch_to_bits(out), torch_to_bits(out_e))
    np.testing.assert_array_equal(torch_to_bits(dX), torch_to_bits(dX_e))
    np.testing.assert_array_equal(dp.cpu().numpy(), dp_e.cpu().numpy())


def test_layer_at_the_expert_limit(gg):
    """1024 experts, the library's maximum, with tokens on eight of them (the
    first, middle and last ids): the permute's histogram table and the
    GEMMs' per-expert tables at their full size, 1016 empty experts."""
    shape = MoeShape("maxe_e1024_h64_f128_t200_k2", E=1024, H=64, F=128, T=200, k=2,
                     routing="uniform", x_std=1.0, w_std=0.05)
    inp = make_inputs(shape, 91)
    rng = np.random.default_rng(92)
    live = np.array([0, 1, 2, 511, 512, 700, 1022, 1023])
    inp.idx[:] = np.stack([rng.choice(live, size=shape.k, replace=False)
                           for _ in range(shape.T)]).astype(np.int32)
    d = _dev(inp)
    layer, out, dX, dprob = _run(gg, shape, d, with_dprob=True)
    fwd = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, shape.P)
    bwd = oracle.moe_backward(inp.dOut, fwd, inp.W1, inp.W2)
    ffw = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, shape.P,
                             faithful=True)
    fbw = oracle.moe_backward(inp.dOut, ffw, inp.W1, inp.W2, faithful=True)
    np.testing.assert_array_equal(layer.view("offsets").cpu().numpy(), fwd["offsets"])
    np.testing.assert_array_equal(layer.view("row_of_slot").cpu().numpy(), fwd["row_of_slot"])
    assert_parity(torch_to_f64(out), fwd["out"], "out", faithful=ffw["out"])
    assert_parity(torch_to_f64(dX), bwd["dX"], "dX", faithful=fbw["dX"])
    assert_parity(dprob.cpu().numpy().astype(np.float64), bwd["dprob"], "dprob",
                  faithful=fbw["dprob"])
