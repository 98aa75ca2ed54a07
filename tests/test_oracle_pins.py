"""Pins of the CPU oracle against things other than itself.

Each check ties the oracle to brute force, a closed form, a library routine or
an invariant that the pages' definitions fix, chosen so that a dropped term, a
wrong sign, a swapped gate/up half, a transposed weight or a wrong row index
in the oracle fails at least one of them. No GPU is used here.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from moe_synth import CONFIGS, f32_to_bf16_bits, make_inputs, normal_bf16


def _bits(a):
    return f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def _val(u16):
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _silu(z):
    return z / (1.0 + math.exp(-z))


# ------------------------------------------------------------------ BF16 rounding

def test_round_to_bf16_matches_torch_on_fp32_values():
    # Library special case: for values that are exactly fp32, rounding fp64 ->
    # bf16 must agree with torch's fp32 -> bf16 conversion (nearest-even).
    rng = np.random.default_rng(7)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-30).astype(np.float32),
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0], np.float32),
    ])
    ours = oracle.round_to_bf16(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_round_to_bf16_ties_to_even():
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0);
    # 1 + 3*2^-8 is halfway between 1 + 2^-7 and 1 + 2^-6: goes to 1 + 2^-6.
    x = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 1 + 2.0 ** -8 + 2.0 ** -30])
    got = oracle.round_to_bf16(x)
    np.testing.assert_array_equal(got, [1.0, 1 + 2.0 ** -6, -1.0, 1 + 2.0 ** -7])


def test_bf16_bits_decode():
    # 0x3F80 = 1.0, 0xC000 = -2.0, 0x3E80 = 0.25, 0x0000 = 0
    np.testing.assert_array_equal(oracle.bf16_bits_to_f64(np.array([0x3F80, 0xC000, 0x3E80, 0], np.uint16)),
                                  [1.0, -2.0, 0.25, 0.0])


# ------------------------------------------------------------------ row map

def _route_brute(idx, E, P):
    """Row map by explicit loops over experts, then tokens, then slots."""
    T, k = idx.shape
    offsets = [0]
    row_of_slot = [-1] * (T * k)
    slot_of_row = [-1] * (T * k + E * (P - 1))
    row = 0
    for e in range(E):
        start = row
        for t in range(T):
            for j in range(k):
                if idx[t, j] == e:
                    row_of_slot[t * k + j] = row
                    slot_of_row[row] = t * k + j
                    row += 1
        cnt = row - start
        row = start + ((cnt + P - 1) // P) * P
        offsets.append(row)
    return np.array(offsets), np.array(row_of_slot), np.array(slot_of_row)


@pytest.mark.parametrize("T,E,k,P", [(0, 4, 2, 1), (1, 1, 1, 1), (3, 4, 2, 1), (7, 5, 3, 4),
                                     (40, 6, 2, 8), (13, 3, 3, 1), (9, 8, 1, 3)])
def test_route_matches_brute_force(T, E, k, P):
    rng = np.random.default_rng(T * 100 + E * 10 + k)
    idx = rng.integers(0, E, size=(T, k)).astype(np.int32)  # duplicates within a token allowed
    off, ros, sor = oracle.route(idx, E, P)
    boff, bros, bsor = _route_brute(idx, E, P)
    np.testing.assert_array_equal(off, boff)
    np.testing.assert_array_equal(ros, bros)
    np.testing.assert_array_equal(sor, bsor)


def test_route_matches_stable_argsort():
    # Library special case: with P = 1 the row order is numpy's stable argsort
    # of the flattened expert ids, and offsets are the cumulative bincount.
    inp = make_inputs(CONFIGS[2].with_tokens(512), 2000, with_weights=False, with_dout=False)
    E = CONFIGS[2].E
    off, ros, sor = oracle.route(inp.idx, E, 1)
    flat = inp.idx.reshape(-1)
    order = np.argsort(flat, kind="stable")
    np.testing.assert_array_equal(sor, order)
    np.testing.assert_array_equal(off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    np.testing.assert_array_equal(ros[order], np.arange(flat.size))


def test_route_zero_token_expert_and_padding():
    idx = np.array([[0, 2], [2, 0], [0, 2]], np.int32)
    off, ros, sor = oracle.route(idx, 4, 4)
    # expert 1 and 3 receive nothing: equal neighbouring offsets
    np.testing.assert_array_equal(off, [0, 4, 4, 8, 8])
    np.testing.assert_array_equal(ros, [0, 4, 5, 1, 2, 6])
    np.testing.assert_array_equal(sor[:8], [0, 3, 4, -1, 1, 2, 5, -1])
    assert np.all(sor[8:] == -1)


def test_route_rejects_bad_ids():
    with pytest.raises(ValueError):
        oracle.route(np.array([[0, 4]], np.int32), 4, 1)
    with pytest.raises(ValueError):
        oracle.route(np.array([[-1, 0]], np.int32), 4, 1)


# ------------------------------------------------------------------ forward

def _brute_forward(x, idx, prob, W1, W2):
    """Dense gated MLP evaluated per token and per routed expert (no grouping)."""
    xv, w1, w2 = _val(x), _val(W1), _val(W2)
    T, k = idx.shape
    F = w1.shape[1] // 2
    out = np.zeros((T, xv.shape[1]))
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            h = np.array([sum(w1[e, n, c] * xv[t, c] for c in range(xv.shape[1])) for n in range(2 * F)])
            a = np.array([_silu(h[i]) * h[F + i] for i in range(F)])
            y = np.array([sum(w2[e, o, i] * a[i] for i in range(F)) for o in range(xv.shape[1])])
            out[t] += float(prob[t, j]) * y
    return out


@pytest.mark.parametrize("T,E,k", [(0, 4, 2), (1, 1, 1), (3, 4, 2), (3, 1, 2), (5, 4, 1)])
def test_forward_matches_brute_force_tiny(T, E, k):
    H, F = 6, 4  # F != H and 2F != H so that a transposed weight cannot pass
    rng = np.random.default_rng(1 + T + 10 * E + 100 * k)
    x = normal_bf16(rng, (T, H), 1.0)
    W1 = normal_bf16(rng, (E, 2 * F, H), 0.5)
    W2 = normal_bf16(rng, (E, H, F), 0.5)
    idx = rng.integers(0, E, size=(T, k)).astype(np.int32)
    prob = rng.uniform(0.1, 1.0, size=(T, k)).astype(np.float32)
    for P in (1, 3):
        fwd = oracle.moe_forward(x, idx, prob, W1, W2, E, P)
        np.testing.assert_allclose(fwd["out"], _brute_forward(x, idx, prob, W1, W2), rtol=1e-12, atol=1e-12)
        assert fwd["out"].shape == (T, H)


def test_forward_matches_brute_force_config1_subset():
    shape = CONFIGS[1]
    inp = make_inputs(shape, 1000)
    fwd = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, shape.P)
    sel = [0, 1, 77, 255]
    ref = np.stack([oracle.token_forward(inp.x[t], inp.idx[t], inp.prob[t], inp.W1, inp.W2) for t in sel])
    np.testing.assert_allclose(fwd["out"][sel], ref, rtol=1e-12, atol=1e-18)
    # and the per-token form itself against explicit loops on two tokens
    sub = _brute_forward(inp.x[:2], inp.idx[:2], inp.prob[:2], inp.W1, inp.W2)
    np.testing.assert_allclose(fwd["out"][:2], sub, rtol=1e-10, atol=1e-18)
    # expert 3 is forced to carry no tokens
    assert fwd["offsets"][3] == fwd["offsets"][4]


def test_worked_example_closed_form():
    # Two tokens, two experts, H=2, F=1, top-2; every value follows by hand from
    # A = silu(g) * u and out = sum_j p_j * W2_e A.
    x = np.array([[1.0, 2.0], [-1.0, 0.5]])
    W1 = np.array([[[1, 0], [0, 1]], [[0, 1], [1, 0]]], np.float64)  # [E, 2F, H]
    W2 = np.array([[[1.0], [2.0]], [[-1.0], [0.5]]])                  # [E, H, F]
    idx = np.array([[1, 0], [0, 1]], np.int32)
    prob = np.array([[0.25, 0.5], [0.75, 0.125]])
    fwd = oracle.moe_forward(_bits(x), idx, prob.astype(np.float32), _bits(W1), _bits(W2), 2, 1)
    s = lambda z: 1.0 / (1.0 + math.exp(-z))  # noqa: E731
    t0 = 0.25 * (2 * s(2) * 1) * np.array([-1.0, 0.5]) + 0.5 * (1 * s(1) * 2) * np.array([1.0, 2.0])
    t1 = 0.75 * (-1 * s(-1) * 0.5) * np.array([1.0, 2.0]) + 0.125 * (0.5 * s(0.5) * -1) * np.array([-1.0, 0.5])
    np.testing.assert_allclose(fwd["out"], np.stack([t0, t1]), rtol=1e-15, atol=0)
    np.testing.assert_array_equal(fwd["offsets"], [0, 2, 4])
    np.testing.assert_array_equal(fwd["row_of_slot"], [2, 0, 1, 3])


def _identity_weights(E, H):
    # gate block = [I; 0], up block = [I; 0], W2 = [I 0] with F = 2H
    F = 2 * H
    W1 = np.zeros((E, 2 * F, H), np.float32)
    W2 = np.zeros((E, H, F), np.float32)
    for e in range(E):
        W1[e, :H, :] = np.eye(H)
        W1[e, F:F + H, :] = np.eye(H)
        W2[e, :, :H] = np.eye(H)
    return _bits(W1), _bits(W2), F


def test_identity_weights_closed_form():
    shape = CONFIGS[1]
    inp = make_inputs(shape, 1000, with_weights=False)
    W1, W2, F = _identity_weights(shape.E, shape.H)
    fwd = oracle.moe_forward(inp.x, inp.idx, inp.prob, W1, W2, shape.E, 1)
    xv = _val(inp.x)
    sig = 1.0 / (1.0 + np.exp(-xv))
    psum = inp.prob.astype(np.float64).sum(axis=1, keepdims=True)
    np.testing.assert_allclose(fwd["out"], psum * xv * (xv * sig), rtol=1e-13, atol=0)
    bwd = oracle.moe_backward(inp.dOut, fwd, W1, W2)
    dv = _val(inp.dOut)
    dsilu = sig + xv * sig * (1 - sig)
    # d/dx [x * silu(x)] = silu(x) + x * silu'(x)
    np.testing.assert_allclose(bwd["dX"], psum * dv * (xv * sig + xv * dsilu), rtol=1e-12, atol=1e-300)
    # every routed slot's expert output is x * silu(x): dprob[t, j] = <dOut_t, x_t silu(x_t)>
    closed = np.sum(dv * xv * (xv * sig), axis=1, keepdims=True) * np.ones_like(bwd["dprob"])
    np.testing.assert_allclose(bwd["dprob"], closed, rtol=1e-12, atol=1e-300)


def test_one_hot_rows_closed_form():
    # Gate row i picks c * x[a_i], up row i picks x[b_i]; W2 = I picks a_i back out.
    E, H, F, T = 1, 8, 8, 5
    rng = np.random.default_rng(3)
    a_sel = rng.integers(0, H, F)
    b_sel = rng.integers(0, H, F)
    c = 2.0
    W1 = np.zeros((E, 2 * F, H), np.float32)
    W1[0, np.arange(F), a_sel] = c
    W1[0, F + np.arange(F), b_sel] = 1.0
    W2 = np.eye(H, F, dtype=np.float32)[None]
    x = normal_bf16(rng, (T, H), 1.0)
    idx = np.zeros((T, 1), np.int32)
    prob = np.ones((T, 1), np.float32)
    fwd = oracle.moe_forward(x, idx, prob, _bits(W1), _bits(W2), E, 1)
    xv = _val(x)
    for t in range(T):
        for i in range(F):
            z = c * xv[t, a_sel[i]]
            assert fwd["A"][t, i] == pytest.approx(_silu(z) * xv[t, b_sel[i]], rel=1e-14, abs=1e-300)
    np.testing.assert_allclose(fwd["out"], fwd["A"][:, :H], rtol=1e-15)


def test_zero_gate_gives_exact_zeros():
    shape = CONFIGS[1]
    inp = make_inputs(shape, 1000)
    W1 = inp.W1.copy()
    W1[:, :shape.F, :] = 0  # silu(0) = 0 exactly
    fwd = oracle.moe_forward(inp.x, inp.idx, inp.prob, W1, inp.W2, shape.E, 1)
    assert np.all(fwd["A"] == 0) and np.all(fwd["out"] == 0)
    bwd = oracle.moe_backward(inp.dOut, fwd, W1, inp.W2)
    # with g = 0: du = dA * silu(0) = 0, and dg = dA * u * 1/2 flows through the zero gate rows -> dX = 0
    assert np.all(bwd["dX"] == 0)
    assert np.all(bwd["dH"][:, shape.F:] == 0)


# ------------------------------------------------------------------ invariants

def test_empty_batch():
    shape = CONFIGS[1].with_tokens(0)
    inp = make_inputs(shape, 1000)
    fwd = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, 1)
    assert fwd["out"].shape == (0, shape.H)
    np.testing.assert_array_equal(fwd["offsets"], np.zeros(shape.E + 1))
    bwd = oracle.moe_backward(inp.dOut, fwd, inp.W1, inp.W2)
    assert bwd["dX"].shape == (0, shape.H)


def test_expert_relabel_invariance():
    shape = CONFIGS[1]
    inp = make_inputs(shape, 1000)
    fwd = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, 1)
    bwd = oracle.moe_backward(inp.dOut, fwd, inp.W1, inp.W2)
    pi = np.array([2, 0, 3, 1])
    W1p = np.empty_like(inp.W1)
    W2p = np.empty_like(inp.W2)
    W1p[pi] = inp.W1
    W2p[pi] = inp.W2
    idxp = pi[inp.idx].astype(np.int32)
    fwd2 = oracle.moe_forward(inp.x, idxp, inp.prob, W1p, W2p, shape.E, 1)
    bwd2 = oracle.moe_backward(inp.dOut, fwd2, W1p, W2p)
    np.testing.assert_allclose(fwd2["out"], fwd["out"], rtol=1e-13, atol=1e-20)
    np.testing.assert_allclose(bwd2["dX"], bwd["dX"], rtol=1e-12, atol=1e-18)


def test_prob_scaling_is_linear():
    shape = CONFIGS[1]
    inp = make_inputs(shape, 1000)
    f1 = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, 1)
    f2 = oracle.moe_forward(inp.x, inp.idx, inp.prob * np.float32(4.0), inp.W1, inp.W2, shape.E, 1)
    np.testing.assert_allclose(f2["out"], 4.0 * f1["out"], rtol=1e-14, atol=0)
    b1 = oracle.moe_backward(inp.dOut, f1, inp.W1, inp.W2)
    b2 = oracle.moe_backward(inp.dOut, f2, inp.W1, inp.W2)
    np.testing.assert_allclose(b2["dX"], 4.0 * b1["dX"], rtol=1e-13, atol=0)


def test_padding_rows_are_zero_and_padding_does_not_change_results():
    shape = CONFIGS[1]
    inp = make_inputs(shape, 1000)
    f1 = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, 1)
    f8 = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, 64)
    pad = f8["slot_of_row"] < 0
    for name in ("Xp", "H1", "A", "Yp"):
        assert np.all(f8[name][pad] == 0), name
    assert np.all(np.diff(f8["offsets"]) % 64 == 0)
    np.testing.assert_array_equal(f8["out"], f1["out"])
    b1 = oracle.moe_backward(inp.dOut, f1, inp.W1, inp.W2)
    b8 = oracle.moe_backward(inp.dOut, f8, inp.W1, inp.W2)
    np.testing.assert_array_equal(b8["dX"], b1["dX"])
    assert np.all(b8["dXp"][pad] == 0)


def test_replacing_one_expert_changes_only_its_tokens():
    shape = CONFIGS[1]
    inp = make_inputs(shape, 1000)
    f1 = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, 1)
    W1 = inp.W1.copy()
    W1[1] = normal_bf16(np.random.default_rng(99), W1[1].shape, 0.02)
    f2 = oracle.moe_forward(inp.x, inp.idx, inp.prob, W1, inp.W2, shape.E, 1)
    touched = np.any(inp.idx == 1, axis=1)
    assert touched.any() and (~touched).any()
    np.testing.assert_array_equal(f2["out"][~touched], f1["out"][~touched])
    assert np.all(np.any(f2["out"][touched] != f1["out"][touched], axis=1))


# ------------------------------------------------------------------ backward

def _torch_forward(x, idx, prob, W1, W2, activation="swiglu", prob_mode="combine"):
    """The same layer in torch float64 ops, token by token (autograd reference).
    The gate uses torch's own silu for SwiGLU and x * sigmoid(1.702 x) for
    QuickGeGLU."""
    T, k = idx.shape
    F = W1.shape[1] // 2
    outs = []
    for t in range(T):
        acc = torch.zeros(x.shape[1], dtype=torch.float64)
        for j in range(k):
            e = int(idx[t, j])
            p = prob[t, j]
            h = W1[e] @ (p * x[t] if prob_mode == "pre_fc1" else x[t])
            gate = (torch.nn.functional.silu(h[:F]) if activation == "swiglu"
                    else h[:F] * torch.sigmoid(1.702 * h[:F]))
            a = gate * h[F:]
            if prob_mode == "activation":
                a = p * a
            y = W2[e] @ a
            acc = acc + (p * y if prob_mode == "combine" else y)
        outs.append(acc)
    return torch.stack(outs)


def test_backward_matches_torch_autograd():
    shape = CONFIGS[1].with_tokens(24)
    inp = make_inputs(shape, 1000)
    inp.W1[:] = normal_bf16(np.random.default_rng(5), inp.W1.shape, 0.2)  # larger scale: non-trivial gate
    inp.W2[:] = normal_bf16(np.random.default_rng(6), inp.W2.shape, 0.2)
    inp.x[:] = normal_bf16(np.random.default_rng(8), inp.x.shape, 1.0)
    fwd = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, 2)
    bwd = oracle.moe_backward(inp.dOut, fwd, inp.W1, inp.W2)
    x = torch.from_numpy(_val(inp.x)).requires_grad_(True)
    p = torch.from_numpy(inp.prob.astype(np.float64)).requires_grad_(True)
    out = _torch_forward(x, inp.idx, p, torch.from_numpy(_val(inp.W1)),
                         torch.from_numpy(_val(inp.W2)))
    np.testing.assert_allclose(fwd["out"], out.detach().numpy(), rtol=1e-11, atol=1e-14)
    out.backward(torch.from_numpy(_val(inp.dOut)))
    np.testing.assert_allclose(bwd["dX"], x.grad.numpy(), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(bwd["dprob"], p.grad.numpy(), rtol=1e-10, atol=1e-13)
    # the per-token backward agrees as well
    for t in (0, 5, 23):
        dx = oracle.token_backward(inp.x[t], inp.dOut[t], inp.idx[t], inp.prob[t], inp.W1, inp.W2)
        np.testing.assert_allclose(dx, x.grad.numpy()[t], rtol=1e-10, atol=1e-13)
        dp = oracle.token_prob_grad(inp.x[t], inp.dOut[t], inp.idx[t], inp.W1, inp.W2)
        np.testing.assert_allclose(dp, p.grad.numpy()[t], rtol=1e-10, atol=1e-13)


def test_backward_matches_finite_differences():
    E, H, F, T, k = 3, 5, 3, 4, 2
    rng = np.random.default_rng(11)
    x = rng.standard_normal((T, H))
    W1 = rng.standard_normal((E, 2 * F, H)) * 0.7
    W2 = rng.standard_normal((E, H, F)) * 0.7
    idx = np.array([[0, 2], [1, 0], [2, 1], [0, 1]], np.int32)
    prob = rng.uniform(0.2, 1.0, (T, k))
    dOut = rng.standard_normal((T, H))
    fwd = oracle.moe_forward(x, idx, prob, W1, W2, E, 1)
    dX = oracle.moe_backward(dOut, fwd, W1, W2)["dX"]
    eps = 1e-6
    num = np.zeros_like(x)
    for t in range(T):
        for c in range(H):
            xp, xm = x.copy(), x.copy()
            xp[t, c] += eps
            xm[t, c] -= eps
            fp = oracle.moe_forward(xp, idx, prob, W1, W2, E, 1)["out"]
            fm = oracle.moe_forward(xm, idx, prob, W1, W2, E, 1)["out"]
            num[t, c] = np.sum(dOut * (fp - fm)) / (2 * eps)
    np.testing.assert_allclose(dX, num, rtol=1e-6, atol=1e-8)
    # and w.r.t. each routing probability (padding P = 4 leaves it unchanged)
    fwd4 = oracle.moe_forward(x, idx, prob, W1, W2, E, 4)
    dprob = oracle.moe_backward(dOut, fwd4, W1, W2)["dprob"]
    num_p = np.zeros_like(prob)
    for t in range(T):
        for j in range(k):
            pp, pm = prob.copy(), prob.copy()
            pp[t, j] += eps
            pm[t, j] -= eps
            fp = oracle.moe_forward(x, idx, pp, W1, W2, E, 1)["out"]
            fm = oracle.moe_forward(x, idx, pm, W1, W2, E, 1)["out"]
            num_p[t, j] = np.sum(dOut * (fp - fm)) / (2 * eps)
    np.testing.assert_allclose(dprob, num_p, rtol=1e-6, atol=1e-8)


def test_swiglu_backward_matches_finite_differences():
    rng = np.random.default_rng(12)
    H1 = rng.standard_normal((3, 8)) * 2
    dA = rng.standard_normal((3, 4))
    ana = oracle.swiglu_backward(dA, H1)
    eps = 1e-6
    num = np.zeros_like(H1)
    for i in range(H1.shape[0]):
        for j in range(H1.shape[1]):
            hp, hm = H1.copy(), H1.copy()
            hp[i, j] += eps
            hm[i, j] -= eps
            num[i, j] = np.sum(dA * (oracle.swiglu(hp) - oracle.swiglu(hm))) / (2 * eps)
    np.testing.assert_allclose(ana, num, rtol=1e-7, atol=1e-9)


def test_faithful_mode_error_budget_config1():
    # The BF16-rounded pipeline stays inside the parity tolerance of the exact
    # pipeline: this sizes the budget the GPU path has to meet.
    shape = CONFIGS[1]
    inp = make_inputs(shape, 1000)
    fe = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, 1)
    ff = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, 1, faithful=True)
    be = oracle.moe_backward(inp.dOut, fe, inp.W1, inp.W2)
    bf = oracle.moe_backward(inp.dOut, ff, inp.W1, inp.W2, faithful=True)
    for a, b in ((ff["out"], fe["out"]), (bf["dX"], be["dX"])):
        rel = np.linalg.norm(a - b) / np.linalg.norm(b)
        assert rel < 5e-3, rel
        assert np.all(np.abs(a - b) <= 1e-2 * np.abs(b) + 1e-3)


# ------------------------------------------------------------------ activation and
# probability variants (QuickGeGLU; probability at the activation or before FC1)

@pytest.mark.parametrize("activation", ["swiglu", "qgeglu"])
@pytest.mark.parametrize("prob_mode", ["combine", "activation", "pre_fc1"])
def test_variants_match_torch_autograd(activation, prob_mode):
    shape = CONFIGS[1].with_tokens(16)
    inp = make_inputs(shape, 1000)
    inp.W1[:] = normal_bf16(np.random.default_rng(5), inp.W1.shape, 0.2)
    inp.W2[:] = normal_bf16(np.random.default_rng(6), inp.W2.shape, 0.2)
    inp.x[:] = normal_bf16(np.random.default_rng(8), inp.x.shape, 1.0)
    fwd = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, 2,
                             activation=activation, prob_mode=prob_mode)
    bwd = oracle.moe_backward(inp.dOut, fwd, inp.W1, inp.W2)
    x = torch.from_numpy(_val(inp.x)).requires_grad_(True)
    p = torch.from_numpy(inp.prob.astype(np.float64)).requires_grad_(True)
    out = _torch_forward(x, inp.idx, p, torch.from_numpy(_val(inp.W1)),
                         torch.from_numpy(_val(inp.W2)), activation, prob_mode)
    np.testing.assert_allclose(fwd["out"], out.detach().numpy(), rtol=1e-11, atol=1e-14)
    out.backward(torch.from_numpy(_val(inp.dOut)))
    np.testing.assert_allclose(bwd["dX"], x.grad.numpy(), rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(bwd["dprob"], p.grad.numpy(), rtol=1e-10, atol=1e-13)
    for t in (0, 7, 15):
        y = oracle.token_forward(inp.x[t], inp.idx[t], inp.prob[t], inp.W1, inp.W2, activation,
                                 prob_mode)
        np.testing.assert_allclose(y, out.detach().numpy()[t], rtol=1e-11, atol=1e-14)
        dx = oracle.token_backward(inp.x[t], inp.dOut[t], inp.idx[t], inp.prob[t], inp.W1,
                                   inp.W2, activation, prob_mode)
        np.testing.assert_allclose(dx, x.grad.numpy()[t], rtol=1e-10, atol=1e-13)
        dp = oracle.token_prob_grad(inp.x[t], inp.dOut[t], inp.idx[t], inp.W1, inp.W2,
                                    activation, prob_mode, probs=inp.prob[t])
        np.testing.assert_allclose(dp, p.grad.numpy()[t], rtol=1e-10, atol=1e-13)


@pytest.mark.parametrize("activation", ["swiglu", "qgeglu"])
def test_probability_at_activation_is_the_combine_function(activation):
    # FC2 is linear and bias-free: p * FC2(act) = FC2(p * act), so both
    # placements give the same output and gradients (exact arithmetic).
    shape = CONFIGS[1]
    inp = make_inputs(shape, 1000)
    res = []
    for mode in ("combine", "activation"):
        f = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, shape.E, 1,
                               activation=activation, prob_mode=mode)
        b = oracle.moe_backward(inp.dOut, f, inp.W1, inp.W2)
        res.append((f["out"], b["dX"], b["dprob"]))
    for a, b in zip(*res):  # equal up to fp64 rounding order
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12 * np.max(np.abs(b)))


def test_qgeglu_identity_weights_closed_form():
    shape = CONFIGS[1]
    inp = make_inputs(shape, 1000, with_weights=False)
    W1, W2, F = _identity_weights(shape.E, shape.H)
    fwd = oracle.moe_forward(inp.x, inp.idx, inp.prob, W1, W2, shape.E, 1, activation="qgeglu")
    xv = _val(inp.x)
    sig = 1.0 / (1.0 + np.exp(-1.702 * xv))
    psum = inp.prob.astype(np.float64).sum(axis=1, keepdims=True)
    np.testing.assert_allclose(fwd["out"], psum * xv * sig * xv, rtol=1e-13, atol=0)
    bwd = oracle.moe_backward(inp.dOut, fwd, W1, W2)
    dv = _val(inp.dOut)
    # d/dx [x * sigmoid(1.702 x) * x] = 2 x s + 1.702 x^2 s (1 - s)
    deriv = 2 * xv * sig + 1.702 * xv * xv * sig * (1 - sig)
    np.testing.assert_allclose(bwd["dX"], psum * dv * deriv, rtol=1e-12, atol=1e-300)


def test_qgeglu_backward_matches_finite_differences():
    rng = np.random.default_rng(13)
    H1 = rng.standard_normal((3, 8)) * 2
    dA = rng.standard_normal((3, 4))
    ana = oracle.glu_backward(dA, H1, "qgeglu")
    eps = 1e-6
    num = np.zeros_like(H1)
    for i in range(H1.shape[0]):
        for j in range(H1.shape[1]):
            hp, hm = H1.copy(), H1.copy()
            hp[i, j] += eps
            hm[i, j] -= eps
            num[i, j] = np.sum(dA * (oracle.glu(hp, "qgeglu") - oracle.glu(hm, "qgeglu"))) / (2 * eps)
    np.testing.assert_allclose(ana, num, rtol=1e-7, atol=1e-9)
    # a planted wrong slope (SiLU's derivative on the QuickGELU gate) is caught
    assert not np.allclose(oracle.glu_backward(dA, H1, "swiglu"), num, rtol=1e-3)


def test_pre_fc1_gradients_match_finite_differences():
    E, H, F, T, k = 3, 5, 3, 4, 2
    rng = np.random.default_rng(17)
    x = rng.standard_normal((T, H))
    W1 = rng.standard_normal((E, 2 * F, H)) * 0.7
    W2 = rng.standard_normal((E, H, F)) * 0.7
    idx = np.array([[0, 2], [1, 0], [2, 1], [0, 1]], np.int32)
    prob = rng.uniform(0.2, 1.0, (T, k))
    dOut = rng.standard_normal((T, H))
    kw = dict(activation="qgeglu", prob_mode="pre_fc1")
    fwd = oracle.moe_forward(x, idx, prob, W1, W2, E, 1, **kw)
    bwd = oracle.moe_backward(dOut, fwd, W1, W2)
    eps = 1e-6

    def loss(xx, pp):
        return np.sum(dOut * oracle.moe_forward(xx, idx, pp, W1, W2, E, 1, **kw)["out"])

    num_x = np.zeros_like(x)
    for t in range(T):
        for c in range(H):
            xp, xm = x.copy(), x.copy()
            xp[t, c] += eps
            xm[t, c] -= eps
            num_x[t, c] = (loss(xp, prob) - loss(xm, prob)) / (2 * eps)
    num_p = np.zeros_like(prob)
    for t in range(T):
        for j in range(k):
            pp, pm = prob.copy(), prob.copy()
            pp[t, j] += eps
            pm[t, j] -= eps
            num_p[t, j] = (loss(x, pp) - loss(x, pm)) / (2 * eps)
    np.testing.assert_allclose(bwd["dX"], num_x, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(bwd["dprob"], num_p, rtol=1e-6, atol=1e-8)
