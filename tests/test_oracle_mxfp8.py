"""Pins of the MXFP8 oracle (``oracle/mxfp8.py``) to things other than itself.

* E4M3 rounding against PyTorch's float8_e4m3fn conversion (an independent
  library routine) over random values, every representable value and every
  midpoint between neighbours (ties to even);
* E4M3 byte encoding against PyTorch's bytes of the same values;
* block exponents against hand-derived cases and the minimality property;
* worked blocks whose codes are derived by hand;
* the half-step error bound of the format;
* the layer against the BF16 oracle: on inputs that MXFP8 represents exactly
  along both axes, the quantisations are the identity, so H1, A and the
  activation gradient must equal the BF16 oracle's (BF16-faithful) values,
  and the later tensors must stay within the format's error;
* the weight quantisation axes, with blocks that lose their small entries
  along one axis but not along the other;
* the combine-mode probability gradient against a central finite difference
  of the forward (exact: out is linear in the probabilities there) and
  against the closed form of identity weights; the weighted-activation
  probability gradient against its closed form on identity weights."""

import numpy as np
import pytest
import torch

import oracle
from oracle import mxfp8 as mxo


def _torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn)


def _all_finite_e4m3():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    return codes, mxo.e4m3_value(codes)


def test_e4m3_values_and_bytes_match_torch():
    codes, vals = _all_finite_e4m3()
    tv = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    np.testing.assert_array_equal(vals, tv)
    assert np.max(vals) == 448.0 and np.min(np.abs(vals[vals != 0])) == 2.0 ** -9
    # the encoder inverts the decoder (signed zeros included)
    np.testing.assert_array_equal(mxo.e4m3_bits(vals), codes)
    # every E4M3 number is a fixed point of the rounding
    np.testing.assert_array_equal(mxo.e4m3_round(vals), vals)


def test_e4m3_round_matches_torch_random_and_midpoints():
    rng = np.random.default_rng(3)
    v = np.concatenate([
        rng.standard_normal(20000) * 60.0,
        rng.uniform(-2.0 ** -5, 2.0 ** -5, 5000),    # subnormal range
        rng.uniform(-463.0, 463.0, 5000),
    ])
    v = v.astype(np.float32).astype(np.float64)      # torch converts from fp32
    np.testing.assert_array_equal(
        mxo.e4m3_round(v), _torch_e4m3(v).float().numpy().astype(np.float64))
    _, vals = _all_finite_e4m3()
    pos = np.unique(vals[vals >= 0])
    mids = (pos[1:] + pos[:-1]) / 2                  # exact ties, fp32-representable
    got = mxo.e4m3_round(np.concatenate([mids, -mids]))
    ref = _torch_e4m3(np.concatenate([mids, -mids])).float().numpy().astype(np.float64)
    np.testing.assert_array_equal(got, ref)
    # a tie goes to the even mantissa: 17 -> 16, 19 -> 20, 2^-10 -> 0
    np.testing.assert_array_equal(mxo.e4m3_round(np.array([17.0, 19.0, 2.0 ** -10])),
                                  [16.0, 20.0, 0.0])
    # saturation above the largest value
    np.testing.assert_array_equal(mxo.e4m3_round(np.array([449.0, 1e6, -1e6])),
                                  [448.0, 448.0, -448.0])


def test_block_exponent_cases_and_minimality():
    cases = {448.0: 0, 448.5: 1, 1.0: -8, 1.75: -8, 1.8: -7, 3.0: -7, 0.0: -127,
             2.0 ** -140: -127, 2.0 ** 130: 122, 2.0 ** 140: 127, 896.0: 1, 2.0 ** -9: -17}
    for amax, e in cases.items():
        assert mxo.block_exponent(np.array([amax]))[0] == e, amax
    rng = np.random.default_rng(4)
    amax = np.exp(rng.uniform(-60, 60, 20000))
    e = mxo.block_exponent(amax)
    assert np.all(amax / np.ldexp(1.0, e) <= 448.0)
    assert np.all(amax / np.ldexp(1.0, e - 1) > 448.0)


def test_worked_blocks():
    v = np.zeros((2, 32))
    v[0, :4] = [448.0, 1.0, -0.5, -0.0]              # e = 0: the values themselves
    v[1, :3] = [3.0, -0.03125, 1e-4]                  # amax 3 = 1.5 * 2^1: e = -7
    q, e = mxo.quantize(v)
    assert e.tolist() == [[0], [-7]]
    bits = mxo.e4m3_bits(q)
    assert bits[0, :4].tolist() == [0x7E, 0x38, 0xB0, 0x80]
    # 3 * 2^7 = 384 = 1.5 * 2^8 -> 0x7C; -0.03125 * 2^7 = -4 -> 0xC8;
    # 1e-4 * 2^7 = 0.0128 -> nearest multiple of 2^-9 is 7 * 2^-9 -> 0x07
    assert bits[1, :3].tolist() == [0x7C, 0xC8, 0x07]
    np.testing.assert_array_equal(bits[:, 4:], np.where(np.signbit(v[:, 4:]), 0x80, 0))


def test_quantisation_error_bound_and_idempotence():
    rng = np.random.default_rng(5)
    v = rng.standard_normal((64, 256)) * np.exp(rng.uniform(-8, 8, (64, 1)))
    q, e = mxo.quantize(v)
    d = mxo.dequantize(q, e)
    scale = np.repeat(np.ldexp(1.0, e), 32, axis=1)
    a = np.abs(v) / scale
    err = np.abs(d - v) / scale
    normal = a >= 2.0 ** -6
    assert np.all(err[normal] <= a[normal] * 2.0 ** -4 + 1e-300)   # half of a 3-bit step
    assert np.all(err[~normal] <= 2.0 ** -10)                       # half the subnormal step
    np.testing.assert_array_equal(mxo.mx(d), d)


def _representable(rng, shape, unit):
    # entries unit * {0, +-0.25, +-0.5, +-1, +-1.5}: every 32-block along any
    # axis has a scale at which all of them are E4M3 numbers
    choices = np.array([0.0, 0.25, -0.25, 0.5, -0.5, 1.0, -1.0, 1.5, -1.5])
    return rng.choice(choices, size=shape) * unit


def test_layer_reduces_to_bf16_oracle_on_representable_inputs():
    rng = np.random.default_rng(6)
    E, H, F, T, k = 4, 64, 96, 40, 2
    x = _representable(rng, (T, H), 1.0)
    W1 = _representable(rng, (E, 2 * F, H), 2.0 ** -4)
    W2 = _representable(rng, (E, H, F), 2.0 ** -4)
    dOut = _representable(rng, (T, H), 0.5)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    prob = rng.uniform(0.1, 1.0, (T, k)).astype(np.float32)
    W = mxo.mx_weights(W1, W2)
    for name, ref in (("W1f", W1), ("W1d", W1), ("W2f", W2), ("W2d", W2)):
        np.testing.assert_array_equal(W[name], ref, err_msg=name)
    for mode in ("combine", "activation"):
        mf = mxo.mx_forward(x, idx, prob, W1, W2, E, 1, prob_mode=mode)
        bf = oracle.moe_forward(x, idx, prob, W1, W2, E, 1, faithful=True, prob_mode=mode)
        np.testing.assert_array_equal(mf["Xq"], bf["Xp"])
        np.testing.assert_array_equal(mf["H1"], bf["H1"])
        np.testing.assert_array_equal(mf["A"], bf["A"])
        rel = np.linalg.norm(mf["out"] - bf["out"]) / np.linalg.norm(bf["out"])
        assert 0 < rel < 0.05, rel                    # only mx(A) differs
        mb = mxo.mx_backward(dOut, mf)
        bb = oracle.moe_backward(dOut, oracle.moe_forward(x, idx, prob, W1, W2, E, 1,
                                                          prob_mode=mode), W1, W2)
        # the activation gradient before the SwiGLU backward: the exact product
        # (the quantisations are the identity here), rounded once to BF16
        dA_ref = oracle.round_to_bf16(oracle.grouped_linear_t(bb["dYp"], W2, mf["offsets"]))
        np.testing.assert_array_equal(mb["dA"], dA_ref * mf["pr"][:, None])
        rel = np.linalg.norm(mb["dX"] - bb["dX"]) / np.linalg.norm(bb["dX"])
        assert rel < 0.05, rel
        rel = np.linalg.norm(mb["dprob"] - bb["dprob"]) / np.linalg.norm(bb["dprob"])
        assert rel < 0.05, rel


def test_layer_error_against_bf16_oracle_is_the_format_error():
    from moe_synth import CONFIGS, make_inputs

    s = CONFIGS[1]
    inp = make_inputs(s, 11)
    for mode in ("combine", "pre_fc1"):
        mf = mxo.mx_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, s.E, s.P, prob_mode=mode)
        bf = oracle.moe_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, s.E, s.P,
                                prob_mode=mode)
        rel = np.linalg.norm(mf["out"] - bf["out"]) / np.linalg.norm(bf["out"])
        assert 0.005 < rel < 0.08, rel                # E4M3 keeps 3 mantissa bits
        mb = mxo.mx_backward(inp.dOut, mf)
        bb = oracle.moe_backward(inp.dOut, bf, inp.W1, inp.W2)
        for name in ("dX", "dprob"):
            rel = np.linalg.norm(mb[name] - bb[name]) / np.linalg.norm(bb[name])
            assert 0.005 < rel < 0.1, (name, rel)


def test_weight_quantisation_axes():
    # W1[e, n, :] (one output row) holds one large entry per 32-block along
    # the input dimension; every other entry is tiny. Along the input
    # dimension the tiny entries fall below the smallest step and vanish;
    # along the output dimension they sit in blocks of tiny values and stay.
    E, F, H = 1, 32, 64
    W1 = np.full((E, 2 * F, H), 2.0 ** -10)
    W1[0, :, ::32] = 2.0 ** 10
    W2 = np.full((E, H, F), 2.0 ** -10)
    W2[0, ::32, :] = 2.0 ** 10
    W = mxo.mx_weights(W1, W2)
    tiny1 = W1 == 2.0 ** -10
    tiny2 = W2 == 2.0 ** -10
    assert np.all(W["W1f"][tiny1] == 0) and np.all(W["W1d"][tiny1] == 2.0 ** -10)
    assert np.all(W["W2d"][tiny2] == 0) and np.all(W["W2f"][tiny2] == 2.0 ** -10)


def test_quantize_rejects_ragged_axis():
    with pytest.raises(ValueError):
        mxo.quantize(np.zeros((2, 48)))


def test_combine_mode_prob_grad_is_the_derivative_of_the_forward():
    # In combine mode out_t = sum_j p_tj * Yp[row(t, j)]: out is linear in
    # every p_tj and no quantiser sits between p and out, so the central
    # difference of L = <dOut, out> through mx_forward is the exact
    # derivative, whatever the step. mx_backward's dprob must equal it.
    from moe_synth import MoeShape, make_inputs

    s = MoeShape("fd_e4_h64_f64_t16_k2", E=4, H=64, F=64, T=16, k=2, x_std=1.0, w_std=0.1)
    inp = make_inputs(s, 71)
    W = mxo.mx_weights(inp.W1, inp.W2)
    f = mxo.mx_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, s.E, weights=W)
    dprob = mxo.mx_backward(inp.dOut, f)["dprob"]
    dOut = oracle.bf16_bits_to_f64(inp.dOut)
    prob = inp.prob.astype(np.float64)
    h = 0.25
    for t, j in [(0, 0), (3, 1), (9, 0), (15, 1)]:
        loss = []
        for sgn in (1.0, -1.0):
            p = prob.copy()
            p[t, j] += sgn * h
            out = mxo.mx_forward(inp.x, inp.idx, p, inp.W1, inp.W2, s.E, weights=W)["out"]
            loss.append(float(np.sum(dOut * out)))
        fd = (loss[0] - loss[1]) / (2 * h)
        assert abs(fd - dprob[t, j]) <= 1e-10 * max(1.0, abs(fd)), (t, j, fd, dprob[t, j])

    # The pin has teeth: the route through the input-gradient GEMM (quantised
    # dOut against the output-dimension quantisation of W2, dotted with the
    # activation) is a different number once the operands are quantised.
    dYp = np.zeros_like(f["Yp"])
    valid = f["slot_of_row"] >= 0
    dYp[valid] = dOut[f["slot_of_row"][valid] // s.k]
    dA0 = oracle.round_to_bf16(oracle.grouped_linear_t(mxo.mx(dYp), W["W2d"], f["offsets"]))
    other_rows = np.sum(dA0 * oracle.glu(f["H1"], "swiglu"), axis=1)
    other = np.zeros(s.T * s.k)
    other[f["slot_of_row"][valid]] = other_rows[valid]
    rel = np.linalg.norm(other - dprob.reshape(-1)) / np.linalg.norm(dprob)
    assert rel > 1e-3, rel


def test_combine_mode_prob_grad_closed_form_on_identity_weights():
    # Gate and up blocks [I; 0] and W2 = [I 0] are exact in MXFP8, and so are
    # inputs x on the representable grid. Then H1 = [x, x], A = bf16(x^2
    # sigmoid(x)) and Yp = mx(A), so in closed form
    # dprob_tj = <dOut_t, mx(bf16(x_t^2 sigmoid(x_t)))> for every pair.
    rng = np.random.default_rng(12)
    E, H, F, T, k = 2, 64, 64, 8, 2
    W1 = np.zeros((E, 2 * F, H))
    W1[:, :H, :] = np.eye(H)
    W1[:, F:F + H, :] = np.eye(H)
    W2 = np.zeros((E, H, F))
    W2[:, :, :H] = np.eye(H)
    x = _representable(rng, (T, H), 1.0)
    dOut = _representable(rng, (T, H), 0.5)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    prob = rng.uniform(0.1, 1.0, (T, k))
    f = mxo.mx_forward(x, idx, prob, W1, W2, E)
    b = mxo.mx_backward(dOut, f)
    sor = f["slot_of_row"]
    valid = sor >= 0
    np.testing.assert_array_equal(f["H1"][valid][:, :H], x[sor[valid] // k])
    np.testing.assert_array_equal(f["H1"][valid][:, F:], x[sor[valid] // k])
    y = mxo.mx(oracle.round_to_bf16(x * x / (1.0 + np.exp(-x))))
    for t in range(T):
        for j in range(k):
            np.testing.assert_allclose(b["dprob"][t, j], np.dot(dOut[t], y[t]), rtol=1e-13,
                                       atol=1e-13)


def test_weighted_activation_prob_grad_closed_form_on_identity_weights():
    # With the probability inside the activation, A = bf16(p * act(H1)) and
    # the quantiser of A passes the gradient straight through, so dprob is
    # the row sum of dA0 * act(H1). With gate and up blocks [I; 0], W2 = [I 0]
    # and representable x and dOut, dA0 = dOut (exact in every format) and
    # act(H1) = x^2 sigmoid(x): dprob_tj = <dOut_t, x_t^2 sigmoid(x_t)>.
    rng = np.random.default_rng(13)
    E, H, F, T, k = 2, 64, 64, 8, 2
    W1 = np.zeros((E, 2 * F, H))
    W1[:, :H, :] = np.eye(H)
    W1[:, F:F + H, :] = np.eye(H)
    W2 = np.zeros((E, H, F))
    W2[:, :, :H] = np.eye(H)
    x = _representable(rng, (T, H), 1.0)
    dOut = _representable(rng, (T, H), 0.5)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    prob = rng.uniform(0.1, 1.0, (T, k))
    f = mxo.mx_forward(x, idx, prob, W1, W2, E, prob_mode="activation")
    b = mxo.mx_backward(dOut, f)
    act = x * x / (1.0 + np.exp(-x))
    for t in range(T):
        for j in range(k):
            np.testing.assert_allclose(b["dprob"][t, j], np.dot(dOut[t], act[t]), rtol=1e-13,
                                       atol=1e-13)
