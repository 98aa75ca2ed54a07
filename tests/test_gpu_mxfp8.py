"""GPU parity of the MXFP8 path (gg_mx_* calls, MxMoeLayer) against the MXFP8
oracle (``oracle/mxfp8.py``).

* quantisers: the permuted activation rows (plain and probability-scaled) and
  the four weight operands, byte for byte (E4M3 codes and E8M0 scales in the
  documented tile layouts);
* each grouped GEMM from the kernels' own inputs: FC1's H1 and FC2's, the
  input-gradient GEMMs' outputs at oracle parity; the E4M3 codes FC1 and the
  SwiGLU-backward epilogue write, against the oracle's quantisation of the
  same BF16 values (the kernel takes that decision in FP32 arithmetic, the
  oracle in FP64: a rare value on a rounding boundary may differ by one step);
* the whole layer, forward and backward, for both activations and the three
  probability placements, on ragged and padded batches, and CUDA-graph
  replay."""

import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_parity, bits_to_torch, torch_to_f64
from moe_synth import MoeShape, make_inputs
from oracle import mxfp8 as mxo

pytestmark = pytest.mark.gpu

# H, F multiples of 128; H = 384 gives a ragged last FC2 / input-gradient
# tile (256 + 128 columns), F = 384 a ragged SwiGLU-backward tile, P = 16
# padding rows
MX_MID = MoeShape("mx_e8_h384_f256_t300_k2", E=8, H=384, F=256, T=300, k=2, routing="uniform",
                  x_std=1.0, w_std=0.05)
MX_PAD = MoeShape("mx_e6_h256_f384_t257_k3_pad16", E=6, H=256, F=384, T=257, k=3, P=16,
                  routing="uniform", x_std=1.0, w_std=0.05)
# H = 2688: a row of 336 16-byte chunks, one full pass of the row quantiser's
# lanes (256 chunks) and a partial one
MX_WIDE = MoeShape("mx_e4_h2688_f128_t70_k4_pad8", E=4, H=2688, F=128, T=70, k=4, P=8,
                   routing="uniform", x_std=1.0, w_std=0.05)
ACTS = {0: "swiglu", 1: "qgeglu"}
MODES = {0: "combine", 1: "activation", 2: "pre_fc1"}


@pytest.fixture(scope="module")
def gg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from moe_expert_grouped_gb300 import build

    build.build()
    import moe_expert_grouped_gb300.gg as mod

    return mod


# ------------------------------------------------------------ scale-tile layouts

def _sf_byte(r, b):
    return (r % 32) * 16 + (r // 32) * 4 + b


def _tiles_before(offsets):
    n = np.diff(offsets)
    t = (n + 127) // 128
    return np.concatenate([[0], np.cumsum(t)]).astype(np.int64)


def _row_tiles(codes, offsets, n_tiles, K):
    """Expected activation scale tiles from per-row codes [R_cap, K/32]."""
    tb = _tiles_before(offsets)
    S = np.zeros((n_tiles, K // 128, 512), np.uint8)
    for e in range(len(offsets) - 1):
        for t in range(tb[e + 1] - tb[e]):
            for r in range(128):
                g = offsets[e] + t * 128 + r
                row = codes[g] if g < offsets[e + 1] else np.zeros(K // 32, np.uint8)
                for blk in range(K // 32):
                    S[tb[e] + t, blk // 4, _sf_byte(r, blk % 4)] = row[blk]
    return S


def _row_codes(S, offsets, R_cap, K):
    """Per-row codes [R_cap, K/32] read back from activation scale tiles."""
    tb = _tiles_before(offsets)
    codes = np.zeros((R_cap, K // 32), np.int64)
    for e in range(len(offsets) - 1):
        for g in range(offsets[e], offsets[e + 1]):
            t = tb[e] + (g - offsets[e]) // 128
            r = (g - offsets[e]) % 128
            for blk in range(K // 32):
                codes[g, blk] = S[t, blk // 4, _sf_byte(r, blk % 4)]
    return codes


def _deq(Q, codes):
    """Exact values of E4M3 bytes Q [R, K] with per-row block codes [R, K/32]."""
    return mxo.dequantize(mxo.e4m3_value(Q), codes.astype(np.int64) - 127)


def _weight_tiles(codes, NT, K, gated_F=0):
    """Expected weight scale tiles [E, NT, K/128, 1024] from codes [E, N, K/32]."""
    E, N, _ = codes.shape
    S = np.zeros((E, NT, K // 128, 1024), np.uint8)
    for n in range(N):
        if gated_F:
            up = n >= gated_F
            j = n - gated_F if up else n
            nt, col = j // 128, j % 128 + (128 if up else 0)
        else:
            nt, col = n // 256, n % 256
        for blk in range(K // 32):
            S[:, nt, blk // 4, (col // 128) * 512 + _sf_byte(col % 128, blk % 4)] = codes[:, n, blk]
    return S


def _quant_bits(v):
    q, e = mxo.quantize(v)
    return mxo.e4m3_bits(q), (e + 127).astype(np.uint8)


def _maps(gg, d, s):
    m = gg.permute(d["x"], d["idx"], d["prob"], s.E, s.P, out={"Xp": None})
    return m, m["offsets"].cpu().numpy().astype(np.int64), m["slot_of_row"].cpu().numpy()


def _dev(inp):
    return dict(x=bits_to_torch(inp.x), idx=torch.from_numpy(inp.idx).cuda(),
                prob=torch.from_numpy(inp.prob).cuda(), W1=bits_to_torch(inp.W1),
                W2=bits_to_torch(inp.W2), dOut=bits_to_torch(inp.dOut))


# ------------------------------------------------------------ quantisers

@pytest.mark.parametrize("shape,scaled", [(MX_MID, False), (MX_PAD, False), (MX_PAD, True),
                                          (MX_WIDE, False), (MX_WIDE, True)])
def test_quantize_rows_bit_exact(gg, shape, scaled):
    s = shape
    inp = make_inputs(s, 31)
    x = inp.x.copy()
    x[0] = 0                                  # an all-zero row: code 0, zero elements
    x[1] = 0x8000                             # negative zeros keep their sign
    x[2] = np.uint16(0x0080)                  # the smallest normal BF16: clamped exponent
    x[3, ::7] = np.uint16(0x7E80)             # one huge value per block group (~8.5e37)
    d = _dev(inp)
    d["x"] = bits_to_torch(x)
    m, off, sor = _maps(gg, d, s)
    rc = gg.r_cap(s.T, s.k, s.E, s.P)
    ws = m["ws"]
    # E4M3 NaN codes and 0xFF scale bytes where nothing is written: padding
    # rows or scale bytes left unwritten fail below
    n_tiles = (rc + 127) // 128 + s.E
    pre = dict(Q=torch.full((rc, s.H), 0x7F, dtype=torch.uint8, device="cuda"),
               S=torch.full((n_tiles, s.H // 128, 512), 0xFF, dtype=torch.uint8, device="cuda"))
    res = gg.mx_quantize_rows(d["x"], m, s.k, s.E, s.P, ws, prob=d["prob"] if scaled else None,
                              n_tiles=n_tiles, out=pre)
    torch.cuda.synchronize()
    assert gg.read_status(ws) == 0
    n = int(off[-1])
    xf = oracle.bf16_bits_to_f64(x)
    src = np.zeros((rc, s.H))
    live = sor[:n] >= 0
    src[:n][live] = xf[sor[:n][live] // s.k]
    if scaled:  # the kernel's order: FP32 product, then BF16 rounding
        por = m["prob_of_row"].cpu().numpy()
        prod = (src[:n].astype(np.float32) * por[:n, None].astype(np.float32)).astype(np.float64)
        src[:n] = oracle.round_to_bf16(prod)
    bits, codes = _quant_bits(src)
    np.testing.assert_array_equal(res["Q"][:n].cpu().numpy(), bits[:n])
    np.testing.assert_array_equal(res["tiles_before"].cpu().numpy(), _tiles_before(off))
    S_ref = _row_tiles(codes, off, res["S"].shape[0], s.H)
    np.testing.assert_array_equal(res["S"].cpu().numpy(), S_ref)


@pytest.mark.parametrize("P", [1, 16])
def test_quantize_rows_empty_batch(gg, P):
    # no tokens: the tile prefix is all zero and every scale byte gets code 0
    # (the buffers start as NaN codes and 0xFF scale bytes)
    E, K, k = 5, 256, 2
    x = torch.empty((0, K), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((0, k), dtype=torch.int32, device="cuda")
    prob = torch.empty((0, k), dtype=torch.float32, device="cuda")
    m = gg.permute(x, idx, prob, E, P, out={"Xp": None})
    rc = gg.r_cap(0, k, E, P)
    n_tiles = (rc + 127) // 128 + E
    pre = dict(Q=torch.full((max(rc, 1), K), 0x7F, dtype=torch.uint8, device="cuda"),
               S=torch.full((n_tiles, K // 128, 512), 0xFF, dtype=torch.uint8, device="cuda"),
               tiles_before=torch.full((E + 1,), 7, dtype=torch.int32, device="cuda"))
    res = gg.mx_quantize_rows(x, m, k, E, P, m["ws"], n_tiles=n_tiles, out=pre)
    torch.cuda.synchronize()
    assert gg.read_status(m["ws"]) == 0
    assert np.all(res["tiles_before"].cpu().numpy() == 0)
    assert np.all(res["S"].cpu().numpy() == 0)


@pytest.mark.parametrize("E,H,F", [(3, 256, 384), (2, 384, 128)])
def test_prepare_weights_bit_exact(gg, E, H, F):
    rng = np.random.default_rng(E * 1000 + F)
    W1 = oracle.round_to_bf16(rng.standard_normal((E, 2 * F, H)) * 0.05)
    W2 = oracle.round_to_bf16(rng.standard_normal((E, H, F)) * 0.05)
    W1[0, 5] = 0.0
    W2[-1, :, 3] = -0.0
    W1[1 % E, 7, :32] = 3.0e4     # one block dominated by a large value
    tb = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).cuda()  # noqa: E731
    mxw, L = gg.mx_prepare_weights(tb(W1), tb(W2))
    torch.cuda.synchronize()
    got = mxw.cpu().numpy()
    ops = {"w1": (W1, F // 128, F), "w2": (W2, (H + 255) // 256, 0),
           "w2t": (np.swapaxes(W2, 1, 2), (F + 255) // 256, 0),
           "w1t": (np.swapaxes(W1, 1, 2), (H + 255) // 256, 0)}
    for name, (Wop, NT, gF) in ops.items():
        Ex, N, K = Wop.shape
        bits, codes = _quant_bits(Wop)
        q = got[L[name]:L[name] + Ex * N * K].reshape(Ex, N, K)
        np.testing.assert_array_equal(q, bits, err_msg=name)
        nb = Ex * NT * (K // 128) * 1024
        S = got[L[name + "_scales"]:L[name + "_scales"] + nb].reshape(Ex, NT, K // 128, 1024)
        np.testing.assert_array_equal(S, _weight_tiles(codes, NT, K, gF), err_msg=name)


# ------------------------------------------------------------ the four GEMMs

def _assert_codes_close(got_q, got_c, ref_q, ref_c, what, max_frac=2e-3):
    """E4M3 codes and block scales equal except on rare rounding boundaries:
    there a value (or, when it is the block maximum, its block's scale) moves
    by one step, so the dequantised values differ by at most a quarter of
    their magnitude plus the block's smallest step."""
    gv = _deq(got_q, got_c)
    rv = _deq(ref_q, ref_c)
    diff = gv != rv
    frac = diff.mean() if diff.size else 0.0
    assert frac <= max_frac, f"{what}: {diff.sum()} of {diff.size} values differ"
    if diff.any():
        tiny = np.repeat(np.ldexp(1.0, ref_c.astype(np.int64) - 127 - 8), 32, axis=1)[diff]
        bound = 0.25 * np.maximum(np.abs(gv[diff]), np.abs(rv[diff])) + tiny
        assert np.all(np.abs(gv[diff] - rv[diff]) <= bound), what


@pytest.mark.parametrize("shape,act", [(MX_MID, 0), (MX_PAD, 1)])
def test_grouped_gemms_match_oracle(gg, shape, act):
    s = shape
    inp = make_inputs(s, 47)
    d = _dev(inp)
    m, off, sor = _maps(gg, d, s)
    rc = gg.r_cap(s.T, s.k, s.E, s.P)
    n = int(off[-1])
    ws = m["ws"]
    mxw, _ = gg.mx_prepare_weights(d["W1"], d["W2"])
    W = mxo.mx_weights(inp.W1, inp.W2)
    xq = gg.mx_quantize_rows(d["x"], m, s.k, s.E, s.P, ws)
    por_t = m["prob_of_row"]
    # FC1 (+ the weighted activation)
    Aq, As, H1 = gg.mx_grouped_gemm(gg.GG_MX_FC1, xq["Q"], xq["S"], mxw, m["offsets"], s.E, rc,
                                    s.H, s.F, ws, activation=act, row_scale=por_t)
    # FC2 on the kernel's own quantised activation
    Yp = gg.mx_grouped_gemm(gg.GG_MX_FC2, Aq, As, mxw, m["offsets"], s.E, rc, s.H, s.F, ws,
                            activation=act)
    # input gradient: dOut rows quantised, FC2's input gradient + activation backward
    dyq = gg.mx_quantize_rows(d["dOut"], m, s.k, s.E, s.P, ws)
    rowdot = torch.zeros((rc, gg.mx_rowdot_stride(s.F)), dtype=torch.float32, device="cuda")
    dHq, dHs = gg.mx_grouped_gemm(gg.GG_MX_DGRAD_FC2, dyq["Q"], dyq["S"], mxw, m["offsets"],
                                  s.E, rc, s.H, s.F, ws, activation=act, H1=H1,
                                  row_scale=por_t, rowdot=rowdot)
    dXp = gg.mx_grouped_gemm(gg.GG_MX_DGRAD_FC1, dHq, dHs, mxw, m["offsets"], s.E, rc, s.H, s.F,
                             ws)
    torch.cuda.synchronize()
    assert gg.read_status(ws) == 0
    name = ACTS[act]
    por = por_t.cpu().numpy().astype(np.float64)[:n, None]

    def rows(Q, S, K):
        """Exact values of the first n rows of a kernel-written E4M3 operand,
        zero rows after them (never written: those buffers start empty)."""
        v = np.zeros((rc, K))
        v[:n] = _deq(Q.cpu().numpy()[:n], _row_codes(S.cpu().numpy(), off, rc, K)[:n])
        return v

    def codes(Q, S, K):
        return Q.cpu().numpy()[:n], _row_codes(S.cpu().numpy(), off, rc, K)[:n]

    # FC1: H1 = bf16(Xq W1f^T)
    H1_ref = oracle.grouped_linear(rows(xq["Q"], xq["S"], s.H), W["W1f"], off)[:n]
    H1k = torch_to_f64(H1[:n])
    assert_parity(H1k, H1_ref, "H1", faithful=oracle.round_to_bf16(H1_ref))
    # the activation codes, from the kernel's own H1
    aq_ref, ac_ref = _quant_bits(oracle.round_to_bf16(oracle.glu(H1k, name) * por))
    _assert_codes_close(*codes(Aq, As, s.F), aq_ref, ac_ref, "A")
    # FC2 from the kernel's codes
    Yp_ref = oracle.grouped_linear(rows(Aq, As, s.F), W["W2f"], off)[:n]
    assert_parity(torch_to_f64(Yp[:n]), Yp_ref, "Yp", faithful=oracle.round_to_bf16(Yp_ref))
    # dgrad FC2 + activation backward from the kernel's dYq and H1
    dA0 = oracle.round_to_bf16(
        oracle.grouped_linear_t(rows(dyq["Q"], dyq["S"], s.H), W["W2d"], off)[:n])
    dq_ref, dc_ref = _quant_bits(oracle.round_to_bf16(oracle.glu_backward(dA0 * por, H1k, name)))
    _assert_codes_close(*codes(dHq, dHs, 2 * s.F), dq_ref, dc_ref, "dH1")
    rd = rowdot.cpu().numpy()[:n, :gg.mx_rowdot_blocks(s.F)].astype(np.float64).sum(axis=1)
    # the kernel pairs the accumulator with the BF16 value of the activation
    assert_parity(rd, np.sum(dA0 * oracle.glu(H1k, name), axis=1), "rowdot",
                  faithful=np.sum(dA0 * oracle.round_to_bf16(oracle.glu(H1k, name)), axis=1))
    # dgrad FC1 from the kernel's dH1 codes
    dXp_ref = oracle.grouped_linear_t(rows(dHq, dHs, 2 * s.F), W["W1d"], off)[:n]
    assert_parity(torch_to_f64(dXp[:n]), dXp_ref, "dXp", faithful=oracle.round_to_bf16(dXp_ref))


# ------------------------------------------------------------ the layer

def _layer(gg, s, d, mxw, act=0, mode=0):
    layer = gg.MxMoeLayer(s.T, s.H, s.F, s.k, s.E, s.P, activation=act, prob_mode=mode)
    out = layer.forward(d["x"], d["idx"], d["prob"], mxw)
    dX, dprob = layer.backward(d["dOut"], mxw, dprob=True)
    torch.cuda.synchronize()
    assert layer.status() == 0
    return layer, out, dX, dprob


@pytest.mark.parametrize("shape,act,mode", [(MX_MID, 0, 0), (MX_MID, 1, 1), (MX_PAD, 0, 2),
                                            (MX_PAD, 1, 0), (MX_PAD, 0, 1), (MX_MID, 1, 2)])
def test_layer_matches_oracle(gg, shape, act, mode):
    s = shape
    inp = make_inputs(s, 53 + act + 3 * mode)
    d = _dev(inp)
    mxw, _ = gg.mx_prepare_weights(d["W1"], d["W2"])
    layer, out, dX, dprob = _layer(gg, s, d, mxw, act, mode)
    kw = dict(activation=ACTS[act], prob_mode=MODES[mode])
    f = mxo.mx_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, s.E, s.P, **kw)
    b = mxo.mx_backward(inp.dOut, f)
    ff = mxo.mx_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, s.E, s.P, faithful=True, **kw)
    fb = mxo.mx_backward(inp.dOut, ff)
    assert_parity(torch_to_f64(out), f["out"], "out", faithful=ff["out"], scope="tensor")
    assert_parity(torch_to_f64(dX), b["dX"], "dX", faithful=fb["dX"], scope="tensor")
    assert_parity(dprob.cpu().numpy().astype(np.float64), b["dprob"], "dprob",
                  faithful=fb["dprob"], scope="tensor")
    n = int(f["offsets"][-1])
    np.testing.assert_array_equal(layer.view("offsets").cpu().numpy(), f["offsets"])
    assert_parity(torch_to_f64(layer.view("H1")[:n]), f["H1"][:n], "H1",
                  faithful=f["H1"][:n])


def test_layer_run_to_run_and_graph_replay(gg):
    s = MX_PAD
    inp = make_inputs(s, 61)
    d = _dev(inp)
    mxw, _ = gg.mx_prepare_weights(d["W1"], d["W2"])
    _, out1, dX1, dp1 = _layer(gg, s, d, mxw)
    _, out2, dX2, dp2 = _layer(gg, s, d, mxw)
    assert torch.equal(out1, out2) and torch.equal(dX1, dX2) and torch.equal(dp1, dp2)
    layer = gg.MxMoeLayer(s.T, s.H, s.F, s.k, s.E, s.P)
    out = torch.empty_like(out1)
    dX = torch.empty_like(dX1)
    dp = torch.empty_like(dp1)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        layer.forward(d["x"], d["idx"], d["prob"], mxw, out=out)
        layer.backward(d["dOut"], mxw, dX=dX, dprob=dp)
    torch.cuda.current_stream().wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(d["x"], d["idx"], d["prob"], mxw, out=out)
        layer.backward(d["dOut"], mxw, dX=dX, dprob=dp)
    out.zero_()
    dX.zero_()
    dp.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(out, out1) and torch.equal(dX, dX1) and torch.equal(dp, dp1)


def test_layer_empty_batch_and_zero_token_experts(gg):
    s = MoeShape("mx_e8_h256_f256_t40_k2_skew", E=8, H=256, F=256, T=40, k=2, routing="uniform",
                 x_std=1.0, w_std=0.05)
    inp = make_inputs(s, 71)
    inp.idx[:] = inp.idx % 3          # experts 3..7 get no tokens
    d = _dev(inp)
    mxw, _ = gg.mx_prepare_weights(d["W1"], d["W2"])
    _, out, dX, dprob = _layer(gg, s, d, mxw)
    f = mxo.mx_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, s.E, s.P)
    ff = mxo.mx_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, s.E, s.P, faithful=True)
    assert_parity(torch_to_f64(out), f["out"], "out", faithful=ff["out"], scope="tensor")
    b, fb = mxo.mx_backward(inp.dOut, f), mxo.mx_backward(inp.dOut, ff)
    assert_parity(torch_to_f64(dX), b["dX"], "dX", faithful=fb["dX"], scope="tensor")
    empty = gg.MxMoeLayer(0, s.H, s.F, s.k, s.E, s.P)
    o = empty.forward(d["x"][:0], d["idx"][:0], d["prob"][:0], mxw)
    g = empty.backward(d["dOut"][:0], mxw)
    torch.cuda.synchronize()
    assert o.shape == (0, s.H) and g.shape == (0, s.H)


def test_layer_fullsize_sampled_parity(gg):
    """The balanced 128-expert layer at full size (the benchmark's workload and
    launch configuration); outputs and gradients of a seeded token sample
    against the MXFP8 oracle run on that sub-batch (rows are independent, the
    weights' quantisation does not depend on the batch)."""
    from moe_synth import CONFIGS

    s = CONFIGS[2]
    inp = make_inputs(s, 2000 + 17)
    d = _dev(inp)
    mxw, _ = gg.mx_prepare_weights(d["W1"], d["W2"])
    layer, out, dX, dprob = _layer(gg, s, d, mxw)
    off, ros, sor = oracle.route(inp.idx, s.E, s.P)
    np.testing.assert_array_equal(layer.view("offsets").cpu().numpy(), off)
    np.testing.assert_array_equal(layer.view("row_of_slot").cpu().numpy(), ros)
    rng = np.random.default_rng(7)
    sel = np.sort(rng.choice(s.T, size=48, replace=False))
    W = mxo.mx_weights(inp.W1, inp.W2)
    f = mxo.mx_forward(inp.x[sel], inp.idx[sel], inp.prob[sel], inp.W1, inp.W2, s.E, 1,
                       weights=W)
    ff = mxo.mx_forward(inp.x[sel], inp.idx[sel], inp.prob[sel], inp.W1, inp.W2, s.E, 1,
                        faithful=True, weights=W)
    b, fb = mxo.mx_backward(inp.dOut[sel], f), mxo.mx_backward(inp.dOut[sel], ff)
    assert_parity(torch_to_f64(out)[sel], f["out"], "out", faithful=ff["out"], scope="tensor")
    assert_parity(torch_to_f64(dX)[sel], b["dX"], "dX", faithful=fb["dX"], scope="tensor")
    assert_parity(dprob.cpu().numpy().astype(np.float64)[sel], b["dprob"], "dprob",
                  faithful=fb["dprob"], scope="tensor")


def test_layer_at_the_expert_limit(gg):
    """The MXFP8 layer with 1024 experts (the maximum), tokens on eight of
    them: scale-tile prefixes and per-expert tables at full size."""
    s = MoeShape("mx_maxe_e1024_h128_f128_t160_k2", E=1024, H=128, F=128, T=160, k=2,
                 routing="uniform", x_std=1.0, w_std=0.05)
    inp = make_inputs(s, 97)
    rng = np.random.default_rng(98)
    live = np.array([0, 1, 2, 511, 512, 700, 1022, 1023])
    inp.idx[:] = np.stack([rng.choice(live, size=s.k, replace=False)
                           for _ in range(s.T)]).astype(np.int32)
    d = _dev(inp)
    mxw, _ = gg.mx_prepare_weights(d["W1"], d["W2"])
    _, out, dX, dprob = _layer(gg, s, d, mxw)
    f = mxo.mx_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, s.E, s.P)
    ff = mxo.mx_forward(inp.x, inp.idx, inp.prob, inp.W1, inp.W2, s.E, s.P, faithful=True)
    b, fb = mxo.mx_backward(inp.dOut, f), mxo.mx_backward(inp.dOut, ff)
    assert_parity(torch_to_f64(out), f["out"], "out", faithful=ff["out"], scope="tensor")
    assert_parity(torch_to_f64(dX), b["dX"], "dX", faithful=fb["dX"], scope="tensor")
    assert_parity(dprob.cpu().numpy().astype(np.float64), b["dprob"], "dprob",
                  faithful=fb["dprob"], scope="tensor")
