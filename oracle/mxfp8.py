"""Plain fp64 CPU oracle of the MXFP8 variant of the expert layer.

TEST INFRASTRUCTURE, like the rest of ``oracle/``: imported only by ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline arm of ``bench.py``; it shares
no code with the CUDA library.

The pages run the routed expert projections in MXFP8 (NVIDIA/Megatron-LM PR
#7333, section "Validation": routed expert projections only in MXFP8, other
modules in BF16; "[Main] Support paged stash with device-initiated
GroupedLinear", NVIDIA/Megatron-LM PR #6828, section "End-to-end GB300
validation": MXFP8 on GB300). They do not spell the format out. Readings
taken here (each also listed in the design notes):

* MXFP8 is the OCP microscaling format with FP8 E4M3 elements: blocks of 32
  consecutive elements along a GEMM's reduction dimension share one E8M0 scale
  (a power of two 2^e, stored as the byte e + 127).
* The scale of a block is the smallest power of two with
  max|v| / 2^e <= 448 (E4M3's largest finite magnitude), so no element of the
  block saturates; e is clamped to [-127, 127] and an all-zero block takes
  e = -127.
* An element is v / 2^e rounded to the nearest E4M3 value, ties to even
  (E4M3: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits, subnormals
  down to 2^-9, no infinities, largest finite 448); a magnitude above 448
  (reachable only at the clamp) saturates to 448, and the sign of zero is
  kept.
* Every GEMM of the layer takes MXFP8 operands quantised along its own
  reduction dimension and accumulates exactly; the weights therefore exist in
  two quantisations: along their input dimension for the forward and along
  their output dimension for the input gradient.
* Every GEMM's result is BF16, and the tensors one GEMM hands to the next are
  BF16 before they are quantised: FC1's output H1 is rounded to BF16 (it is
  also what the backward reads), the gated activation is applied to those
  BF16 values and its result rounded to BF16, and only then quantised for
  FC2; the input gradient of FC2 (the activation's output gradient) is
  rounded to BF16 before the activation's backward, whose result dH1 is
  rounded to BF16 before it is quantised for the second input-gradient GEMM.
  The quantised codes are decided on these BF16 values, which both this
  oracle and the kernels compute.

Shapes follow ``moe_oracle``: W1[E, 2F, H], W2[E, H, F], x[T, H].
"""

from __future__ import annotations

import numpy as np
import torch

from . import moe_oracle as _mo

# The elementwise steps below run as plain PyTorch CPU ops on views of the
# numpy arrays (same arithmetic, fp64; PyTorch spreads them over the host
# cores, which matters for the full-size weights).

BLOCK = 32
E4M3_MAX = 448.0
E8M0_BIAS = 127


# ---------------------------------------------------------------- E4M3 elements

def e4m3_round(v: np.ndarray) -> np.ndarray:
    """Nearest E4M3 value of each fp64 entry, ties to even, saturating at 448.

    Normal E4M3 numbers 2^E * (1 + m/8) cover exponents E in [-6, 8]; below
    2^-6 the grid is the subnormal step 2^-9."""
    v = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float64))
    a = v.abs()
    _, p = torch.frexp(a)                   # a = f * 2^p, f in [0.5, 1)
    E = torch.clamp(p - 1, min=-6)          # binade of a; subnormals share E = -6
    step = torch.ldexp(torch.ones_like(a), E - 3)   # 3 mantissa bits
    q = torch.round(a / step) * step        # torch.round rounds half to even
    q = torch.clamp(q, max=E4M3_MAX)
    return torch.copysign(q, v).numpy()


def e4m3_bits(q: np.ndarray) -> np.ndarray:
    """Byte encoding (sign, 4-bit exponent with bias 7, 3-bit mantissa) of
    E4M3 values (entries must already be E4M3 numbers)."""
    q = np.asarray(q, dtype=np.float64)
    sign = np.signbit(q).astype(np.uint8) << 7
    a = np.abs(q)
    _, p = np.frexp(a)
    E = p - 1
    normal = a >= 2.0 ** -6
    exp_field = np.where(normal, E + 7, 0)
    mant = np.where(normal, a / np.ldexp(1.0, E) * 8 - 8, a / 2.0 ** -9)
    if np.any(mant != np.rint(mant)) or np.any(a > E4M3_MAX):
        raise ValueError("not E4M3 values")
    return (sign | (exp_field.astype(np.uint8) << 3) | mant.astype(np.uint8)).astype(np.uint8)


def e4m3_value(bits: np.ndarray) -> np.ndarray:
    """Exact value of E4M3 bytes (0x7F / 0xFF, the NaN codes, are rejected)."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    if np.any((b & 0x7F) == 0x7F):
        raise ValueError("E4M3 NaN code")
    exp_field = (b >> 3) & 0xF
    mant = b & 7
    mag = np.where(exp_field == 0, mant * 2.0 ** -9,
                   np.ldexp(1.0 + mant / 8.0, exp_field - 7))
    return np.where(b & 0x80, -mag, mag)


# ---------------------------------------------------------------- block scales

def block_exponent(amax: np.ndarray) -> np.ndarray:
    """Smallest e with amax / 2^e <= 448, clamped to [-127, 127] (-127 for 0).

    With amax = (1 + f) * 2^q, 448 = 1.75 * 2^8: e = q - 8 when 1 + f <= 1.75,
    else q - 7."""
    amax = torch.from_numpy(np.ascontiguousarray(amax, dtype=np.float64))
    f, p = torch.frexp(amax)                # amax = f * 2^p, f in [0.5, 1)
    q = p.to(torch.int64) - 1
    e = q - 8 + (2.0 * f > 1.75).to(torch.int64)
    e = torch.where(amax > 0, e, torch.full_like(e, -E8M0_BIAS))
    return torch.clamp(e, -E8M0_BIAS, E8M0_BIAS).numpy()


def quantize(v: np.ndarray):
    """MXFP8 quantisation of the last axis (length a multiple of 32).

    Returns (elements, exponents): the E4M3 values v / 2^e (fp64 holding E4M3
    numbers, same shape as v) and the block exponents e (shape [..., K/32])."""
    v = np.asarray(v, dtype=np.float64)
    K = v.shape[-1]
    if K % BLOCK:
        raise ValueError("the quantised axis must be a multiple of 32")
    blocks = torch.from_numpy(np.ascontiguousarray(v)).reshape(v.shape[:-1] + (K // BLOCK, BLOCK))
    e = block_exponent(blocks.abs().amax(dim=-1).numpy())
    scale = torch.ldexp(torch.ones(e.shape, dtype=torch.float64), torch.from_numpy(e))
    q = e4m3_round((blocks / scale[..., None]).numpy())
    return q.reshape(v.shape), e


def dequantize(q: np.ndarray, e: np.ndarray) -> np.ndarray:
    """Exact value of MXFP8 data: element times its block's 2^e."""
    q = torch.from_numpy(np.ascontiguousarray(q, dtype=np.float64))
    K = q.shape[-1]
    blocks = q.reshape(q.shape[:-1] + (K // BLOCK, BLOCK))
    e = torch.from_numpy(np.ascontiguousarray(e, dtype=np.int64))
    scale = torch.ldexp(torch.ones(e.shape, dtype=torch.float64), e)
    return (blocks * scale[..., None]).reshape(q.shape).numpy()


def mx(v: np.ndarray) -> np.ndarray:
    """Quantise-dequantise along the last axis: the value a GEMM sees."""
    return dequantize(*quantize(v))


def mx_weights(W1, W2):
    """The four weight quantisations of the layer (exact values, fp64).

    W1f[E, 2F, H], W2f[E, H, F]: along the input dimension (forward GEMMs);
    W1d[E, 2F, H] quantised along 2F and W2d[E, H, F] along H (input-gradient
    GEMMs, which reduce over the weights' output dimension)."""
    W1 = _mo._as_f64(W1)
    W2 = _mo._as_f64(W2)
    W1f = mx(W1)
    W2f = mx(W2)
    W1d = np.swapaxes(mx(np.swapaxes(W1, 1, 2)), 1, 2)
    W2d = np.swapaxes(mx(np.swapaxes(W2, 1, 2)), 1, 2)
    return dict(W1f=W1f, W2f=W2f, W1d=W1d, W2d=W2d)


# ---------------------------------------------------------------- the layer

def mx_forward(x, idx, prob, W1, W2, E: int, P: int = 1, activation: str = "swiglu",
               prob_mode: str = "combine", faithful: bool = False, weights=None) -> dict:
    """MXFP8 expert layer, forward (readings in the module docstring).

    Xq = mx(x rows), H1 = bf16(Xq W1f^T), A = bf16(act(H1)) (times the
    probability in ``activation`` mode), Yp = mx(A) W2f^T exactly, out =
    the probability-weighted (``combine``) or plain sum of the k rows. The
    pre-FC1 probability mode scales x before its quantisation. With
    ``faithful``, Yp and out are also rounded to BF16 (where the GPU path
    stores them); that only sizes the error budget of a parity test.
    ``weights`` may pass the result of ``mx_weights(W1, W2)`` to reuse it."""
    if prob_mode not in ("combine", "activation", "pre_fc1"):
        raise ValueError(prob_mode)
    x = _mo._as_f64(x)
    idx = np.asarray(idx)
    prob = np.asarray(prob, dtype=np.float64)
    T, k = idx.shape
    W = mx_weights(W1, W2) if weights is None else weights
    offsets, row_of_slot, slot_of_row = _mo.route(idx, E, P)
    R_cap = slot_of_row.shape[0]
    pr = np.zeros(R_cap)
    valid = slot_of_row >= 0
    pr[valid] = prob.reshape(-1)[slot_of_row[valid]]
    Xp = np.zeros((R_cap, x.shape[1]))
    Xp[valid] = x[slot_of_row[valid] // k]
    if prob_mode == "pre_fc1":
        Xp = _mo.round_to_bf16(Xp * pr[:, None])
    Xq = mx(Xp)
    H1 = _mo.round_to_bf16(_mo.grouped_linear(Xq, W["W1f"], offsets))
    A = _mo.glu(H1, activation)
    if prob_mode == "activation":
        A = A * pr[:, None]
    A = _mo.round_to_bf16(A)
    Aq = mx(A)
    rnd = _mo.round_to_bf16 if faithful else (lambda v: v)
    Yp = rnd(_mo.grouped_linear(Aq, W["W2f"], offsets))
    if prob_mode == "combine":
        out = rnd(_mo.combine(Yp, row_of_slot, prob, T, k))
    else:
        out = rnd(_mo.combine(Yp, row_of_slot, None, T, k))
    return dict(out=out, offsets=offsets, row_of_slot=row_of_slot, slot_of_row=slot_of_row,
                Xq=Xq, H1=H1, A=A, Aq=Aq, Yp=Yp, W=W, x=x, prob=prob, pr=pr,
                activation=activation, prob_mode=prob_mode, k=k, faithful=faithful)


def mx_backward(dOut, fwd: dict) -> dict:
    """MXFP8 expert layer, input gradient and probability gradient.

    dYq = mx(dOut rows) (each row of the permuted gradient is its token's
    dOut), dA0 = bf16(dYq W2d), dA = dA0 times the probability (``combine`` and
    ``activation`` modes: the probability scales the activation's output, or
    equivalently FC2's), dH1 = bf16(act'(H1) applied to dA), dXp = mx(dH1)
    W1d, dX = the plain sum of the k rows (probability-weighted in
    ``pre_fc1`` mode). The quantisers pass gradients straight through.

    dprob is taken where the probability enters the forward:
      * ``combine``: out_t = sum_j p_tj * Yp[row(t, j)] is linear in p and no
        quantiser lies between p and out, so dprob_tj = <dOut_t, Yp[row(t, j)]>
        exactly, with the forward's Yp (the probability gradient at the
        combine, "[Main] Support paged stash with device-initiated
        GroupedLinear", "What does this PR do?": the probability boundary);
      * ``activation``: A = bf16(p * act(H1)) is quantised for FC2, whose
        quantiser passes the gradient straight through, so dprob is the row
        sum of dA0 * act(H1), dA0 being the gradient that reaches A;
      * ``pre_fc1``: <x_t, dXp[row]>.
    With a ``faithful`` forward (whose Yp is already BF16), dXp, dX and the
    activation in the ``activation``-mode sum are rounded to BF16 as well."""
    dOut = _mo._as_f64(dOut)
    k = fwd["k"]
    T = dOut.shape[0]
    offsets, ros, sor = fwd["offsets"], fwd["row_of_slot"], fwd["slot_of_row"]
    W = fwd["W"]
    pr = fwd["pr"]
    mode = fwd["prob_mode"]
    R_cap = sor.shape[0]
    valid = sor >= 0
    dYp = np.zeros((R_cap, dOut.shape[1]))
    dYp[valid] = dOut[sor[valid] // k]
    dA0 = _mo.round_to_bf16(_mo.grouped_linear_t(mx(dYp), W["W2d"], offsets))
    dprob_rows = np.zeros(R_cap)
    rnd = _mo.round_to_bf16 if fwd.get("faithful") else (lambda v: v)
    if mode == "combine":
        dA = dA0 * pr[:, None]
        dprob_rows[valid] = np.sum(dYp[valid] * fwd["Yp"][valid], axis=1)
    elif mode == "activation":
        dA = dA0 * pr[:, None]
        act = rnd(_mo.glu(fwd["H1"], fwd["activation"]))
        dprob_rows[valid] = np.sum(dA0[valid] * act[valid], axis=1)
    else:
        dA = dA0
    dH1 = _mo.round_to_bf16(_mo.glu_backward(dA, fwd["H1"], fwd["activation"]))
    dXp = rnd(_mo.grouped_linear_t(mx(dH1), W["W1d"], offsets))
    if mode == "pre_fc1":
        x = fwd["x"]
        dprob_rows[valid] = np.sum(x[sor[valid] // k] * dXp[valid], axis=1)
        dX = rnd(_mo.combine(dXp, ros, fwd["prob"], T, k))
    else:
        dX = rnd(_mo.combine(dXp, ros, None, T, k))
    dprob = np.zeros(T * k)
    dprob[sor[valid]] = dprob_rows[valid]
    return dict(dX=dX, dprob=dprob.reshape(T, k), dYp=dYp, dA=dA, dH1=dH1, dXp=dXp)
