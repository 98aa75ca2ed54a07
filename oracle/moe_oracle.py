"""Plain fp64 CPU oracle of the grouped expert MLP: forward and input gradient.

TEST INFRASTRUCTURE. Imported only by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline / reference arm of ``bench.py``. It shares no code with the
CUDA library (no kernels, headers, tables or helpers) and is written to be
checked by eye against the pages it follows:

* "perf(moe): add frozen grouped GEMM for adapter training" (AlignmentResearch/
  Megatron-LM PR #3), sections "Why this change" and "Why existing behavior
  remains safe": the frozen, bias-free BF16 expert weights of all local experts
  are applied by one grouped GEMM over ragged per-expert token groups; experts
  with zero tokens are legal; the weights receive no gradient, only the input
  does.
* "[Main] Support paged stash with device-initiated GroupedLinear" (NVIDIA/
  Megatron-LM PR #6828), section "What does this PR do?": grouped FC1, a fused
  gated activation (SwiGLU) with GLU interleaving disabled, grouped FC2, and the
  routing probability applied at the activation / combine boundary.
* NVIDIA/Megatron-LM PR #7333, section "Summary": expert rows padded to a fixed
  multiple (256) with device-resident per-expert metadata.

Notation: T tokens, k routed slots per token, R = T*k routed rows, E experts,
H hidden, F expert FFN width (FC1 produces 2F columns), P the per-expert row
padding multiple and R_cap = T*k + E*(P-1). Weights are row-major per expert
in nn.Linear [out, in] layout: W1[E, 2F, H], W2[E, H, F].

Readings taken where the pages are silent (each also listed in the design notes):
* gate/up order: GLU interleaving is disabled, so the 2F FC1 outputs are two
  contiguous halves; the first F columns are the gate (SiLU side), the last F
  the linear "up" side.
* permutation order: expert-ascending, then (token, slot)-ascending, i.e. a
  stable sort of the flattened pairs by expert id.
* offsets: int32, E+1 entries, exclusive prefix sum of the padded counts.
* the routing probability multiplies each expert's output in the combine (FC2
  is linear and bias-free, so this equals weighting at the activation).
* padding rows hold zeros and carry slot id -1.

Two modes: exact fp64 (the pass/fail reference) and ``faithful=True``, which
rounds to BF16 (nearest-even) exactly where the GPU path stores BF16. The
faithful mode only sizes the error budget; it is never the parity reference.

All functions take BF16 tensors as uint16 bit patterns or as float64 arrays
that already hold BF16-representable values.
"""

from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------- BF16 helpers

def bf16_bits_to_f64(u16: np.ndarray) -> np.ndarray:
    """Exact value of BF16 bit patterns (BF16 is the top half of an fp32)."""
    u32 = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest BF16 value, ties to even.

    BF16 keeps 8 significant bits. Writing x = m * 2**e with 0.5 <= |m| < 1,
    the BF16 grid spacing near x is 2**(e-8); below the smallest normal
    exponent the spacing stays at the subnormal step 2**-133. Overflow is not
    handled (the workloads stay far from it).
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, -125)
    scale = np.ldexp(1.0, 8 - e)
    return np.rint(x * scale) / scale


def _as_f64(a: np.ndarray) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return bf16_bits_to_f64(a)
    return a.astype(np.float64)


def _sigmoid(z: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-z))


# ---------------------------------------------------------------- row mapping

def route(idx: np.ndarray, E: int, P: int = 1):
    """Expert-contiguous row map of the routed (token, slot) pairs.

    Expert e's rows are the pairs (t, j) with idx[t, j] == e, in ascending
    (t, j) order, followed by zero rows up to a multiple of P. Returns
    ``offsets[E+1]`` (exclusive prefix of padded counts), ``row_of_slot[T*k]``
    (row of pair t*k+j) and ``slot_of_row[R_cap]`` (pair id of a row, -1 for
    padding and for rows past offsets[E]).
    """
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape if idx.ndim == 2 else (0, 1)
    flat = idx.reshape(-1)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert id out of range")
    R_cap = T * k + E * (P - 1)
    offsets = np.zeros(E + 1, dtype=np.int64)
    row_of_slot = np.full(T * k, -1, dtype=np.int64)
    slot_of_row = np.full(R_cap, -1, dtype=np.int64)
    for e in range(E):
        pairs = np.nonzero(flat == e)[0]  # ascending pair id = ascending (t, j)
        cnt = pairs.size
        padded = -(-cnt // P) * P
        base = offsets[e]
        row_of_slot[pairs] = base + np.arange(cnt)
        slot_of_row[base:base + cnt] = pairs
        offsets[e + 1] = base + padded
    return offsets.astype(np.int32), row_of_slot.astype(np.int32), slot_of_row.astype(np.int32)


def permute(x, idx, prob, E: int, P: int = 1):
    """Gather the routed token rows into expert-contiguous order.

    Returns Xp[R_cap, H] (fp64, zero on padding and unused rows), the row maps
    and prob_of_row[R_cap] (the pair's probability, 0 on padding).
    """
    xf = _as_f64(x)
    T, H = xf.shape
    k = np.asarray(idx).shape[1]
    offsets, row_of_slot, slot_of_row = route(np.asarray(idx).reshape(T, k), E, P)
    R_cap = slot_of_row.size
    Xp = np.zeros((R_cap, H), dtype=np.float64)
    prob_of_row = np.zeros(R_cap, dtype=np.float64)
    live = slot_of_row >= 0
    Xp[live] = xf[slot_of_row[live] // k]
    prob_of_row[live] = np.asarray(prob, dtype=np.float64).reshape(-1)[slot_of_row[live]]
    return Xp, offsets, row_of_slot, slot_of_row, prob_of_row


# ---------------------------------------------------------------- grouped GEMMs

def grouped_linear(Xp: np.ndarray, W, offsets) -> np.ndarray:
    """Y[rows of e] = Xp[rows of e] @ W[e]^T for every expert (nn.Linear)."""
    E, N, K = np.shape(W)
    Y = np.zeros((Xp.shape[0], N), dtype=np.float64)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            Y[r0:r1] = Xp[r0:r1] @ _as_f64(W[e]).T
    return Y


def grouped_linear_t(dY: np.ndarray, W, offsets) -> np.ndarray:
    """Input gradient of ``grouped_linear``: dX[rows of e] = dY[rows of e] @ W[e]."""
    E, N, K = np.shape(W)
    dX = np.zeros((dY.shape[0], K), dtype=np.float64)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 > r0:
            dX[r0:r1] = dY[r0:r1] @ _as_f64(W[e])
    return dX


# ---------------------------------------------------------------- activation
#
# Gated activations of "[Main] Support paged stash with device-initiated
# GroupedLinear" (NVIDIA/Megatron-LM PR #6828, "What does this PR do?"): fused
# SwiGLU or QuickGeGLU with GLU interleaving disabled. Both are
# act(g) * u with act(g) = g * sigmoid(alpha * g): alpha = 1 is SiLU; the
# page names QuickGeGLU without defining it, read here as the QuickGELU gate
# x * sigmoid(1.702 x) of the usual definition.

GLU_ALPHA = {"swiglu": 1.0, "qgeglu": 1.702}


def glu(H1: np.ndarray, activation: str = "swiglu") -> np.ndarray:
    """A = g * sigmoid(alpha g) * u, g the first and u the second half of FC1's output."""
    a = GLU_ALPHA[activation]
    F = H1.shape[1] // 2
    g, u = H1[:, :F], H1[:, F:]
    return g * _sigmoid(a * g) * u


def glu_backward(dA: np.ndarray, H1: np.ndarray, activation: str = "swiglu") -> np.ndarray:
    """Gradient of ``glu`` w.r.t. its input [g, u], given dA.

    d/dg [g * s] = s + a*g*s*(1-s) = s*(1 + a*g*(1-s)) with s = sigmoid(a*g);
    dL/dg = dA * u * s*(1 + a*g*(1-s)),  dL/du = dA * g*s.
    """
    a = GLU_ALPHA[activation]
    F = H1.shape[1] // 2
    g, u = H1[:, :F], H1[:, F:]
    s = _sigmoid(a * g)
    dg = dA * u * s * (1.0 + a * g * (1.0 - s))
    du = dA * g * s
    return np.concatenate([dg, du], axis=1)


def swiglu(H1: np.ndarray) -> np.ndarray:
    """A = silu(g) * u (``glu`` with SiLU)."""
    return glu(H1, "swiglu")


def swiglu_backward(dA: np.ndarray, H1: np.ndarray) -> np.ndarray:
    """Gradient of ``swiglu`` w.r.t. [g, u] (``glu_backward`` with SiLU)."""
    return glu_backward(dA, H1, "swiglu")


# ---------------------------------------------------------------- combine

def combine(Yp: np.ndarray, row_of_slot, prob, T: int, k: int) -> np.ndarray:
    """out[t] = sum_j prob[t, j] * Yp[row_of_slot[t*k + j]], slots in order.

    ``prob=None`` gives the unweighted sum (the input-gradient combine).
    """
    H = Yp.shape[1]
    out = np.zeros((T, H), dtype=np.float64)
    rows = np.asarray(row_of_slot, dtype=np.int64).reshape(T, k)
    p = None if prob is None else np.asarray(prob, dtype=np.float64).reshape(T, k)
    for j in range(k):
        term = Yp[rows[:, j]]
        out += term if p is None else p[:, j:j + 1] * term
    return out


# ---------------------------------------------------------------- full layer

def prob_grad(dOut: np.ndarray, Yp: np.ndarray, row_of_slot, T: int, k: int) -> np.ndarray:
    """Gradient of the combine w.r.t. the routing probabilities.

    out_t = sum_j prob[t, j] * Yp[row(t, j)] is linear in each prob[t, j], so
    dL/dprob[t, j] = <dOut_t, Yp[row(t, j)]> (0 for a slot without a row).
    The probabilities are taken as given: the router that produced them is
    outside the layer. (The same pairing of a token-major row with a permuted
    row gives the pre-FC1 form <x_t, dXp[row(t, j)]>.)
    """
    dO = _as_f64(dOut)
    rows = np.asarray(row_of_slot, dtype=np.int64).reshape(T, k)
    dp = np.zeros((T, k), dtype=np.float64)
    for t in range(T):
        for j in range(k):
            r = rows[t, j]
            if r >= 0:
                dp[t, j] = float(np.dot(dO[t], Yp[r]))
    return dp


PROB_MODES = ("combine", "activation", "pre_fc1")


def moe_forward(x, idx, prob, W1, W2, E: int, P: int = 1, faithful: bool = False,
                activation: str = "swiglu", prob_mode: str = "combine"):
    """Forward of the expert layer. Returns a dict of every intermediate.

    Steps: permute -> FC1 (grouped) -> gated activation -> FC2 (grouped) ->
    combine, with the routing probability p of each (token, slot) pair applied
    at one of the three places PR #6828 ("What does this PR do?") names:
      "combine":    out_t = sum_j p * Yp[row]          (A = act, Yp = FC2(A));
      "activation": A = p * act(H1) (the weighted gated activation), the
                    combine sums Yp unweighted; FC2 is linear and bias-free, so
                    this is the same function as "combine";
      "pre_fc1":    Xp[row] = p * x_t before FC1 (a different function), the
                    combine sums unweighted.
    With ``faithful`` the values are rounded to BF16 where the GPU path stores
    BF16 (Xp, H1, A, Yp, out).
    """
    if prob_mode not in PROB_MODES:
        raise ValueError(prob_mode)
    rnd = round_to_bf16 if faithful else (lambda v: v)
    idx = np.asarray(idx)
    T = _as_f64(x).shape[0]
    k = idx.shape[1] if idx.ndim == 2 else 1
    Xp, offsets, row_of_slot, slot_of_row, prob_of_row = permute(x, idx, prob, E, P)
    if prob_mode == "pre_fc1":
        Xp = rnd(prob_of_row[:, None] * Xp)
    H1 = rnd(grouped_linear(Xp, W1, offsets))
    act = glu(H1, activation)
    A = rnd(prob_of_row[:, None] * act if prob_mode == "activation" else act)
    Yp = rnd(grouped_linear(A, W2, offsets))
    out = rnd(combine(Yp, row_of_slot, prob if prob_mode == "combine" else None, T, k))
    return dict(Xp=Xp, offsets=offsets, row_of_slot=row_of_slot, slot_of_row=slot_of_row,
                prob_of_row=prob_of_row, H1=H1, A=A, Yp=Yp, out=out, T=T, k=k, E=E, P=P,
                x=_as_f64(x), prob=np.asarray(prob, dtype=np.float64).reshape(T, k),
                activation=activation, prob_mode=prob_mode)


def moe_backward(dOut, fwd: dict, W1, W2, faithful: bool = False):
    """Input gradient dX of ``moe_forward`` (weights are frozen: no dW), and the
    routing-probability gradient dprob.

    dYp[r] = dOut[t] for the pair (t, j) of row r (0 on padding). The gradient
    w.r.t. the activation output is dA = p_r * (dYp @ W2_e) ("combine" and
    "activation": the probability multiplies the activation or the FC2 output)
    or dYp @ W2_e ("pre_fc1"); dH = act'(H1) applied to dA; dXp = dH @ W1_e;
    dX[t] = sum_j dXp[row(t, j)], weighted by p for "pre_fc1".
    dprob[t, j] = <dOut_t, FC2(act(H1))[row]> for "combine" / "activation"
    (``prob_grad``: the FC2 output is linear in p) and <x_t, dXp[row]> for
    "pre_fc1" (Xp[row] = p * x_t). With ``faithful`` the values are rounded to
    BF16 where the GPU path stores BF16 (dH, dXp, dX); dprob stays fp32 and
    pairs dOut with the FC2 output of the BF16 activation before that output
    is rounded (the path forms it from FC2's fp32 accumulation against the
    stored activation and never reads a rounded Yp for it).
    """
    rnd = round_to_bf16 if faithful else (lambda v: v)
    dO = _as_f64(dOut)
    T, k = fwd["T"], fwd["k"]
    act_name, mode = fwd["activation"], fwd["prob_mode"]
    slot_of_row = fwd["slot_of_row"]
    offsets = fwd["offsets"]
    p_row = fwd["prob_of_row"][:, None]
    live = slot_of_row >= 0
    dYp = np.zeros((slot_of_row.size, dO.shape[1]), dtype=np.float64)
    dYp[live] = dO[slot_of_row[live] // k]
    # gradient w.r.t. the activation output act(H1): p * (dYp @ W2_e) unless p
    # was applied before FC1
    dact = grouped_linear_t(dYp, W2, offsets)
    dA = dact if mode == "pre_fc1" else p_row * dact
    dH = rnd(glu_backward(dA, fwd["H1"], act_name))
    dXp = rnd(grouped_linear_t(dH, W1, offsets))
    if mode == "pre_fc1":
        # Xp[row] = p * x_t: dX_t = sum_j p * dXp[row], dprob = <x_t, dXp[row]>
        dX = rnd(combine(dXp, fwd["row_of_slot"], fwd["prob"], T, k))
        dprob = prob_grad(fwd["x"], dXp, fwd["row_of_slot"], T, k)
    else:
        dX = rnd(combine(dXp, fwd["row_of_slot"], None, T, k))
        # dprob = <dOut_t, FC2 output of the unweighted activation>
        if mode == "combine" and not faithful:
            Yu = fwd["Yp"]
        elif mode == "combine":
            Yu = grouped_linear(fwd["A"], W2, offsets)
        else:
            Yu = grouped_linear(rnd(glu(fwd["H1"], act_name)), W2, offsets)
        dprob = prob_grad(dO, Yu, fwd["row_of_slot"], T, k)
    return dict(dYp=dYp, dH=dH, dXp=dXp, dX=dX, dprob=dprob)


# ---------------------------------------------------------------- one token

def token_forward(x_t, experts, probs, W1, W2, activation: str = "swiglu",
                  prob_mode: str = "combine") -> np.ndarray:
    """Output of one token: sum over its routed experts of FC2(act(FC1 x)) with
    the probability p applied per ``prob_mode`` (see ``moe_forward``).

    ``W1``/``W2`` may be the full [E, ...] BF16 arrays (uint16 bits); only the
    routed experts are converted. Used for sampled checks at full size.
    """
    al = GLU_ALPHA[activation]
    xt = _as_f64(x_t).reshape(-1)
    y = np.zeros_like(xt)
    for e, p in zip(np.asarray(experts).reshape(-1), np.asarray(probs, dtype=np.float64).reshape(-1)):
        w1 = _as_f64(W1[int(e)])
        w2 = _as_f64(W2[int(e)])
        h = w1 @ (p * xt if prob_mode == "pre_fc1" else xt)
        F = h.size // 2
        a = h[:F] * _sigmoid(al * h[:F]) * h[F:]
        y += (w2 @ a) if prob_mode == "pre_fc1" else p * (w2 @ a)
    return y


def _token_expert_grads(xt, do, p, w1, w2, al, prob_mode):
    """For one routed expert of one token: (gradient w.r.t. x_t, dprob)."""
    xin = p * xt if prob_mode == "pre_fc1" else xt
    h = w1 @ xin
    F = h.size // 2
    g, u = h[:F], h[F:]
    s = _sigmoid(al * g)
    dact = do @ w2
    da = dact if prob_mode == "pre_fc1" else p * dact
    dh = np.concatenate([da * u * s * (1.0 + al * g * (1.0 - s)), da * g * s])
    dxin = dh @ w1
    if prob_mode == "pre_fc1":
        return p * dxin, float(np.dot(xt, dxin))
    return dxin, float(np.dot(dact, g * s * u))


def token_backward(x_t, dout_t, experts, probs, W1, W2, activation: str = "swiglu",
                   prob_mode: str = "combine") -> np.ndarray:
    """Input gradient of ``token_forward`` for one token, given dOut[t]."""
    xt = _as_f64(x_t).reshape(-1)
    do = _as_f64(dout_t).reshape(-1)
    dx = np.zeros_like(xt)
    for e, p in zip(np.asarray(experts).reshape(-1), np.asarray(probs, dtype=np.float64).reshape(-1)):
        dx += _token_expert_grads(xt, do, p, _as_f64(W1[int(e)]), _as_f64(W2[int(e)]),
                                  GLU_ALPHA[activation], prob_mode)[0]
    return dx


def token_prob_grad(x_t, dout_t, experts, W1, W2, activation: str = "swiglu",
                    prob_mode: str = "combine", probs=None) -> np.ndarray:
    """dL/dprob of one token's k slots: <dOut_t, FC2(act(FC1 x_t))> per expert, or
    for "pre_fc1" <x_t, d/dXp> at Xp = p * x_t (``probs`` required there)."""
    xt = _as_f64(x_t).reshape(-1)
    do = _as_f64(dout_t).reshape(-1)
    ex = np.asarray(experts).reshape(-1)
    ps = np.ones(ex.size) if probs is None else np.asarray(probs, dtype=np.float64).reshape(-1)
    if prob_mode == "pre_fc1" and probs is None:
        raise ValueError("pre_fc1 needs the probabilities")
    return np.asarray([_token_expert_grads(xt, do, p, _as_f64(W1[int(e)]), _as_f64(W2[int(e)]),
                                           GLU_ALPHA[activation], prob_mode)[1]
                       for e, p in zip(ex, ps)])
