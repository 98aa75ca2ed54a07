"""Seeded synthetic inputs for the grouped expert MLP.

This module is shared by the CPU oracle's tests, the CUDA path's tests and the
benchmark. It only draws random numbers and lays them out: it holds none of the
expert-MLP arithmetic (no permutation, no GEMM, no activation, no combine).

Every tensor that the expert path consumes is produced here as host numpy data:
BF16 tensors as ``uint16`` bit patterns (round-to-nearest-even from fp32), the
routing as ``int32`` expert ids ``idx[T, k]`` and ``float32`` probabilities
``prob[T, k]``. Oracle and GPU therefore see identical bits.

Routing recipe (the pages give none; "top-k from seeded softmax logits" is the
workload's own wording):
  * logits ~ N(0, 1) iid in fp32, shape [T, E]; experts forced to carry no
    tokens get -inf;
  * probabilities are the softmax over all E experts; the k largest logits are
    kept (ties go to the lower expert id) together with their softmax values,
    without renormalisation;
  * skewed loads (Zipf, Dirichlet) add log-weights to Gumbel noise and take the
    top k of the sum (Gumbel-top-k: sampling k distinct experts without
    replacement in proportion to the weights); the probabilities are the
    softmax of the same perturbed logits.

Seeds follow ``base = 1000 * cfg``: x -> base+1, W1 -> base+2, W2 -> base+3,
routing -> base+4, dOut -> base+5 (numpy PCG64 via ``default_rng``).
"""

from __future__ import annotations

import dataclasses

import numpy as np

__all__ = [
    "CONFIGS",
    "MoeShape",
    "MoeInputs",
    "f32_to_bf16_bits",
    "normal_bf16",
    "route_softmax_topk",
    "route_gumbel_topk",
    "make_inputs",
    "make_shared_expert_pair",
]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> BF16 bit patterns with round-to-nearest-even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def normal_bf16(rng: np.random.Generator, shape, std: float, chunk_rows: int = 4096) -> np.ndarray:
    """N(0, std^2) samples rounded to BF16, returned as uint16 bits.

    Drawn in fp32 row chunks along the first axis so that multi-GB weight
    tensors never need an fp64 temporary of the full size.
    """
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16)
    if out.size == 0:
        return out
    flat = out.reshape(shape[0], -1)
    inner = flat.shape[1]
    step = max(1, (1 << 24) // max(inner, 1))
    step = min(step, max(chunk_rows, 1) * 64)
    for r0 in range(0, shape[0], step):
        r1 = min(shape[0], r0 + step)
        v = rng.standard_normal((r1 - r0, inner), dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        flat[r0:r1] = f32_to_bf16_bits(v)
    return out


def _topk_desc(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest scores per row, ties to the lower index."""
    # stable argsort of the negated scores keeps equal scores in index order
    order = np.argsort(-scores, axis=1, kind="stable")
    return order[:, :k].astype(np.int32)


def _softmax_rows(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.float64)
    m = np.max(z, axis=1, keepdims=True)
    e = np.exp(z - m)
    return e / np.sum(e, axis=1, keepdims=True)


def route_softmax_topk(rng: np.random.Generator, T: int, E: int, k: int, zero_experts=()):
    """Top-k routing from iid N(0,1) logits (uniform random k-subsets)."""
    logits = rng.standard_normal((T, E), dtype=np.float32).astype(np.float64)
    for e in zero_experts:
        logits[:, e] = -np.inf
    idx = _topk_desc(logits, k)
    p = _softmax_rows(logits) if T else np.zeros((0, E))
    prob = np.take_along_axis(p, idx.astype(np.int64), axis=1).astype(np.float32)
    return idx, prob


def route_gumbel_topk(rng: np.random.Generator, T: int, k: int, log_w: np.ndarray):
    """Top-k of log-weights plus Gumbel noise (k distinct experts per token)."""
    E = log_w.shape[0]
    g = rng.gumbel(size=(T, E))
    logits = log_w[None, :] + g
    idx = _topk_desc(logits, k)
    p = _softmax_rows(logits) if T else np.zeros((0, E))
    prob = np.take_along_axis(p, idx.astype(np.int64), axis=1).astype(np.float32)
    return idx, prob


@dataclasses.dataclass(frozen=True)
class MoeShape:
    name: str
    E: int
    H: int
    F: int
    T: int
    k: int
    P: int = 1  # per-expert row padding multiple
    routing: str = "uniform"  # uniform | softmax_zero3 | zipf | dirichlet
    x_std: float = 1.0
    w_std: float = 0.02

    @property
    def R(self) -> int:
        return self.T * self.k

    @property
    def R_cap(self) -> int:
        return self.T * self.k + self.E * (self.P - 1)

    def flop_fwd(self) -> float:
        return 6.0 * self.R * self.H * self.F

    def flop_dgrad(self) -> float:
        return 6.0 * self.R * self.H * self.F

    def with_tokens(self, T: int) -> "MoeShape":
        """The same workload with T tokens; the name carries the new T."""
        import re

        if re.search(r"_t\d+", self.name):
            name = re.sub(r"_t\d+", f"_t{T}", self.name, count=1)
        else:
            name = re.sub(r"_k(\d+)", rf"_t{T}_k\1", self.name, count=1)
        return dataclasses.replace(self, T=T, name=name)


# The five workloads: a tiny correctness case, the balanced 128-expert layer,
# skewed routing with empty experts and 256-row padding, one expert-parallel
# rank's shard (32 experts, 30272 tokens), and the large-token sweep family.
CONFIGS = {
    1: MoeShape("tiny_e4_h64_f128_t256_k2", E=4, H=64, F=128, T=256, k=2,
                routing="softmax_zero3", x_std=0.02, w_std=0.02),
    2: MoeShape("balanced_e128_h2048_f768_t16384_k8", E=128, H=2048, F=768, T=16384, k=8),
    3: MoeShape("zipf_e128_h2048_f768_t4096_k8_pad256", E=128, H=2048, F=768, T=4096, k=8,
                P=256, routing="zipf"),
    4: MoeShape("ep4shard_e32_h4096_f2048_t30272_k8", E=32, H=4096, F=2048, T=30272, k=8,
                routing="dirichlet"),
    5: MoeShape("sweep_e128_h2688_f1856_k8", E=128, H=2688, F=1856, T=1024, k=8),
}

SWEEP_ROWS = [8192 << i for i in range(8)]  # 8192 ... 1048576 routed rows


@dataclasses.dataclass
class MoeInputs:
    shape: MoeShape
    x: np.ndarray      # uint16 [T, H]   BF16 bits
    idx: np.ndarray    # int32  [T, k]
    prob: np.ndarray   # float32 [T, k]
    W1: np.ndarray     # uint16 [E, 2F, H] BF16 bits (gate rows 0..F-1, up rows F..2F-1)
    W2: np.ndarray     # uint16 [E, H, F]  BF16 bits
    dOut: np.ndarray   # uint16 [T, H]   BF16 bits


def _routing(shape: MoeShape, rng: np.random.Generator):
    T, E, k = shape.T, shape.E, shape.k
    if shape.routing == "uniform":
        return route_softmax_topk(rng, T, E, k)
    if shape.routing == "softmax_zero3":
        return route_softmax_topk(rng, T, E, k, zero_experts=(3,))
    if shape.routing == "zipf":
        # Zipf(s=1.2) weights over the live experts, ranks assigned by a seeded
        # permutation; 16 seeded experts carry no tokens.
        n_dead = min(16, E - k)
        perm = rng.permutation(E)
        dead = perm[:n_dead]
        live = perm[n_dead:]
        log_w = np.full(E, -np.inf)
        ranks = np.arange(1, live.size + 1, dtype=np.float64)
        log_w[live] = -1.2 * np.log(ranks)
        return route_gumbel_topk(rng, T, k, log_w)
    if shape.routing == "dirichlet":
        w = rng.dirichlet(np.full(E, 2.0))
        return route_gumbel_topk(rng, T, k, np.log(w))
    raise ValueError(f"unknown routing {shape.routing!r}")


def make_inputs(shape: MoeShape, seed_base: int, with_weights: bool = True,
                with_dout: bool = True) -> MoeInputs:
    """All inputs of one workload, seeded from ``seed_base`` (= 1000 * cfg)."""
    H, F, E, T = shape.H, shape.F, shape.E, shape.T
    x = normal_bf16(np.random.default_rng(seed_base + 1), (T, H), shape.x_std)
    if with_weights:
        W1 = normal_bf16(np.random.default_rng(seed_base + 2), (E, 2 * F, H), shape.w_std)
        W2 = normal_bf16(np.random.default_rng(seed_base + 3), (E, H, F), shape.w_std)
    else:
        W1 = np.zeros((0,), np.uint16)
        W2 = np.zeros((0,), np.uint16)
    idx, prob = _routing(shape, np.random.default_rng(seed_base + 4))
    dOut = (normal_bf16(np.random.default_rng(seed_base + 5), (T, H), 1.0)
            if with_dout else np.zeros((0,), np.uint16))
    return MoeInputs(shape, x, idx, prob, W1, W2, dOut)


def make_shared_expert_pair(a: MoeInputs, e_star: int, seed: int) -> MoeInputs:
    """A second load draw that routes exactly the same token rows to ``e_star``.

    Every (token, slot) pair that ``a`` sends to ``e_star`` is kept: same token
    index, same x row, same probability, same dOut row. All other slots are
    re-drawn among the other experts (distinct within a token), and every token
    with no ``e_star`` slot gets a fresh x row and dOut row. The per-expert
    counts of all other experts therefore change, which moves ``e_star``'s rows
    to a different place in the permuted buffer.
    """
    s = a.shape
    rng = np.random.default_rng(seed)
    idx = a.idx.copy()
    prob = a.prob.copy()
    x = a.x.copy()
    dOut = a.dOut.copy()
    has = np.any(idx == e_star, axis=1)
    others = np.array([e for e in range(s.E) if e != e_star], dtype=np.int32)
    for t in range(s.T):
        keep = idx[t] == e_star
        n_new = int(np.sum(~keep))
        choice = rng.choice(others, size=n_new, replace=False)
        idx[t, ~keep] = choice
        prob[t, ~keep] = rng.uniform(0.0, 0.2, size=n_new).astype(np.float32)
    fresh = ~has
    n_fresh = int(np.sum(fresh))
    if n_fresh:
        x[fresh] = normal_bf16(rng, (n_fresh, s.H), s.x_std)
        dOut[fresh] = normal_bf16(rng, (n_fresh, s.H), 1.0)
    return MoeInputs(s, x, idx, prob, a.W1, a.W2, dOut)
