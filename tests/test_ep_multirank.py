"""Expert parallelism on CPU: two gloo ranks, each owning half of the experts.

The orchestration of ``moe_expert_grouped_gb300.ep.ExpertParallelLayer`` (the
grouping of pairs by owning rank, the count exchange, the row and expert-id
all-to-all, the reverse all-to-all of outputs and gradients, the weighted
recombination and the probability-gradient gather) runs unchanged; its
rank-local steps are the oracle's plain definitions in fp64. Each rank's
output, input gradient and probability gradient must equal the oracle run on
that rank's tokens with all experts' weights."""

import os
import socket

import numpy as np
import torch
import torch.multiprocessing as mp

import oracle
from moe_synth import MoeShape, make_inputs

SHAPE = MoeShape("ep_e8_h64_f128_k3", E=8, H=64, F=128, T=48, k=3, routing="uniform",
                 x_std=1.0, w_std=0.1)


class OracleOps:
    """The rank-local steps by their definitions (fp64, CPU)."""

    def __init__(self, El: int):
        self.El = El
        self._fwd = None

    def split_ids(self, idx, El, world):
        return (torch.div(idx, El, rounding_mode="floor").to(torch.int32),
                torch.remainder(idx, El).to(torch.int32))

    def gather(self, src, index):
        return src[index.long()]

    def group_by_rank(self, x, dest, prob, world):
        off, ros, sor = oracle.route(dest.numpy(), world, 1)
        k = dest.shape[1]
        rows = x[torch.from_numpy(sor.astype(np.int64)) // k]
        return dict(Xp=rows, offsets=torch.from_numpy(off.astype(np.int64)),
                    row_of_slot=torch.from_numpy(ros.astype(np.int64)),
                    slot_of_row=torch.from_numpy(sor.astype(np.int64)), ws=None)

    def to_send_order(self, src, maps, k, world):
        return src[maps["slot_of_row"] // k]

    def local_forward(self, rows, eid, W1, W2):
        n = rows.shape[0]
        self._fwd = oracle.moe_forward(rows.numpy(), eid.numpy().reshape(n, 1), np.ones((n, 1)),
                                       W1, W2, self.El, 1)
        return torch.from_numpy(self._fwd["out"])

    def local_backward(self, d_rows, W1, W2):
        bwd = oracle.moe_backward(d_rows.numpy(), self._fwd, W1, W2)
        return torch.from_numpy(bwd["dX"]), torch.from_numpy(bwd["dprob"].reshape(-1))

    def combine(self, rows, maps, prob, T, k):
        return torch.from_numpy(oracle.combine(rows.numpy(), maps["row_of_slot"].numpy(),
                                               prob.numpy(), T, k))


def _tokens(rank):
    # rank-specific token counts and routing; the same global weights
    shape = SHAPE.with_tokens(SHAPE.T + 7 * rank)
    return shape, make_inputs(shape, 9000 + rank, with_weights=False)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    from moe_expert_grouped_gb300.ep import ExpertParallelLayer

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = make_inputs(SHAPE, 8000)  # global weights, identical on every rank
        shape, inp = _tokens(rank)
        El = SHAPE.E // world
        W1 = oracle.bf16_bits_to_f64(w.W1)
        W2 = oracle.bf16_bits_to_f64(w.W2)
        W1l, W2l = W1[rank * El:(rank + 1) * El], W2[rank * El:(rank + 1) * El]
        try:
            ExpertParallelLayer(SHAPE.H, SHAPE.F, SHAPE.k, 7, ops=OracleOps(El))
            uneven_rejected = False
        except ValueError:
            uneven_rejected = True
        layer = ExpertParallelLayer(SHAPE.H, SHAPE.F, SHAPE.k, SHAPE.E, ops=OracleOps(El))
        x = torch.from_numpy(oracle.bf16_bits_to_f64(inp.x))
        idx = torch.from_numpy(inp.idx)
        prob = torch.from_numpy(inp.prob.astype(np.float64))
        out = layer.forward(x, idx, prob, W1l, W2l)
        dX, dprob = layer.backward(torch.from_numpy(oracle.bf16_bits_to_f64(inp.dOut)), W1l, W2l)
        fwd = oracle.moe_forward(inp.x, inp.idx, inp.prob, W1, W2, SHAPE.E, 1)
        bwd = oracle.moe_backward(inp.dOut, fwd, W1, W2)
        errs = [float(np.max(np.abs(a.numpy() - b)) / max(1e-300, float(np.max(np.abs(b)))))
                for a, b in ((out, fwd["out"]), (dX, bwd["dX"]), (dprob, bwd["dprob"]))]
        # the exchange really moved rows between the ranks
        sent = (layer._ctx[0]["offsets"][1:] - layer._ctx[0]["offsets"][:-1]).tolist()
        q.put((rank, errs, sent, uneven_rejected))
    finally:
        dist.destroy_process_group()


def test_expert_parallel_two_ranks_matches_single_process():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, errs, sent, uneven_rejected in res:
        assert uneven_rejected  # 7 experts do not split over 2 ranks
        assert max(errs) < 1e-12, (rank, errs)
        assert all(s > 0 for s in sent), sent  # both ranks send rows to both ranks


def test_expert_parallel_single_rank_without_torch_distributed():
    from moe_expert_grouped_gb300.ep import ExpertParallelLayer

    w = make_inputs(SHAPE, 8000)
    shape, inp = _tokens(0)
    W1 = oracle.bf16_bits_to_f64(w.W1)
    W2 = oracle.bf16_bits_to_f64(w.W2)
    layer = ExpertParallelLayer(SHAPE.H, SHAPE.F, SHAPE.k, SHAPE.E, ops=OracleOps(SHAPE.E))
    assert layer.world == 1 and layer.El == SHAPE.E
    out = layer.forward(torch.from_numpy(oracle.bf16_bits_to_f64(inp.x)),
                        torch.from_numpy(inp.idx), torch.from_numpy(inp.prob.astype(np.float64)),
                        W1, W2)
    fwd = oracle.moe_forward(inp.x, inp.idx, inp.prob, W1, W2, SHAPE.E, 1)
    np.testing.assert_allclose(out.numpy(), fwd["out"], rtol=1e-12, atol=1e-14)
