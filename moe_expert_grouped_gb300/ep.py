"""Expert parallelism around the grouped expert layer.

Each of W ranks owns E / W experts (rank r: experts [r*El, (r+1)*El)) and their
weights. A rank's routed (token, slot) pairs are grouped by the rank that owns
their expert, the rows are exchanged with one all-to-all (counts first, then
rows and local expert ids), every rank runs the grouped expert MLP on the rows
it received (one slot per row, no probability), the outputs travel back with
the reverse all-to-all and the sending rank combines them with the routing
probabilities. The backward mirrors it: the output gradient goes out in the
same order, the input-gradient rows and the per-row probability gradients
come back, and the sender sums the rows weighted by the probabilities
("perf(moe): add frozen grouped GEMM for adapter training",
AlignmentResearch/Megatron-LM PR #3, "B200 throughput evidence": ordinary
all-to-all dispatch around the local grouped GEMM).

The exchange uses torch.distributed (NCCL between GPUs, gloo on CPU); the
rank-local steps come from an ``ops`` object: ``GgOps`` runs them with this
library's kernels on the rank's GPU (the split of the expert ids by rank, the
grouping by rank, the gathers into send and token order, the expert MLP and
the combines). Counts are read on the host once per exchange (uneven
all-to-all splits need them).
"""

from __future__ import annotations

from typing import Optional

import torch
import torch.distributed as dist


def _a2a(x: torch.Tensor, out_counts, in_counts, group) -> torch.Tensor:
    """Uneven all-to-all along dim 0 (identity on one rank)."""
    if group is None and not dist.is_initialized():
        return x
    out = x.new_empty((int(sum(out_counts)),) + tuple(x.shape[1:]))
    dist.all_to_all_single(out, x.contiguous(), list(out_counts), list(in_counts), group=group)
    return out


def _exchange_counts(send_counts: torch.Tensor, group) -> torch.Tensor:
    if group is None and not dist.is_initialized():
        return send_counts.clone()
    recv = torch.empty_like(send_counts)
    dist.all_to_all_single(recv, send_counts.contiguous(), group=group)
    return recv


class GgOps:
    """Rank-local steps with the library's kernels (CUDA tensors)."""

    def __init__(self, H: int, F: int, El: int, activation: int = 0):
        from . import gg  # the CUDA library: loaded only when these ops are used

        self.gg = gg
        self.H, self.F, self.El, self.activation = H, F, El, activation
        self._layer = None
        self._ws = None  # the forward's workspace: status word of its routing calls

    def split_ids(self, idx, El: int, world: int):
        T, k = idx.shape
        self._ws = self.gg.workspace(T, k, world, idx.device)
        return self.gg.ep_split_ids(idx.contiguous(), El, world, self._ws)

    def group_by_rank(self, x, dest, prob, world: int) -> dict:
        # the stable counting sort of the pairs by destination rank is the
        # permute with the ranks as "experts"
        return self.gg.permute(x, dest, prob, world, 1, ws=self._ws)

    def gather(self, src, index) -> torch.Tensor:
        return self.gg.gather_rows32(src.contiguous(), index, self._ws)

    def status(self) -> int:
        return self.gg.read_status(self._ws) if self._ws is not None else 0

    def to_send_order(self, src, maps: dict, k: int, world: int) -> torch.Tensor:
        n = src.shape[0] * k
        return self.gg.permute_rows(src, maps["row_of_slot"], maps["slot_of_row"],
                                    maps["offsets"], k, world, 1, n, maps["ws"])

    def local_forward(self, rows, local_eid, W1, W2) -> torch.Tensor:
        n = rows.shape[0]
        # One device buffer serves every forward; it is replaced (by one for
        # the next power of two rows, at least 1024) only when a batch does
        # not fit it.
        L = self._layer
        if L is None or L.device != rows.device or not L.fits(n):
            cap = 1 << max(10, (max(n, 1) - 1).bit_length())
            L = self.gg.MoeLayer(cap, self.H, self.F, 1, self.El, 1, device=rows.device,
                                 activation=self.activation)
            self._layer = L
        ones = torch.ones((n, 1), dtype=torch.float32, device=rows.device)
        return L.forward(rows, local_eid.view(n, 1), ones, W1, W2)

    def local_backward(self, d_rows, W1, W2):
        dX, dprob = self._layer.backward(d_rows, W1, W2, dprob=True)
        return dX, dprob.view(-1)

    def combine(self, rows, maps: dict, prob, T: int, k: int) -> torch.Tensor:
        return self.gg.unpermute_combine(rows, maps["row_of_slot"], prob, T, k, maps["ws"])


class ExpertParallelLayer:
    """The expert layer over ``E`` experts spread evenly over the ranks of
    ``group`` (one rank when torch.distributed is not initialised).

    forward(x [T, H], idx [T, k] global expert ids, prob [T, k], W1_local
    [E/W, 2F, H], W2_local [E/W, H, F]) -> out [T, H]; backward(dOut) ->
    (dX [T, H], dprob [T, k]) after a forward, the probability applied at the
    combine.
    """

    def __init__(self, H: int, F: int, k: int, E: int, group=None, ops=None):
        self.group = group
        distributed = group is not None or dist.is_initialized()
        self.world = dist.get_world_size(group) if distributed else 1
        self.rank = dist.get_rank(group) if distributed else 0
        if E % self.world != 0:
            raise ValueError(f"{E} experts do not split evenly over {self.world} ranks")
        self.H, self.F, self.k, self.E = H, F, k, E
        self.El = E // self.world
        self.ops = ops if ops is not None else GgOps(H, F, self.El)
        self._ctx: Optional[tuple] = None

    def forward(self, x, idx, prob, W1_local, W2_local):
        T, k, W, El = x.shape[0], self.k, self.world, self.El
        dest, local_eid = self.ops.split_ids(idx, El, W)
        maps = self.ops.group_by_rank(x, dest, prob, W)
        n = T * k
        off = maps["offsets"].tolist()  # the one host read: uneven splits need the counts
        send_l = [off[r + 1] - off[r] for r in range(W)]
        recv = _exchange_counts(torch.tensor(send_l, dtype=torch.int64,
                                             device=maps["offsets"].device), self.group)
        recv_l = recv.tolist()
        # local expert id of every sent row (row r carries pair slot_of_row[r])
        eid = self.ops.gather(local_eid.reshape(-1), maps["slot_of_row"][:n])
        rows = _a2a(maps["Xp"][:n], recv_l, send_l, self.group)
        eids = _a2a(eid, recv_l, send_l, self.group)
        y = self.ops.local_forward(rows, eids, W1_local, W2_local)
        y_back = _a2a(y, send_l, recv_l, self.group)
        self._ctx = (maps, send_l, recv_l, prob, T)
        return self.ops.combine(y_back, maps, prob, T, k)

    def backward(self, dOut, W1_local, W2_local):
        if self._ctx is None:
            raise RuntimeError("backward needs a forward first")
        maps, send_l, recv_l, prob, T = self._ctx
        k, n = self.k, T * self.k
        d_send = self.ops.to_send_order(dOut, maps, k, self.world)[:n]
        d_rows = _a2a(d_send, recv_l, send_l, self.group)
        dx_rows, dp_rows = self.ops.local_backward(d_rows, W1_local, W2_local)
        dx_back = _a2a(dx_rows, send_l, recv_l, self.group)
        dp_back = _a2a(dp_rows, send_l, recv_l, self.group)
        # the remote rows carry no probability: weight them in the sum
        dX = self.ops.combine(dx_back, maps, prob, T, k)
        dprob = self.ops.gather(dp_back, maps["row_of_slot"]).view(T, k)
        return dX, dprob
