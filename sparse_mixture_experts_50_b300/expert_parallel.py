"""Expert-parallel form of the layer: the experts split over ranks, the
routed rows exchanged between them.

The Mixtral pages deploy the 8x7B model on two GPUs (youtublog.net page,
deployment setup: 2 GPUs x 80 GB, BF16).  With the E experts split over G
ranks - rank g holds experts g*El .. (g+1)*El - 1, El = E / G - each rank
routes and dispatches its own tokens over all E experts, sends every routed
row to the rank that holds its expert, runs its own experts' grouped GEMMs on
the rows it received, sends the results back, and combines its tokens.  The
arithmetic per token is the single-GPU layer's; only where each expert's
GEMM runs changes.

One forward, for one rank (compute in libmoe's kernels, exchange through a
communicator, e.g. ``TorchComm`` over torch.distributed):
  route     moe_router_topk + moe_permute of the local tokens over all E
            experts; x_perm is expert-major, so the rows for rank g are the
            contiguous block of experts g*El .. (g+1)*El - 1.
  counts    all-to-all of El per-expert counts per rank pair ->
            ``ExchangePlan`` (host: the split sizes must be known to post
            the row exchange, so the counts come to the host once per call).
  rows      all-to-all of the routed rows (received rank-major), then
            moe_gather_rows regroups them expert-major: for each local
            expert, the rows of rank 0, then of rank 1, ... - the order a
            single-GPU dispatch of all ranks' tokens, concatenated in rank
            order, gives that expert.
  experts   moe_expert_ffn_ws on the local experts' weights.
  back      moe_gather_rows back to rank-major, the reverse all-to-all (each
            row returns to where x_perm held it), moe_combine.
The rows land in local memory before the grouped GEMMs read them; no kernel
reads a peer's memory.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass
class ExchangePlan:
    """The row exchange of one forward on one rank, from the counts.

    counts_send[g, j]: rows this rank sends for expert j of rank g (its own
    dispatch counts, reshaped [G, El]); counts_recv[s, j]: rows rank s sends
    for this rank's local expert j.  Everything else follows:
      send_splits[g]   rows to rank g (a contiguous block of x_perm)
      recv_splits[s]   rows from rank s (the receive buffer is rank-major;
                       within a rank, expert-major, as its x_perm)
      local_offsets    [El+1] boundaries of the local experts' rows after
                       regrouping (expert-major, ranks in order within one)
      regroup_src[q]   receive-buffer row of expert-major row q
      ungroup_src[p]   expert-major row of receive-buffer row p (the inverse)
    """

    counts_send: np.ndarray
    counts_recv: np.ndarray
    send_splits: list
    recv_splits: list
    local_offsets: np.ndarray
    regroup_src: np.ndarray
    ungroup_src: np.ndarray

    @classmethod
    def build(cls, counts_send, counts_recv) -> "ExchangePlan":
        cs = np.asarray(counts_send, dtype=np.int64)
        cr = np.asarray(counts_recv, dtype=np.int64)
        if cs.ndim != 2 or cs.shape != cr.shape or (cs < 0).any() or (cr < 0).any():
            raise ValueError("counts must be two non-negative [G, El] arrays")
        G, El = cr.shape
        # Receive buffer: rank s's block starts at recv_base[s]; within it,
        # expert j's rows start at recv_base[s] + sum(cr[s, :j]).
        recv_base = np.concatenate([[0], np.cumsum(cr.sum(axis=1))])
        within = np.concatenate([np.zeros((G, 1), dtype=np.int64), np.cumsum(cr, axis=1)[:, :-1]], axis=1)
        local_counts = cr.sum(axis=0)
        regroup = []
        for j in range(El):
            for s in range(G):
                start = recv_base[s] + within[s, j]
                regroup.append(np.arange(start, start + cr[s, j], dtype=np.int64))
        regroup_src = np.concatenate(regroup) if regroup else np.zeros(0, dtype=np.int64)
        ungroup_src = np.empty_like(regroup_src)
        ungroup_src[regroup_src] = np.arange(regroup_src.size, dtype=np.int64)
        return cls(counts_send=cs, counts_recv=cr,
                   send_splits=[int(v) for v in cs.sum(axis=1)], recv_splits=[int(v) for v in cr.sum(axis=1)],
                   local_offsets=np.concatenate([[0], np.cumsum(local_counts)]).astype(np.int64),
                   regroup_src=regroup_src, ungroup_src=ungroup_src)


class TorchComm:
    """The exchanges over torch.distributed (NCCL for CUDA tensors, gloo for
    CPU tensors): all-to-all of counts and of rows with given split sizes."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)

    def all_to_all_counts(self, counts_send: torch.Tensor) -> torch.Tensor:
        """counts_send [G*El] int64 (block g for rank g) -> counts_recv [G*El]
        (block s from rank s)."""
        out = torch.empty_like(counts_send)
        self.dist.all_to_all_single(out, counts_send, group=self.group)
        return out

    def all_to_all_rows(self, rows: torch.Tensor, send_splits, recv_splits) -> torch.Tensor:
        """rows [sum(send_splits), d], block g to rank g -> [sum(recv_splits), d],
        block s from rank s."""
        out = rows.new_empty((int(sum(recv_splits)),) + tuple(rows.shape[1:]))
        self.dist.all_to_all_single(out, rows.contiguous(), output_split_sizes=list(recv_splits),
                                    input_split_sizes=list(send_splits), group=self.group)
        return out


@dataclass
class _Routed:
    T: int
    w: torch.Tensor
    slot_pos: torch.Tensor
    x_perm: torch.Tensor
    counts: np.ndarray


class ExpertParallelMoE:
    """The bf16 layer with this rank's share of the experts.

    Wg [E, d] is every rank's (the router sees all experts); W1l, W3l
    [El, dff, d] and W2l [El, d, dff] are this rank's experts, global ids
    rank*El .. rank*El + El - 1.  ``forward(x)`` must be called by every rank
    of the communicator together.  The steps are also callable one by one
    (``route``, ``experts``, ``combine``) around exchanges done elsewhere."""

    def __init__(self, Wg, W1l, W3l, W2l, k, comm, rank=None, world=None):
        from . import binding
        self.B = binding
        self.Wg, self.W1l, self.W3l, self.W2l, self.k = Wg, W1l, W3l, W2l, k
        self.comm = comm
        self.rank = comm.rank if rank is None else rank
        self.world = comm.world if world is None else world
        self.E = Wg.shape[0]
        self.El = W1l.shape[0]
        if self.El * self.world != self.E:
            raise ValueError(f"{self.E} experts do not split into {self.world} ranks of {self.El}")

    def route(self, x) -> _Routed:
        """Router and dispatch of the local tokens over all E experts."""
        idx, w = self.B.moe_router_topk(x, self.Wg, self.k)
        counts, _, _, slot_pos, x_perm = self.B.moe_permute(x, idx, self.E)
        return _Routed(T=x.shape[0], w=w, slot_pos=slot_pos, x_perm=x_perm,
                       counts=counts.cpu().numpy().astype(np.int64))

    def plan(self, routed: _Routed, counts_recv) -> ExchangePlan:
        return ExchangePlan.build(routed.counts.reshape(self.world, self.El),
                                  np.asarray(counts_recv, dtype=np.int64).reshape(self.world, self.El))

    def experts(self, x_recv, plan: ExchangePlan):
        """Regroup the received rows expert-major, run the local experts'
        grouped GEMMs, and put the results back in receive order."""
        dev = x_recv.device
        n = x_recv.shape[0]
        if n == 0:
            return x_recv.new_empty((0, self.W2l.shape[1]))
        regroup = torch.from_numpy(plan.regroup_src.astype(np.int32)).to(dev)
        ungroup = torch.from_numpy(plan.ungroup_src.astype(np.int32)).to(dev)
        offsets = torch.from_numpy(plan.local_offsets.astype(np.int32)).to(dev)
        x_loc = self.B.moe_gather_rows(x_recv, regroup)
        _, y_loc = self.B.moe_expert_ffn_ws(x_loc, offsets, self.W1l, self.W3l, self.W2l)
        return self.B.moe_gather_rows(y_loc, ungroup)

    def combine(self, routed: _Routed, y_perm):
        return self.B.moe_combine(y_perm, routed.slot_pos, routed.w, routed.T)

    def forward(self, x):
        routed = self.route(x)
        counts_recv = self.comm.all_to_all_counts(torch.from_numpy(routed.counts).to(x.device))
        plan = self.plan(routed, counts_recv.cpu().numpy())
        x_recv = self.comm.all_to_all_rows(routed.x_perm, plan.send_splits, plan.recv_splits)
        y_recv = self.experts(x_recv, plan)
        y_perm = self.comm.all_to_all_rows(y_recv, plan.recv_splits, plan.send_splits)
        return self.combine(routed, y_perm)
