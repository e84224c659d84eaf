"""The expert-parallel exchange on the CPU: world_size 2, gloo backend.

Each rank routes and dispatches its own tokens with the oracle's step
functions (standing in for the GPU kernels, which these CPU ranks cannot
run), then exchanges counts and rows with the library's ``TorchComm`` and
regroups them with its ``ExchangePlan``.  The rows each rank ends up with for
its own experts must equal, bit for bit, the rows a single dispatch of all
ranks' tokens (concatenated in rank order) gives those experts; after the
experts run and the results travel back, each rank's output must equal the
whole layer's on its tokens.
"""
import os
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_mixture_experts_50_b300.expert_parallel import ExchangePlan  # noqa: E402

E, K, D, F = 8, 2, 16, 24
TOKENS = (37, 58)  # rank 0, rank 1


def _layer(seed=5):
    r = np.random.default_rng(seed)
    return dict(Wg=r.standard_normal((E, D)) / 4, W1=r.standard_normal((E, F, D)) / 4,
                W3=r.standard_normal((E, F, D)) / 4, W2=r.standard_normal((E, D, F)) / 5)


def _tokens(rank):
    return np.random.default_rng(100 + rank).standard_normal((TOKENS[rank], D))


def test_plan_regroups_expert_major():
    """Three ranks, two local experts each: a receive buffer labelled (source,
    expert, i) comes out expert-major, sources in order, i ascending; the
    inverse puts it back; splits and offsets are the sums they must be."""
    r = np.random.default_rng(3)
    G, El = 3, 2
    cs = r.integers(0, 5, (G, El))
    cr = r.integers(0, 5, (G, El))
    cr[1, 0] = 0  # an empty (source, expert) block
    p = ExchangePlan.build(cs, cr)
    assert p.send_splits == [int(v) for v in cs.sum(1)] and p.recv_splits == [int(v) for v in cr.sum(1)]
    labels = [(s, j, i) for s in range(G) for j in range(El) for i in range(cr[s, j])]
    regrouped = [labels[q] for q in p.regroup_src]
    assert regrouped == [(s, j, i) for j in range(El) for s in range(G) for i in range(cr[s, j])]
    assert list(p.local_offsets) == [0] + list(np.cumsum(cr.sum(0)))
    assert np.array_equal(p.regroup_src[p.ungroup_src], np.arange(len(labels)))
    with pytest.raises(ValueError):
        ExchangePlan.build(cs, cr[:, :1])


def test_plan_with_no_rows():
    p = ExchangePlan.build(np.zeros((2, 4), dtype=np.int64), np.zeros((2, 4), dtype=np.int64))
    assert p.regroup_src.size == 0 and list(p.local_offsets) == [0] * 5


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import oracle.moe_oracle as O
    from sparse_mixture_experts_50_b300.expert_parallel import ExchangePlan, TorchComm
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        comm = TorchComm()
        El = E // world
        mine = slice(rank * El, (rank + 1) * El)
        L = _layer()
        x = _tokens(rank)
        # route + dispatch of the local tokens (the oracle standing in for the kernels)
        w, idx, _ = O.router(x, L["Wg"], K)
        counts, _, row_src, slot_pos = O.dispatch(idx, E)
        x_perm = torch.from_numpy(x[row_src])
        counts_recv = comm.all_to_all_counts(torch.from_numpy(counts.astype(np.int64)))
        plan = ExchangePlan.build(counts.reshape(world, El), counts_recv.numpy().reshape(world, El))
        x_recv = comm.all_to_all_rows(x_perm, plan.send_splits, plan.recv_splits)
        x_loc = x_recv.numpy()[plan.regroup_src]
        # What a single dispatch of all ranks' tokens gives this rank's experts.
        X = np.concatenate([_tokens(r) for r in range(world)])
        _, idx_all, _ = O.router(X, L["Wg"], K)
        c_all, off_all, src_all, _ = O.dispatch(idx_all, E)
        want = X[src_all[off_all[rank * El]:off_all[(rank + 1) * El]]]
        rows_ok = bool(np.array_equal(x_loc, want))
        offs_ok = bool(np.array_equal(plan.local_offsets, off_all[rank * El:(rank + 1) * El + 1] - off_all[rank * El]))
        # this rank's experts, then the way back
        lo = plan.local_offsets
        h = O.gate_up_projection(x_loc, lo, L["W1"][mine], L["W3"][mine])
        y_loc = O.down_projection(h, lo, L["W2"][mine])
        y_perm = comm.all_to_all_rows(torch.from_numpy(y_loc[plan.ungroup_src]), plan.recv_splits, plan.send_splits)
        out = O.combine(y_perm.numpy(), slot_pos, w)
        ref, _, _, _ = O.moe_forward(x, L["Wg"], L["W1"], L["W3"], L["W2"], K)
        err = float(np.max(np.abs(out - ref)) / np.max(np.abs(ref)))
        q.put((rank, rows_ok, offs_ok, err, plan.send_splits, plan.recv_splits))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_exchange_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 30500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, rows_ok, offs_ok, err, send, recv in got:
        assert rows_ok, f"rank {rank}: regrouped rows differ from the single-dispatch rows"
        assert offs_ok, f"rank {rank}: local expert offsets differ"
        assert err < 1e-12, f"rank {rank}: output differs from the whole layer by {err:.2e}"
        assert sum(send) == TOKENS[rank] * K
    # what rank 0 sends to rank 1 is what rank 1 receives from rank 0, and back
    assert got[0][4][1] == got[1][5][0] and got[1][4][0] == got[0][5][1]
