"""The expert-parallel layer's GPU steps on one GPU (GPU).

Two (or four) ranks are emulated in one process: their routing, experts and
combine run through the library's kernels one rank after another, and the
exchanges between them are done here by slicing and concatenating the
blocks each rank sends, in the order torch.distributed's all-to-all would
deliver them.  Each rank's output must match the single-GPU layer's on its
own tokens and the oracle.  The layer's own forward also runs over NCCL
with one rank (the all-to-alls are then the identity), and so does the
bench's expert-parallel leg.  The exchange between several ranks over
torch.distributed is covered on CPU ranks with gloo.
"""
import numpy as np
import pytest
import torch

import moe_workloads as mw
import oracle.moe_oracle as O
from parity import check_close, check_routing, effective_routing, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from sparse_mixture_experts_50_b300 import binding
    binding.lib()
    binding.moe_get_device_status(reset=True)
    return binding


def test_gather_rows_bit_exact(B):
    r = np.random.default_rng(7)
    src = torch.from_numpy(r.standard_normal((300, 72))).to(torch.bfloat16)
    idx = r.integers(0, 300, 777).astype(np.int32)
    got = B.moe_gather_rows(src.to(DEV), torch.from_numpy(idx).to(DEV))
    assert B.moe_get_device_status(reset=True) == 0
    assert torch.equal(got.cpu(), src[torch.from_numpy(idx).long()])


def emulate(B, layers, xs):
    """One forward of every emulated rank, exchanges done by slicing."""
    from sparse_mixture_experts_50_b300.expert_parallel import ExchangePlan
    G = len(layers)
    El = layers[0].El
    routed = [L.route(x) for L, x in zip(layers, xs)]
    plans = []
    for g in range(G):
        counts_recv = np.stack([routed[s].counts[g * El:(g + 1) * El] for s in range(G)])
        plans.append(layers[g].plan(routed[g], counts_recv.reshape(-1)))

    def block(buf, splits, g):
        a = int(sum(splits[:g]))
        return buf[a:a + splits[g]]

    x_recv = [torch.cat([block(routed[s].x_perm, plans[s].send_splits, g) for s in range(G)]) for g in range(G)]
    y_recv = [layers[g].experts(x_recv[g], plans[g]) for g in range(G)]
    y_perm = [torch.cat([block(y_recv[g], plans[g].recv_splits, s) for g in range(G)]) for s in range(G)]
    return [layers[s].combine(routed[s], y_perm[s]) for s in range(G)], plans


@pytest.mark.parametrize("G,tokens", [(2, (37, 300)), (4, (5, 0, 129, 64)), (2, (16, 16))])
def test_expert_parallel_matches_layer(B, G, tokens):
    from sparse_mixture_experts_50_b300.expert_parallel import ExpertParallelMoE
    wl = mw.get("small_bf16")
    t = mw.make_inputs(wl)
    g = {n: v.to(DEV) for n, v in t.items()}
    El = wl.E // G
    r = np.random.default_rng(sum(tokens))
    xs_cpu = [torch.from_numpy(r.standard_normal((n, wl.d))).to(torch.bfloat16) for n in tokens]
    xs = [x.to(DEV) for x in xs_cpu]
    layers = [ExpertParallelMoE(g["Wg"], g["W1"][s * El:(s + 1) * El].contiguous(),
                                g["W3"][s * El:(s + 1) * El].contiguous(), g["W2"][s * El:(s + 1) * El].contiguous(),
                                wl.k, comm=None, rank=s, world=G) for s in range(G)]
    outs, plans = emulate(B, layers, xs)
    assert B.moe_get_device_status(reset=True) == 0
    for s in range(G):
        assert sum(plans[s].send_splits) == tokens[s] * wl.k
        if tokens[s] == 0:
            assert outs[s].shape == (0, wl.d)
            continue
        ref_gpu = B.moe_forward(xs[s], g["Wg"], g["W1"], g["W3"], g["W2"], wl.k)
        check_close(to_np(outs[s]), to_np(ref_gpu), "bf16", f"rank {s} vs the single-GPU layer")
        ref, ora_w, ora_idx, logits = O.moe_forward(xs_cpu[s], t["Wg"], t["W1"], t["W3"], t["W2"], wl.k)
        gidx, gw = B.moe_router_topk(xs[s], g["Wg"], wl.k)
        check_routing(to_np(gidx), to_np(gw), ora_idx, ora_w, logits, wl.k)
        w_eff, idx_eff = effective_routing(to_np(gidx), ora_w, ora_idx, logits)
        if not np.array_equal(idx_eff, ora_idx):
            ref = O.moe_forward_with_routing(xs_cpu[s], t["W1"], t["W3"], t["W2"], w_eff, idx_eff)
        check_close(to_np(outs[s]), ref, "bf16", f"rank {s} vs the oracle")


def _nccl_rank(q):
    import os
    import sys
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(31500 + os.getpid() % 1000), RANK="0",
                      WORLD_SIZE="1")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    sys.path.insert(0, os.path.join(root, "tests"))
    import torch
    import torch.distributed as dist

    import moe_workloads as mw
    from sparse_mixture_experts_50_b300 import binding
    from sparse_mixture_experts_50_b300.expert_parallel import ExpertParallelMoE, TorchComm
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda:0"))
    try:
        wl = mw.get("small_bf16")
        g = {n: v.to("cuda:0") for n, v in mw.make_inputs(wl).items()}
        layer = ExpertParallelMoE(g["Wg"], g["W1"], g["W3"], g["W2"], wl.k, TorchComm())
        out = layer.forward(g["x"])
        ref = binding.moe_forward(g["x"], g["Wg"], g["W1"], g["W3"], g["W2"], wl.k)
        torch.cuda.synchronize()
        q.put((bool(torch.equal(out, ref)), binding.moe_get_device_status(reset=True)))
    finally:
        dist.destroy_process_group()


def test_expert_parallel_forward_over_nccl_one_rank(B):
    """ExpertParallelMoE.forward with TorchComm over NCCL (one rank, device
    tensors): the exchange is the identity, so the output must equal
    moe_forward's bit for bit."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    p = ctx.Process(target=_nccl_rank, args=(q,))
    p.start()
    p.join(timeout=300)
    assert p.exitcode == 0
    same, status = q.get(timeout=5)
    assert status == 0 and same


def test_bench_expert_parallel_leg_one_rank(B):
    """bench.py --expert-parallel at one rank (NCCL world of one): the leg
    runs the Mixtral-shape decode through ExpertParallelMoE and prints one
    well-formed JSON line."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--expert-parallel", "--steps", "3",
                        "--warmup", "3"], cwd=root, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = r.stdout.strip().splitlines()
    assert lines and lines[-1].startswith("{"), r.stdout[-500:]
    line = json.loads(lines[-1])
    assert line["n_gpus"] == 1 and line["steps"] == 3 and line["value"] > 0
    assert line["config"]["parallelism"].startswith("expert-parallel x1")
    assert line["roofline"]["bound"] == "hbm" and line["roofline"]["achieved"] > 0
