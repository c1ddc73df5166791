"""The data-parallel exchange of the MLP backward on two CPU ranks (gloo).

Under data parallelism each rank runs the backward on its own slice of the
tokens and accumulates fp32 weight gradients; one all-reduce (sum) of dWg,
dWu, dWd then equals the single-process gradient, and the dx rows stay
local.  This checks that invariant with a real gloo all-reduce over the
oracle's per-shard gradients (the GPU path is one process per GPU and
writes into the same fp32 accumulate buffers)."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def shard(M, rank, world):
    """Contiguous token slice of `rank` (the first M % world ranks get one more)."""
    base, rem = divmod(M, world)
    start = rank * base + min(rank, rem)
    return start, start + base + (1 if rank < rem else 0)


def _worker(rank, world, port, result_path):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from activated_mlp_gemms_gb300.workloads import make_inputs, to_f64
    from oracle import mlp_backward

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    M, H, I = 37, 16, 24
    t = {k: to_f64(v) for k, v in make_inputs(M, H, I, "swiglu", seed=3).items() if v is not None}
    a, b = shard(M, rank, world)
    loc = mlp_backward(t["dout"][a:b], t["x"][a:b], t["Wg"], t["Wu"], t["Wd"], "swiglu", 1.125, 2.0)
    grads = {k: torch.tensor(loc[k]) for k in ("dWg", "dWu", "dWd")}
    for v in grads.values():
        dist.all_reduce(v, op=dist.ReduceOp.SUM)
    # gather the local dx rows (padded to the largest shard: gloo gathers equal sizes)
    rows = [shard(M, r, world)[1] - shard(M, r, world)[0] for r in range(world)]
    dx = torch.zeros(max(rows), H, dtype=torch.float64)
    dx[: b - a] = torch.tensor(loc["dx"])
    parts = [torch.zeros_like(dx) for _ in range(world)]
    dist.all_gather(parts, dx)
    parts = [p[:n] for p, n in zip(parts, rows)]
    if rank == 0:
        full = mlp_backward(t["dout"], t["x"], t["Wg"], t["Wu"], t["Wd"], "swiglu", 1.125, 2.0)
        errs = {k: float(np.max(np.abs(grads[k].numpy() - full[k]))) for k in grads}
        errs["dx"] = float(np.max(np.abs(torch.cat(parts).numpy() - full["dx"])))
        with open(result_path, "w") as f:
            f.write(repr(errs))
    dist.barrier()
    dist.destroy_process_group()


def test_shard_covers_tokens():
    for M in (1, 7, 37, 2048):
        for world in (1, 2, 3, 8):
            spans = [shard(M, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == M
            assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))


def test_two_rank_gradient_allreduce_equals_single_process(tmp_path):
    path = str(tmp_path / "errs.txt")
    mp.start_processes(_worker, args=(2, _free_port(), path), nprocs=2, join=True,
                       start_method="spawn")
    errs = eval(open(path).read())  # noqa: S307 (our own file)
    for k, e in errs.items():
        assert e < 1e-12, (k, e)
