"""World-size-2 gloo checks of the multi-rank path (CPU only).

bench.py runs one replica of the layer per rank on that rank's own tokens and
reports the maximum time over ranks.  Here two gloo ranks check the host-side
pieces (barrier, max-over-ranks) and that sharding tokens across ranks is
exact: concatenated per-rank outputs equal the single-batch oracle, and the
weight gradients summed in rank order equal the single-batch ones.
"""
import json
import os
import socket
import subprocess
import sys

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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    from mixture_experts_layer_19_gb300.workload import LayerShape, make_inputs, to_f64
    from oracle import moe_ref
    try:
        bench.init_dist(world, "gloo")
        ws, r, _ = bench.dist_env()
        assert (ws, r) == (world, rank)
        bench.barrier(ws)
        m = bench.max_over_ranks(1.5 + rank, ws, torch.device("cpu"))
        # token sharding: rank r takes tokens [r*T/2, (r+1)*T/2)
        T, d, F, E, k = 32, 32, 32, 4, 2
        inp = make_inputs(LayerShape(T, d, F, E, k), seed=3, alpha=1.1)
        X, L, Wg, Wu, Wd, dY = (to_f64(getattr(inp, n)) for n in ("X", "logits", "Wg", "Wu", "Wd", "dY"))
        sl = slice(rank * T // world, (rank + 1) * T // world)
        Y, ctx = moe_ref.forward(X[sl], L[sl], Wg, Wu, Wd, k)
        g = moe_ref.backward(dY[sl], X[sl], L[sl], Wg, Wu, Wd, ctx)
        parts = [torch.zeros_like(torch.from_numpy(Y)) for _ in range(world)]
        dist.all_gather(parts, torch.from_numpy(Y))
        dw = [torch.zeros(E, F, d, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(dw, torch.from_numpy(g["dWg"]))
        if rank == 0:
            Yf, cf = moe_ref.forward(X, L, Wg, Wu, Wd, k)
            gf = moe_ref.backward(dY, X, L, Wg, Wu, Wd, cf)
            ycat = torch.cat(parts).numpy()
            dsum = dw[0].numpy().copy()
            for i in range(1, world):
                dsum += dw[i].numpy()
            q.put((m, float(np.abs(ycat - Yf).max()), float(np.abs(dsum - gf["dWg"]).max() / np.abs(gf["dWg"]).max())))
        bench.barrier(ws)
        dist.destroy_process_group()
    except Exception as e:  # report instead of hanging the parent
        q.put(("error", repr(e)))


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = q.get(timeout=240)
    for p in procs:
        p.join(timeout=60)
    assert res[0] != "error", res
    m, yerr, dwerr = res
    assert m == 2.5
    assert yerr == 0.0
    assert dwerr < 1e-13


def test_bench_launches_its_own_ranks():
    """`bench.py --gpus 2` outside any launcher starts two ranks itself
    (torch.distributed.run on 127.0.0.1); the dry run exchanges their timings
    over gloo and rank 0 alone prints one line with the max over ranks."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--dry-run"],
                       capture_output=True, text=True, timeout=240, env=env, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    assert out["n_gpus"] == 2 and out["config"]["parallelism"] == "replicas2"
    assert out["max_rank_ms"] >= 20.0          # rank 1 waits 20 ms, rank 0 10 ms: the max is taken
