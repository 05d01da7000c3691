"""Multi-process paths on the CPU (gloo, world size 2), no GPU.

1. bench.py's cross-rank timing: every rank gets the slowest rank's time and
   the whole-job rate counts the units of all ranks.
2. The data-parallel recipe the C ABI is built for: each rank holds a slice of
   the tokens and a replica of W, computes its per-row losses and its dW with
   the upstream gradient 1/n_valid of the WHOLE batch, then sums dW and
   (sum of losses, n_valid) across ranks. The result must equal the unsharded
   computation. The per-rank arithmetic here is the CPU oracle (test
   infrastructure), so this checks the composition rule, not the kernels.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)


def _timing_worker(rank, port, q):
    import bench
    _init(rank, port)
    try:
        ms = [120.0, 180.0][rank]
        worst = bench.max_over_ranks(ms, WORLD, "cpu")
        q.put((rank, worst, bench.job_rate(32768, WORLD, 10, worst)))
    finally:
        dist.destroy_process_group()


def _problem(seed=0, N=40, D=12, V=50, K=5, T=1.5):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, D))
    W = rng.standard_normal((V, D)) / np.sqrt(D)
    idx = np.stack([rng.choice(V, size=K, replace=False) for _ in range(N)]).astype(np.int64)
    t = np.sort(2.0 * rng.standard_normal((N, K)), axis=1)[:, ::-1].copy()
    mask = (rng.random(N) > 0.2).astype(np.uint8)
    return H, W, idx, t, mask, T


def _dp_worker(rank, port, q):
    _init(rank, port)
    try:
        H, W, idx, t, mask, T = _problem()
        N = H.shape[0]
        lo, hi = rank * N // WORLD, (rank + 1) * N // WORLD
        sl = slice(lo, hi)
        # global n_valid first: one all-reduce of the local count
        nv = torch.tensor([float(mask[sl].sum())], dtype=torch.float64)
        dist.all_reduce(nv)
        n_valid = int(nv.item())
        loss, _lse, _ = oracle.kd_forward(H[sl], W, idx[sl], t[sl], mask[sl], T)
        g = mask[sl].astype(np.float64) / n_valid
        dH, dW = oracle.kd_backward(H[sl], W, idx[sl], t[sl], mask[sl], T, g)
        tot = torch.tensor([loss.sum()], dtype=torch.float64)
        dist.all_reduce(tot)
        dWt = torch.from_numpy(dW)
        dist.all_reduce(dWt)
        q.put((rank, lo, float(tot.item()) / n_valid, dH, dWt.numpy()))
    finally:
        dist.destroy_process_group()


def _run(worker):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=worker, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(WORLD)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out, key=lambda x: x[0])


def test_bench_timing_takes_the_slowest_rank():
    out = _run(_timing_worker)
    for _rank, worst, rate in out:
        assert worst == 180.0
        assert rate == pytest.approx(2 * 32768 * 10 / 0.180)


def test_token_sharded_dp_matches_unsharded():
    out = _run(_dp_worker)
    H, W, idx, t, mask, T = _problem()
    loss, _lse, nv = oracle.kd_forward(H, W, idx, t, mask, T)
    g = mask.astype(np.float64) / nv
    dH, dW = oracle.kd_backward(H, W, idx, t, mask, T, g)
    mean = oracle.mean_loss(loss, nv)
    N = H.shape[0]
    for rank, lo, mean_r, dH_r, dW_r in out:
        assert mean_r == pytest.approx(mean, rel=1e-12)
        np.testing.assert_allclose(dH_r, dH[lo:lo + dH_r.shape[0]], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(dW_r, dW, rtol=1e-10, atol=1e-14)
    assert sum(o[3].shape[0] for o in out) == N
