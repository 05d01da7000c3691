"""Multi-process paths on the CPU (gloo, world size 2), no GPU.

1. bench.py's cross-rank timing: every rank gets the slowest rank's time and
   the whole-job rate counts the units of all ranks.
2. The product's multi-GPU orchestration (``top_kl_loss_lm_b300.sharded``):
   the token-sharded (data-parallel) step and the vocabulary-sharded step,
   each rank running its part and the ranks exchanging counts, partial
   logsumexps, dW or dH with the module's own collectives. The compute calls
   are the oracle-backed stand-ins of ``tests/_oracle_ops`` (the kernels cannot
   run here), so this checks the sharding and the reductions: every rank's
   result must equal the unsharded oracle.
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
    idx = np.stack([rng.choice(V, size=K, replace=False) for _ in range(N)]).astype(np.int32)
    t = np.sort(2.0 * rng.standard_normal((N, K)), axis=1)[:, ::-1].copy()
    mask = (rng.random(N) > 0.2).astype(np.uint8)
    t[mask == 0] = np.nan  # masked rows' teacher entries are never read
    return H, W, idx, t, mask, T


def _tensors(H, W, idx, t, mask):
    return (torch.from_numpy(H), torch.from_numpy(W), torch.from_numpy(idx), torch.from_numpy(t),
            torch.from_numpy(mask))


def _fp64(head, *names):
    for n in names:
        setattr(head, n, torch.zeros(getattr(head, n).shape, dtype=torch.float64))


def _token_worker(rank, port, q):
    from tests import _oracle_ops
    from top_kl_loss_lm_b300 import sharded
    _init(rank, port)
    try:
        H, W, idx, t, mask, T = _problem()
        N, D = H.shape
        lo, hi = sharded.token_range(N, rank, WORLD)
        Ht, Wt, it, tt, mt = _tensors(H[lo:hi], W, idx[lo:hi], t[lo:hi], mask[lo:hi])
        head = sharded.TokenShardedHead(hi - lo, D, W.shape[0], idx.shape[1], T, "cpu",
                                        ops=_oracle_ops)
        _fp64(head, "loss", "lse", "dloss", "dH", "dW")  # the CPU stand-in computes in fp64
        loss_sum, nv = head.step(Ht, Wt, it, tt, mt)
        q.put((rank, lo, sharded.mean_loss(loss_sum, nv), int(nv.item()), head.dH.numpy(),
               head.dW.numpy(), head.loss.numpy()))
    finally:
        dist.destroy_process_group()


def _vocab_worker(rank, port, q):
    from tests import _oracle_ops
    from top_kl_loss_lm_b300 import sharded
    _init(rank, port)
    try:
        H, W, idx, t, mask, T = _problem()
        N, D = H.shape
        V = W.shape[0]
        head = sharded.VocabShardedHead(N, D, V, idx.shape[1], T, "cpu", ops=_oracle_ops, align=8)
        _fp64(head, "local", "parts", "ent", "loss", "lse", "dloss", "dH", "dW_shard")
        Ht, Wt, it, tt, mt = _tensors(H, W[head.v0:head.v1], idx, t, mask)
        loss_sum, nv = head.step(Ht, Wt, it, tt, mt)
        q.put((rank, head.v0, sharded.mean_loss(loss_sum, nv), head.loss.numpy(), head.lse.numpy(),
               head.dH.numpy(), head.dW_shard.numpy()))
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


def _reference():
    H, W, idx, t, mask, T = _problem()
    loss, lse, nv = oracle.kd_forward(H, W, idx, t, mask, T)
    g = mask.astype(np.float64) / nv
    dH, dW = oracle.kd_backward(H, W, idx, t, mask, T, g)
    return H, W, loss, lse, nv, dH, dW


def test_token_sharded_step_matches_unsharded():
    out = _run(_token_worker)
    H, W, loss, lse, nv, dH, dW = _reference()
    mean = oracle.mean_loss(loss, nv)
    rows = 0
    for rank, lo, mean_r, nv_r, dH_r, dW_r, loss_r in out:
        assert nv_r == nv                                    # the count is global on every rank
        assert mean_r == pytest.approx(mean, rel=1e-12)
        np.testing.assert_allclose(loss_r, loss[lo:lo + loss_r.shape[0]], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(dH_r, dH[lo:lo + dH_r.shape[0]], rtol=1e-12, atol=1e-15)
        np.testing.assert_allclose(dW_r, dW, rtol=1e-10, atol=1e-14)  # summed over the ranks
        rows += dH_r.shape[0]
    assert rows == H.shape[0]


def test_vocab_sharded_step_matches_unsharded():
    out = _run(_vocab_worker)
    H, W, loss, lse, nv, dH, dW = _reference()
    mean = oracle.mean_loss(loss, nv)
    cols = 0
    for rank, v0, mean_r, loss_r, lse_r, dH_r, dW_r in out:
        assert mean_r == pytest.approx(mean, rel=1e-12)
        np.testing.assert_allclose(loss_r, loss, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse_r, lse, rtol=1e-13)
        np.testing.assert_allclose(dH_r, dH, rtol=1e-10, atol=1e-14)   # summed over the shards
        np.testing.assert_allclose(dW_r, dW[v0:v0 + dW_r.shape[0]], rtol=1e-12, atol=1e-15)
        cols += dW_r.shape[0]
    assert cols == W.shape[0]
    # every rank merged the same gathered parts into the same bits
    assert all(np.array_equal(o[3], out[0][3]) for o in out)


def test_shard_ranges_cover_disjointly():
    from top_kl_loss_lm_b300 import sharded
    for N, world in ((32768, 8), (301, 3), (5, 4)):
        spans = [sharded.token_range(N, r, world) for r in range(world)]
        assert spans[0][0] == 0 and spans[-1][1] == N
        assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
    for V, world in ((201088, 8), (151936, 3), (1000, 4), (300, 2)):
        spans = [sharded.vocab_range(V, r, world) for r in range(world)]
        assert spans[0][0] == 0 and spans[-1][1] == V
        assert all(a[1] == b[0] and a[1] > a[0] for a, b in zip(spans, spans[1:]))
        assert all(v0 % 256 == 0 for v0, _ in spans)
    with pytest.raises(ValueError):
        sharded.vocab_range(300, 0, 3)  # two 256-wide tiles cannot make three shards
