"""Guard bands around every buffer the library writes (compute-sanitizer is not
available on these GPUs, so out-of-bounds writes are caught this way).

Each output and the workspace is carved out of a larger allocation whose bytes
before and after it are set to a sentinel; after the call the sentinels must be
intact, and the inputs must be unchanged. The shapes are ragged on purpose: N,
V and D off the tile multiples, a short last backward chunk and forward chunk,
K = 1 and K = 256, vocabulary shards that start mid-tile, so the TMA boxes past
V and N, the dZ row padding and the selection kernel's candidate arrays all sit
next to a guard band.
"""
import pytest
import torch

from top_kl_loss_lm_b300 import binding
from workloads import make_problem, mean_upstream_grad

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
GUARD = 4096   # bytes on each side; a multiple of 256 keeps every view's alignment
SENTINEL = 0x5A


class Guarded:
    """A tensor of the given shape and dtype with sentinel bands around it."""

    def __init__(self, shape, dtype, fill=float("nan")):
        n = 1
        for d in shape:
            n *= d
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((GUARD + nbytes + GUARD,), SENTINEL, dtype=torch.uint8, device=DEV)
        self.t = self.raw[GUARD:GUARD + nbytes].view(dtype).view(shape)
        if dtype.is_floating_point:
            self.t.fill_(fill)
        else:
            self.t.fill_(-1 if dtype != torch.uint8 else 0xEE)

    def check(self, name):
        torch.cuda.synchronize()
        lo = self.raw[:GUARD]
        hi = self.raw[self.raw.numel() - GUARD:]
        assert torch.all(lo == SENTINEL) and torch.all(hi == SENTINEL), f"{name}: guard band overwritten"


def _inputs_unchanged(before, after):
    # byte for byte: masked rows carry NaN teacher logits, which never compare equal
    for name, (a, b) in zip(("H", "W", "idx", "t", "mask"), zip(before, after)):
        assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8)), \
            f"input {name} written"


def _fwd_bwd(p, chunk, accumulate=False):
    N, D, V, K = p.N, p.D, p.V, p.K
    snap = [x.clone() for x in (p.H, p.W, p.idx, p.t, p.mask)]
    ws = Guarded((binding.kd_topk_kl_workspace_size(N, D, V, K, chunk),), torch.uint8)
    loss, lse = Guarded((N,), torch.float32), Guarded((N,), torch.float32)
    nv = Guarded((1,), torch.int64)
    dH = Guarded((N, D), torch.bfloat16)
    dW = Guarded((V, D), torch.float32, fill=0.0)
    binding.kd_topk_kl_fwd(p.H, p.W, p.idx, p.t, p.mask, p.T, loss.t, lse.t, nv.t, ws.t)
    g = mean_upstream_grad(p.mask).to(DEV)
    binding.kd_topk_kl_bwd(p.H, p.W, p.idx, p.t, p.mask, lse.t, g, p.T, chunk, accumulate, dH.t, dW.t,
                           ws.t)
    for name, b in (("ws", ws), ("loss", loss), ("lse", lse), ("n_valid", nv), ("dH", dH), ("dW", dW)):
        b.check(name)
    assert binding.kd_get_status() == 0
    _inputs_unchanged(snap, (p.H, p.W, p.idx, p.t, p.mask))
    assert torch.isfinite(loss.t).all() and torch.isfinite(dH.t.float()).all()


@pytest.mark.parametrize("N,D,V,K,chunk", [
    (300, 136, 1000, 16, 128),        # everything ragged, short last chunk
    (2 * 4096 + 300, 72, 1800, 1, 1536),  # three forward chunks, K = 1
    (140, 264, 3000, 256, 0),         # K = 256, two hidden tiles of 144
    (513, 8, 257, 5, 256),            # D = 8 (one k-block), V one past a tile
])
def test_head_writes_stay_inside_their_buffers(N, D, V, K, chunk):
    p = make_problem(N, D, V, K, 1.3, seed=51, mask="frac", mask_frac=0.1, garbage_masked=True,
                     device=DEV)
    _fwd_bwd(p, chunk)
    _fwd_bwd(p, chunk, accumulate=True)


def test_shards_write_inside_their_buffers():
    p = make_problem(300, 136, 1000, 16, 1.1, seed=52, mask="frac", mask_frac=0.1, garbage_masked=True,
                     device=DEV)
    N, D, V, K = p.N, p.D, p.V, p.K
    for a, b in ((0, 333), (333, 334), (334, 1000)):
        ws = Guarded((binding.kd_topk_kl_shard_workspace_size(N, D, b - a, K, 128),), torch.uint8)
        parts, ent = Guarded((N, 2), torch.float32), Guarded((N,), torch.float32)
        nv = Guarded((1,), torch.int64)
        binding.kd_topk_kl_fwd_shard(p.H, p.W[a:b], a, V, p.idx, p.t, p.mask, p.T, parts.t, ent.t, nv.t,
                                     ws.t)
        loss, lse = Guarded((N,), torch.float32), Guarded((N,), torch.float32)
        binding.kd_topk_kl_shard_merge(parts.t.view(1, N, 2), ent.t, p.mask, p.T, loss.t, lse.t)
        dloss = Guarded((N,), torch.float32)
        s = Guarded((1,), torch.float64)
        binding.kd_topk_kl_mean_grad(loss.t, p.mask, nv.t, dloss.t, s.t)
        dH = Guarded((N, D), torch.float32, fill=0.0)
        dW = Guarded((b - a, D), torch.float32, fill=0.0)
        binding.kd_topk_kl_bwd_shard(p.H, p.W[a:b], a, V, p.idx, p.t, p.mask, lse.t, dloss.t, p.T, 128,
                                     False, True, dH.t, dW.t, ws.t)
        for name, buf in (("ws", ws), ("parts", parts), ("ent", ent), ("n_valid", nv), ("loss", loss),
                          ("lse", lse), ("dloss", dloss), ("loss_sum", s), ("dH", dH), ("dW", dW)):
            buf.check(f"shard [{a}, {b}) {name}")
    assert binding.kd_get_status() == 0


@pytest.mark.parametrize("N,V,K,grad", [(300, 1000, 16, True), (77, 4104, 256, True), (129, 520, 1, False)])
def test_logits_writes_stay_inside_their_buffers(N, V, K, grad):
    p = make_problem(N, 8, V, K, 0.9, seed=53, mask="frac", mask_frac=0.1, garbage_masked=True, device=DEV)
    Z = (3.0 * torch.randn(N, V, device=DEV)).to(torch.bfloat16)
    Zc = Z.clone()
    ws = Guarded((binding.kd_topk_kl_logits_workspace_size(N, K),), torch.uint8)
    loss, lse = Guarded((N,), torch.float32), Guarded((N,), torch.float32)
    nv = Guarded((1,), torch.int64)
    dZ = Guarded((N, V), torch.bfloat16) if grad else None
    g = mean_upstream_grad(p.mask).to(DEV) if grad else None
    binding.kd_topk_kl_logits(Z, p.idx, p.t, p.mask, p.T, loss.t, lse.t, nv.t, ws.t, dloss=g,
                              dZ=dZ.t if grad else None)
    for name, buf in (("ws", ws), ("loss", loss), ("lse", lse), ("n_valid", nv)) + ((("dZ", dZ),) if grad else ()):
        buf.check(name)
    assert torch.equal(Z.view(torch.uint8), Zc.view(torch.uint8)), "logits written"
    assert binding.kd_get_status() == 0


@pytest.mark.parametrize("N,D,V,K", [(300, 136, 1000, 16), (70, 64, 5000, 256), (4100, 72, 520, 1),
                                     (301, 72, 20001 * 8 // 8, 100)])
def test_teacher_topk_writes_stay_inside_their_buffers(N, D, V, K):
    p = make_problem(N, D, V, 1, 1.0, seed=54, device=DEV)
    ws = Guarded((binding.kd_teacher_topk_workspace_size(N, D, V, K),), torch.uint8)
    ids = Guarded((N, K), torch.int32)
    vals = Guarded((N, K), torch.float32)
    binding.kd_teacher_topk(p.H, p.W, ids.t, vals.t, ws.t)
    for name, buf in (("ws", ws), ("ids", ids), ("logits", vals)):
        buf.check(name)
    assert binding.kd_get_status() == 0
    assert int(ids.t.min()) >= 0 and int(ids.t.max()) < V
