"""The checked build (libkdtopk_checked.so, -DKD_CHECKED) at ragged shapes.

It stands in for a memory sanitizer, which cannot run on these GPUs: every
bulk-tensor copy checks its coordinates first, the selection kernels their
shared-memory slots, and a failed check records KD_ERR_BOUNDS and skips the
access. Each call here runs through both builds on the same inputs; the
checked build must report no failed check and give the same bits.
"""
import importlib.util
import os

import pytest
import torch

from top_kl_loss_lm_b300 import binding
from top_kl_loss_lm_b300.build import LIB_CHECKED, build_library
from workloads import make_problem, mean_upstream_grad

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def checked():
    build_library(checked=True)
    spec = importlib.util.spec_from_file_location("binding_checked", binding.__file__)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.library_path = lambda: LIB_CHECKED
    assert os.path.exists(LIB_CHECKED)
    return mod


def _head(b, p, chunk):
    N, D, V, K = p.N, p.D, p.V, p.K
    ws = torch.empty(b.kd_topk_kl_workspace_size(N, D, V, K, chunk), dtype=torch.uint8, device=DEV)
    loss, lse = torch.empty(N, device=DEV), torch.empty(N, device=DEV)
    nv = torch.empty(1, dtype=torch.int64, device=DEV)
    b.kd_topk_kl_fwd(p.H, p.W, p.idx, p.t, p.mask, p.T, loss, lse, nv, ws)
    g = torch.empty(N, device=DEV)
    s = torch.empty(1, dtype=torch.float64, device=DEV)
    b.kd_topk_kl_mean_grad(loss, p.mask, nv, g, s)
    dH = torch.empty_like(p.H)
    dW = torch.empty(V, D, device=DEV)
    b.kd_topk_kl_bwd(p.H, p.W, p.idx, p.t, p.mask, lse, g, p.T, chunk, False, dH, dW, ws)
    torch.cuda.synchronize()
    return b.kd_get_status(), [loss, lse, nv, g, s, dH.view(torch.int16), dW]


@pytest.mark.parametrize("N,D,V,K,chunk", [(300, 136, 1000, 16, 128), (2 * 4096 + 300, 72, 1800, 1, 1536),
                                           (140, 264, 3000, 256, 0), (513, 8, 257, 5, 256)])
def test_head_passes_every_check(checked, N, D, V, K, chunk):
    p = make_problem(N, D, V, K, 1.3, seed=61, mask="frac", mask_frac=0.1, garbage_masked=True,
                     device=DEV)
    st_c, out_c = _head(checked, p, chunk)
    st_n, out_n = _head(binding, p, chunk)
    assert st_c == 0, binding.STATUS.get(st_c)
    assert st_n == 0
    for a, b in zip(out_c, out_n):
        assert torch.equal(a, b)


def test_shards_logits_and_teacher_pass_every_check(checked):
    p = make_problem(300, 136, 1000, 16, 1.1, seed=62, mask="frac", mask_frac=0.1, garbage_masked=True,
                     device=DEV)
    N, D, V, K = p.N, p.D, p.V, p.K
    outs = []
    for b in (checked, binding):
        got = []
        for a, e in ((0, 333), (333, 334), (334, 1000)):
            ws = torch.empty(b.kd_topk_kl_shard_workspace_size(N, D, e - a, K, 128), dtype=torch.uint8,
                             device=DEV)
            parts, ent = torch.empty(N, 2, device=DEV), torch.empty(N, device=DEV)
            nv = torch.empty(1, dtype=torch.int64, device=DEV)
            b.kd_topk_kl_fwd_shard(p.H, p.W[a:e], a, V, p.idx, p.t, p.mask, p.T, parts, ent, nv, ws)
            dH = torch.zeros(N, D, device=DEV)
            dW = torch.empty(e - a, D, device=DEV)
            lse = torch.full((N,), 7.0, device=DEV)
            g = mean_upstream_grad(p.mask).to(DEV)
            b.kd_topk_kl_bwd_shard(p.H, p.W[a:e], a, V, p.idx, p.t, p.mask, lse, g, p.T, 128, False, False,
                                   dH, dW, ws)
            got += [parts, ent, dH, dW]
        Z = (3.0 * torch.randn(77, 4104, device=DEV, generator=torch.Generator(device=DEV).manual_seed(5))
             ).to(torch.bfloat16)
        q = make_problem(77, 8, 4104, 256, 0.9, seed=63, mask="frac", mask_frac=0.1, device=DEV)
        ws = torch.empty(b.kd_topk_kl_logits_workspace_size(77, 256), dtype=torch.uint8, device=DEV)
        loss, lse2 = torch.empty(77, device=DEV), torch.empty(77, device=DEV)
        nv = torch.empty(1, dtype=torch.int64, device=DEV)
        dZ = torch.empty_like(Z)
        b.kd_topk_kl_logits(Z, q.idx, q.t, q.mask, q.T, loss, lse2, nv, ws,
                            dloss=mean_upstream_grad(q.mask).to(DEV), dZ=dZ)
        got += [loss, lse2, dZ.view(torch.int16)]
        for (n, d, v, k) in ((300, 136, 1000, 16), (301, 72, 20001, 100)):
            r = make_problem(n, d, v, 1, 1.0, seed=64, device=DEV)
            ws = torch.empty(b.kd_teacher_topk_workspace_size(n, d, v, k), dtype=torch.uint8, device=DEV)
            ids = torch.empty(n, k, dtype=torch.int32, device=DEV)
            vals = torch.empty(n, k, device=DEV)
            b.kd_teacher_topk(r.H, r.W, ids, vals, ws)
            got += [ids, vals]
        torch.cuda.synchronize()
        assert b.kd_get_status() == 0
        outs.append(got)
    for a, b2 in zip(*outs):
        assert torch.equal(a, b2)
