"""Parity of kd_topk_kl_logits (loss and logit gradient from materialised logits)
with the CPU fp64 oracle's kd_from_logits, through the C ABI.

Small cases compare every element; every cluster size (one row split over 1,
2, 4 or 8 CTAs), with one or two CTAs per SM, is exercised by a vocabulary
size that needs it; the full-size case (N = 32,768
rows of the 201,088-token head) is checked on sampled rows plus the property
that every counted row of dZ sums to zero.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import _parity as P
from top_kl_loss_lm_b300 import binding
from workloads import make_problem, mean_upstream_grad

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _logits_problem(N, V, K, T, seed, scale=4.0, **kw):
    p = make_problem(N, 8, V, K, T, seed=seed, device=DEV, **kw)
    g = torch.Generator(device=DEV).manual_seed(seed + 101)
    Z = (torch.randn(N, V, device=DEV, generator=g) * scale).to(torch.bfloat16)
    return p, Z


def _run(p, Z, grad=True, in_place=False):
    N, V, K = Z.shape[0], Z.shape[1], p.K
    ws = torch.empty(binding.kd_topk_kl_logits_workspace_size(N, K), dtype=torch.uint8, device=DEV)
    loss = torch.full((N,), float("nan"), device=DEV)
    lse = torch.full((N,), float("nan"), device=DEV)
    nv = torch.full((1,), -1, dtype=torch.int64, device=DEV)
    g = mean_upstream_grad(p.mask).to(DEV) if grad else None
    Zin = Z.clone() if in_place else Z
    dZ = None
    if grad:
        dZ = Zin if in_place else torch.full_like(Z, float("nan"))
    binding.kd_topk_kl_logits(Zin, p.idx, p.t, p.mask, p.T, loss, lse, nv, ws, dloss=g, dZ=dZ)
    torch.cuda.synchronize()
    return dict(loss=loss, lse=lse, n_valid=nv, dZ=dZ, g=g, status=binding.kd_get_status())


def _compare(p, Z, out, rows=None):
    Zc = Z.double().cpu().numpy()
    idx, t, m = p.idx.cpu().numpy(), p.t.double().cpu().numpy(), p.mask.cpu().numpy()
    g = out["g"].double().cpu().numpy() if out["g"] is not None else None
    if rows is not None:
        Zc, idx, t, m = Zc[rows], idx[rows], t[rows], m[rows]
        g = g[rows] if g is not None else None
    loss, lse, nv, dZ = oracle.kd_from_logits(Zc, idx, t, m, p.T, g)
    sel = slice(None) if rows is None else rows
    assert out["status"] == 0, binding.STATUS.get(out["status"])
    if rows is None:
        assert int(out["n_valid"].item()) == nv
    P.assert_rows_close(out["loss"].cpu().numpy()[sel], loss, "loss")
    P.assert_lse_close(out["lse"].cpu().numpy()[sel], lse, "lse")
    if dZ is not None:
        P.assert_grad_close(out["dZ"].double().cpu().numpy()[sel], dZ, "dZ")


def test_small_every_element():
    p, Z = _logits_problem(300, 1000, 16, 1.3, seed=1, mask="frac", mask_frac=0.1,
                           garbage_masked=True)
    _compare(p, Z, _run(p, Z))


# (V, cluster size x CTAs per SM the library picks for it, rows: ~8+ per cluster)
@pytest.mark.parametrize("V,shape,N", [(4096, "1x2", 2400), (40000, "2x2", 1200),
                                       (100000, "4x2", 600), (201088, "8x2", 300),
                                       (300000, "8x1", 200), (400000, "8x1", 150)])
def test_cluster_sizes(V, shape, N):
    # one row is split over a cluster of CTAs whose slices meet through distributed
    # shared memory; more rows than clusters, so every ring buffer is reused
    p, Z = _logits_problem(N, V, 64, 1.0, seed=V % 97, mask="frac", mask_frac=0.05)
    _compare(p, Z, _run(p, Z))


def test_gradient_in_place_and_loss_only():
    p, Z = _logits_problem(257, 2056, 32, 0.8, seed=7, mask="frac", mask_frac=0.05)
    ref = _run(p, Z)
    inplace = _run(p, Z, in_place=True)
    assert torch.equal(ref["dZ"], inplace["dZ"])
    only = _run(p, Z, grad=False)  # a different kernel shape: same values up to fp32 order
    assert only["status"] == 0
    assert torch.allclose(only["loss"], ref["loss"], rtol=1e-5, atol=1e-6)
    assert torch.allclose(only["lse"], ref["lse"], rtol=1e-6, atol=1e-6)
    _compare(p, Z, ref)
    _compare(p, Z, only)


def test_k_extremes_duplicates_and_empty():
    p, Z = _logits_problem(130, 800, 1, 1.0, seed=8)
    _compare(p, Z, _run(p, Z))
    p, Z = _logits_problem(70, 3000, 256, 2.0, seed=9, mask="frac", mask_frac=0.1)
    _compare(p, Z, _run(p, Z))
    p, Z = _logits_problem(96, 512, 8, 1.3, seed=10)
    p.idx[::3, 1] = p.idx[::3, 0]
    _compare(p, Z, _run(p, Z))
    p, Z = _logits_problem(50, 640, 8, 1.0, seed=11)
    p.mask.zero_()
    p.t.fill_(float("nan"))
    out = _run(p, Z)
    assert out["status"] == 0 and int(out["n_valid"].item()) == 0
    assert torch.all(out["loss"] == 0) and torch.all(out["dZ"].float() == 0)


def test_strided_rows_and_argument_errors():
    p, Zbig = _logits_problem(64, 1032, 16, 1.0, seed=12)
    Z = Zbig[:, :1024]  # rows 1,032 apart
    p.idx.clamp_(max=1023)
    out = _run(p, Z)
    _compare(p, Z, out)
    with pytest.raises(binding.KdError):  # V not a multiple of 8
        _run(p, Zbig[:, :1020])


@pytest.mark.parametrize("V", [4096, 201088])
def test_loss_only_shapes(V):
    # without the gradient the library runs lighter CTAs, four per SM, one row buffer
    p, Z = _logits_problem(700, V, 256, 1.3, seed=17, mask="frac", mask_frac=0.05)
    _compare(p, Z, _run(p, Z, grad=False))


@pytest.mark.slow
def test_full_size_sampled_rows():
    N, V, K = 32768, 201088, 64
    p, Z = _logits_problem(N, V, K, 1.0, seed=13, scale=3.0, mask="frac", mask_frac=0.02)
    out = _run(p, Z)
    assert out["status"] == 0
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.choice(N, 48, replace=False), [0, N - 1]]))
    _compare(p, Z, out, rows=rows)
    # every counted row of dZ sums to zero (softmax minus a normalised teacher)
    s = out["dZ"].float().sum(dim=1)
    scale = out["dZ"].float().abs().sum(dim=1).clamp_min(1e-30)
    assert torch.all((s.abs() / scale) < 2e-2)
    assert int(out["n_valid"].item()) == int(p.mask.sum().item())
