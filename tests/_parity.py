"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI,
run the CPU fp64 oracle on the same inputs, and compare with the tolerances
the loss is specified to (bf16 operands, fp32 accumulation):

  per-row loss:  |gpu - ref| <= 1e-3 |ref| where |ref| >= 0.1, and <= 1e-4 nats
                 where |ref| < 0.1 (a relative bound means nothing at a loss of 0;
                 masked rows and rows whose teacher matches the student are there)
  lse:           |gpu - ref| <= 1e-5 max(|ref|, 1): fp32 accumulation of the
                 logits and of the sum of exponentials, nothing looser
  mean loss:     relative 1e-3
  dH, dW:        max|gpu - ref| / max|ref| <= 2e-2 and
                 ||gpu - ref||_F / ||ref||_F <= 5e-3
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from top_kl_loss_lm_b300 import binding
from workloads import Problem, mean_upstream_grad

LOSS_RTOL = 1e-3
LOSS_FLOOR_BELOW = 0.1   # |ref| under this gets the absolute bound instead
LOSS_ATOL = 1e-4
LSE_RTOL = 1e-5
GRAD_MAXREL = 2e-2
GRAD_NORMREL = 5e-3


def run_gpu(p: Problem, chunk_tokens: int = 0, g: torch.Tensor = None, accumulate: bool = False,
            dW_init: torch.Tensor = None, backward: bool = True):
    dev = p.H.device
    N, D, V, K = p.N, p.D, p.V, p.K
    ws = torch.empty(max(binding.kd_topk_kl_workspace_size(N, D, V, K, chunk_tokens), 256),
                     dtype=torch.uint8, device=dev)
    loss = torch.full((N,), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((N,), float("nan"), dtype=torch.float32, device=dev)
    nv = torch.full((1,), -1, dtype=torch.int64, device=dev)
    binding.kd_topk_kl_fwd(p.H, p.W, p.idx, p.t, p.mask, p.T, loss, lse, nv, ws)
    out = dict(loss=loss, lse=lse, n_valid=nv)
    if backward:
        if g is None:
            g = mean_upstream_grad(p.mask).to(dev)
        dH = torch.full_like(p.H, float("nan"))
        dW = dW_init.clone() if dW_init is not None else torch.full((V, D), float("nan"),
                                                                     dtype=torch.float32, device=dev)
        binding.kd_topk_kl_bwd(p.H, p.W, p.idx, p.t, p.mask, lse, g, p.T, chunk_tokens, accumulate,
                               dH, dW, ws)
        out.update(dH=dH, dW=dW, g=g)
    torch.cuda.synchronize()
    out["status"] = binding.kd_get_status()
    return out


def host(p: Problem):
    return dict(H=p.H.double().cpu().numpy(), W=p.W.double().cpu().numpy(),
                idx=p.idx.cpu().numpy(), t=p.t.double().cpu().numpy(), mask=p.mask.cpu().numpy())


def run_oracle(p: Problem, g: np.ndarray = None, rows=None, backward=True):
    """Oracle on all rows, or on the listed rows only (row-local outputs)."""
    h = host(p)
    if rows is not None:
        rows = np.asarray(rows)
        sub = {k: (v[rows] if k != "W" else v) for k, v in h.items()}
    else:
        sub = h
    loss, lse, nv = oracle.kd_forward(sub["H"], sub["W"], sub["idx"], sub["t"], sub["mask"], p.T)
    out = dict(loss=loss, lse=lse, n_valid=nv)
    if backward:
        gg = g if rows is None else g[rows]
        dH, dW = oracle.kd_backward(sub["H"], sub["W"], sub["idx"], sub["t"], sub["mask"], p.T, gg)
        out.update(dH=dH, dW=dW)
    return out


def assert_rows_close(got, ref, name):
    """Per-row loss bound; returns how many rows were judged by the absolute floor."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    small = np.abs(ref) < LOSS_FLOOR_BELOW
    bound = np.where(small, LOSS_ATOL, LOSS_RTOL * np.abs(ref))
    bad = np.nonzero(~(err <= bound))[0]
    assert bad.size == 0, (f"{name}: {bad.size} rows off, worst {err.max():.3e} at {int(np.argmax(err))} "
                           f"({int(small.sum())} of {ref.size} rows under the absolute floor)")
    return int(small.sum())


def assert_lse_close(got, ref, name="lse"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    rel = err / np.maximum(np.abs(ref), 1.0)
    bad = np.nonzero(~(rel <= LSE_RTOL))[0]
    assert bad.size == 0, f"{name}: {bad.size} rows off, worst relative {rel.max():.3e}"


def assert_grad_close(got, ref, name):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    scale = np.max(np.abs(ref))
    if scale == 0.0:
        assert np.max(np.abs(got)) == 0.0, f"{name}: expected all zeros"
        return
    maxrel = np.max(np.abs(got - ref)) / scale
    normrel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert maxrel <= GRAD_MAXREL and normrel <= GRAD_NORMREL, \
        f"{name}: max-abs-rel {maxrel:.3e}, normwise {normrel:.3e}"


def compare_full(p: Problem, gpu: dict, backward=True):
    g = gpu["g"].double().cpu().numpy() if backward else None
    ref = run_oracle(p, g, backward=backward)
    assert gpu["status"] == 0, binding.STATUS.get(gpu["status"])
    assert int(gpu["n_valid"].item()) == ref["n_valid"]
    assert_rows_close(gpu["loss"].cpu().numpy(), ref["loss"], "loss")
    assert_lse_close(gpu["lse"].cpu().numpy(), ref["lse"], "lse")
    nv = ref["n_valid"]
    gm = float(gpu["loss"].double().sum().item()) / nv if nv else 0.0
    rm = oracle.mean_loss(ref["loss"], nv)
    assert abs(gm - rm) <= LOSS_RTOL * abs(rm) + 1e-7, (gm, rm)
    if backward:
        assert_grad_close(gpu["dH"].double().cpu().numpy(), ref["dH"], "dH")
        assert_grad_close(gpu["dW"].double().cpu().numpy(), ref["dW"], "dW")
    return ref
