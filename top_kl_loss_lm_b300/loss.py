"""torch.autograd wrapper around the C ABI (allocation and marshalling only).

``fused_topk_kl(H, W, topk_idx, topk_logit, mask, T)`` returns the per-row
loss (zero at masked rows) and the number of counted rows; the mean loss is
``loss.sum() / n_valid``. Backward calls ``kd_topk_kl_bwd`` with the incoming
per-row gradient. The workspace is allocated here, with torch, once per call.
"""
from __future__ import annotations

import torch

from . import binding


class FusedTopKKL(torch.autograd.Function):
    @staticmethod
    def forward(ctx, H, W, topk_idx, topk_logit, mask, T: float, chunk_tokens: int = 0):
        N, D = H.shape
        V = W.shape[0]
        K = topk_idx.shape[1]
        dev = H.device
        ws = torch.empty(binding.kd_topk_kl_workspace_size(N, D, V, K, chunk_tokens),
                         dtype=torch.uint8, device=dev)
        loss = torch.empty(N, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
        n_valid = torch.empty(1, dtype=torch.int64, device=dev)
        binding.kd_topk_kl_fwd(H, W, topk_idx, topk_logit, mask, T, loss, lse, n_valid, ws)
        ctx.save_for_backward(H, W, topk_idx, topk_logit, mask, lse)
        ctx.T = float(T)
        ctx.chunk_tokens = int(chunk_tokens)
        ctx.ws = ws
        ctx.mark_non_differentiable(lse, n_valid)
        return loss, lse, n_valid

    @staticmethod
    def backward(ctx, dloss, _dlse, _dnv):
        H, W, topk_idx, topk_logit, mask, lse = ctx.saved_tensors
        dH = torch.empty_like(H)
        dW = torch.empty(W.shape, dtype=torch.float32, device=W.device)
        binding.kd_topk_kl_bwd(H, W, topk_idx, topk_logit, mask, lse,
                               dloss.to(torch.float32).contiguous(), ctx.T, ctx.chunk_tokens, False,
                               dH, dW, ctx.ws)
        return dH, dW, None, None, None, None, None


def fused_topk_kl(H, W, topk_idx, topk_logit, mask=None, T: float = 1.0, chunk_tokens: int = 0):
    """Per-row top-K KL loss with the fused kernels; returns (loss[N], n_valid[1])."""
    loss, _lse, n_valid = FusedTopKKL.apply(H, W, topk_idx, topk_logit, mask, T, chunk_tokens)
    return loss, n_valid
