"""A stand-in for the library's compute calls, backed by the CPU oracle.

Test infrastructure: it lets the multi-process tests run the product's
multi-GPU orchestration (``top_kl_loss_lm_b300.sharded``: shard ranges, the
collectives and their order) on CPU ranks with gloo, where the CUDA kernels
cannot run. Each function has the binding's signature and fills the given
output tensors from ``oracle`` (fp64), so the orchestration's results can be
compared with the unsharded oracle. The kernels themselves are checked against
the oracle on the GPU (tests/test_gpu_shards.py).
"""
import numpy as np
import torch

import oracle


def _np(x):
    return None if x is None else x.detach().to(torch.float64).numpy()


def _put(dst, value):
    dst.copy_(torch.as_tensor(np.asarray(value)).to(dst.dtype).reshape(dst.shape))


def _full_W(W_shard, v0, V):
    Ws = _np(W_shard)
    W = np.zeros((V, Ws.shape[1]))
    W[v0:v0 + Ws.shape[0]] = Ws
    return W


def kd_topk_kl_workspace_size(N, D, V, K, chunk_tokens=0):
    return 256


kd_topk_kl_shard_workspace_size = kd_topk_kl_workspace_size


def kd_topk_kl_fwd(H, W, idx, t, mask, T, loss, lse, n_valid, ws, stream=None):
    l, s, nv = oracle.kd_forward(_np(H), _np(W), idx.numpy(), _np(t), mask.numpy(), T)
    _put(loss, l)
    _put(lse, s)
    _put(n_valid, [nv])


def kd_topk_kl_mean_grad(loss, mask, n_valid, dloss=None, loss_sum=None, stream=None):
    nv = int(n_valid.item())
    if dloss is not None:
        _put(dloss, mask.numpy().astype(np.float64) / nv if nv > 0 else np.zeros(mask.shape[0]))
    if loss_sum is not None:
        _put(loss_sum, [float(np.sum(_np(loss)))])


def kd_topk_kl_bwd(H, W, idx, t, mask, lse, dloss, T, chunk_tokens, accumulate_dW, dH, dW, ws,
                   stream=None):
    gH, gW = oracle.kd_backward(_np(H), _np(W), idx.numpy(), _np(t), mask.numpy(), T, _np(dloss))
    _put(dH, gH)
    _put(dW, gW + (_np(dW) if accumulate_dW else 0.0))


def kd_topk_kl_fwd_shard(H, W_shard, v0, V, idx, t, mask, T, parts, ent, n_valid, ws, stream=None):
    v1 = v0 + W_shard.shape[0]
    lse_s, x_s, e = oracle.kd_forward_shard(_np(H), _full_W(W_shard, v0, V), idx.numpy(), _np(t),
                                            mask.numpy(), T, v0, v1)
    _put(parts, np.stack([lse_s, x_s], axis=1))
    _put(ent, e)
    _put(n_valid, [int(mask.numpy().astype(bool).sum())])


def kd_topk_kl_shard_merge(parts, ent, mask, T, loss, lse, stream=None):
    p = _np(parts)
    m = p[:, :, 0].max(axis=0)
    s = m + np.log(np.sum(np.exp(p[:, :, 0] - m), axis=0))
    x = np.sum(p[:, :, 1], axis=0)
    _put(lse, s)
    _put(loss, np.where(mask.numpy().astype(bool), _np(ent) - x / T + s, 0.0))


def kd_topk_kl_bwd_shard(H, W_shard, v0, V, idx, t, mask, lse, dloss, T, chunk_tokens,
                         accumulate_dW, accumulate_dH, dH, dW_shard, ws, stream=None):
    v1 = v0 + W_shard.shape[0]
    gH, gW = oracle.kd_backward_shard(_np(H), _full_W(W_shard, v0, V), idx.numpy(), _np(t),
                                      mask.numpy(), T, _np(dloss), _np(lse), v0, v1)
    _put(dH, gH + (_np(dH) if accumulate_dH else 0.0))
    _put(dW_shard, gW + (_np(dW_shard) if accumulate_dW else 0.0))
