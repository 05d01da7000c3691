"""The fused top-K KL head on several GPUs, one process per GPU.

The pages leave multi-GPU communication as the method's open question (news
article "Offline Top-K Distillation Removes the Need for a Resident Teacher
Model...", closing caveats: whether communication replaces GPU memory as the
bottleneck). Two splits of the same computation, each exact:

* ``TokenShardedHead`` (data parallelism). Every rank holds a slice of the
  batch's tokens and the whole W. The per-row loss, lse and dH stay local; the
  mean needs the global count of counted rows, and dW is a sum over tokens.
  Exchange per step: an all-reduce of n_valid (8 bytes) before the backward,
  and of dW (V x D fp32) and the loss sum (8 bytes) after it.
* ``VocabShardedHead``. Every rank holds all tokens and a slice of W's rows
  (as a tensor-parallel output head does). Each per-row quantity is a sum or
  a logsumexp over vocabulary columns, so each rank computes its shard's
  (lse, cross term) per row, the ranks all-gather them (8 bytes a row per
  rank) and merge them in shard order, identically on every rank; the
  backward takes the merged lse, each rank keeps its rows of dW, and dH (a sum
  over shards) is all-reduced (N x D fp32).

Collectives are torch.distributed calls on the given process group (NCCL
between GPUs). Every step of the loss itself runs in the library's kernels
through ``ops``, the ctypes binding; nothing here does arithmetic on the data.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch
import torch.distributed as dist

from . import binding as _binding

__all__ = ["token_range", "vocab_range", "group_size_rank", "TokenShardedHead", "VocabShardedHead",
           "mean_loss"]


def token_range(N: int, rank: int, world: int) -> Tuple[int, int]:
    """Rows [lo, hi) of an N-token batch that `rank` of `world` holds (contiguous, balanced)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of world {world}")
    return N * rank // world, N * (rank + 1) // world


def vocab_range(V: int, rank: int, world: int, align: int = 256) -> Tuple[int, int]:
    """Vocabulary ids [v0, v1) of `rank`'s shard: boundaries on multiples of `align`
    (the GEMM's 256-wide vocabulary tile, so only the last shard has a ragged tile),
    as even as that allows. Every shard is non-empty when world <= ceil(V / align)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of world {world}")
    tiles = -(-V // align)
    if world > tiles:
        raise ValueError(f"{world} shards of a {V}-token vocabulary in {align}-wide tiles")
    t0, t1 = tiles * rank // world, tiles * (rank + 1) // world
    return min(V, t0 * align), min(V, t1 * align)


def group_size_rank(group=None) -> Tuple[int, int]:
    """(world size, rank) of the process group; (1, 0) without torch.distributed."""
    if dist.is_available() and dist.is_initialized():
        return dist.get_world_size(group), dist.get_rank(group)
    return 1, 0


class TokenShardedHead:
    """One rank's part of a token-sharded (data-parallel) step.

    Holds the rank's outputs and workspace for N_local tokens. ``step`` runs
    forward, mean gradient and backward of the GLOBAL mean loss over all
    ranks' counted rows: after it, ``dH`` holds this rank's rows of dH (bf16)
    and ``dW`` the full dW summed over ranks (fp32); ``loss_sum`` / ``n_valid``
    are the global sum and count (device tensors, mean = loss_sum / n_valid).
    """

    def __init__(self, N_local: int, D: int, V: int, K: int, T: float, device,
                 chunk_tokens: int = 0, group=None, ops=None):
        self.ops = ops if ops is not None else _binding
        self.group = group
        self.world, self.rank = group_size_rank(group)
        self.T = float(T)
        self.chunk = int(chunk_tokens)
        dev = torch.device(device)
        self.ws = torch.empty(max(self.ops.kd_topk_kl_workspace_size(N_local, D, V, K, chunk_tokens), 256),
                              dtype=torch.uint8, device=dev)
        self.loss = torch.empty(N_local, dtype=torch.float32, device=dev)
        self.lse = torch.empty(N_local, dtype=torch.float32, device=dev)
        self.n_valid = torch.zeros(1, dtype=torch.int64, device=dev)
        self.dloss = torch.empty(N_local, dtype=torch.float32, device=dev)
        self.loss_sum = torch.zeros(1, dtype=torch.float64, device=dev)
        self.dH = torch.empty(N_local, D, dtype=torch.bfloat16, device=dev)
        self.dW = torch.empty(V, D, dtype=torch.float32, device=dev)

    def step(self, H, W, idx, t, mask):
        ops = self.ops
        ops.kd_topk_kl_fwd(H, W, idx, t, mask, self.T, self.loss, self.lse, self.n_valid, self.ws)
        if self.world > 1:
            dist.all_reduce(self.n_valid, group=self.group)   # global count of counted rows
        ops.kd_topk_kl_mean_grad(self.loss, mask, self.n_valid, self.dloss, self.loss_sum)
        ops.kd_topk_kl_bwd(H, W, idx, t, mask, self.lse, self.dloss, self.T, self.chunk, False,
                           self.dH, self.dW, self.ws)
        if self.world > 1:
            dist.all_reduce(self.dW, group=self.group)        # dW is a sum over all tokens
            dist.all_reduce(self.loss_sum, group=self.group)
        return self.loss_sum, self.n_valid


class VocabShardedHead:
    """One rank's vocabulary shard of a step over all N tokens.

    The rank holds rows [v0, v1) of W (``vocab_range``). After ``step``: ``loss``
    and ``lse`` are the whole vocabulary's (the same bits on every rank), ``dH``
    the full dH (fp32, all-reduced over shards), ``dW_shard`` this shard's rows
    of dW (fp32), ``loss_sum`` / ``n_valid`` the sum and count of the mean.
    """

    def __init__(self, N: int, D: int, V: int, K: int, T: float, device, chunk_tokens: int = 0,
                 group=None, ops=None, align: int = 256):
        self.ops = ops if ops is not None else _binding
        self.group = group
        self.world, self.rank = group_size_rank(group)
        self.V = int(V)
        self.v0, self.v1 = vocab_range(V, self.rank, self.world, align)
        self.T = float(T)
        self.chunk = int(chunk_tokens)
        dev = torch.device(device)
        Vs = self.v1 - self.v0
        self.ws = torch.empty(max(self.ops.kd_topk_kl_shard_workspace_size(N, D, Vs, K, chunk_tokens), 256),
                              dtype=torch.uint8, device=dev)
        self.local = torch.empty(N, 2, dtype=torch.float32, device=dev)                # this shard's
        self.parts = (torch.empty(self.world * N, 2, dtype=torch.float32, device=dev)  # [R x N, 2]
                      if self.world > 1 else self.local)
        self.ent = torch.empty(N, dtype=torch.float32, device=dev)
        self.n_valid = torch.zeros(1, dtype=torch.int64, device=dev)
        self.loss = torch.empty(N, dtype=torch.float32, device=dev)
        self.lse = torch.empty(N, dtype=torch.float32, device=dev)
        self.dloss = torch.empty(N, dtype=torch.float32, device=dev)
        self.loss_sum = torch.zeros(1, dtype=torch.float64, device=dev)
        self.dH = torch.empty(N, D, dtype=torch.float32, device=dev)
        self.dW_shard = torch.empty(Vs, D, dtype=torch.float32, device=dev)
        self.N = N

    def step(self, H, W_shard, idx, t, mask):
        ops, N = self.ops, self.N
        ops.kd_topk_kl_fwd_shard(H, W_shard, self.v0, self.V, idx, t, mask, self.T, self.local,
                                 self.ent, self.n_valid, self.ws)
        if self.world > 1:
            dist.all_gather_into_tensor(self.parts, self.local, group=self.group)
        ops.kd_topk_kl_shard_merge(self.parts.view(self.world, N, 2), self.ent, mask, self.T,
                                   self.loss, self.lse)
        # every rank holds all rows: its own count is the global one
        ops.kd_topk_kl_mean_grad(self.loss, mask, self.n_valid, self.dloss, self.loss_sum)
        ops.kd_topk_kl_bwd_shard(H, W_shard, self.v0, self.V, idx, t, mask, self.lse, self.dloss,
                                 self.T, self.chunk, False, False, self.dH, self.dW_shard, self.ws)
        if self.world > 1:
            dist.all_reduce(self.dH, group=self.group)        # dH is a sum over the shards
        return self.loss_sum, self.n_valid


def mean_loss(loss_sum: torch.Tensor, n_valid: torch.Tensor) -> float:
    """The mean loss from the device sum and count (one host read; 0 with no counted rows)."""
    nv = int(n_valid.item())
    return float(loss_sum.item()) / nv if nv > 0 else 0.0
