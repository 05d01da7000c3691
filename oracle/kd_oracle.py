"""CPU fp64 oracle for the top-K KL distillation loss on a student output head.

TEST INFRASTRUCTURE ONLY. This module is imported by ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``. The
product (the CUDA library and its Python binding) never imports or calls it,
and it shares no code with that path: it is a plain, slow, obviously correct
restatement of what the method computes, written with numpy in float64.

What it restates (source: "Efficient Knowledge Distillation for LLMs: Offline
Top-K Logits and a Fused Chunked KL Loss" and the blog post "Making Knowledge
Distillation Cheap Enough to Run at Scale"):

* The teacher is known only through its cached top-K (token id, logit) pairs
  per position (blog, "Two systems changes", offline distillation paragraph).
  Its distribution is the softmax of those K logits; every other token has
  probability zero. This is the teacher grid the dense-KL bullet rebuilds
  "from the cached top-100 logits".
* The student distribution is the softmax of the full-vocabulary logits
  Z = H W^T that the output projection produces (blog, fused chunked KL
  bullet: the projection from hidden states to logits is part of the loss).
* The loss per position is KL(teacher || student); the three variants in the
  blog (dense, forward-chunked, fused chunked) are stated to be mathematically
  equivalent, so the plain dense definition is the oracle for all of them.
* The reported loss is the mean over counted (unmasked) positions.

Readings where the pages are silent (each is listed with its reason in the
design notes): both distributions use the same temperature T (student
softmax(Z/T), teacher softmax(t/T)); there is no T^2 factor; ``lse`` is the
natural-log logsumexp of Z/T; a duplicated teacher id is one grid entry
whose probability is the sum of its cached entries (as in the dense teacher
grid); masked rows give zero loss and zero gradient and their teacher entries
are never read; with no counted rows the mean is 0.

Row blocks (``row_chunk``) exist only to bound memory: every row is computed
independently and the same way whatever the block size.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "teacher_log_probs",
    "student_logits",
    "logsumexp_rows",
    "kd_forward",
    "kd_backward",
    "mean_loss",
    "dense_teacher_grid",
    "kd_from_logits",
    "teacher_topk",
    "kd_forward_shard",
    "kd_backward_shard",
]


def logsumexp_rows(a: np.ndarray) -> np.ndarray:
    """Natural-log logsumexp along the last axis, max-shifted (fp64)."""
    m = np.max(a, axis=-1, keepdims=True)
    return (m + np.log(np.sum(np.exp(a - m), axis=-1, keepdims=True)))[..., 0]


def teacher_log_probs(t_rows: np.ndarray, T: float) -> np.ndarray:
    """log p_k = t_k/T - logsumexp_k(t/T) over the K cached logits of each row.

    Teacher distribution over its cached top-K only (blog "Two systems changes",
    dense-KL bullet: the teacher grid comes from the cached top-K logits).
    """
    b = np.asarray(t_rows, dtype=np.float64) / T
    return b - logsumexp_rows(b)[:, None]


def student_logits(H_rows: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Z = H W^T, the student's output-head logits (one row per position)."""
    return np.asarray(H_rows, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T


def dense_teacher_grid(idx_rows: np.ndarray, logp_rows: np.ndarray, V: int) -> np.ndarray:
    """p~[n, j] = sum of p_k over the cached entries k of row n with idx_k = j.

    The dense teacher-probability grid of the dense-KL bullet; zero outside
    the cached ids. Used by the backward for the teacher term of dZ.
    """
    n = idx_rows.shape[0]
    grid = np.zeros((n, V), dtype=np.float64)
    rows = np.repeat(np.arange(n), idx_rows.shape[1])
    np.add.at(grid, (rows, idx_rows.reshape(-1).astype(np.int64)), np.exp(logp_rows).reshape(-1))
    return grid


def _blocks(n: int, row_chunk: int):
    step = max(1, int(row_chunk))
    for r0 in range(0, n, step):
        yield r0, min(n, r0 + step)


def kd_forward(H, W, idx, t, mask, T: float, row_chunk: int = 64):
    """Per-row KL(teacher_topK || student) and logsumexp of Z/T.

    For each row n (fp64, exact bf16 values of H and W):
      a = (H[n] W^T)/T,   lse_n = logsumexp(a),   log q = a - lse_n
      P = dense teacher grid of row n (softmax of t[n]/T placed at idx[n])
      loss_n = sum_{j: P_j > 0} P_j (log P_j - log q_j)      if mask_n
             = 0                                              otherwise
    This is the dense-KL bullet's computation (blog "Two systems changes"),
    the pages' correctness baseline. lse is returned for every row (it does
    not depend on the teacher).
    Returns (loss[N], lse[N], n_valid).
    """
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    idx = np.asarray(idx)
    t = np.asarray(t)
    mask = np.asarray(mask).astype(bool)
    N = H.shape[0]
    loss = np.zeros(N, dtype=np.float64)
    lse = np.zeros(N, dtype=np.float64)
    for r0, r1 in _blocks(N, row_chunk):
        a = student_logits(H[r0:r1], W) / T
        lse[r0:r1] = logsumexp_rows(a)
        valid = np.nonzero(mask[r0:r1])[0]
        if valid.size == 0:
            continue
        logp = teacher_log_probs(t[r0:r1][valid], T)
        P = dense_teacher_grid(idx[r0:r1][valid].astype(np.int64), logp, W.shape[0])
        log_q = a[valid] - lse[r0:r1][valid][:, None]
        pos = P > 0
        terms = np.zeros_like(P)
        terms[pos] = P[pos] * (np.log(P[pos]) - log_q[pos])
        loss[r0 + valid] = np.sum(terms, axis=1)
    return loss, lse, int(mask.sum())


def mean_loss(loss: np.ndarray, n_valid: int) -> float:
    """Mean of the per-row loss over counted rows (0 when nothing is counted)."""
    return float(np.sum(np.asarray(loss, dtype=np.float64)) / n_valid) if n_valid > 0 else 0.0


def kd_backward(H, W, idx, t, mask, T: float, g, row_chunk: int = 64):
    """Gradients of sum_n g_n * loss_n with respect to H and W.

    With q = softmax(Z/T) over the full vocabulary and p~ the dense teacher grid,
      dZ[n, j] = (g_n / T) * (q[n, j] - p~[n, j])   (0 on masked rows)
      dH = dZ W,   dW = dZ^T H
    (blog "Two systems changes", fused chunked bullet: the backward recomputes
    each chunk's logits rather than storing them). Returns (dH[N,D], dW[V,D]).
    """
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    idx = np.asarray(idx)
    t = np.asarray(t)
    mask = np.asarray(mask).astype(bool)
    g = np.asarray(g, dtype=np.float64)
    N, D = H.shape
    V = W.shape[0]
    dH = np.zeros((N, D), dtype=np.float64)
    dW = np.zeros((V, D), dtype=np.float64)
    for r0, r1 in _blocks(N, row_chunk):
        valid = np.nonzero(mask[r0:r1])[0]
        if valid.size == 0:
            continue
        rows = r0 + valid
        a = student_logits(H[rows], W) / T
        q = np.exp(a - logsumexp_rows(a)[:, None])
        ptil = dense_teacher_grid(idx[rows].astype(np.int64), teacher_log_probs(t[rows], T), V)
        dZ = (g[rows] / T)[:, None] * (q - ptil)
        dH[rows] = dZ @ W
        dW += dZ.T @ H[rows]
    return dH, dW


def kd_from_logits(Z, idx, t, mask, T: float, g=None, row_chunk: int = 64):
    """The same loss and its logit gradient, from logits that were already computed.

    The forward-chunked bullet (blog "Two systems changes") keeps the teacher
    sparse and computes the loss one slice of positions at a time from the
    student's logits, which the output layer has produced in full beforehand.
    Per row n of Z (fp64):
      a = Z[n]/T,  lse_n = logsumexp(a),  loss_n = sum_{P_j > 0} P_j (log P_j - (a_j - lse_n))
      dZ[n, j] = (g_n/T) (exp(a_j - lse_n) - p~[n, j])   (0 on masked rows)
    with P / p~ the dense teacher grid of the row, exactly as in kd_forward and
    kd_backward. Returns (loss[N], lse[N], n_valid, dZ[N, V] or None when g is None).
    """
    Z = np.asarray(Z, dtype=np.float64)
    idx = np.asarray(idx)
    t = np.asarray(t)
    mask = np.asarray(mask).astype(bool)
    N, V = Z.shape
    loss = np.zeros(N, dtype=np.float64)
    lse = np.zeros(N, dtype=np.float64)
    dZ = None if g is None else np.zeros((N, V), dtype=np.float64)
    for r0, r1 in _blocks(N, row_chunk):
        a = Z[r0:r1] / T
        lse[r0:r1] = logsumexp_rows(a)
        valid = np.nonzero(mask[r0:r1])[0]
        if valid.size == 0:
            continue
        logp = teacher_log_probs(t[r0:r1][valid], T)
        P = dense_teacher_grid(idx[r0:r1][valid].astype(np.int64), logp, V)
        log_q = a[valid] - lse[r0:r1][valid][:, None]
        pos = P > 0
        terms = np.zeros_like(P)
        terms[pos] = P[pos] * (np.log(P[pos]) - log_q[pos])
        loss[r0 + valid] = np.sum(terms, axis=1)
        if dZ is not None:
            gv = np.asarray(g, dtype=np.float64)[r0 + valid]
            dZ[r0 + valid] = (gv / T)[:, None] * (np.exp(log_q) - P)
    return loss, lse, int(mask.sum()), dZ


def teacher_topk(H, W, K: int, row_chunk: int = 64):
    """The teacher's cached top-K: per row, the K largest logits of H W^T and their ids.

    Offline distillation caches, once per training position, the teacher's K most
    likely tokens and their logits, so the teacher never has to be resident while
    the student trains (blog "Two systems changes", offline-distillation paragraph;
    the pages' cache holds the top 100). Per row n (fp64, exact bf16 inputs):
      z = H[n] W^T;  ids = the K positions of the largest z, in descending order of z
    Ties at the boundary make several id sets correct; this returns the one a
    stable descending sort gives (lower id first among equal logits).
    Returns (ids[N, K] int64, logits[N, K] fp64).
    """
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    N = H.shape[0]
    ids = np.zeros((N, K), dtype=np.int64)
    vals = np.zeros((N, K), dtype=np.float64)
    for r0, r1 in _blocks(N, row_chunk):
        z = student_logits(H[r0:r1], W)
        order = np.argsort(-z, axis=1, kind="stable")[:, :K]
        ids[r0:r1] = order
        vals[r0:r1] = np.take_along_axis(z, order, axis=1)
    return ids, vals


def kd_forward_shard(H, W, idx, t, mask, T: float, v0: int, v1: int, row_chunk: int = 64):
    """The per-row pieces of the loss that a slice [v0, v1) of the vocabulary holds.

    The loss is a sum over vocabulary columns plus a logsumexp over them, so
    it splits over any partition of the vocabulary (the pages leave multi-GPU
    communication open: news article "Offline Top-K Distillation Removes the
    Need for a Resident Teacher Model...", closing caveats). Per row n (fp64,
    W the FULL [V x D] weight, only its rows v0..v1-1 used):
      lse_s[n] = logsumexp_{v0 <= j < v1} (H[n] W[j]^T / T)
      x_s[n]   = sum_{v0 <= j < v1} P[n, j] * (H[n] W[j]^T)     (0 on masked rows)
      ent[n]   = sum_{j: P[n, j] > 0} P[n, j] log P[n, j]      (0 on masked rows)
    with P the dense teacher grid of the whole vocabulary. Over a partition,
    lse = logsumexp_s lse_s and loss = ent - (sum_s x_s) / T + lse.
    Returns (lse_s[N], x_s[N], ent[N]).
    """
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    idx = np.asarray(idx)
    t = np.asarray(t)
    mask = np.asarray(mask).astype(bool)
    N, V = H.shape[0], W.shape[0]
    lse_s = np.zeros(N, dtype=np.float64)
    x_s = np.zeros(N, dtype=np.float64)
    ent = np.zeros(N, dtype=np.float64)
    for r0, r1 in _blocks(N, row_chunk):
        z = student_logits(H[r0:r1], W[v0:v1])
        lse_s[r0:r1] = logsumexp_rows(z / T)
        valid = np.nonzero(mask[r0:r1])[0]
        if valid.size == 0:
            continue
        P = dense_teacher_grid(idx[r0:r1][valid].astype(np.int64),
                               teacher_log_probs(t[r0:r1][valid], T), V)
        x_s[r0 + valid] = np.sum(P[:, v0:v1] * z[valid], axis=1)
        pos = P > 0
        terms = np.zeros_like(P)
        terms[pos] = P[pos] * np.log(P[pos])
        ent[r0 + valid] = np.sum(terms, axis=1)
    return lse_s, x_s, ent


def kd_backward_shard(H, W, idx, t, mask, T: float, g, lse, v0: int, v1: int, row_chunk: int = 64):
    """The slice [v0, v1) of the vocabulary's share of the gradients.

    With the logsumexp of the WHOLE vocabulary, lse[n], per row (fp64):
      dZ_s[n, j] = (g_n / T) (exp(H[n] W[j]^T / T - lse[n]) - P[n, j])   for v0 <= j < v1
    (0 on masked rows), and
      dH_s = dZ_s W[v0:v1]      (the full dH is the sum over the slices)
      dW_s = dZ_s^T H           (rows v0..v1-1 of the full dW)
    Returns (dH_s[N, D], dW_s[v1 - v0, D]).
    """
    H = np.asarray(H, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    idx = np.asarray(idx)
    t = np.asarray(t)
    mask = np.asarray(mask).astype(bool)
    g = np.asarray(g, dtype=np.float64)
    lse = np.asarray(lse, dtype=np.float64)
    N, D = H.shape
    V = W.shape[0]
    dH = np.zeros((N, D), dtype=np.float64)
    dW = np.zeros((v1 - v0, D), dtype=np.float64)
    for r0, r1 in _blocks(N, row_chunk):
        valid = np.nonzero(mask[r0:r1])[0]
        if valid.size == 0:
            continue
        rows = r0 + valid
        z = student_logits(H[rows], W[v0:v1])
        q = np.exp(z / T - lse[rows][:, None])
        P = dense_teacher_grid(idx[rows].astype(np.int64), teacher_log_probs(t[rows], T), V)
        dZ = (g[rows] / T)[:, None] * (q - P[:, v0:v1])
        dH[rows] = dZ @ W[v0:v1]
        dW += dZ.T @ H[rows]
    return dH, dW
