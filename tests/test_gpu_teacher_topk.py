"""The teacher's top-K cache (kd_teacher_topk) through the C ABI, against the CPU
fp64 oracle's teacher_topk.

The GPU decides the top-K on fp32 logits; near-equal logits at the boundary may
therefore come out in a different but equally correct set. So the checks are:
ids valid and distinct, logits in descending order, each returned logit equal
to the exact logit of its id within the fp32 accumulation error, no id left out
whose exact logit beats the smallest returned one by more than that error, and
the returned values equal the oracle's top-K values within it. Ties are
exercised on purpose (repeated rows of W, an all-zero hidden state); tied
logits go to the smallest ids, so repeated calls return the same cache.

Vocabularies of 16,384 and more take the fused path (a threshold per row from a
strided sample of W's rows, the GEMM keeping only the logits that reach it);
its fallback for rows whose threshold keeps too few or too many logits is
forced on purpose below, and must give the same exact cache.
"""
import numpy as np
import pytest
import torch

import oracle
from top_kl_loss_lm_b300 import binding
from workloads import make_problem

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _run(H, W, K):
    N, D = H.shape
    V = W.shape[0]
    ws = torch.empty(binding.kd_teacher_topk_workspace_size(N, D, V, K), dtype=torch.uint8,
                     device=DEV)
    ids = torch.full((N, K), -1, dtype=torch.int32, device=DEV)
    vals = torch.full((N, K), float("nan"), device=DEV)
    binding.kd_teacher_topk(H, W, ids, vals, ws)
    torch.cuda.synchronize()
    assert binding.kd_get_status() == 0
    return ids.cpu().numpy().astype(np.int64), vals.double().cpu().numpy()


def _check(H, W, K, ids, vals, rows=None):
    Hn = H.double().cpu().numpy()
    Wn = W.double().cpu().numpy()
    rows = np.arange(Hn.shape[0]) if rows is None else np.asarray(rows)
    Z = Hn[rows] @ Wn.T
    V = Wn.shape[0]
    ref_ids, ref_vals = oracle.teacher_topk(Hn[rows], Wn, K)
    for i, n in enumerate(rows):
        z = Z[i]
        tol = 1e-5 * max(1.0, float(np.abs(z).max()))  # fp32 accumulation of D bf16 products
        g_ids, g_vals = ids[n], vals[n]
        assert np.all((g_ids >= 0) & (g_ids < V)), n
        assert len(set(g_ids.tolist())) == K, n
        assert np.all(np.diff(g_vals) <= 0), n
        assert np.all(np.abs(g_vals - z[g_ids]) <= tol), n
        rest = np.delete(z, g_ids)
        if rest.size:
            assert rest.max() <= z[g_ids].min() + 2 * tol, n
        assert np.all(np.abs(g_vals - ref_vals[i]) <= 2 * tol), n


def _problem(N, D, V, seed):
    p = make_problem(N, D, V, 1, 1.0, seed=seed, device=DEV)
    return p.H, p.W


def test_small_every_row():
    H, W = _problem(300, 136, 1000, seed=1)
    _check(H, W, 16, *_run(H, W, 16))


@pytest.mark.parametrize("K", [1, 100, 256])
def test_k_range_and_ragged_vocabulary(K):
    H, W = _problem(130, 64, 1001, seed=2)  # V not a multiple of 4 or 8
    _check(H, W, K, *_run(H, W, K))


@pytest.mark.parametrize("V", [600, 5000])
def test_ties_and_all_equal_row(V):
    # V = 5,000: row 5's 5,000 equal logits overflow the shared-memory candidate
    # list, so the later radix levels read the row again
    H, W = _problem(64, 64, V, seed=3)
    W[7] = W[3]
    W[100:140] = W[50]      # 41 equal logits in every row
    H[5] = 0                # every logit of row 5 is 0
    ids, vals = _run(H, W, 32)
    _check(H, W, 32, ids, vals)
    assert np.all(vals[5] == 0)
    # ties go to the smallest ids, so the cache is the same on every call
    assert list(ids[5]) == list(range(32))
    ids2, vals2 = _run(H, W, 32)
    assert np.array_equal(ids, ids2) and np.array_equal(vals, vals2)


def test_several_row_chunks():
    H, W = _problem(2 * 4096 + 123, 32, 700, seed=4)
    _check(H, W, 8, *_run(H, W, 8))


def test_cache_feeds_the_loss():
    # distilling a student from its own complete cache (K = V) gives zero KL
    H, W = _problem(96, 64, 200, seed=5)
    ids, vals = (torch.as_tensor(x, device=DEV) for x in _run(H, W, 200))
    N, V, K = 96, 200, 200
    ws = torch.empty(binding.kd_topk_kl_workspace_size(N, 64, V, K, 0), dtype=torch.uint8, device=DEV)
    loss = torch.empty(N, device=DEV)
    lse = torch.empty(N, device=DEV)
    nv = torch.empty(1, dtype=torch.int64, device=DEV)
    binding.kd_topk_kl_fwd(H, W, ids.to(torch.int32), vals.to(torch.float32), None, 1.0, loss, lse,
                           nv, ws)
    torch.cuda.synchronize()
    assert binding.kd_get_status() == 0
    assert float(loss.abs().max()) < 1e-4


@pytest.mark.parametrize("K", [1, 100, 256])
def test_fused_path_every_row(K):
    H, W = _problem(300, 136, 20000, seed=7)
    _check(H, W, K, *_run(H, W, K))


def test_fused_path_over_several_chunks():
    H, W = _problem(4096 + 123, 32, 16384 + 77, seed=8)
    _check(H, W, 8, *_run(H, W, 8), rows=np.r_[0:64, 4060:4219])


def test_fused_path_falls_back_exactly():
    # V = 20,000 samples every 9th row of W. Row 5 is all ties (every logit 0: far
    # more than the candidate list holds); on row 9 the sampled rows of W dominate
    # (too few logits reach the threshold). Both force the chunk's exact fallback.
    H, W = _problem(200, 64, 20000, seed=9)
    H[5] = 0
    Wf = W.float()
    Wf[::9] *= 50.0
    W2 = Wf.to(torch.bfloat16)
    H2 = H.clone()
    H2[9] = W2[0]  # z = <W[0], W[j]>: the sampled rows (x 50) tower over the rest
    ids, vals = _run(H2, W2, 100)
    _check(H2, W2, 100, ids, vals)
    assert list(ids[5]) == list(range(100)) and np.all(vals[5] == 0)
    ids2, vals2 = _run(H2, W2, 100)
    assert np.array_equal(ids, ids2) and np.array_equal(vals, vals2)


def test_fused_select_many_equal_candidates():
    # Rows 1,000..1,600 of W repeat row 999, and row 3 of H points along it: that
    # row's 602 largest logits are equal. All of them are candidates, more than the
    # short sort after the histogram holds, so the row sorts its whole list; the K
    # kept go to the smallest ids. Row 4 sees them among ordinary logits.
    H, W = _problem(64, 64, 20000, seed=10)
    W[1000:1601] = W[999]
    H2 = H.clone()
    H2[3] = W[999] * 4
    ids, vals = _run(H2, W, 100)
    _check(H2, W, 100, ids, vals)
    assert list(ids[3]) == list(range(999, 1099))
    assert np.all(vals[3] == vals[3][0])


@pytest.mark.slow
def test_gptoss_teacher_head_sampled_rows():
    # the pages cache the top 100 over the 201,088-token vocabulary
    H, W = _problem(4096 + 512, 2880, 201088, seed=6)
    K = 100
    ids, vals = _run(H, W, K)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([rng.choice(H.shape[0], 24, replace=False), [0, H.shape[0] - 1]]))
    _check(H, W, K, ids, vals, rows=rows)


@pytest.mark.slow
def test_gptoss_teacher_head_k256_sampled_rows():
    # the largest K the cache supports over the full vocabulary, with a ragged last chunk
    H, W = _problem(2 * 4096 + 300, 2880, 201088, seed=16)
    K = 256
    ids, vals = _run(H, W, K)
    rng = np.random.default_rng(1)
    rows = np.unique(np.concatenate([rng.choice(H.shape[0], 20, replace=False), [0, 4095, 4096, H.shape[0] - 1]]))
    _check(H, W, K, ids, vals, rows=rows)
