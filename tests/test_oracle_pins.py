"""Pins for the CPU fp64 oracle, checked against things other than itself.

Each pin uses an independent route to the same number: a library routine
(torch's kl_div / log_softmax / cross_entropy / autograd in float64), a closed
form worked by hand, central finite differences, or an invariant the
mathematics fixes. ``test_planted_mistakes_are_caught`` plants mistakes in the
oracle's helpers and checks that the pins notice.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import kd_oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand_problem(seed, N, D, V, K, *, masked=(), dup_row=None, scale=1.0):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, D)) * scale
    W = rng.standard_normal((V, D)) / math.sqrt(D)
    idx = np.stack([rng.permutation(V)[:K] for _ in range(N)]).astype(np.int32)
    if dup_row is not None and K >= 2:
        idx[dup_row, 1] = idx[dup_row, 0]
    t = np.sort(rng.standard_normal((N, K)) * 3.0, axis=1)[:, ::-1].copy()
    mask = np.ones(N, dtype=np.uint8)
    for r in masked:
        mask[r] = 0
    return H, W, idx, t, mask


def _library_dense_kl(H, W, idx, t, mask, T, g=None):
    """KL(P || softmax(Z/T)) per row with torch's kl_div on a dense teacher grid.

    The grid is filled entry by entry from torch.softmax of the cached logits,
    so duplicates add up. Returns (loss rows, dH, dW) via torch autograd.
    """
    Ht = torch.tensor(H, dtype=torch.float64, requires_grad=True)
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    N, V = H.shape[0], W.shape[0]
    P = torch.zeros(N, V, dtype=torch.float64)
    for n in range(N):
        if not mask[n]:
            continue
        pk = torch.softmax(torch.tensor(t[n], dtype=torch.float64) / T, dim=0)
        for k in range(idx.shape[1]):
            P[n, int(idx[n, k])] += pk[k]
    logq = torch.log_softmax((Ht @ Wt.T) / T, dim=1)
    kl = torch.nn.functional.kl_div(logq, P, reduction="none").sum(dim=1)
    kl = torch.where(torch.tensor(mask.astype(bool)), kl, torch.zeros_like(kl))
    gg = torch.ones(N, dtype=torch.float64) if g is None else torch.tensor(g, dtype=torch.float64)
    (kl * gg).sum().backward()
    return kl.detach().numpy(), Ht.grad.numpy(), Wt.grad.numpy()


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# ----------------------------------------------------------------------------- pins


def _pin_library(seed=0, T=1.7, dup=True):
    H, W, idx, t, mask = _rand_problem(seed, 6, 5, 13, 4, masked=(2,), dup_row=4 if dup else None)
    g = np.linspace(0.5, 2.0, 6)
    loss, lse, nv = oracle.kd_forward(H, W, idx, t, mask, T, row_chunk=4)
    dH, dW = oracle.kd_backward(H, W, idx, t, mask, T, g, row_chunk=4)
    lib, ldH, ldW = _library_dense_kl(H, W, idx, t, mask, T, g)
    lse_lib = torch.logsumexp(torch.tensor(H @ W.T) / T, dim=1).numpy()
    return dict(loss=_rel(loss, lib), lse=_rel(lse, lse_lib), dH=_rel(dH, ldH), dW=_rel(dW, ldW),
                nv=(nv == 5))


@pytest.mark.parametrize("T", [1.0, 1.7, 0.5])
def test_matches_library_dense_kl_and_autograd(T):
    r = _pin_library(seed=3, T=T)
    assert r["nv"]
    assert r["loss"] < 1e-12 and r["lse"] < 1e-12
    assert r["dH"] < 1e-12 and r["dW"] < 1e-12


def test_k_equals_v_brute_force():
    # K = V: the teacher covers the whole vocabulary
    H, W, idx, t, mask = _rand_problem(1, 5, 4, 9, 9)
    loss, _, _ = oracle.kd_forward(H, W, idx, t, mask, 1.3)
    lib, _, _ = _library_dense_kl(H, W, idx, t, mask, 1.3)
    assert _rel(loss, lib) < 1e-12


@pytest.mark.parametrize("T", [1.0, 2.0, 0.7])
def test_zero_when_teacher_equals_student(T):
    H, W, _, _, mask = _rand_problem(2, 4, 6, 10, 10)
    Z = H @ W.T
    idx = np.tile(np.arange(10, dtype=np.int32), (4, 1))
    rng = np.random.default_rng(0)
    perm = np.stack([rng.permutation(10) for _ in range(4)])
    idx = np.take_along_axis(idx, perm, 1)
    t = np.take_along_axis(Z, perm, 1)
    loss, _, _ = oracle.kd_forward(H, W, idx, t, mask, T)
    dH, dW = oracle.kd_backward(H, W, idx, t, mask, T, np.ones(4))
    assert np.max(np.abs(loss)) < 1e-13
    assert np.max(np.abs(dH)) < 1e-13 and np.max(np.abs(dW)) < 1e-13


def test_nonnegative():
    for seed in range(8):
        H, W, idx, t, mask = _rand_problem(seed, 7, 6, 20, 5, scale=3.0)
        loss, _, _ = oracle.kd_forward(H, W, idx, t, mask, 1.0 + 0.25 * seed)
        assert np.all(loss >= -1e-14)


@pytest.mark.parametrize("T", [1.0, 2.5])
def test_k1_is_cross_entropy(T):
    H, W, idx, _, mask = _rand_problem(4, 6, 5, 11, 1)
    t = np.random.default_rng(1).standard_normal((6, 1))  # any value: p = 1
    loss, _, _ = oracle.kd_forward(H, W, idx, t, mask, T)
    ce = torch.nn.functional.cross_entropy(torch.tensor(H @ W.T) / T,
                                           torch.tensor(idx[:, 0], dtype=torch.int64),
                                           reduction="none").numpy()
    assert _rel(loss, ce) < 1e-12


def test_two_class_closed_form():
    # V = K = 2: KL between two Bernoulli laws, written out by hand
    H = np.array([[0.3, -1.1], [2.0, 0.5]])
    W = np.array([[0.7, 0.2], [-0.4, 0.9]])
    idx = np.array([[1, 0], [0, 1]], dtype=np.int32)
    t = np.array([[0.25, -0.75], [1.5, 1.0]])
    T = 1.6
    loss, _, _ = oracle.kd_forward(H, W, idx, t, np.ones(2, np.uint8), T)
    for n in range(2):
        z0 = H[n] @ W[0]
        z1 = H[n] @ W[1]
        q1 = 1.0 / (1.0 + math.exp(-(z1 - z0) / T))                 # student P(token 1)
        t_of = {int(idx[n, 0]): t[n, 0], int(idx[n, 1]): t[n, 1]}
        p1 = 1.0 / (1.0 + math.exp(-(t_of[1] - t_of[0]) / T))       # teacher P(token 1)
        want = p1 * math.log(p1 / q1) + (1 - p1) * math.log((1 - p1) / (1 - q1))
        assert abs(loss[n] - want) < 1e-14


def test_hand_worked_example():
    # Z = (0, ln 2, ln 3) -> q = (1, 2, 3)/6; teacher ids (2, 0) with logits
    # (ln 3, 0) -> p = (3/4 at id 2, 1/4 at id 0). KL = ln 1.5 exactly;
    # dZ = q - p~ = (-1/12, 1/3, -1/4); dH = dZ W; dW = dZ^T H.
    H = np.array([[1.0]])
    W = np.array([[0.0], [math.log(2.0)], [math.log(3.0)]])
    idx = np.array([[2, 0]], dtype=np.int32)
    t = np.array([[math.log(3.0), 0.0]])
    m = np.ones(1, np.uint8)
    loss, lse, nv = oracle.kd_forward(H, W, idx, t, m, 1.0)
    assert abs(loss[0] - math.log(1.5)) < 1e-15
    assert abs(lse[0] - math.log(6.0)) < 1e-15 and nv == 1
    dH, dW = oracle.kd_backward(H, W, idx, t, m, 1.0, np.ones(1))
    assert abs(dH[0, 0] - (math.log(2.0) / 3.0 - math.log(3.0) / 4.0)) < 1e-15
    assert np.allclose(dW[:, 0], [-1.0 / 12.0, 1.0 / 3.0, -0.25], rtol=0, atol=1e-15)


def test_finite_differences():
    H, W, idx, t, mask = _rand_problem(5, 3, 4, 7, 3, masked=(1,), dup_row=2)
    g = np.array([0.7, 1.3, -0.4])
    for T in (1.0, 2.0):
        dH, dW = oracle.kd_backward(H, W, idx, t, mask, T, g)

        def f(Hx, Wx):
            loss, _, _ = oracle.kd_forward(Hx, Wx, idx, t, mask, T)
            return float(np.dot(g, loss))

        h = 1e-6
        num_H = np.zeros_like(H)
        for i in range(H.shape[0]):
            for j in range(H.shape[1]):
                Hp = H.copy(); Hp[i, j] += h
                Hm = H.copy(); Hm[i, j] -= h
                num_H[i, j] = (f(Hp, W) - f(Hm, W)) / (2 * h)
        num_W = np.zeros_like(W)
        for i in range(W.shape[0]):
            for j in range(W.shape[1]):
                Wp = W.copy(); Wp[i, j] += h
                Wm = W.copy(); Wm[i, j] -= h
                num_W[i, j] = (f(H, Wp) - f(H, Wm)) / (2 * h)
        assert _rel(dH, num_H) < 1e-7
        assert _rel(dW, num_W) < 1e-7


def test_scaling_shift_and_permutation():
    H, W, idx, t, mask = _rand_problem(6, 5, 4, 12, 6)
    T = 2.0
    base, _, _ = oracle.kd_forward(H, W, idx, t, mask, T)
    scaled, _, _ = oracle.kd_forward(H / T, W, idx, t / T, mask, 1.0)
    assert _rel(base, scaled) < 1e-12
    shifted, _, _ = oracle.kd_forward(H, W, idx, t + np.arange(5)[:, None] * 3.7, mask, T)
    assert _rel(base, shifted) < 1e-12
    perm = np.random.default_rng(2).permutation(6)
    permuted, _, _ = oracle.kd_forward(H, W, idx[:, perm], t[:, perm], mask, T)
    assert _rel(base, permuted) < 1e-12


def test_row_sum_invariant():
    H, W, idx, t, mask = _rand_problem(7, 6, 5, 15, 4, masked=(0,))
    dH, dW = oracle.kd_backward(H, W, idx, t, mask, 1.4, np.linspace(-1, 1, 6))
    assert np.max(np.abs(dW.sum(axis=0))) < 1e-13


def test_masked_rows_are_never_read():
    H, W, idx, t, mask = _rand_problem(8, 6, 5, 15, 4, masked=(1, 4))
    loss, lse, nv = oracle.kd_forward(H, W, idx, t, mask, 1.0)
    dH, dW = oracle.kd_backward(H, W, idx, t, mask, 1.0, np.ones(6))
    idx2, t2 = idx.copy(), t.copy()
    idx2[[1, 4]] = -99999
    t2[[1, 4]] = np.nan
    loss2, lse2, nv2 = oracle.kd_forward(H, W, idx2, t2, mask, 1.0)
    dH2, dW2 = oracle.kd_backward(H, W, idx2, t2, mask, 1.0, np.ones(6))
    assert nv == nv2 == 4
    assert np.array_equal(loss, loss2) and np.array_equal(lse, lse2)
    assert np.array_equal(dH, dH2) and np.array_equal(dW, dW2)
    assert loss[1] == 0.0 and loss[4] == 0.0 and not np.any(dH[[1, 4]])


def test_no_counted_rows():
    H, W, idx, t, _ = _rand_problem(9, 3, 4, 8, 2)
    mask = np.zeros(3, np.uint8)
    loss, lse, nv = oracle.kd_forward(H, W, idx, t, mask, 1.0)
    assert nv == 0 and oracle.mean_loss(loss, nv) == 0.0
    dH, dW = oracle.kd_backward(H, W, idx, t, mask, 1.0, np.zeros(3))
    assert not np.any(dH) and not np.any(dW)
    assert np.all(np.isfinite(lse))


def test_row_chunk_invariance():
    H, W, idx, t, mask = _rand_problem(10, 9, 5, 14, 3, masked=(3,))
    g = np.linspace(0.1, 0.9, 9)
    ref = oracle.kd_forward(H, W, idx, t, mask, 1.2, row_chunk=9)
    refb = oracle.kd_backward(H, W, idx, t, mask, 1.2, g, row_chunk=9)
    for c in (1, 7):
        out = oracle.kd_forward(H, W, idx, t, mask, 1.2, row_chunk=c)
        outb = oracle.kd_backward(H, W, idx, t, mask, 1.2, g, row_chunk=c)
        assert _rel(out[0], ref[0]) < 1e-12 and _rel(out[1], ref[1]) < 1e-12
        assert _rel(outb[0], refb[0]) < 1e-12 and _rel(outb[1], refb[1]) < 1e-12


# ------------------------------------------------------------- planted mistakes


def _mut_teacher_no_T(t_rows, T):
    b = np.asarray(t_rows, dtype=np.float64)
    return b - kd_oracle.logsumexp_rows(b)[:, None]


def _mut_teacher_unnormalised(t_rows, T):
    return np.asarray(t_rows, dtype=np.float64) / T


def _mut_lse_max_only(a):
    return np.max(a, axis=-1)


_orig_student = kd_oracle.student_logits


def _mut_student_shifted_rows(H_rows, W):
    return _orig_student(H_rows, np.roll(np.asarray(W), 1, axis=0))


def _mut_grid_assign(idx_rows, logp_rows, V):
    n = idx_rows.shape[0]
    grid = np.zeros((n, V))
    for r in range(n):
        grid[r, idx_rows[r]] = np.exp(logp_rows[r])  # duplicates overwrite instead of adding
    return grid


@pytest.mark.parametrize("name,fn", [
    ("teacher_log_probs", _mut_teacher_no_T),
    ("teacher_log_probs", _mut_teacher_unnormalised),
    ("logsumexp_rows", _mut_lse_max_only),
    ("student_logits", _mut_student_shifted_rows),
    ("dense_teacher_grid", _mut_grid_assign),
])
def test_planted_mistakes_are_caught(monkeypatch, name, fn):
    monkeypatch.setattr(kd_oracle, name, fn)
    r = _pin_library(seed=11, T=1.7, dup=True)
    worst = max(r["loss"], r["lse"], r["dH"], r["dW"])
    assert worst > 1e-6, f"mutation of {name} went unnoticed"


def test_dense_grid_bytes_match_pages_example():
    # The blog's worked size: a 4 x 201,088 x 32,768 bf16 teacher grid is about
    # 50 GB (the fixture records the figures and where they are printed); the
    # memory sweep of bench.py reports this size beside the fused head's peak.
    fx = {}
    with open(__file__.replace("test_oracle_pins.py", "golden/pages_dense_grid.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                fx[k] = float(v)
    from bench import dense_grid_bytes
    b = dense_grid_bytes(int(fx["batch"]) * int(fx["seq"]), int(fx["vocab"]), int(fx["bytes_per_elem"]))
    assert b == 4 * 201088 * 32768 * 2
    assert abs(b / 1e9 - fx["approx_gb"]) / fx["approx_gb"] < 0.1


# ----------------------------------------------------------------------------- logits-input form


def _library_dense_kl_logits(Z, idx, t, mask, T, g):
    """torch kl_div of the dense teacher grid against log_softmax(Z/T), autograd wrt Z."""
    Zt = torch.tensor(Z, dtype=torch.float64, requires_grad=True)
    N, V = Z.shape
    P = torch.zeros(N, V, dtype=torch.float64)
    for n in range(N):
        if not mask[n]:
            continue
        pk = torch.softmax(torch.tensor(t[n], dtype=torch.float64) / T, dim=0)
        for k in range(idx.shape[1]):
            P[n, int(idx[n, k])] += pk[k]
    kl = torch.nn.functional.kl_div(torch.log_softmax(Zt / T, dim=1), P, reduction="none").sum(dim=1)
    kl = torch.where(torch.tensor(mask.astype(bool)), kl, torch.zeros_like(kl))
    (kl * torch.tensor(g, dtype=torch.float64)).sum().backward()
    return kl.detach().numpy(), Zt.grad.numpy()


@pytest.mark.parametrize("T", [0.6, 1.5])
def test_logits_form_matches_library(T):
    H, W, idx, t, mask = _rand_problem(21, 7, 5, 17, 4, masked=(3,), dup_row=5)
    Z = H @ W.T * 2.0
    g = np.linspace(-1.0, 2.0, 7)
    loss, lse, nv, dZ = oracle.kd_from_logits(Z, idx, t, mask, T, g, row_chunk=3)
    lib, ldZ = _library_dense_kl_logits(Z, idx, t, mask, T, g)
    assert _rel(loss, lib) < 1e-12
    assert _rel(lse, torch.logsumexp(torch.tensor(Z) / T, dim=1).numpy()) < 1e-13
    assert _rel(dZ, ldZ) < 1e-12
    assert nv == 6


def test_logits_form_chains_to_head_gradients():
    # with Z = H W^T the logit gradient must give the head oracle's dH = dZ W and dW = dZ^T H
    H, W, idx, t, mask = _rand_problem(22, 9, 6, 23, 5, masked=(0, 4), dup_row=2)
    g = np.linspace(0.1, 1.0, 9)
    for T in (1.0, 1.8):
        loss, lse, nv, dZ = oracle.kd_from_logits(H @ W.T, idx, t, mask, T, g)
        l2, lse2, nv2 = oracle.kd_forward(H, W, idx, t, mask, T)
        dH, dW = oracle.kd_backward(H, W, idx, t, mask, T, g)
        assert _rel(loss, l2) < 1e-13 and _rel(lse, lse2) < 1e-13 and nv == nv2
        assert _rel(dZ @ W, dH) < 1e-12 and _rel(dZ.T @ H, dW) < 1e-12
        assert np.all(dZ[mask == 0] == 0)


def test_logits_form_finite_differences():
    rng = np.random.default_rng(23)
    Z = rng.standard_normal((3, 8)) * 2.0
    idx = np.array([[1, 5, 5], [0, 2, 7], [3, 4, 6]])  # row 0 repeats an id
    t = np.sort(rng.standard_normal((3, 3)), axis=1)[:, ::-1].copy()
    mask = np.array([1, 0, 1], dtype=np.uint8)
    g = np.array([0.9, 1.1, -0.6])
    for T in (1.0, 0.7):
        _, _, _, dZ = oracle.kd_from_logits(Z, idx, t, mask, T, g)

        def f(Zx):
            return float(np.dot(g, oracle.kd_from_logits(Zx, idx, t, mask, T)[0]))

        h = 1e-6
        num = np.zeros_like(Z)
        for i in range(Z.shape[0]):
            for j in range(Z.shape[1]):
                Zp = Z.copy(); Zp[i, j] += h
                Zm = Z.copy(); Zm[i, j] -= h
                num[i, j] = (f(Zp) - f(Zm)) / (2 * h)
        assert _rel(dZ, num) < 1e-7


# ----------------------------------------------------------------------------- teacher top-K cache


def test_teacher_topk_brute_force_and_invariants():
    rng = np.random.default_rng(31)
    H = rng.standard_normal((5, 6))
    W = rng.standard_normal((40, 6))
    W[7] = W[3]  # two tokens with equal logits in every row
    K = 9
    ids, vals = oracle.teacher_topk(H, W, K, row_chunk=2)
    for n in range(H.shape[0]):
        z = [float(sum(H[n, d] * W[j, d] for d in range(6))) for j in range(40)]
        ranked = sorted(range(40), key=lambda j: (-z[j], j))  # brute force, python sort
        assert list(ids[n]) == ranked[:K]
        assert np.allclose(vals[n], [z[j] for j in ranked[:K]], rtol=0, atol=1e-12)
        assert np.all(np.diff(vals[n]) <= 0)
        rest = np.delete(np.array(z), ids[n])
        assert rest.max() <= vals[n, -1]
    # K = V returns a full descending permutation
    ids_all, vals_all = oracle.teacher_topk(H[:2], W, 40)
    assert sorted(ids_all[0]) == list(range(40))


def test_teacher_topk_feeds_the_loss_at_k_equals_v():
    # caching all V logits and distilling from the cache is the exact dense KL:
    # with the student equal to the teacher the loss is zero
    H, W, _, _, _ = _rand_problem(32, 3, 5, 11, 1)
    ids, vals = oracle.teacher_topk(H, W, 11)
    loss, _, _ = oracle.kd_forward(H, W, ids, vals, np.ones(3, dtype=np.uint8), 1.3)
    assert np.max(np.abs(loss)) < 1e-12


# ----------------------------------------------------------------------------- vocabulary shards


def _shard_problem():
    # three uneven slices; row 1 repeats an id, row 3 is masked (NaN teacher logits)
    H, W, idx, t, mask = _rand_problem(21, 7, 6, 23, 5, masked=(3,), dup_row=1)
    t[3] = np.nan
    idx[5] = [0, 1, 2, 3, 4]  # every teacher id of row 5 in the first slice
    return H, W, idx, t, mask, [(0, 8), (8, 9), (9, 23)]


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_vocab_shards_recombine_to_the_whole_vocabulary(T):
    # logsumexp and sums over a partition of the columns give back kd_forward /
    # kd_backward exactly (up to fp64 rounding), for any split
    H, W, idx, t, mask, cuts = _shard_problem()
    loss, lse, _ = oracle.kd_forward(H, W, idx, t, mask, T)
    g = np.linspace(0.3, 1.1, H.shape[0])
    dH, dW = oracle.kd_backward(H, W, idx, t, mask, T, g)
    parts = [oracle.kd_forward_shard(H, W, idx, t, mask, T, a, b) for a, b in cuts]
    lse_m = np.logaddexp.reduce(np.stack([p[0] for p in parts]), axis=0)
    x = np.sum([p[1] for p in parts], axis=0)
    for p in parts:
        np.testing.assert_array_equal(p[2], parts[0][2])  # entropy: the whole grid, every shard
    loss_m = np.where(mask.astype(bool), parts[0][2] - x / T + lse_m, 0.0)
    assert _rel(lse_m, lse) < 1e-13
    assert _rel(loss_m, loss) < 1e-12
    grads = [oracle.kd_backward_shard(H, W, idx, t, mask, T, g, lse, a, b) for a, b in cuts]
    assert _rel(np.sum([gr[0] for gr in grads], axis=0), dH) < 1e-12
    assert _rel(np.concatenate([gr[1] for gr in grads], axis=0), dW) < 1e-12


def test_vocab_shard_pieces_match_torch():
    # each piece on its own, by an independent route: torch's logsumexp over the
    # slice, the dense grid filled entry by entry, -entr(P) summed for the entropy
    T = 1.3
    H, W, idx, t, mask, cuts = _shard_problem()
    Z = torch.tensor(H) @ torch.tensor(W).T
    for a, b in cuts:
        lse_s, x_s, ent = oracle.kd_forward_shard(H, W, idx, t, mask, T, a, b)
        np.testing.assert_allclose(lse_s, torch.logsumexp(Z[:, a:b] / T, dim=1).numpy(), rtol=1e-13)
        for n in range(H.shape[0]):
            if not mask[n]:
                assert x_s[n] == 0.0 and ent[n] == 0.0
                continue
            pk = torch.softmax(torch.tensor(t[n]) / T, dim=0)
            P = torch.zeros(W.shape[0], dtype=torch.float64)
            for k in range(idx.shape[1]):
                P[int(idx[n, k])] += pk[k]
            assert x_s[n] == pytest.approx(float((P[a:b] * Z[n, a:b]).sum()), rel=1e-12, abs=1e-14)
            assert ent[n] == pytest.approx(float(-torch.special.entr(P).sum()), rel=1e-12)
