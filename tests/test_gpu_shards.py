"""Vocabulary shards and the device-side mean gradient, through the C ABI.

The head split over the vocabulary: each shard runs kd_topk_kl_fwd_shard on
its rows of W, the shards' (lse, cross term) parts are merged by
kd_topk_kl_shard_merge, and kd_topk_kl_bwd_shard gives each shard's part of dH
and its rows of dW. On one GPU the shards run one after another (a rank per
shard does the same work in parallel); the merged loss / lse and the summed
dH / stacked dW must match the CPU oracle of the WHOLE vocabulary, element by
element, and each shard's parts must match the oracle's shard restatement.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import _parity as P
from top_kl_loss_lm_b300 import binding
from workloads import config_problem, make_problem, mean_upstream_grad

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run_shards(p, cuts, chunk=0, g=None):
    """Forward, merge, mean gradient and backward over the shards `cuts`."""
    N, D, V, K = p.N, p.D, p.V, p.K
    R = len(cuts)
    ws = torch.empty(max(binding.kd_topk_kl_shard_workspace_size(N, D, b - a, K, chunk)
                         for a, b in cuts), dtype=torch.uint8, device=DEV)
    parts = torch.full((R, N, 2), float("nan"), device=DEV)
    ents = torch.full((R, N), float("nan"), device=DEV)
    nvs = torch.full((R, 1), -1, dtype=torch.int64, device=DEV)
    for r, (a, b) in enumerate(cuts):
        binding.kd_topk_kl_fwd_shard(p.H, p.W[a:b], a, V, p.idx, p.t, p.mask, p.T, parts[r], ents[r],
                                     nvs[r], ws)
    loss = torch.full((N,), float("nan"), device=DEV)
    lse = torch.full((N,), float("nan"), device=DEV)
    binding.kd_topk_kl_shard_merge(parts, ents[0], p.mask, p.T, loss, lse)
    dloss = torch.full((N,), float("nan"), device=DEV)
    loss_sum = torch.full((1,), float("nan"), dtype=torch.float64, device=DEV)
    binding.kd_topk_kl_mean_grad(loss, p.mask, nvs[0], dloss, loss_sum)
    gg = dloss if g is None else g
    dH = torch.full((N, D), float("nan"), device=DEV)
    dW = torch.full((V, D), float("nan"), device=DEV)
    for r, (a, b) in enumerate(cuts):
        binding.kd_topk_kl_bwd_shard(p.H, p.W[a:b], a, V, p.idx, p.t, p.mask, lse, gg, p.T, chunk,
                                     False, r > 0, dH, dW[a:b], ws)
    torch.cuda.synchronize()
    return dict(parts=parts, ents=ents, nvs=nvs, loss=loss, lse=lse, dloss=dloss,
                loss_sum=loss_sum, g=gg, dH=dH, dW=dW, status=binding.kd_get_status())


def check_against_oracle(p, cuts, out):
    h = P.host(p)
    assert out["status"] == 0, binding.STATUS.get(out["status"])
    nv = int(p.mask.sum().item())
    assert all(int(x) == nv for x in out["nvs"].cpu())
    g = out["g"].double().cpu().numpy()
    ref_loss, ref_lse, _ = oracle.kd_forward(h["H"], h["W"], h["idx"], h["t"], h["mask"], p.T)
    P.assert_rows_close(out["loss"].cpu().numpy(), ref_loss, "merged loss")
    P.assert_lse_close(out["lse"].cpu().numpy(), ref_lse, "merged lse")
    for r, (a, b) in enumerate(cuts):
        lse_s, x_s, ent = oracle.kd_forward_shard(h["H"], h["W"], h["idx"], h["t"], h["mask"], p.T, a, b)
        P.assert_lse_close(out["parts"][r, :, 0].cpu().numpy(), lse_s, f"shard {r} lse")
        got_x = out["parts"][r, :, 1].double().cpu().numpy()
        assert np.all(np.abs(got_x - x_s) <= 1e-5 * np.abs(x_s) + 1e-4), f"shard {r} cross term"
        P.assert_rows_close(out["ents"][r].cpu().numpy(), ent, f"shard {r} entropy")
    ref_dH, ref_dW = oracle.kd_backward(h["H"], h["W"], h["idx"], h["t"], h["mask"], p.T, g)
    P.assert_grad_close(out["dH"].double().cpu().numpy(), ref_dH, "dH (sum over shards)")
    P.assert_grad_close(out["dW"].double().cpu().numpy(), ref_dW, "dW (stacked shards)")
    return ref_loss


@pytest.mark.parametrize("cuts", [
    [(0, 256), (256, 512), (512, 1000)],    # tile-aligned
    [(0, 333), (333, 334), (334, 1000)],    # ragged, one single-column shard
    [(0, 1000)],                            # one shard is the whole vocabulary
])
def test_small_shards_match_oracle(cuts):
    p = make_problem(300, 136, 1000, 16, 1.5, seed=41, mask="frac", mask_frac=0.1,
                     garbage_masked=True, device=DEV)
    out = run_shards(p, cuts, chunk=128)
    check_against_oracle(p, cuts, out)
    # the mean gradient came from the device count
    want = mean_upstream_grad(p.mask).to(DEV)
    assert torch.equal(out["dloss"], want)
    assert abs(out["loss_sum"].item() - out["loss"].double().sum().item()) <= 1e-9 * abs(out["loss_sum"].item())


def test_shards_agree_with_the_unsharded_library():
    p = make_problem(700, 256, 5000, 32, 1.0, seed=42, mask="frac", mask_frac=0.05, device=DEV)
    cuts = [(0, 1792), (1792, 3584), (3584, 5000)]
    out = run_shards(p, cuts, chunk=256)
    full = P.run_gpu(p, chunk_tokens=256, g=out["g"])
    assert full["status"] == 0
    np.testing.assert_allclose(out["loss"].cpu().numpy(), full["loss"].cpu().numpy(), rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(out["lse"].cpu().numpy(), full["lse"].cpu().numpy(), rtol=1e-6)
    P.assert_grad_close(out["dW"].double().cpu().numpy(), full["dW"].double().cpu().numpy(), "dW vs unsharded")
    P.assert_grad_close(out["dH"].double().cpu().numpy(), full["dH"].double().cpu().numpy(), "dH vs unsharded")


def test_shard_without_teacher_ids_and_edge_rows():
    # every teacher id in [0, 64): the second shard holds none of them; K = 1 and a
    # repeated id on some rows; masked rows with junk
    p = make_problem(200, 64, 2000, 4, 0.8, seed=43, mask="frac", mask_frac=0.2,
                     garbage_masked=True, device=DEV)
    counted = p.mask.bool()
    p.idx[counted] = torch.randint(0, 64, (int(counted.sum()), 4), device=DEV, dtype=torch.int32)
    p.idx[::7, 1] = p.idx[::7, 0]
    cuts = [(0, 100), (100, 2000)]
    out = run_shards(p, cuts)
    check_against_oracle(p, cuts, out)
    assert torch.all(out["parts"][1, :, 1] == 0)  # no teacher entry in the second shard


def test_invalid_id_is_reported_by_every_shard():
    p = make_problem(64, 64, 300, 4, 1.0, seed=44, device=DEV)
    p.idx[5, 2] = p.V + 3
    out = run_shards(p, [(0, 150), (150, 300)])
    assert out["status"] == 5  # KD_ERR_INDEX
    assert binding.kd_get_status() == 0


def test_mean_grad_with_no_counted_rows():
    N = 1000
    loss = torch.zeros(N, device=DEV)
    mask = torch.zeros(N, dtype=torch.uint8, device=DEV)
    nv = torch.zeros(1, dtype=torch.int64, device=DEV)
    dloss = torch.full((N,), float("nan"), device=DEV)
    s = torch.full((1,), float("nan"), dtype=torch.float64, device=DEV)
    binding.kd_topk_kl_mean_grad(loss, mask, nv, dloss, s)
    torch.cuda.synchronize()
    assert torch.all(dloss == 0) and s.item() == 0.0


@pytest.mark.slow
def test_gptoss_head_in_two_shards_sampled_rows():
    p = config_problem("gptoss_4k", device=DEV)
    V = p.V
    cuts = [(0, 100608), (100608, V)]
    out = run_shards(p, cuts)
    assert out["status"] == 0
    rng = np.random.default_rng(3)
    m = p.mask.cpu().numpy().astype(bool)
    rows = np.unique(np.concatenate([rng.choice(np.nonzero(m)[0], 24, replace=False),
                                     rng.choice(np.nonzero(~m)[0], 4, replace=False)]))
    ref = P.run_oracle(p, out["g"].double().cpu().numpy(), rows=rows, backward=True)
    P.assert_rows_close(out["loss"].cpu().numpy()[rows], ref["loss"], "loss (sampled rows)")
    P.assert_lse_close(out["lse"].cpu().numpy()[rows], ref["lse"], "lse (sampled rows)")
    P.assert_grad_close(out["dH"].double().cpu().numpy()[rows], ref["dH"], "dH (sampled rows)")


def test_sharded_steps_on_one_gpu_match_the_oracle():
    # the product's step classes with world size 1 (no collectives): the
    # token-sharded step's forward / mean gradient / backward, and the vocabulary
    # step's shard forward / merge / shard backward over the whole vocabulary
    from top_kl_loss_lm_b300 import sharded
    p = make_problem(500, 136, 3000, 16, 1.2, seed=45, mask="frac", mask_frac=0.1,
                     garbage_masked=True, device=DEV)
    h = P.host(p)
    nv = int(p.mask.sum().item())
    g = p.mask.cpu().numpy().astype(np.float64) / nv
    ref_loss, ref_lse, _ = oracle.kd_forward(h["H"], h["W"], h["idx"], h["t"], h["mask"], p.T)
    ref_dH, ref_dW = oracle.kd_backward(h["H"], h["W"], h["idx"], h["t"], h["mask"], p.T, g)
    ref_mean = oracle.mean_loss(ref_loss, nv)

    tok = sharded.TokenShardedHead(p.N, p.D, p.V, p.K, p.T, DEV, chunk_tokens=256)
    loss_sum, n_valid = tok.step(p.H, p.W, p.idx, p.t, p.mask)
    assert int(n_valid.item()) == nv
    assert abs(sharded.mean_loss(loss_sum, n_valid) - ref_mean) <= 1e-3 * abs(ref_mean)
    P.assert_rows_close(tok.loss.cpu().numpy(), ref_loss, "token-sharded loss")
    P.assert_grad_close(tok.dH.double().cpu().numpy(), ref_dH, "token-sharded dH")
    P.assert_grad_close(tok.dW.double().cpu().numpy(), ref_dW, "token-sharded dW")

    voc = sharded.VocabShardedHead(p.N, p.D, p.V, p.K, p.T, DEV, chunk_tokens=256)
    assert (voc.v0, voc.v1) == (0, p.V)
    loss_sum, n_valid = voc.step(p.H, p.W[voc.v0:voc.v1], p.idx, p.t, p.mask)
    assert abs(sharded.mean_loss(loss_sum, n_valid) - ref_mean) <= 1e-3 * abs(ref_mean)
    P.assert_rows_close(voc.loss.cpu().numpy(), ref_loss, "vocabulary-sharded loss")
    P.assert_lse_close(voc.lse.cpu().numpy(), ref_lse, "vocabulary-sharded lse")
    P.assert_grad_close(voc.dH.double().cpu().numpy(), ref_dH, "vocabulary-sharded dH")
    P.assert_grad_close(voc.dW_shard.double().cpu().numpy(), ref_dW, "vocabulary-sharded dW")
    assert binding.kd_get_status() == 0
