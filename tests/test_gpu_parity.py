"""Parity of the CUDA path (through the C ABI) with the CPU fp64 oracle.

Small cases compare every output element; the full-size workloads compare
sampled rows the oracle can afford (loss, lse and dH are row-local; dW is
checked with a second backward whose upstream gradient is non-zero only on
the sampled rows) plus properties that hold at any size.
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


def _full(p, chunk=0, **kw):
    gpu = P.run_gpu(p, chunk_tokens=chunk, **kw)
    return gpu, P.compare_full(p, gpu)


# ------------------------------------------------------------------ small, every element

def test_tiny_config():
    p = config_problem("tiny", device=DEV)
    _full(p)


def test_ragged_shapes_masked_garbage():
    # N, V, D not multiples of the tiles; masked rows carry NaN logits / junk ids
    p = make_problem(300, 136, 1000, 16, 1.5, seed=1, mask="frac", mask_frac=0.1,
                     garbage_masked=True, device=DEV)
    _full(p, chunk=128)


def test_several_tiles_and_chunks():
    p = make_problem(1000, 512, 20000, 64, 1.0, seed=2, mask="frac", mask_frac=0.02, device=DEV)
    _full(p, chunk=384)


def test_forward_row_chunks_with_ragged_tail():
    # the forward is launched per 4,096 rows: two full chunks and a ragged third one,
    # with the backward's chunks (1,536 rows) cutting across the forward's
    p = make_problem(2 * 4096 + 300, 72, 1800, 16, 1.2, seed=15, mask="frac", mask_frac=0.03,
                     garbage_masked=True, device=DEV)
    _full(p, chunk=1536)


@pytest.mark.parametrize("T", [0.1, 0.7, 2.0])
def test_teacher_covers_vocabulary(T):
    p = make_problem(64, 64, 200, 200, T, seed=3, device=DEV)
    _full(p)


def test_k1_and_k256():
    _full(make_problem(130, 64, 777, 1, 1.0, seed=4, device=DEV))
    _full(make_problem(140, 72, 3000, 256, 2.0, seed=5, mask="frac", mask_frac=0.05, device=DEV))


def test_duplicate_ids_merge():
    p = make_problem(96, 64, 500, 8, 1.3, seed=6, device=DEV)
    p.idx[::3, 1] = p.idx[::3, 0]
    p.idx[1::5, 7] = p.idx[1::5, 2]
    _full(p)


def test_single_row_and_extreme_logits():
    _full(make_problem(1, 64, 300, 4, 1.0, seed=7, device=DEV))
    p = make_problem(200, 128, 2048, 32, 1.0, seed=8, device=DEV)
    p.H = (p.H.float() * 30.0).to(torch.bfloat16)  # logits of size ~100: lse must not overflow
    _full(p)


def test_no_counted_rows():
    p = make_problem(150, 64, 600, 8, 1.0, seed=9, device=DEV)
    p.mask.zero_()
    p.t.fill_(float("nan"))
    gpu = P.run_gpu(p)
    assert gpu["status"] == 0
    assert int(gpu["n_valid"].item()) == 0
    assert torch.all(gpu["loss"] == 0)
    assert torch.all(gpu["dH"].float() == 0) and torch.all(gpu["dW"] == 0)
    ref = P.run_oracle(p, backward=False)
    P.assert_lse_close(gpu["lse"].cpu().numpy(), ref["lse"], "lse")


def test_chunk_size_invariance():
    p = make_problem(700, 96, 1500, 16, 1.0, seed=10, mask="frac", mask_frac=0.05, device=DEV)
    a = P.run_gpu(p, chunk_tokens=128)
    b = P.run_gpu(p, chunk_tokens=4096)
    assert torch.equal(a["loss"], b["loss"]) and torch.equal(a["lse"], b["lse"])
    P.compare_full(p, a)
    P.compare_full(p, b)
    rel = (a["dW"] - b["dW"]).abs().max() / b["dW"].abs().max()
    assert rel.item() < 1e-3


def test_accumulate_dw():
    p = make_problem(200, 64, 900, 8, 1.0, seed=11, device=DEV)
    init = torch.randn(p.V, p.D, device=DEV) * 1e-3
    gpu = P.run_gpu(p, accumulate=True, dW_init=init)
    ref = P.run_oracle(p, gpu["g"].double().cpu().numpy())
    P.assert_grad_close((gpu["dW"] - init).double().cpu().numpy(), ref["dW"], "dW accumulated")


def test_accumulate_dw_over_several_dw_groups():
    # 1,000 rows in 256-row chunks: dW is contracted over two chunks per launch,
    # so this runs two groups (the second ending in a short chunk) and adds onto dW_init
    p = make_problem(1000, 72, 1300, 8, 1.4, seed=16, mask="frac", mask_frac=0.05, device=DEV)
    init = torch.randn(p.V, p.D, device=DEV) * 1e-3
    gpu = P.run_gpu(p, chunk_tokens=256, accumulate=True, dW_init=init)
    ref = P.run_oracle(p, gpu["g"].double().cpu().numpy())
    P.assert_grad_close(gpu["dH"].double().cpu().numpy(), ref["dH"], "dH")
    P.assert_grad_close((gpu["dW"] - init).double().cpu().numpy(), ref["dW"], "dW accumulated")


def test_invalid_id_at_counted_row_is_reported():
    p = make_problem(64, 64, 300, 4, 1.0, seed=12, mask="frac", mask_frac=0.25, device=DEV)
    masked = torch.nonzero(p.mask == 0)[0, 0].item()
    p.idx[masked, 0] = 10 ** 6          # ignored: row is masked
    gpu = P.run_gpu(p, backward=False)
    assert gpu["status"] == 0
    counted = torch.nonzero(p.mask == 1)[0, 0].item()
    p.idx[counted, 1] = p.V + 5
    gpu = P.run_gpu(p, backward=False)
    assert gpu["status"] == 5           # KD_ERR_INDEX
    assert binding.kd_get_status() == 0  # cleared by the read


def test_bounded_wait_reports_timeout_and_context_survives():
    binding.kd_debug_wait_timeout(2_000_000)  # 2 ms on a barrier nothing arrives on
    assert binding.kd_get_status() == 6       # KD_ERR_TIMEOUT
    assert binding.kd_get_status() == 0
    _full(make_problem(64, 64, 300, 4, 1.0, seed=13, device=DEV))


def test_autograd_wrapper():
    from top_kl_loss_lm_b300.loss import fused_topk_kl
    p = make_problem(130, 64, 700, 8, 1.0, seed=14, mask="frac", mask_frac=0.1, device=DEV)
    H = p.H.clone().requires_grad_(True)
    W = p.W.clone().requires_grad_(True)
    loss, nv = fused_topk_kl(H, W, p.idx, p.t, p.mask, p.T)
    (loss.sum() / nv.float()).backward()
    g = mean_upstream_grad(p.mask).double().cpu().numpy()
    ref = P.run_oracle(p, g)
    P.assert_rows_close(loss.detach().cpu().numpy(), ref["loss"], "loss")
    P.assert_grad_close(H.grad.double().cpu().numpy(), ref["dH"], "dH")
    # W is bf16, so its grad is rounded to bf16 on the way out of autograd
    P.assert_grad_close(W.grad.double().cpu().numpy(), ref["dW"], "dW")


# ------------------------------------------------------------------ full-size, sampled rows

def _sample_rows(p, n_counted=48, n_masked=8, seed=0):
    rng = np.random.default_rng(seed)
    m = p.mask.cpu().numpy().astype(bool)
    counted = np.nonzero(m)[0]
    masked = np.nonzero(~m)[0]
    rows = list(rng.choice(counted, size=min(n_counted, counted.size), replace=False))
    if masked.size:
        rows += list(rng.choice(masked, size=min(n_masked, masked.size), replace=False))
    rows += [0, p.N - 1]
    return np.unique(np.array(rows))


def _check_sampled(p, chunk=0):
    gpu = P.run_gpu(p, chunk_tokens=chunk)
    assert gpu["status"] == 0
    rows = _sample_rows(p)
    g = gpu["g"].double().cpu().numpy()
    ref = P.run_oracle(p, g, rows=rows, backward=True)
    assert int(gpu["n_valid"].item()) == int(p.mask.sum().item())
    P.assert_rows_close(gpu["loss"].cpu().numpy()[rows], ref["loss"], "loss (sampled rows)")
    P.assert_lse_close(gpu["lse"].cpu().numpy()[rows], ref["lse"], "lse (sampled rows)")
    P.assert_grad_close(gpu["dH"].double().cpu().numpy()[rows], ref["dH"], "dH (sampled rows)")
    # full-size property: sum_v dW[v, :] = sum_n (sum_j dZ[n, j]) H[n, :] = 0
    dW = gpu["dW"]
    assert torch.isfinite(dW).all()
    # (what is left comes from rounding dZ to bf16 before the contraction: about
    # 1e-6 of a column's absolute sum at these sizes)
    ratio = dW.double().sum(0).abs().max().item() / dW.double().abs().sum(0).max().item()
    assert ratio <= 1e-4, ratio
    # dW over the sampled rows alone: upstream gradient only there
    gs = torch.zeros_like(gpu["g"])
    gs[torch.as_tensor(rows, device=gs.device)] = gpu["g"][torch.as_tensor(rows, device=gs.device)]
    gpu2 = P.run_gpu(p, chunk_tokens=chunk, g=gs)
    assert gpu2["status"] == 0
    P.assert_grad_close(gpu2["dW"].double().cpu().numpy(), ref["dW"], "dW (sampled rows)")
    return gpu


@pytest.mark.slow
def test_gptoss_head_4k():
    _check_sampled(config_problem("gptoss_4k", device=DEV))


@pytest.mark.slow
def test_gptoss_head_32k():
    _check_sampled(config_problem("gptoss_32k", device=DEV))


@pytest.mark.slow
@pytest.mark.parametrize("K", [8, 64, 256])
@pytest.mark.parametrize("T", [1.0, 2.0])
def test_packed_documents(K, T):
    _check_sampled(config_problem("packed_qwen", device=DEV, K=K, T=T))


@pytest.mark.slow
@pytest.mark.parametrize("N", [131072, 262144])
def test_gptoss_head_long_sweep(N):
    # the largest sizes of the memory / rate sweep, sampled rows + row-sum property
    _check_sampled(config_problem("gptoss_32k", device=DEV, N=N))


@pytest.mark.slow
def test_peak_memory_linear_in_tokens():
    D, V, K = 2880, 201088, 64
    peaks = []
    Ns = [8192, 32768, 65536]  # every N holds two backward chunks (one dW group)
    for N in Ns:
        p = make_problem(N, D, V, K, 1.0, seed=20, device=DEV)
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats()
        base = torch.cuda.memory_allocated()
        gpu = P.run_gpu(p, chunk_tokens=4096)
        assert gpu["status"] == 0
        peaks.append(torch.cuda.max_memory_allocated() - base)
        del gpu, p
        torch.cuda.empty_cache()
    per_token = [(peaks[i + 1] - peaks[i]) / (Ns[i + 1] - Ns[i]) for i in range(len(Ns) - 1)]
    assert abs(per_token[1] - per_token[0]) <= 0.05 * per_token[0]
    # a dense N x V bf16 grid costs V * 2 bytes per token; the fused head's growth is
    # H, dH and the teacher cache (a few KB), and the fixed part (W, dW, W^T, the dZ
    # chunks) is a small fraction of one grid at 65,536 tokens
    assert per_token[-1] < 0.05 * V * 2
    assert peaks[-1] < Ns[-1] * V * 2 / 3
