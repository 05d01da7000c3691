"""The allocation-free forward, kd_topk_kl_fwd_noalloc.

Some callers cannot allocate device memory: a plugin running inside a process
whose own allocator already holds the GPU's memory, or a hot path where a
cudaMalloc (which may synchronise the device) is not allowed. For them the
library keeps the forward's scratch in a fixed array of its own. This file
checks, through the C ABI, that two calls in a row give bit for bit what the
regular forward gives with a caller workspace, that the largest size the
array holds runs, and that one token more, or a size far beyond the array, is
refused before anything runs. It is collected last on purpose.
"""
import ctypes

import pytest
import torch

from tests import _parity as P
from top_kl_loss_lm_b300 import binding
from workloads import make_problem

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _regular(p):
    ws = torch.empty(binding.kd_topk_kl_workspace_size(p.N, p.D, p.V, p.K, 0), dtype=torch.uint8,
                     device=DEV)
    out = [torch.empty(p.N, device=DEV), torch.empty(p.N, device=DEV),
           torch.empty(1, dtype=torch.int64, device=DEV)]
    binding.kd_topk_kl_fwd(p.H, p.W, p.idx, p.t, p.mask, p.T, *out, ws)
    return out


def _noalloc(p):
    out = [torch.full((p.N,), float("nan"), device=DEV), torch.full((p.N,), float("nan"), device=DEV),
           torch.full((1,), -1, dtype=torch.int64, device=DEV)]
    binding.kd_topk_kl_fwd_noalloc(p.H, p.W, p.idx, p.t, p.mask, p.T, *out)
    return out


def test_two_calls_in_a_row_match_the_workspace_forward():
    # a larger problem first, then a smaller one over the stale scratch; both entry
    # points run the same kernels in the same order, so the results agree bit for bit
    probs = [make_problem(1500, 256, 20000, 64, 1.3, seed=31, mask="frac", mask_frac=0.05,
                          garbage_masked=True, device=DEV),
             make_problem(300, 136, 1000, 16, 1.0, seed=32, mask="frac", mask_frac=0.1, device=DEV)]
    results = [(_noalloc(p), _regular(p)) for p in probs]
    torch.cuda.synchronize()
    assert binding.kd_get_status() == 0
    for (got, want), p in zip(results, probs):
        assert torch.equal(got[0], want[0]), "loss"
        assert torch.equal(got[1], want[1]), "lse"
        assert int(got[2].item()) == int(want[2].item()) == int(p.mask.sum().item())


SCRATCH_BYTES = 64 << 20


def _a256(x):
    return (x + 255) // 256 * 256


def _scratch_needed(N, V, K):
    # the forward's scratch as the header states it: sorted teacher pairs (8 K),
    # teacher entropy (4), (max, sum) partials (8 min(ceil(V / 256), 64)) and the
    # gathered logits (4 K) bytes per token, each region 256-byte aligned
    slots = min(-(-V // 256), 64)
    return _a256(N * K * 8) + _a256(N * 4) + _a256(N * slots * 8) + _a256(N * K * 4)


def _largest_n(V, K):
    n = SCRATCH_BYTES // (12 * K + 4 + 8 * min(-(-V // 256), 64))
    while _scratch_needed(n + 1, V, K) <= SCRATCH_BYTES:
        n += 1
    while _scratch_needed(n, V, K) > SCRATCH_BYTES:
        n -= 1
    return n


def test_largest_size_that_fits_runs_and_one_more_is_refused():
    D, V, K = 64, 512, 256
    n_max = _largest_n(V, K)
    assert 20000 < n_max < 23000
    p = make_problem(n_max, D, V, K, 1.0, seed=33, mask="frac", mask_frac=0.02, device=DEV)
    got, want = _noalloc(p), _regular(p)
    torch.cuda.synchronize()
    assert binding.kd_get_status() == 0
    assert torch.equal(got[0], want[0]) and torch.equal(got[1], want[1])
    lib = binding.lib()
    dummy = torch.zeros(16, dtype=torch.uint8, device=DEV)
    ptr = dummy.data_ptr()
    code = lib.kd_topk_kl_fwd_noalloc(ptr, ptr, ptr, ptr, None, n_max + 1, D, V, K,
                                      ctypes.c_float(1.0), ptr, ptr, ptr, None)
    assert code == 4  # KD_ERR_WORKSPACE, nothing launched


def test_size_beyond_the_fixed_scratch_is_refused():
    lib = binding.lib()
    dummy = torch.zeros(16, dtype=torch.uint8, device=DEV)
    ptr = dummy.data_ptr()
    # 200K tokens at K = 64 over a 201,088 vocabulary needs ~257 MB of forward scratch
    code = lib.kd_topk_kl_fwd_noalloc(ptr, ptr, ptr, ptr, None, 200000, 2880, 201088, 64,
                                      ctypes.c_float(1.0), ptr, ptr, ptr, None)
    assert code == 4  # KD_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert binding.kd_get_status() == 0
