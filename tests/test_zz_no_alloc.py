"""The allocation-free forward, kd_topk_kl_fwd_noalloc.

Some callers cannot allocate device memory: a plugin running inside a process
whose own allocator already holds the GPU's memory, or a hot path where a
cudaMalloc (which may synchronise the device) is not allowed. For them the
library keeps the forward's scratch in a fixed array of its own. This file
checks, through the C ABI, that two calls in a row give what the regular
forward gives with a caller workspace, and that a size beyond the fixed array
is refused before anything runs. It is collected last on purpose.
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
    # a larger problem first, then a smaller one over the stale scratch
    probs = [make_problem(1500, 256, 20000, 64, 1.3, seed=31, mask="frac", mask_frac=0.05,
                          garbage_masked=True, device=DEV),
             make_problem(300, 136, 1000, 16, 1.0, seed=32, mask="frac", mask_frac=0.1, device=DEV)]
    results = [(_noalloc(p), _regular(p)) for p in probs]
    torch.cuda.synchronize()
    assert binding.kd_get_status() == 0
    for (got, want), p in zip(results, probs):
        P.assert_rows_close(got[0].cpu().numpy(), want[0].cpu().numpy(), "loss")
        P.assert_rows_close(got[1].cpu().numpy(), want[1].cpu().numpy(), "lse")
        assert int(got[2].item()) == int(want[2].item()) == int(p.mask.sum().item())


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
