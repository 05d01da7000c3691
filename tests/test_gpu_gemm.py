"""The tcgen05/TMA mainloop on its own, as a plain GEMM against torch.matmul in
fp32 on the same bf16 operands, for every operand layout: both K-major (the
logits, and dH = dZ W with W transposed), A MN-major with B K-major (dW = dZ^T H
with H transposed), B MN-major and both MN-major, in the CTA-pair form
(cta_group::2, 256-row tiles) the loss runs and in the single-CTA form.
"""
import pytest
import torch

from top_kl_loss_lm_b300 import binding

pytestmark = pytest.mark.gpu


def _ref(A, B, a_mn, b_mn):
    Af = A.float().T if a_mn else A.float()
    Bf = B.float() if b_mn else B.float().T
    return Af @ Bf


@pytest.mark.parametrize("cta_pair", [True, False])
@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (True, False), (False, True), (True, True)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 128), (200, 264, 136),
                                   (128, 240, 64), (1024, 2880, 1024), (384, 1000, 8)])
def test_gemm_matches_torch(a_mn, b_mn, M, N, K, cta_pair):
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N * 3 + K)
    A = torch.randn((K, M) if a_mn else (M, K), device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn((K, N) if b_mn else (N, K), device="cuda", generator=g).to(torch.bfloat16)
    C = torch.full((M, N), float("nan"), device="cuda")
    binding.kd_debug_gemm_bf16(A, B, C, a_mn, b_mn, cta_pair)
    torch.cuda.synchronize()
    assert binding.kd_get_status() == 0
    R = _ref(A, B, a_mn, b_mn)
    assert torch.isfinite(C).all()
    err = (C - R).abs().max().item() / R.abs().max().item()
    assert err < 1e-4, err
