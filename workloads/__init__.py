"""Seeded synthetic inputs for the fused top-K KL distillation head.

This module only draws random numbers and lays them out. It holds none of the
loss arithmetic: the CPU oracle (``oracle/``) and the CUDA library both take
what it returns as plain inputs.

Shapes and distributions follow the workloads named for the method's output
head (gpt-oss-style vocabulary V=201,088, hidden D=2,880, cached teacher top-K):

* ``H ~ N(0, 1)`` and ``W ~ N(0, 1/D)`` drawn in fp32, rounded to bf16.
* Teacher top-K indices: K distinct token ids per row, uniform in [0, V).
* Teacher top-K logits, sorted descending per row, either ``8 * N(0, 1)``
  (``"normal8"``) or ``N(0, 4) + Gumbel(0, 1)`` (``"gumbel"``).
* Mask: all rows, an exact fraction chosen without replacement, or packed
  documents whose last position and trailing padding are masked.

The teacher cache stands in for the offline top-K cache the method trains
against (Efficient Knowledge Distillation for LLMs: Offline Top-K Logits and a
Fused Chunked KL Loss, abstract; blog "Two systems changes", offline
distillation paragraph). No dataset, model or checkpoint is involved.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

__all__ = ["Problem", "make_problem", "CONFIGS", "config_problem", "packed_mask",
           "mean_upstream_grad"]


@dataclasses.dataclass
class Problem:
    """One synthetic head problem. Tensors live on ``device``."""
    H: torch.Tensor          # N x D bf16, row-major
    W: torch.Tensor          # V x D bf16, row-major (lm-head weight)
    idx: torch.Tensor        # N x K int32 teacher token ids (cache order)
    t: torch.Tensor          # N x K fp32 teacher logits (cache order)
    mask: torch.Tensor       # N uint8, 1 = row counted
    T: float
    name: str = ""

    @property
    def N(self) -> int:
        return self.H.shape[0]

    @property
    def D(self) -> int:
        return self.H.shape[1]

    @property
    def V(self) -> int:
        return self.W.shape[0]

    @property
    def K(self) -> int:
        return self.idx.shape[1]


def _gen(seed: int, offset: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000003 + int(offset))
    return g


def _distinct_indices(N: int, V: int, K: int, g: torch.Generator, device) -> torch.Tensor:
    """K distinct ids per row, uniform over [0, V), in random (cache) order."""
    if K > V:
        raise ValueError("K must not exceed V")
    if K * K > V:
        # many collisions expected: a random permutation prefix per row
        keys = torch.rand(N, V, generator=g, device=device)
        return keys.argsort(dim=1)[:, :K].to(torch.int32).contiguous()
    idx = torch.randint(0, V, (N, K), generator=g, device=device, dtype=torch.int64)
    for _ in range(1000):
        s = idx.sort(dim=1).values
        dup = (s[:, 1:] == s[:, :-1]).any(dim=1)
        nd = int(dup.sum().item())
        if nd == 0:
            return idx.to(torch.int32).contiguous()
        idx[dup] = torch.randint(0, V, (nd, K), generator=g, device=device, dtype=torch.int64)
    raise RuntimeError("could not draw distinct indices")


def _teacher_logits(N: int, K: int, dist: str, g: torch.Generator, device) -> torch.Tensor:
    if dist == "normal8":
        x = 8.0 * torch.randn(N, K, generator=g, device=device)
    elif dist == "gumbel":
        u = torch.rand(N, K, generator=g, device=device).clamp_(1e-12, 1.0 - 1e-7)
        x = 2.0 * torch.randn(N, K, generator=g, device=device) - torch.log(-torch.log(u))
    else:
        raise ValueError(dist)
    return x.sort(dim=1, descending=True).values.to(torch.float32).contiguous()


def packed_mask(N: int, g: torch.Generator, lo: int = 256, hi: int = 4096) -> torch.Tensor:
    """Mask for documents of length U[lo, hi] packed whole, in order, into N slots.

    Each document's last position (the boundary) is masked; the slots left
    after the last document that fits are padding and are masked too.
    Returned on the CPU as uint8.
    """
    m = torch.zeros(N, dtype=torch.uint8)
    pos = 0
    while True:
        L = int(torch.randint(lo, hi + 1, (1,), generator=g).item())
        if pos + L > N:
            break
        m[pos:pos + L - 1] = 1
        pos += L
    return m


def make_problem(N: int, D: int, V: int, K: int, T: float = 1.0, *, seed: int = 0,
                 teacher: str = "gumbel", mask: str = "none", mask_frac: float = 0.0,
                 garbage_masked: bool = False, device="cpu", name: str = "") -> Problem:
    """Draw one problem. ``mask`` is ``"none"``, ``"frac"`` or ``"packed"``."""
    device = torch.device(device)
    gH, gW, gI, gT, gM = (_gen(seed, o, device) for o in (1, 2, 3, 4, 5))
    H = torch.randn(N, D, generator=gH, device=device).to(torch.bfloat16).contiguous()
    W = (torch.randn(V, D, generator=gW, device=device) * (1.0 / D) ** 0.5).to(torch.bfloat16).contiguous()
    idx = _distinct_indices(N, V, K, gI, device)
    t = _teacher_logits(N, K, teacher, gT, device)
    if mask == "none":
        m = torch.ones(N, dtype=torch.uint8, device=device)
    elif mask == "frac":
        nm = int(round(mask_frac * N))
        gm = _gen(seed, 6, "cpu")
        perm = torch.randperm(N, generator=gm)[:nm]
        m = torch.ones(N, dtype=torch.uint8)
        m[perm] = 0
        m = m.to(device)
    elif mask == "packed":
        m = packed_mask(N, _gen(seed, 6, "cpu")).to(device)
    else:
        raise ValueError(mask)
    if garbage_masked:
        bad = m == 0
        nb = int(bad.sum().item())
        if nb:
            # masked rows carry junk that must never be read
            junk = torch.randint(-5 * V, 5 * V, (nb, K), generator=gM, device=device, dtype=torch.int64)
            idx[bad] = junk.to(torch.int32)
            t[bad] = float("nan")
    return Problem(H=H, W=W, idx=idx, t=t, mask=m.contiguous(), T=float(T), name=name)


def mean_upstream_grad(mask: torch.Tensor) -> torch.Tensor:
    """Upstream gradient of the mean over counted rows: 1/n_valid there, 0 elsewhere."""
    nv = int(mask.sum().item())
    g = mask.to(torch.float32)
    return g / nv if nv > 0 else g


# Named workloads: (N, D, V, K, T, teacher, mask, mask_frac, garbage_masked)
CONFIGS = {
    "tiny": dict(N=256, D=256, V=4096, K=32, T=1.0, teacher="normal8", mask="none"),
    "gptoss_4k": dict(N=4096, D=2880, V=201088, K=64, T=1.0, teacher="gumbel", mask="frac",
                      mask_frac=0.02),
    "gptoss_32k": dict(N=32768, D=2880, V=201088, K=64, T=1.0, teacher="gumbel", mask="frac",
                       mask_frac=0.02),
    # small profiling case: same D and K as the gpt-oss head, W still larger than L2
    "profile_small": dict(N=4096, D=2880, V=32768, K=64, T=1.0, teacher="gumbel", mask="frac",
                          mask_frac=0.02),
    # profiling case for DRAM traffic: the gpt-oss head's D, K and launch sizes (4,096
    # rows per forward / dZ / dH launch, 8,192 tokens per dW launch: one store, one add)
    # over a third of its vocabulary, ~3 GB on the device
    "profile_medium": dict(N=16384, D=2880, V=65536, K=64, T=1.0, teacher="gumbel", mask="frac",
                           mask_frac=0.02),
    "packed_qwen": dict(N=32768, D=4096, V=151936, K=64, T=1.0, teacher="gumbel", mask="packed",
                        garbage_masked=True),
}


def config_problem(name: str, *, seed: int = 0, device="cpu", N: Optional[int] = None,
                   K: Optional[int] = None, T: Optional[float] = None) -> Problem:
    c = dict(CONFIGS[name])
    if N is not None:
        c["N"] = N
    if K is not None:
        c["K"] = K
    if T is not None:
        c["T"] = T
    return make_problem(seed=seed, device=device, name=name, **c)
