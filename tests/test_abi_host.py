"""Host-side checks of libkdtopk that need no GPU: the library loads and exports
every symbol its headers declare, argument errors come back before any CUDA
call, the workspace grows linearly in N (never N x V), and the work schedule
visits every (row block, column tile, k-block) exactly once.
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from top_kl_loss_lm_b300 import binding
from top_kl_loss_lm_b300.build import build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    build_library()
    return binding.lib()


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(INCLUDE)):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(INCLUDE, fn)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(kd_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert "kd_topk_kl_fwd" in names and "kd_topk_kl_bwd" in names and "kd_get_status" in names
    for n in names:
        assert hasattr(lib, n), n
        ctypes.cast(getattr(lib, n), ctypes.c_void_p)


def test_status_strings(lib):
    for code in range(9):
        s = binding.kd_status_string(code)
        assert isinstance(s, str) and s
    assert binding.kd_status_string(0) == "ok"


def _fwd_raw(lib, H=16, W=16, idx=16, t=16, N=4, D=8, V=16, K=2, T=1.0, ws=256):
    return lib.kd_topk_kl_fwd(H, W, idx, t, None, N, D, V, K, ctypes.c_float(T), 16, 16, 16, ws,
                              1 << 20, None)


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers: host-only argument checks")
def test_argument_errors_without_gpu(lib):
    assert _fwd_raw(lib, K=0) == 1
    assert _fwd_raw(lib, K=257) == 1
    assert _fwd_raw(lib, D=12) == 1
    assert _fwd_raw(lib, T=0.0) == 1
    assert _fwd_raw(lib, T=float("nan")) == 1
    assert _fwd_raw(lib, N=-1) == 1
    assert _fwd_raw(lib, H=0) == 1
    assert _fwd_raw(lib, H=8) == 2
    assert _fwd_raw(lib, idx=2) == 2
    assert _fwd_raw(lib, ws=16) == 2
    # arguments are valid: the call reaches CUDA, finds no device, and says so
    assert _fwd_raw(lib) in (3, 7)
    assert lib.kd_get_status(None) in (3, 7)


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake pointers: host-only argument checks")
def test_shard_and_mean_grad_argument_errors_without_gpu(lib):
    f = ctypes.c_float(1.0)

    def fwd_shard(v0, Vs, V=16, parts=16):
        return lib.kd_topk_kl_fwd_shard(16, 16, v0, Vs, V, 16, 16, None, 4, 8, 2, f, parts, 16, 16, 256,
                                        1 << 20, None)
    assert fwd_shard(8, 9) == 1      # the shard runs past V
    assert fwd_shard(-1, 4) == 1
    assert fwd_shard(0, 0) == 1
    assert fwd_shard(0, 16, parts=4) == 2  # parts must be 8-byte aligned
    assert fwd_shard(4, 8) in (3, 7)       # valid: reaches CUDA, finds no device
    assert lib.kd_topk_kl_shard_merge(16, 0, 16, None, 4, f, 16, 16, None) == 1   # R = 0
    assert lib.kd_topk_kl_shard_merge(16, 2, 16, None, 4, ctypes.c_float(0.0), 16, 16, None) == 1
    assert lib.kd_topk_kl_mean_grad(16, None, 4, None, 16, 16, None) == 1         # no n_valid
    assert lib.kd_topk_kl_mean_grad(16, None, 4, 16, None, None, None) == 1       # no output
    assert lib.kd_topk_kl_bwd_shard(16, 16, 12, 8, 16, 16, 16, None, 16, 16, 4, 8, 2, f, 0, 0, 0,
                                    16, 16, 256, 1 << 20, None) == 1             # past V


def test_workspace_linear_in_tokens(lib):
    D, V, K = 2880, 201088, 64
    Ns = [4096, 16384, 65536, 131072, 262144]
    ws = [binding.kd_topk_kl_workspace_size(n, D, V, K, 4096) for n in Ns]
    assert all(w > 0 for w in ws)
    # per-token growth is a small constant once N holds two chunks; the only
    # vocabulary-sized part (two 4096-token dZ chunks, one per dW group slot) is fixed
    slopes = [(ws[i + 1] - ws[i]) / (Ns[i + 1] - Ns[i]) for i in range(1, len(Ns) - 1)]
    assert max(slopes) < 2 * 1024 and max(slopes) - min(slopes) < 64
    for n, w in zip(Ns, ws):
        # two dZ chunks, the transposed copies of W (V x D bf16) and of a dW
        # group's H (2 chunks x D bf16) and the dH split partials (at most 8 x
        # chunk x D fp32) are vocabulary- or chunk-sized, all fixed in N
        fixed = 2 * 4096 * V * 2 + V * D * 2 + 2 * 4096 * D * 2 + 8 * 4096 * D * 4
        assert w < fixed + n * 2048
        if n >= 65536:
            assert w < n * V * 2 / 3  # well below one dense N x V bf16 grid
    assert binding.kd_topk_kl_workspace_size(0, D, V, K, 0) > 0
    assert binding.kd_topk_kl_workspace_size(16, 12, V, K, 0) == 0
    assert binding.kd_topk_kl_workspace_size(16, D, V, 0, 0) == 0


SHAPES = [
    (0, 256, 4096, 256),        # tiny forward
    (0, 300, 1000, 136),        # ragged forward
    (0, 4096, 201088, 2880),    # gpt-oss head forward
    (0, 8192, 151936, 4096),
    (1, 4096, 2880, 201088),    # dH of one 4096-token chunk
    (1, 300, 136, 1000),
    (2, 201088, 2880, 4096),    # dW of one chunk
    (2, 201088, 2880, 8192),    # dW of a two-chunk group
    (2, 1000, 136, 300),
]


@pytest.mark.parametrize("kind,rows,cols,depth", SHAPES)
@pytest.mark.parametrize("sms,tile_rows", [(74, 256), (66, 256), (148, 128), (7, 256)])
def test_schedule_visits_each_tile_once(lib, kind, rows, cols, depth, sms, tile_rows):
    info, counts = binding.kd_debug_schedule(kind, rows, cols, depth, sms, tile_rows)
    assert counts.min() == 1 and counts.max() == 1
    assert info["grid"] == min(sms, info["units"])
    if kind == 0:
        assert info["max_slots"] <= min(64, info["NB"])
        assert info["KB"] == -(-depth // 64)


def test_forward_schedule_is_balanced_on_gptoss_shapes(lib):
    for N in (4096, 16384, 32768, 65536, 262144):
        info, _ = binding.kd_debug_schedule(0, N, 201088, 2880, 74, 256, with_counts=False)
        assert info["units"] % 74 == 0, (N, info)
        info, _ = binding.kd_debug_schedule(0, N, 201088, 2880, 148, 128, with_counts=False)
        assert info["units"] % 148 == 0, (N, info)


def test_dh_split_fills_the_last_wave(lib):
    info, _ = binding.kd_debug_schedule(1, 4096, 2880, 201088, 74, 256, with_counts=False)
    units = info["units"]
    assert info["k_splits"] > 1
    assert units / (-(-units // 74) * 74) > 0.95


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    # no CPU or library fallback: without libkdtopk.so every call raises
    monkeypatch.setattr(binding, "_LIB", None)
    monkeypatch.setattr(binding, "library_path", lambda: str(tmp_path / "libkdtopk.so"))
    with pytest.raises(RuntimeError, match="missing"):
        binding.kd_topk_kl_workspace_size(16, 8, 32, 2)
    with pytest.raises(RuntimeError, match="missing"):
        binding.lib()


def test_binding_refuses_host_tensors_and_mixed_devices():
    # the library launches on the current device and refuses other memory; the
    # binding therefore needs every tensor of a call on one CUDA device and makes
    # that device current around the call
    from types import SimpleNamespace
    N, D, V, K = 4, 8, 16, 2
    H = torch.zeros(N, D, dtype=torch.bfloat16)
    W = torch.zeros(V, D, dtype=torch.bfloat16)
    idx = torch.zeros(N, K, dtype=torch.int32)
    t = torch.zeros(N, K)
    out = [torch.zeros(N), torch.zeros(N), torch.zeros(1, dtype=torch.int64)]
    ws = torch.zeros(256, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensors"):
        binding.kd_topk_kl_fwd(H, W, idx, t, None, 1.0, *out, ws)
    with pytest.raises(ValueError, match="CUDA tensors"):
        binding.kd_topk_kl_fwd_noalloc(H, W, idx, t, None, 1.0, *out)
    a = SimpleNamespace(is_cuda=True, device=torch.device("cuda", 0))
    b = SimpleNamespace(is_cuda=True, device=torch.device("cuda", 1))
    assert binding.call_device(a, None, a) == torch.device("cuda", 0)
    with pytest.raises(ValueError, match="different devices"):
        binding.call_device(a, b)


def test_issued_width_factor():
    # a GEMM pays for its output columns in 256-wide MMA instructions: the hidden
    # size for dH and dW, the vocabulary for the forward and dZ
    import bench
    assert bench.issued_width_factor("dw_gemm", 2880, 201088) == 3072 / 2880
    assert bench.issued_width_factor("dh_gemm", 2880, 201088) == 3072 / 2880
    assert bench.issued_width_factor("dw_gemm", 4096, 151936) == 1.0
    assert bench.issued_width_factor("fwd_gemm", 2880, 201088) == 201216 / 201088
    assert bench.issued_width_factor("dz_gemm", 4096, 151936) == 152064 / 151936


def test_per_clock_fraction():
    # the same work per clock gives the same fraction on a slower-clocked box
    import bench
    peaks = {"clocks_under_load": {"sm_mhz_median": 1200.0}}
    same = bench.per_clock_fraction(1300.0, 1400.0, {"sm_mhz": 1200.0, "samples": 9}, peaks)
    assert abs(same - 1300.0 / 1400.0) < 1e-12
    slow = bench.per_clock_fraction(1300.0 * 1100 / 1200, 1400.0, {"sm_mhz": 1100.0, "samples": 9}, peaks)
    assert abs(slow - 1300.0 / 1400.0) < 1e-12
    assert bench.per_clock_fraction(1300.0, 1400.0, None, peaks) is None
    assert bench.per_clock_fraction(1300.0, 1400.0, {"sm_mhz": 1200.0, "samples": 9}, {}) is None
    assert bench.per_clock_fraction(1300.0, 1400.0, {"sm_mhz": 1200.0, "samples": 2}, peaks) is None
