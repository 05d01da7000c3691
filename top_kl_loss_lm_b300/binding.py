"""ctypes binding of libkdtopk (include/kd_topk_kl.h), same names as the C ABI.

This layer only marshals: it checks dtypes, shapes and devices of torch
tensors, passes their data pointers and the current CUDA stream, and turns a
non-zero kd_status into ``KdError``. Every step of the loss runs in the CUDA
library; there is no fallback. If ``libkdtopk.so`` is missing the first call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

__all__ = [
    "KdError", "lib", "library_path",
    "kd_topk_kl_workspace_size", "kd_topk_kl_fwd", "kd_topk_kl_bwd", "kd_topk_kl_fwd_noalloc",
    "kd_topk_kl_logits_workspace_size", "kd_topk_kl_logits", "kd_topk_kl_mean_grad",
    "kd_topk_kl_shard_workspace_size", "kd_topk_kl_fwd_shard", "kd_topk_kl_shard_merge",
    "kd_topk_kl_bwd_shard", "call_device",
    "kd_teacher_topk_workspace_size", "kd_teacher_topk",
    "kd_get_status", "kd_status_string",
    "kd_debug_gemm_bf16", "kd_debug_wait_timeout", "kd_debug_schedule",
    "kd_debug_profile", "kd_debug_profile_read", "PROFILE_CATEGORIES",
    "STATUS",
]

STATUS = {
    0: "KD_OK", 1: "KD_ERR_ARG", 2: "KD_ERR_ALIGN", 3: "KD_ERR_UNSUPPORTED",
    4: "KD_ERR_WORKSPACE", 5: "KD_ERR_INDEX", 6: "KD_ERR_TIMEOUT", 7: "KD_ERR_CUDA",
    8: "KD_ERR_BOUNDS",
}

_LIB = None
_LOCK = threading.Lock()


def library_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkdtopk.so")


class KdError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {STATUS.get(self.code, self.code)} ({kd_status_string(self.code)})")


def lib() -> ctypes.CDLL:
    """Load libkdtopk.so (once) and declare its signatures."""
    global _LIB
    if _LIB is not None:
        return _LIB
    with _LOCK:
        if _LIB is not None:
            return _LIB
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with `python -m top_kl_loss_lm_b300.build`")
        L = ctypes.CDLL(path)
        vp, i64, i32, f32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.kd_topk_kl_workspace_size.argtypes = [i64, i32, i32, i32, i64]
        L.kd_topk_kl_workspace_size.restype = sz
        L.kd_topk_kl_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, f32, vp, vp, vp, vp, sz, vp]
        L.kd_topk_kl_fwd.restype = i32
        L.kd_topk_kl_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, f32, i64, i32,
                                     vp, vp, vp, sz, vp]
        L.kd_topk_kl_bwd.restype = i32
        L.kd_topk_kl_fwd_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i32, i32, i32, f32, vp, vp, vp, vp]
        L.kd_topk_kl_fwd_noalloc.restype = i32
        L.kd_topk_kl_mean_grad.argtypes = [vp, vp, i64, vp, vp, vp, vp]
        L.kd_topk_kl_mean_grad.restype = i32
        L.kd_topk_kl_shard_workspace_size.argtypes = [i64, i32, i32, i32, i64]
        L.kd_topk_kl_shard_workspace_size.restype = sz
        L.kd_topk_kl_fwd_shard.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, i64, i32, i32, f32, vp,
                                           vp, vp, vp, sz, vp]
        L.kd_topk_kl_fwd_shard.restype = i32
        L.kd_topk_kl_shard_merge.argtypes = [vp, i32, vp, vp, i64, f32, vp, vp, vp]
        L.kd_topk_kl_shard_merge.restype = i32
        L.kd_topk_kl_bwd_shard.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp, vp, vp, i64, i32, i32,
                                           f32, i64, i32, i32, vp, vp, vp, sz, vp]
        L.kd_topk_kl_bwd_shard.restype = i32
        L.kd_topk_kl_logits_workspace_size.argtypes = [i64, i32]
        L.kd_topk_kl_logits_workspace_size.restype = sz
        L.kd_topk_kl_logits.argtypes = [vp, i64, vp, vp, vp, vp, i64, i32, i32, f32, vp, vp, vp, vp,
                                        i64, vp, sz, vp]
        L.kd_topk_kl_logits.restype = i32
        L.kd_teacher_topk_workspace_size.argtypes = [i64, i32, i32, i32]
        L.kd_teacher_topk_workspace_size.restype = sz
        L.kd_teacher_topk.argtypes = [vp, vp, i64, i32, i32, i32, vp, vp, vp, sz, vp]
        L.kd_teacher_topk.restype = i32
        L.kd_get_status.argtypes = [vp]
        L.kd_get_status.restype = i32
        L.kd_status_string.argtypes = [i32]
        L.kd_status_string.restype = ctypes.c_char_p
        L.kd_debug_gemm_bf16.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp]
        L.kd_debug_gemm_bf16.restype = i32
        L.kd_debug_wait_timeout.argtypes = [ctypes.c_uint64, vp]
        L.kd_debug_wait_timeout.restype = i32
        L.kd_debug_schedule.argtypes = [i32, i64, i64, i64, i32, i32, vp, vp]
        L.kd_debug_schedule.restype = i32
        L.kd_debug_profile.argtypes = [i32]
        L.kd_debug_profile.restype = i32
        L.kd_debug_profile_read.argtypes = [vp, vp, i32]
        L.kd_debug_profile_read.restype = i32
        _LIB = L
        return L


def _stream(stream, device=None) -> Optional[int]:
    """The stream handle to launch on: the given one, else the current stream of
    `device` (the device the call's tensors live on)."""
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def call_device(*tensors) -> torch.device:
    """The one CUDA device every given tensor (None entries skipped) lives on.

    The library launches on the CURRENT device and refuses memory of any other,
    so each wrapper makes this device current around its call."""
    dev = None
    for t in tensors:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError(f"tensor on {t.device}: the library needs CUDA tensors")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"tensors on different devices ({dev} and {t.device})")
    if dev is None:
        raise ValueError("no tensor given")
    return dev


def _ptr(t: Optional[torch.Tensor], dtype, shape, name: str, device=None):
    if t is None:
        return None
    if t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if not t.is_cuda or (device is not None and t.device != device):
        raise ValueError(f"{name}: must be on {device or 'a CUDA device'}")
    return t.data_ptr()


def _check(code: int, where: str):
    if code != 0:
        raise KdError(code, where)


def kd_status_string(code: int) -> str:
    return lib().kd_status_string(int(code)).decode()


def kd_topk_kl_workspace_size(N: int, D: int, V: int, K: int, chunk_tokens: int = 0) -> int:
    return int(lib().kd_topk_kl_workspace_size(N, D, V, K, chunk_tokens))


def kd_topk_kl_fwd(H, W, topk_idx, topk_logit, mask, T: float, loss, lse, n_valid, ws, stream=None):
    """Forward into caller-owned tensors (see kd_topk_kl_fwd in the header)."""
    N, D = H.shape
    V = W.shape[0]
    K = topk_idx.shape[1]
    dev = call_device(H, W, topk_idx, topk_logit, mask, loss, lse, n_valid, ws)
    args = (
        _ptr(H, torch.bfloat16, (N, D), "H", dev), _ptr(W, torch.bfloat16, (V, D), "W", dev),
        _ptr(topk_idx, torch.int32, (N, K), "topk_idx", dev),
        _ptr(topk_logit, torch.float32, (N, K), "topk_logit", dev),
        _ptr(mask, torch.uint8, (N,), "mask", dev),
        N, D, V, K, float(T),
        _ptr(loss, torch.float32, (N,), "loss", dev), _ptr(lse, torch.float32, (N,), "lse", dev),
        _ptr(n_valid, torch.int64, (1,), "n_valid", dev),
        _ptr(ws, torch.uint8, (ws.numel(),), "ws", dev), ws.numel(), _stream(stream, dev),
    )
    with torch.cuda.device(dev):
        _check(lib().kd_topk_kl_fwd(*args), "kd_topk_kl_fwd")


def kd_topk_kl_fwd_noalloc(H, W, topk_idx, topk_logit, mask, T: float, loss, lse, n_valid,
                           stream=None):
    """Forward that needs no workspace: the library uses its own fixed device scratch.

    For callers that cannot allocate device memory (see kd_topk_kl_fwd_noalloc in
    the header for the size limit and the sharing rules).
    """
    N, D = H.shape
    V = W.shape[0]
    K = topk_idx.shape[1]
    dev = call_device(H, W, topk_idx, topk_logit, mask, loss, lse, n_valid)
    args = (
        _ptr(H, torch.bfloat16, (N, D), "H", dev), _ptr(W, torch.bfloat16, (V, D), "W", dev),
        _ptr(topk_idx, torch.int32, (N, K), "topk_idx", dev),
        _ptr(topk_logit, torch.float32, (N, K), "topk_logit", dev),
        _ptr(mask, torch.uint8, (N,), "mask", dev),
        N, D, V, K, float(T),
        _ptr(loss, torch.float32, (N,), "loss", dev), _ptr(lse, torch.float32, (N,), "lse", dev),
        _ptr(n_valid, torch.int64, (1,), "n_valid", dev), _stream(stream, dev),
    )
    with torch.cuda.device(dev):
        _check(lib().kd_topk_kl_fwd_noalloc(*args), "kd_topk_kl_fwd_noalloc")


def kd_topk_kl_bwd(H, W, topk_idx, topk_logit, mask, lse, dloss, T: float, chunk_tokens: int,
                   accumulate_dW: bool, dH, dW, ws, stream=None):
    """Backward into caller-owned dH (bf16) and dW (fp32)."""
    N, D = H.shape
    V = W.shape[0]
    K = topk_idx.shape[1]
    dev = call_device(H, W, topk_idx, topk_logit, mask, lse, dloss, dH, dW, ws)
    args = (
        _ptr(H, torch.bfloat16, (N, D), "H", dev), _ptr(W, torch.bfloat16, (V, D), "W", dev),
        _ptr(topk_idx, torch.int32, (N, K), "topk_idx", dev),
        _ptr(topk_logit, torch.float32, (N, K), "topk_logit", dev),
        _ptr(mask, torch.uint8, (N,), "mask", dev),
        _ptr(lse, torch.float32, (N,), "lse", dev), _ptr(dloss, torch.float32, (N,), "dloss", dev),
        N, D, V, K, float(T), int(chunk_tokens), 1 if accumulate_dW else 0,
        _ptr(dH, torch.bfloat16, (N, D), "dH", dev), _ptr(dW, torch.float32, (V, D), "dW", dev),
        _ptr(ws, torch.uint8, (ws.numel(),), "ws", dev), ws.numel(), _stream(stream, dev),
    )
    with torch.cuda.device(dev):
        _check(lib().kd_topk_kl_bwd(*args), "kd_topk_kl_bwd")


def kd_topk_kl_mean_grad(loss, mask, n_valid, dloss=None, loss_sum=None, stream=None):
    """dloss = mask / n_valid (n_valid read on the device) and loss_sum = sum(loss), fp64."""
    N = loss.shape[0]
    dev = call_device(loss, mask, n_valid, dloss, loss_sum)
    args = (
        _ptr(loss, torch.float32, (N,), "loss", dev), _ptr(mask, torch.uint8, (N,), "mask", dev), N,
        _ptr(n_valid, torch.int64, (1,), "n_valid", dev), _ptr(dloss, torch.float32, (N,), "dloss", dev),
        _ptr(loss_sum, torch.float64, (1,), "loss_sum", dev), _stream(stream, dev),
    )
    with torch.cuda.device(dev):
        _check(lib().kd_topk_kl_mean_grad(*args), "kd_topk_kl_mean_grad")


def kd_topk_kl_shard_workspace_size(N: int, D: int, V_shard: int, K: int, chunk_tokens: int = 0) -> int:
    return int(lib().kd_topk_kl_shard_workspace_size(N, D, V_shard, K, chunk_tokens))


def kd_topk_kl_fwd_shard(H, W_shard, v0: int, V: int, topk_idx, topk_logit, mask, T: float, parts,
                         ent, n_valid, ws, stream=None):
    """Forward of the vocabulary shard [v0, v0 + W_shard.shape[0]) of V: parts [N, 2], ent [N]."""
    N, D = H.shape
    Vs = W_shard.shape[0]
    K = topk_idx.shape[1]
    dev = call_device(H, W_shard, topk_idx, topk_logit, mask, parts, ent, n_valid, ws)
    args = (
        _ptr(H, torch.bfloat16, (N, D), "H", dev), _ptr(W_shard, torch.bfloat16, (Vs, D), "W_shard", dev),
        int(v0), Vs, int(V),
        _ptr(topk_idx, torch.int32, (N, K), "topk_idx", dev),
        _ptr(topk_logit, torch.float32, (N, K), "topk_logit", dev),
        _ptr(mask, torch.uint8, (N,), "mask", dev), N, D, K, float(T),
        _ptr(parts, torch.float32, (N, 2), "parts", dev), _ptr(ent, torch.float32, (N,), "ent", dev),
        _ptr(n_valid, torch.int64, (1,), "n_valid", dev),
        _ptr(ws, torch.uint8, (ws.numel(),), "ws", dev), ws.numel(), _stream(stream, dev),
    )
    with torch.cuda.device(dev):
        _check(lib().kd_topk_kl_fwd_shard(*args), "kd_topk_kl_fwd_shard")


def kd_topk_kl_shard_merge(parts, ent, mask, T: float, loss, lse, stream=None):
    """loss, lse [N] from the shards' parts stacked as [R, N, 2] (shard order)."""
    R, N = parts.shape[0], parts.shape[1]
    dev = call_device(parts, ent, mask, loss, lse)
    args = (
        _ptr(parts, torch.float32, (R, N, 2), "parts", dev), R,
        _ptr(ent, torch.float32, (N,), "ent", dev), _ptr(mask, torch.uint8, (N,), "mask", dev), N,
        float(T), _ptr(loss, torch.float32, (N,), "loss", dev), _ptr(lse, torch.float32, (N,), "lse", dev),
        _stream(stream, dev),
    )
    with torch.cuda.device(dev):
        _check(lib().kd_topk_kl_shard_merge(*args), "kd_topk_kl_shard_merge")


def kd_topk_kl_bwd_shard(H, W_shard, v0: int, V: int, topk_idx, topk_logit, mask, lse, dloss,
                         T: float, chunk_tokens: int, accumulate_dW: bool, accumulate_dH: bool, dH,
                         dW_shard, ws, stream=None):
    """The shard's gradients: dH [N, D] fp32 (its part of the sum over shards), dW_shard fp32."""
    N, D = H.shape
    Vs = W_shard.shape[0]
    K = topk_idx.shape[1]
    dev = call_device(H, W_shard, topk_idx, topk_logit, mask, lse, dloss, dH, dW_shard, ws)
    args = (
        _ptr(H, torch.bfloat16, (N, D), "H", dev), _ptr(W_shard, torch.bfloat16, (Vs, D), "W_shard", dev),
        int(v0), Vs, int(V),
        _ptr(topk_idx, torch.int32, (N, K), "topk_idx", dev),
        _ptr(topk_logit, torch.float32, (N, K), "topk_logit", dev),
        _ptr(mask, torch.uint8, (N,), "mask", dev),
        _ptr(lse, torch.float32, (N,), "lse", dev), _ptr(dloss, torch.float32, (N,), "dloss", dev),
        N, D, K, float(T), int(chunk_tokens), 1 if accumulate_dW else 0, 1 if accumulate_dH else 0,
        _ptr(dH, torch.float32, (N, D), "dH", dev), _ptr(dW_shard, torch.float32, (Vs, D), "dW_shard", dev),
        _ptr(ws, torch.uint8, (ws.numel(),), "ws", dev), ws.numel(), _stream(stream, dev),
    )
    with torch.cuda.device(dev):
        _check(lib().kd_topk_kl_bwd_shard(*args), "kd_topk_kl_bwd_shard")


def kd_topk_kl_logits_workspace_size(N: int, K: int) -> int:
    return int(lib().kd_topk_kl_logits_workspace_size(N, K))


def _rows_ptr(t: torch.Tensor, name: str, N: int, V: int, device):
    """Data pointer and row stride of an N x V bf16 matrix whose rows are contiguous."""
    if t.dtype != torch.bfloat16 or tuple(t.shape) != (N, V):
        raise ValueError(f"{name}: expected bfloat16 of shape {(N, V)}, got {t.dtype} {tuple(t.shape)}")
    if t.stride(1) != 1 or (N > 1 and t.stride(0) < V):
        raise ValueError(f"{name}: rows must be contiguous")
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name}: must be on {device}")
    return t.data_ptr(), (t.stride(0) if N > 1 else V)


def kd_topk_kl_logits(Z, topk_idx, topk_logit, mask, T: float, loss, lse, n_valid, ws,
                      dloss=None, dZ=None, stream=None):
    """Loss (and dZ when dloss and dZ are given) from materialised bf16 logits Z [N x V]."""
    N, V = Z.shape
    K = topk_idx.shape[1]
    dev = call_device(Z, topk_idx, topk_logit, mask, loss, lse, n_valid, ws, dloss, dZ)
    zp, ldz = _rows_ptr(Z, "Z", N, V, dev)
    dp, lddz = (None, 0) if dZ is None else _rows_ptr(dZ, "dZ", N, V, dev)
    args = (
        zp, ldz, _ptr(topk_idx, torch.int32, (N, K), "topk_idx", dev),
        _ptr(topk_logit, torch.float32, (N, K), "topk_logit", dev),
        _ptr(mask, torch.uint8, (N,), "mask", dev),
        _ptr(dloss, torch.float32, (N,), "dloss", dev),
        N, V, K, float(T),
        _ptr(loss, torch.float32, (N,), "loss", dev), _ptr(lse, torch.float32, (N,), "lse", dev),
        _ptr(n_valid, torch.int64, (1,), "n_valid", dev), dp, lddz,
        _ptr(ws, torch.uint8, (ws.numel(),), "ws", dev), ws.numel(), _stream(stream, dev),
    )
    with torch.cuda.device(dev):
        _check(lib().kd_topk_kl_logits(*args), "kd_topk_kl_logits")


def kd_teacher_topk_workspace_size(N: int, D: int, V: int, K: int) -> int:
    return int(lib().kd_teacher_topk_workspace_size(N, D, V, K))


def kd_teacher_topk(H, W, topk_idx, topk_logit, ws, stream=None):
    """The teacher's top-K cache (ids int32, logits fp32) of H W^T into caller tensors."""
    N, D = H.shape
    V = W.shape[0]
    K = topk_idx.shape[1]
    dev = call_device(H, W, topk_idx, topk_logit, ws)
    args = (
        _ptr(H, torch.bfloat16, (N, D), "H", dev), _ptr(W, torch.bfloat16, (V, D), "W", dev),
        N, D, V, K,
        _ptr(topk_idx, torch.int32, (N, K), "topk_idx", dev),
        _ptr(topk_logit, torch.float32, (N, K), "topk_logit", dev),
        _ptr(ws, torch.uint8, (ws.numel(),), "ws", dev), ws.numel(), _stream(stream, dev),
    )
    with torch.cuda.device(dev):
        _check(lib().kd_teacher_topk(*args), "kd_teacher_topk")


def kd_get_status(stream=None, device=None) -> int:
    """Synchronise the stream and return (and clear) the status word of `device`
    (default: the current device)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(lib().kd_get_status(_stream(stream, dev)))


def kd_debug_gemm_bf16(A, B, C, a_mn: bool, b_mn: bool, cta_pair: bool = True, stream=None):
    """C = A·B^T through the tcgen05 mainloop (see kd_topk_kl_testing.h)."""
    if a_mn:
        K, M = A.shape
    else:
        M, K = A.shape
    N = B.shape[1] if b_mn else B.shape[0]
    dev = call_device(A, B, C)
    _ptr(A, torch.bfloat16, tuple(A.shape), "A", dev)
    _ptr(B, torch.bfloat16, tuple(B.shape), "B", dev)
    _ptr(C, torch.float32, (M, N), "C", dev)
    with torch.cuda.device(dev):
        _check(lib().kd_debug_gemm_bf16(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                        int(a_mn), int(b_mn), int(cta_pair), _stream(stream, dev)),
               "kd_debug_gemm_bf16")


def kd_debug_wait_timeout(timeout_ns: int, stream=None):
    _check(lib().kd_debug_wait_timeout(int(timeout_ns), _stream(stream)), "kd_debug_wait_timeout")


def kd_debug_schedule(kind: int, rows: int, cols: int, depth: int, grid_units: int,
                      tile_rows: int = 256, with_counts=True):
    """Host-only: the work schedule as (info dict, per-(m, n, k-block) visit counts or None)."""
    import numpy as np
    info = np.zeros(8, dtype=np.int64)
    code = lib().kd_debug_schedule(kind, rows, cols, depth, grid_units, tile_rows, None,
                                   info.ctypes.data)
    _check(code, "kd_debug_schedule")
    counts = None
    if with_counts:
        MB, NB, KB = int(info[2]), int(info[3]), int(info[4])
        counts = np.zeros(MB * NB * KB, dtype=np.int32)
        info2 = np.zeros(8, dtype=np.int64)
        _check(lib().kd_debug_schedule(kind, rows, cols, depth, grid_units, tile_rows,
                                       counts.ctypes.data, info2.ctypes.data), "kd_debug_schedule")
        counts = counts.reshape(MB, NB, KB)
    keys = ["units", "grid", "MB", "NB", "KB", "BN", "max_slots", "k_splits"]
    return {k: int(v) for k, v in zip(keys, info)}, counts


PROFILE_CATEGORIES = ["prep", "fwd_gemm", "combine", "dz_gemm", "dh_gemm", "dh_sum", "dw_gemm",
                      "logits", "topk_gemm", "topk_select", "transpose"]


def kd_debug_profile(enable: bool):
    _check(lib().kd_debug_profile(1 if enable else 0), "kd_debug_profile")


def kd_debug_profile_read():
    """{category: (total_ms, launches)} for the records since kd_debug_profile(True)."""
    import numpy as np
    n = len(PROFILE_CATEGORIES)
    ms = np.zeros(n, dtype=np.float64)
    cnt = np.zeros(n, dtype=np.int64)
    _check(lib().kd_debug_profile_read(ms.ctypes.data, cnt.ctypes.data, n), "kd_debug_profile_read")
    return {c: (float(ms[i]), int(cnt[i])) for i, c in enumerate(PROFILE_CATEGORIES)}
