"""GB300-native paged KV-cache decode attention.

Python face of the C ABI in ``include/pkv.h`` (library
``_lib/libpkv_gb300.so``, built by ``_build.build_library``).  This module only
marshals arguments: it reads shapes from tensor metadata, hands raw device
pointers and the current CUDA stream to the library, and lets PyTorch own the
device memory (including the split-K workspace).  All computation happens in
the library's CUDA kernels; there is no CPU or PyTorch fallback, and a
missing library is an error.

    store_kvcache(k, v, k_cache, v_cache, slot_mapping)
    paged_attn_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out)

Layouts: k, v ``[N, Hkv, D]``; caches ``[NB, bs, Hkv, D]``; q, out
``[B, Hq, D]`` (all bf16, contiguous, on one CUDA device); slot_mapping int64
``[N]`` (-1 = skip); block_tables int32 ``[B, MBS]``; context_lens int32 ``[B]``.
"""

from __future__ import annotations

import ctypes
import os
import threading

from . import _build

__all__ = [
    "store_kvcache",
    "paged_attn_decode",
    "store_kvcache_fp8",
    "paged_prefill",
    "paged_attn_decode_fp8",
    "decode_workspace_bytes",
    "load_library",
    "library_path",
    "PkvError",
    "FLAG_BAD_SLOT",
    "FLAG_BAD_BLOCK",
    "FLAG_BAD_CONTEXT_LEN",
    "FLAG_TIMEOUT",
    "FLAG_V_RANGE",
]

FLAG_BAD_SLOT = 0x1
FLAG_BAD_BLOCK = 0x2
FLAG_BAD_CONTEXT_LEN = 0x4
FLAG_TIMEOUT = 0x8
FLAG_V_RANGE = 0x10  # paged_prefill: a V value beyond f16's range was clamped

_STATUS = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_UNSUPPORTED",
           3: "PKV_ERR_WORKSPACE", 4: "PKV_ERR_CUDA"}


class PkvError(RuntimeError):
    """A library call returned a non-OK status."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is missing; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                ctypes.c_float, ctypes.c_size_t)
        lib.pkv_store_kvcache.restype = i32
        lib.pkv_store_kvcache.argtypes = [P, P, P, P, P, i64, i32, i32, i64, i32, P, P]
        lib.pkv_decode_workspace_bytes.restype = sz
        lib.pkv_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32]
        lib.pkv_paged_attn_decode.restype = i32
        lib.pkv_paged_attn_decode.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i64, i32,
                                              f32, P, P, sz, i32, P, P]
        lib.pkv_store_kvcache_fp8.restype = i32
        lib.pkv_store_kvcache_fp8.argtypes = [P, P, P, P, P, i64, i32, i32, i64, i32, f32, f32, P, P]
        lib.pkv_paged_attn_decode_fp8.restype = i32
        lib.pkv_paged_attn_decode_fp8.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i64, i32,
                                                  f32, f32, f32, P, P, sz, i32, P, P]
        lib.pkv_paged_prefill.restype = i32
        lib.pkv_paged_prefill.argtypes = [P, P, P, P, i32, P, P, i32, i64, i32, i32, i32, i32,
                                          i64, i32, f32, P, P, P]
        lib.pkv_last_error.restype = ctypes.c_char_p
        lib.pkv_last_error.argtypes = []
        lib.pkv_version.restype = i32
        lib.pkv_version.argtypes = []
        _lib = lib
        return lib


def _check(status: int):
    if status != 0:
        msg = load_library().pkv_last_error().decode(errors="replace")
        raise PkvError(status, msg)


def _require(t, name, dtype, ndim, host_ok=False):
    """A contiguous tensor the kernels can address: CUDA memory or, where
    ``host_ok`` (an output the kernels write once), pinned host memory."""
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    addressable = t.is_cuda or (host_ok and t.device.type == "cpu" and t.is_pinned())
    if t.dtype != dtype or t.dim() != ndim or not addressable or not t.is_contiguous():
        where = "CUDA or pinned host" if host_ok else "CUDA"
        raise ValueError(f"{name} must be a contiguous {where} {dtype} tensor with {ndim} dims; "
                         f"got {t.dtype}, shape {tuple(t.shape)}, device {t.device}, "
                         f"contiguous={t.is_contiguous()}")


def _raw_stream(device_index: int):
    """Handle of the current CUDA stream on `device_index` (no Python Stream object)."""
    import torch

    get = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if get is not None:
        return get(device_index)
    return torch.cuda.current_stream(device_index).cuda_stream


def _on_device(index: int):
    """Context that makes `index` the current CUDA device only when it is not already."""
    import contextlib

    import torch

    if torch.cuda.current_device() == index:
        return contextlib.nullcontext()
    return torch.cuda.device(index)


def store_kvcache(k, v, k_cache, v_cache, slot_mapping, err_flag=None):
    """Scatter new K/V rows into the paged caches through ``slot_mapping``."""
    import torch

    _require(k, "k", torch.bfloat16, 3)
    _require(v, "v", torch.bfloat16, 3)
    _require(k_cache, "k_cache", torch.bfloat16, 4)
    _require(v_cache, "v_cache", torch.bfloat16, 4)
    _require(slot_mapping, "slot_mapping", torch.int64, 1)
    N, Hkv, D = k.shape
    NB, bs, Hkv2, D2 = k_cache.shape
    if v.shape != k.shape or v_cache.shape != k_cache.shape or (Hkv2, D2) != (Hkv, D):
        raise ValueError("store_kvcache: shape mismatch between k/v and the caches")
    if slot_mapping.shape[0] != N:
        raise ValueError("store_kvcache: slot_mapping length != number of rows")
    if err_flag is not None:
        _require(err_flag, "err_flag", torch.int32, 1)
    lib = _lib or load_library()
    idx = k.get_device()
    with _on_device(idx):
        _check(lib.pkv_store_kvcache(
            k.data_ptr(), v.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
            slot_mapping.data_ptr(), N, Hkv, D, NB, bs,
            err_flag.data_ptr() if err_flag is not None else None, _raw_stream(idx)))


def decode_workspace_bytes(B, Hq, Hkv, D, MBS, bs, max_ctas=0) -> int:
    """Workspace bytes paged_attn_decode needs for these sizes (0 when B == 0)."""
    return int(load_library().pkv_decode_workspace_bytes(B, Hq, Hkv, D, MBS, bs, max_ctas))


_ws_cache: dict = {}


def _workspace(device, stream_handle, nbytes):
    import torch

    if nbytes == 0:
        return None
    key = (device.index, stream_handle)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def paged_attn_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                      max_ctas=0, workspace=None, err_flag=None):
    """One decode step of paged attention; writes ``out`` in place and returns it.

    ``out`` may be a CUDA tensor or a pinned CPU tensor, which the kernels
    then write directly over the host link.
    """
    import torch

    _require(q, "q", torch.bfloat16, 3)
    _require(k_cache, "k_cache", torch.bfloat16, 4)
    _require(v_cache, "v_cache", torch.bfloat16, 4)
    _require(block_tables, "block_tables", torch.int32, 2)
    _require(context_lens, "context_lens", torch.int32, 1)
    _require(out, "out", torch.bfloat16, 3, host_ok=True)
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    if v_cache.shape != k_cache.shape or D2 != D:
        raise ValueError("paged_attn_decode: cache shapes do not match q")
    if out.shape != q.shape:
        raise ValueError("paged_attn_decode: out must have q's shape")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("paged_attn_decode: block_tables/context_lens batch != q batch")
    MBS = block_tables.shape[1]
    if err_flag is not None:
        _require(err_flag, "err_flag", torch.int32, 1)
    lib = _lib or load_library()
    idx = q.get_device()
    with _on_device(idx):
        stream = _raw_stream(idx)
        if workspace is None:
            need = int(lib.pkv_decode_workspace_bytes(B, Hq, Hkv, D, max(MBS, 1), bs, max_ctas))
            workspace = _workspace(q.device, stream, need)
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        _check(lib.pkv_paged_attn_decode(
            q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
            max(MBS, 1), context_lens.data_ptr(), B, Hq, Hkv, D, NB, bs, float(scale),
            out.data_ptr(), ws_ptr, ws_bytes, int(max_ctas),
            err_flag.data_ptr() if err_flag is not None else None, stream))
    return out


# ---------------------------------------------------------------- FP8 cache


def _require_fp8_cache(t, name):
    import torch

    ok = t.dtype == torch.uint8 or t.dtype == getattr(torch, "float8_e4m3fn", None)
    if not isinstance(t, torch.Tensor) or not ok or t.dim() != 4 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA uint8 (or float8_e4m3fn) tensor "
                         f"[NB, bs, Hkv, D]")


def store_kvcache_fp8(k, v, k_cache, v_cache, slot_mapping, k_scale, v_scale, err_flag=None):
    """Quantize new bf16 K/V rows to E4M3 (per-tensor scales) into FP8 caches."""
    import torch

    _require(k, "k", torch.bfloat16, 3)
    _require(v, "v", torch.bfloat16, 3)
    _require_fp8_cache(k_cache, "k_cache")
    _require_fp8_cache(v_cache, "v_cache")
    _require(slot_mapping, "slot_mapping", torch.int64, 1)
    N, Hkv, D = k.shape
    NB, bs, Hkv2, D2 = k_cache.shape
    if v.shape != k.shape or v_cache.shape != k_cache.shape or (Hkv2, D2) != (Hkv, D):
        raise ValueError("store_kvcache_fp8: shape mismatch between k/v and the caches")
    if slot_mapping.shape[0] != N:
        raise ValueError("store_kvcache_fp8: slot_mapping length != number of rows")
    lib = _lib or load_library()
    idx = k.get_device()
    with _on_device(idx):
        _check(lib.pkv_store_kvcache_fp8(
            k.data_ptr(), v.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
            slot_mapping.data_ptr(), N, Hkv, D, NB, bs, float(k_scale), float(v_scale),
            err_flag.data_ptr() if err_flag is not None else None, _raw_stream(idx)))


def paged_attn_decode_fp8(q, k_cache, v_cache, block_tables, context_lens, scale, k_scale,
                          v_scale, out, max_ctas=0, workspace=None, err_flag=None):
    """Decode attention over FP8 (E4M3) caches; writes ``out`` and returns it."""
    import torch

    _require(q, "q", torch.bfloat16, 3)
    _require_fp8_cache(k_cache, "k_cache")
    _require_fp8_cache(v_cache, "v_cache")
    _require(block_tables, "block_tables", torch.int32, 2)
    _require(context_lens, "context_lens", torch.int32, 1)
    _require(out, "out", torch.bfloat16, 3, host_ok=True)
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    if v_cache.shape != k_cache.shape or D2 != D or out.shape != q.shape:
        raise ValueError("paged_attn_decode_fp8: shapes do not match")
    if block_tables.shape[0] != B or context_lens.shape[0] != B:
        raise ValueError("paged_attn_decode_fp8: block_tables/context_lens batch != q batch")
    MBS = block_tables.shape[1]
    lib = _lib or load_library()
    idx = q.get_device()
    with _on_device(idx):
        stream = _raw_stream(idx)
        if workspace is None:
            need = int(lib.pkv_decode_workspace_bytes(B, Hq, Hkv, D, max(MBS, 1), bs, max_ctas))
            workspace = _workspace(q.device, stream, need)
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        _check(lib.pkv_paged_attn_decode_fp8(
            q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
            max(MBS, 1), context_lens.data_ptr(), B, Hq, Hkv, D, NB, bs, float(scale),
            float(k_scale), float(v_scale), out.data_ptr(), ws_ptr, ws_bytes, int(max_ctas),
            err_flag.data_ptr() if err_flag is not None else None, stream))
    return out


# ---------------------------------------------------------------- prefill


def paged_prefill(q, k_cache, v_cache, block_tables, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                  scale, out, err_flag=None):
    """Causal attention of a prefill step's new tokens over their paged contexts.

    q / out are [Tq, Hq, D] bf16 (the sequences' new tokens, concatenated);
    cu_seqlens_q / cu_seqlens_k are int32 [B + 1] on the device; new token i
    of sequence b attends to context positions 0 .. k_len_b - q_len_b + i.
    Store the new tokens' K/V first (``store_kvcache``).  ``out`` may be a
    CUDA tensor or a pinned CPU tensor, which the kernel then writes directly
    over the host link.  Returns ``out``.
    """
    import torch

    _require(q, "q", torch.bfloat16, 3)
    _require(k_cache, "k_cache", torch.bfloat16, 4)
    _require(v_cache, "v_cache", torch.bfloat16, 4)
    _require(block_tables, "block_tables", torch.int32, 2)
    _require(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _require(cu_seqlens_k, "cu_seqlens_k", torch.int32, 1)
    _require(out, "out", torch.bfloat16, 3, host_ok=True)
    Tq, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    if v_cache.shape != k_cache.shape or D2 != D or out.shape != q.shape:
        raise ValueError("paged_prefill: shapes do not match")
    B = cu_seqlens_q.shape[0] - 1
    if B < 0 or cu_seqlens_k.shape[0] != B + 1 or block_tables.shape[0] != B:
        raise ValueError("paged_prefill: cu_seqlens / block_tables batch sizes differ")
    lib = _lib or load_library()
    idx = q.get_device()
    with _on_device(idx):
        _check(lib.pkv_paged_prefill(
            q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
            max(block_tables.shape[1], 1), cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), B, Tq,
            int(max_seqlen_q), Hq, Hkv, D, NB, bs, float(scale), out.data_ptr(),
            err_flag.data_ptr() if err_flag is not None else None, _raw_stream(idx)))
    return out
