"""CPU oracle for paged decode attention (test infrastructure).

Only tests, the smoke check and the benchmark's CPU-baseline leg may import
this package.  The product path (the CUDA library and its Python binding)
never imports, loads or calls it, and it imports nothing from the product.

The arithmetic lives in ``pkv_oracle.c`` (plain C, fp64, one loop per term of
the definition); this module compiles it with gcc on first use and marshals
numpy arrays into it.  bf16 tensors are uint16 arrays of raw bf16 bits.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no FMA contraction) if stale."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    stale = force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    )
    if stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
             "-std=c11", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
            lib.oracle_store_kvcache.restype = i64
            lib.oracle_store_kvcache.argtypes = [P, P, P, P, P, i64, i32, i32, i64, i32]
            lib.oracle_paged_attn_decode_pairs.restype = i64
            lib.oracle_paged_attn_decode_pairs.argtypes = [
                P, P, P, P, i32, P, i32, i32, i32, i32, i64, i32, f32, P, i64, P]
            lib.oracle_paged_attn_decode.restype = i64
            lib.oracle_paged_attn_decode.argtypes = [
                P, P, P, P, i32, P, i32, i32, i32, i32, i64, i32, f32, P]
            lib.oracle_paged_prefill_pairs.restype = i64
            lib.oracle_paged_prefill_pairs.argtypes = [
                P, P, P, P, i32, P, P, i32, i32, i32, i32, i64, i32, f32, P, i64, P]
            lib.oracle_dense_causal_attn.restype = None
            lib.oracle_dense_causal_attn.argtypes = [P, P, P, i32, i32, i32, i32, i32, f32, P]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_e4m3_encode.argtypes = [f32]
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_store_kvcache_fp8.restype = i64
            lib.oracle_store_kvcache_fp8.argtypes = [P, P, P, P, P, i64, i32, i32, i64, i32, f32, f32]
            lib.oracle_dequant_fp8.restype = None
            lib.oracle_dequant_fp8.argtypes = [P, i64, f32, P]
            lib.oracle_paged_attn_decode_pairs_f64kv.restype = i64
            lib.oracle_paged_attn_decode_pairs_f64kv.argtypes = [
                P, P, P, P, i32, P, i32, i32, i32, i64, i32, f32, P, i64, P]
            lib.oracle_dense_attn.restype = None
            lib.oracle_dense_attn.argtypes = [P, P, P, i32, i32, i32, i32, f32, P]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _run_pairs(call, pairs: np.ndarray, out: np.ndarray, threads: int) -> int:
    """Run ``call(pairs_chunk, out_chunk) -> status`` over disjoint chunks of
    the (row, head) pairs, on up to ``threads`` host threads.

    Each pair's result depends only on the inputs, so splitting the pair list
    changes nothing in the arithmetic: the C routine computes every row on its
    own, and ctypes releases the GIL while it runs.  Returns the smallest
    status (negative = an allocation failed in some chunk).
    """
    n = pairs.shape[0]
    threads = max(1, min(int(threads), n))
    if threads == 1:
        return int(call(pairs, out))
    # more chunks than threads, so that uneven rows (long and short contexts) balance
    bounds = np.linspace(0, n, 4 * threads + 1).astype(np.int64)
    chunks = [(int(a), int(b)) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        res = list(ex.map(lambda ab: int(call(np.ascontiguousarray(pairs[ab[0]:ab[1]]),
                                              out[ab[0]:ab[1]])), chunks))
    return min(res)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def store_kvcache(k, v, k_cache, v_cache, slot_mapping):
    """Scatter new K/V rows into copies of the caches.

    Returns ``(k_cache_out, v_cache_out, n_out_of_range)``; inputs untouched.
    """
    lib = _load()
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    kc = np.array(k_cache, dtype=np.uint16, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint16, copy=True, order="C")
    slots = _c(slot_mapping, np.int64)
    NB, bs, Hkv, D = kc.shape
    N = slots.shape[0]
    assert k.shape == (N, Hkv, D) and v.shape == (N, Hkv, D)
    bad = lib.oracle_store_kvcache(_ptr(k), _ptr(v), _ptr(kc), _ptr(vc), _ptr(slots),
                                   N, Hkv, D, NB, bs)
    return kc, vc, int(bad)


def store_kvcache_(k, v, k_cache, v_cache, slot_mapping) -> int:
    """In-place variant of store_kvcache: writes into ``k_cache`` / ``v_cache``.

    The caches must be C-contiguous uint16 arrays.  Returns the number of
    out-of-range slots (skipped).
    """
    lib = _load()
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    slots = _c(slot_mapping, np.int64)
    for c in (k_cache, v_cache):
        if c.dtype != np.uint16 or not c.flags["C_CONTIGUOUS"] or not c.flags["WRITEABLE"]:
            raise ValueError("caches must be writeable C-contiguous uint16 arrays")
    NB, bs, Hkv, D = k_cache.shape
    N = slots.shape[0]
    assert k.shape == (N, Hkv, D) and v.shape == (N, Hkv, D) and v_cache.shape == k_cache.shape
    return int(lib.oracle_store_kvcache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(slots), N, Hkv, D, NB, bs))


def paged_attn_decode(q, k_cache, v_cache, block_tables, context_lens, scale, pairs=None,
                      threads=1):
    """fp64 decode attention.

    Without ``pairs`` returns ``[B, Hq, D]``; with ``pairs`` (an ``[n, 2]``
    array of (b, h)) returns ``[n, D]`` for just those rows.  ``threads > 1``
    splits the pairs over host threads (same results).
    """
    lib = _load()
    q = _c(q, np.uint16)
    kc = _c(k_cache, np.uint16)
    vc = _c(v_cache, np.uint16)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = kc.shape
    assert D2 == D and vc.shape == kc.shape and Hq % Hkv == 0
    MBS = bt.shape[1]
    if pairs is None:
        out = np.zeros((B, Hq, D), dtype=np.float64)
        bad = lib.oracle_paged_attn_decode(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), MBS, _ptr(cl),
                                           B, Hq, Hkv, D, NB, bs, float(scale), _ptr(out))
    else:
        pr = _c(pairs, np.int32).reshape(-1, 2)
        out = np.zeros((pr.shape[0], D), dtype=np.float64)
        bad = _run_pairs(
            lambda pc, oc: lib.oracle_paged_attn_decode_pairs(
                _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), MBS, _ptr(cl), B, Hq, Hkv, D, NB, bs,
                float(scale), _ptr(pc), pc.shape[0], _ptr(oc)),
            pr, out, threads)
    if bad < 0:
        raise MemoryError("oracle allocation failed")
    return out


def dense_attn(q, k, v, scale):
    """fp64 attention over contiguous K/V ``[n, Hkv, D]`` for one sequence's ``q [Hq, D]``."""
    lib = _load()
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    Hq, D = q.shape
    n, Hkv, D2 = k.shape
    assert D2 == D and v.shape == k.shape
    out = np.zeros((Hq, D), dtype=np.float64)
    lib.oracle_dense_attn(_ptr(q), _ptr(k), _ptr(v), n, Hq, Hkv, D, float(scale), _ptr(out))
    return out


# ---------------------------------------------------------------- FP8 cache


def e4m3_encode(x: float) -> int:
    """OCP E4M3 code of an fp32 value (nearest, ties to even, saturating)."""
    return int(_load().oracle_e4m3_encode(float(np.float32(x))))


def e4m3_decode(code: int) -> float:
    return float(_load().oracle_e4m3_decode(int(code)))


def store_kvcache_fp8(k, v, k_cache, v_cache, slot_mapping, k_scale, v_scale):
    """Quantize new bf16 K/V rows into copies of uint8 (E4M3) caches."""
    lib = _load()
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    kc = np.array(k_cache, dtype=np.uint8, copy=True, order="C")
    vc = np.array(v_cache, dtype=np.uint8, copy=True, order="C")
    slots = _c(slot_mapping, np.int64)
    NB, bs, Hkv, D = kc.shape
    N = slots.shape[0]
    bad = lib.oracle_store_kvcache_fp8(_ptr(k), _ptr(v), _ptr(kc), _ptr(vc), _ptr(slots), N, Hkv,
                                       D, NB, bs, float(k_scale), float(v_scale))
    return kc, vc, int(bad)


def e4m3_table(scale):
    """Code of every bf16 bit pattern x for x * (1/scale), as store_kvcache_fp8 writes it.

    The code depends only on x once the scale is fixed, so this is the plain
    quantizer memoised over all 65536 inputs (one row through the oracle's
    own store); ``table[bits]`` then quantizes whole caches quickly.
    """
    x = np.arange(65536, dtype=np.uint16).reshape(1, 1, 65536)
    cache = np.zeros((1, 1, 1, 65536), np.uint8)
    kc, _, bad = store_kvcache_fp8(x, x, cache, cache, np.zeros(1, np.int64), scale, scale)
    assert bad == 0
    return kc.reshape(65536)


def quantize_bf16(bits, scale):
    """E4M3 codes of bf16 values (uint16 bits) for a per-tensor scale."""
    return e4m3_table(scale)[np.asarray(bits, dtype=np.uint16)]


def dequant_fp8(codes, scale):
    """fp64 values of E4M3 codes times scale."""
    lib = _load()
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib.oracle_dequant_fp8(_ptr(c), c.size, float(scale), _ptr(out))
    return out


def paged_attn_decode_values(q, k_vals, v_vals, block_tables, context_lens, scale, pairs=None,
                             threads=1):
    """fp64 decode attention over caches holding fp64 values [NB, bs, Hkv, D]."""
    lib = _load()
    q = _c(q, np.uint16)
    kv = _c(k_vals, np.float64)
    vv = _c(v_vals, np.float64)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = kv.shape
    assert D2 == D and vv.shape == kv.shape and Hq % Hkv == 0
    if pairs is None:
        pr = np.array([(b, h) for b in range(B) for h in range(Hq)], np.int32)
    else:
        pr = _c(pairs, np.int32).reshape(-1, 2)
    out = np.zeros((pr.shape[0], D), dtype=np.float64)
    bad = _run_pairs(
        lambda pc, oc: lib.oracle_paged_attn_decode_pairs_f64kv(
            _ptr(q), _ptr(kv), _ptr(vv), _ptr(bt), bt.shape[1], _ptr(cl), Hq, Hkv, D, NB, bs,
            float(scale), _ptr(pc), pc.shape[0], _ptr(oc)),
        pr, out, threads)
    if bad < 0:
        raise MemoryError("oracle allocation failed")
    return out.reshape(B, Hq, D) if pairs is None else out


def paged_attn_decode_fp8(q, k_cache, v_cache, block_tables, context_lens, scale, k_scale,
                          v_scale, pairs=None, threads=1):
    """fp64 decode attention over FP8 caches (dequantized K and V)."""
    kd = dequant_fp8(k_cache, k_scale)
    vd = dequant_fp8(v_cache, v_scale)
    return paged_attn_decode_values(q, kd, vd, block_tables, context_lens, scale, pairs=pairs,
                                    threads=threads)


# ---------------------------------------------------------------- prefill


def paged_prefill(q, k_cache, v_cache, block_tables, cu_seqlens_q, cu_seqlens_k, scale,
                  pairs=None, threads=1):
    """fp64 causal prefill attention over the paged cache.

    q is [Tq, Hq, D] (the sequences' new tokens, concatenated); query i of
    sequence b sits at position k_len_b - q_len_b + i and attends to positions
    0 .. that one.  Returns [Tq, Hq, D], or [len(pairs), D] for the listed
    (token row, head) pairs.  ``threads > 1`` splits the pairs over host
    threads (same results).
    """
    lib = _load()
    q = _c(q, np.uint16)
    kc = _c(k_cache, np.uint16)
    vc = _c(v_cache, np.uint16)
    bt = _c(block_tables, np.int32)
    cq = _c(cu_seqlens_q, np.int32)
    ck = _c(cu_seqlens_k, np.int32)
    Tq, Hq, D = q.shape
    NB, bs, Hkv, D2 = kc.shape
    B = cq.shape[0] - 1
    assert D2 == D and vc.shape == kc.shape and Hq % Hkv == 0 and ck.shape[0] == B + 1
    if pairs is None:
        pr = np.stack(np.meshgrid(np.arange(Tq), np.arange(Hq), indexing="ij"), -1)
        pr = np.ascontiguousarray(pr.reshape(-1, 2).astype(np.int32))
    else:
        pr = _c(pairs, np.int32).reshape(-1, 2)
    out = np.zeros((pr.shape[0], D), dtype=np.float64)
    bad = _run_pairs(
        lambda pc, oc: lib.oracle_paged_prefill_pairs(
            _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), bt.shape[1], _ptr(cq), _ptr(ck), B, Hq, Hkv,
            D, NB, bs, float(scale), _ptr(pc), pc.shape[0], _ptr(oc)),
        pr, out, threads)
    if bad < 0:
        raise MemoryError("oracle allocation failed")
    return out.reshape(Tq, Hq, D) if pairs is None else out


def dense_causal_attn(q, k, v, scale):
    """fp64 causal attention of one sequence over contiguous K/V.

    q [Lq, Hq, D], k/v [Lk, Hkv, D] bf16 bits; query i at position Lk - Lq + i.
    """
    lib = _load()
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    Lq, Hq, D = q.shape
    Lk, Hkv, D2 = k.shape
    assert D2 == D and v.shape == k.shape and Lq <= Lk
    out = np.zeros((Lq, Hq, D), dtype=np.float64)
    lib.oracle_dense_causal_attn(_ptr(q), _ptr(k), _ptr(v), Lq, Lk, Hq, Hkv, D, float(scale),
                                 _ptr(out))
    return out
