"""The C-ABI library builds, loads without a GPU and exports every declared symbol."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_two_operations():
    names = _declared()
    assert "pkv_store_kvcache" in names and "pkv_paged_attn_decode" in names


def test_library_exports_every_declared_symbol(cuda_lib_path):
    lib = ctypes.CDLL(cuda_lib_path)
    for name in _declared():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", cuda_lib_path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (pkv_\w+)", out))
    assert set(_declared()) <= exported


def test_library_needs_no_cuda_shared_objects(cuda_lib_path):
    out = subprocess.run(["ldd", cuda_lib_path], capture_output=True, text=True).stdout
    assert "libcudart" not in out and "libcuda.so" not in out


def test_host_only_entry_points(cuda_lib_path):
    lib = ctypes.CDLL(cuda_lib_path)
    lib.pkv_version.restype = ctypes.c_int
    assert lib.pkv_version() >= 100
    f = lib.pkv_decode_workspace_bytes
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 7
    hdr = lambda B: (8 + B + 1) * 4 + (-(8 + B + 1) * 4) % 256
    # Two partial slots of G x (D + 4) floats per worker; workers are bounded by
    # boxes + 7 (4 seqs x 2 KV heads x 19 boxes = 152 boxes -> 159), by 2048, and by
    # max_ctas CTAs of up to 8 workers.
    assert f(4, 4, 2, 64, 19, 16, 0) == hdr(4) + 159 * 2 * 2 * 68 * 4
    assert f(64, 16, 8, 128, 16, 256, 0) == hdr(64) + 2048 * 2 * 2 * 132 * 4
    assert f(64, 16, 8, 128, 16, 256, 10) == hdr(64) + 80 * 2 * 2 * 132 * 4
    assert f(64, 64, 8, 128, 16, 256, 10) == hdr(64) + 80 * 2 * 8 * 132 * 4
    assert f(-1, 4, 2, 64, 19, 16, 0) == 0
    assert f(0, 4, 2, 64, 19, 16, 0) == 0
    assert f(4, 6, 4, 64, 19, 16, 0) == 0  # Hq not a multiple of Hkv
    lib.pkv_status_string.restype = ctypes.c_char_p
    assert lib.pkv_status_string(3) == b"PKV_ERR_WORKSPACE"


def test_argument_errors_need_no_gpu(cuda_lib_path):
    """Bad sizes are rejected on the host, before any CUDA call."""
    lib = ctypes.CDLL(cuda_lib_path)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.pkv_paged_attn_decode.restype = i32
    lib.pkv_paged_attn_decode.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i64, i32,
                                          f32, P, P, sz, i32, P, P]
    lib.pkv_last_error.restype = ctypes.c_char_p
    # Hq not a multiple of Hkv
    st = lib.pkv_paged_attn_decode(None, None, None, None, 1, None, 1, 6, 4, 64, 1, 16, 1.0,
                                   None, None, 0, 0, None, None)
    assert st == 1 and b"multiple" in lib.pkv_last_error()
    # head_dim 96 not built
    st = lib.pkv_paged_attn_decode(None, None, None, None, 1, None, 1, 4, 4, 96, 1, 16, 1.0,
                                   None, None, 0, 0, None, None)
    assert st == 2
    # block size not a multiple of 16
    st = lib.pkv_paged_attn_decode(None, None, None, None, 1, None, 1, 4, 4, 64, 1, 8, 1.0,
                                   None, None, 0, 0, None, None)
    assert st == 2
    # B == 0 is a no-op
    st = lib.pkv_paged_attn_decode(None, None, None, None, 1, None, 0, 4, 4, 64, 1, 16, 1.0,
                                   None, None, 0, 0, None, None)
    assert st == 0
    lib.pkv_store_kvcache.restype = i32
    lib.pkv_store_kvcache.argtypes = [P, P, P, P, P, i64, i32, i32, i64, i32, P, P]
    assert lib.pkv_store_kvcache(None, None, None, None, None, 0, 2, 64, 4, 16, None, None) == 0
    assert lib.pkv_store_kvcache(None, None, None, None, None, 3, 2, 64, 4, 16, None, None) == 1


def test_fp8_argument_errors_need_no_gpu(cuda_lib_path):
    lib = ctypes.CDLL(cuda_lib_path)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.pkv_last_error.restype = ctypes.c_char_p
    st8 = lib.pkv_store_kvcache_fp8
    st8.restype = i32
    st8.argtypes = [P, P, P, P, P, i64, i32, i32, i64, i32, f32, f32, P, P]
    assert st8(None, None, None, None, None, 0, 2, 64, 4, 16, 1.0, 1.0, None, None) == 0
    assert st8(None, None, None, None, None, 0, 1, 8, 4, 16, 1.0, 1.0, None, None) == 2  # Hkv*D % 16
    assert st8(None, None, None, None, None, 0, 2, 64, 4, 16, 0.0, 1.0, None, None) == 1
    assert st8(None, None, None, None, None, 0, 2, 64, 4, 16, 1.0, float("nan"), None, None) == 1
    assert b"scales" in lib.pkv_last_error()
    assert st8(None, None, None, None, None, 3, 2, 64, 4, 16, 1.0, 1.0, None, None) == 1  # null
    dec8 = lib.pkv_paged_attn_decode_fp8
    dec8.restype = i32
    dec8.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i64, i32, f32, f32, f32, P, P, sz, i32,
                     P, P]
    assert dec8(None, None, None, None, 1, None, 1, 6, 4, 64, 1, 16, 1.0, 1.0, 1.0,
                None, None, 0, 0, None, None) == 1
    assert dec8(None, None, None, None, 1, None, 1, 4, 4, 96, 1, 16, 1.0, 1.0, 1.0,
                None, None, 0, 0, None, None) == 2
    assert dec8(None, None, None, None, 1, None, 1, 4, 4, 64, 1, 16, 1.0, -1.0, 1.0,
                None, None, 0, 0, None, None) == 1
    assert dec8(None, None, None, None, 1, None, 0, 4, 4, 64, 1, 16, 1.0, 1.0, 1.0,
                None, None, 0, 0, None, None) == 0


def test_prefill_argument_errors_need_no_gpu(cuda_lib_path):
    lib = ctypes.CDLL(cuda_lib_path)
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    lib.pkv_last_error.restype = ctypes.c_char_p
    f = lib.pkv_paged_prefill
    f.restype = i32
    f.argtypes = [P, P, P, P, i32, P, P, i32, i64, i32, i32, i32, i32, i64, i32, f32, P, P, P]
    # (q, kc, vc, tables, MBS, cu_q, cu_k, B, Tq, max_q, Hq, Hkv, D, NB, bs, scale, out, err, stream)
    assert f(None, None, None, None, 4, None, None, 2, 10, 5, 6, 4, 64, 8, 16, 1.0, None, None, None) == 1
    assert b"multiple" in lib.pkv_last_error()
    assert f(None, None, None, None, 4, None, None, 2, 10, 5, 4, 4, 96, 8, 16, 1.0, None, None, None) == 2
    assert f(None, None, None, None, 4, None, None, 2, 10, 5, 4, 4, 64, 8, 8, 1.0, None, None, None) == 2
    assert f(None, None, None, None, 4, None, None, 2, 10, 5, 12, 4, 64, 8, 16, 1.0, None, None, None) == 2
    assert f(None, None, None, None, 4, None, None, 2, 10, 5, 4, 4, 64, 8, 16, float("inf"), None, None, None) == 1
    assert f(None, None, None, None, 4, None, None, -1, 10, 5, 4, 4, 64, 8, 16, 1.0, None, None, None) == 1
    # nothing to do: no launch, no device needed
    assert f(None, None, None, None, 4, None, None, 0, 0, 0, 4, 4, 64, 8, 16, 1.0, None, None, None) == 0
    assert f(None, None, None, None, 4, None, None, 2, 10, 5, 4, 4, 64, 8, 16, 1.0, None, None, None) == 1  # null


def test_selftest_rejects_bad_limits_on_the_host(cuda_lib_path):
    """The bounded-wait self-test refuses limits outside (0, 0.1 s] and a
    missing err_flag before any launch (no GPU needed)."""
    lib = ctypes.CDLL(cuda_lib_path)
    f = lib.pkv_selftest_bounded_wait
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    assert f(0, 0, ctypes.c_void_p(16), None, None) == 1
    assert f(200_000_000, 0, ctypes.c_void_p(16), None, None) == 1
    assert f(1000, 0, None, None, None) == 1
