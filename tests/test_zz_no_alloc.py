"""The allocation-free decode entry point matches the regular one and the oracle.

pkv_paged_attn_decode_noalloc is for callers that cannot allocate device
memory when they run attention (a custom allocator or memory pool that must
not be re-entered, a runtime that only owns the step's input and output
buffers): it keeps its scratch in a fixed array inside the library instead
of a caller workspace.  These tests call it through the C ABI, two calls in
a row on different steps, and check each result
  - bit for bit against pkv_paged_attn_decode with max_ctas = 0 (the fixed
    array holds the partial results of the full grid for these shapes, so
    both calls launch the same grid and split the contexts at the same
    places), and
  - against the fp64 oracle within the attention tolerance (max-abs 1e-2,
    mean-abs 1e-3), so that a bug shared by both entry points cannot pass.
A bad block id must set the error flag through the new entry point as it does
through the regular one.  The file is named so pytest runs it last.
"""

import ctypes

import numpy as np
import pytest

import oracle
from paged_kv_cache_85_gb300 import workload as wl

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-2
MEAN_ABS = 1e-3
FLAG_BAD_BLOCK = 0x2


@pytest.fixture(scope="module")
def lib(cuda_lib_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = ctypes.CDLL(cuda_lib_path)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    lib.pkv_paged_attn_decode.restype = i32
    lib.pkv_paged_attn_decode.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i64, i32,
                                          f32, P, P, sz, i32, P, P]
    lib.pkv_paged_attn_decode_noalloc.restype = i32
    lib.pkv_paged_attn_decode_noalloc.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i64,
                                                  i32, f32, P, P, P]
    lib.pkv_decode_workspace_bytes.restype = sz
    lib.pkv_decode_workspace_bytes.argtypes = [i32] * 7
    lib.pkv_last_error.restype = ctypes.c_char_p
    return lib


def _dev(w):
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return dict(q=bf(w.q), kc=bf(w.k_cache), vc=bf(w.v_cache),
                tables=torch.from_numpy(w.block_tables).cuda(),
                lens=torch.from_numpy(w.context_lens).cuda())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _regular(lib, w, d, err=None):
    out = torch.empty_like(d["q"])
    n = lib.pkv_decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, w.MBS, w.bs, 0)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    st = lib.pkv_paged_attn_decode(d["q"].data_ptr(), d["kc"].data_ptr(), d["vc"].data_ptr(),
                                   d["tables"].data_ptr(), w.MBS, d["lens"].data_ptr(), w.B, w.Hq,
                                   w.Hkv, w.D, w.NB, w.bs, w.scale, out.data_ptr(), ws.data_ptr(),
                                   n, 0, None if err is None else err.data_ptr(), _stream())
    assert st == 0, lib.pkv_last_error()
    return out


def _noalloc(lib, w, d, err=None):
    out = torch.empty_like(d["q"])
    st = lib.pkv_paged_attn_decode_noalloc(d["q"].data_ptr(), d["kc"].data_ptr(), d["vc"].data_ptr(),
                                           d["tables"].data_ptr(), w.MBS, d["lens"].data_ptr(), w.B,
                                           w.Hq, w.Hkv, w.D, w.NB, w.bs, w.scale, out.data_ptr(),
                                           None if err is None else err.data_ptr(), _stream())
    assert st == 0, lib.pkv_last_error()
    return out


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


def _close(got, ref):
    x = got.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(x).all()
    err = np.abs(x - ref)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (err.max(), err.mean())


def _steps():
    ctx = [1, 7, 16, 33, 100, 257, 600, 1024, 1500, 2048, 3001, 4096]
    return [
        # GQA 4, head_dim 128: two four-worker CTAs per SM
        wl.make_workload("g4", B=12, Hq=16, Hkv=4, D=128, bs=16, context_lens=ctx,
                         rng=np.random.default_rng(21)),
        # GQA 8, head_dim 128: one eight-worker CTA per SM
        wl.make_workload("g8", B=12, Hq=32, Hkv=4, D=128, bs=16, context_lens=ctx[::-1],
                         rng=np.random.default_rng(22)),
        wl.config_workload(0),
    ]


def test_noalloc_matches_regular_entry_point_and_oracle_on_calls_in_a_row(lib):
    for w in _steps():
        d = _dev(w)
        got = _noalloc(lib, w, d)
        again = _noalloc(lib, w, d)  # the array keeps the last call's contents: same result
        ref = _regular(lib, w, d)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(_bits(got), _bits(ref))
        np.testing.assert_array_equal(_bits(again), _bits(ref))
        _close(got, oracle.paged_attn_decode(w.q, w.k_cache, w.v_cache, w.block_tables,
                                             w.context_lens, w.scale))


def test_noalloc_reports_bad_block_ids(lib):
    w = _steps()[0]
    d = _dev(w)
    tables = d["tables"].clone()
    tables[5, 0] = w.NB + 7  # a needed entry out of range
    d["tables"] = tables
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _noalloc(lib, w, d, err=err)
    err_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = _regular(lib, w, d, err=err_ref)
    torch.cuda.synchronize()
    assert int(err.item()) & FLAG_BAD_BLOCK
    assert int(err.item()) == int(err_ref.item())
    np.testing.assert_array_equal(_bits(got), _bits(ref))
    assert torch.isfinite(got.float()).all()
