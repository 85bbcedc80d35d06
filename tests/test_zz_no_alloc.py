"""The allocation-free decode entry point matches the regular one.

pkv_paged_attn_decode_noalloc is for callers that cannot allocate device
memory when they run attention (a custom allocator or memory pool that must
not be re-entered, a runtime that only owns the step's input and output
buffers): it keeps its scratch in a fixed array inside the library instead
of a caller workspace.  This test calls it through the C ABI twice in a row,
on two different steps, and checks each result against
pkv_paged_attn_decode on the same inputs, within the attention tolerance
(max-abs 1e-2, mean-abs 1e-3).  The file is named so pytest runs it last.
"""

import ctypes

import numpy as np
import pytest

from paged_kv_cache_85_gb300 import workload as wl

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-2
MEAN_ABS = 1e-3


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


def _regular(lib, w, d, stream):
    out = torch.empty_like(d["q"])
    n = lib.pkv_decode_workspace_bytes(w.B, w.Hq, w.Hkv, w.D, w.MBS, w.bs, 0)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    st = lib.pkv_paged_attn_decode(d["q"].data_ptr(), d["kc"].data_ptr(), d["vc"].data_ptr(),
                                   d["tables"].data_ptr(), w.MBS, d["lens"].data_ptr(), w.B, w.Hq,
                                   w.Hkv, w.D, w.NB, w.bs, w.scale, out.data_ptr(), ws.data_ptr(),
                                   n, 0, None, stream)
    assert st == 0, lib.pkv_last_error()
    return out


def _noalloc(lib, w, d, stream):
    out = torch.empty_like(d["q"])
    st = lib.pkv_paged_attn_decode_noalloc(d["q"].data_ptr(), d["kc"].data_ptr(), d["vc"].data_ptr(),
                                           d["tables"].data_ptr(), w.MBS, d["lens"].data_ptr(), w.B,
                                           w.Hq, w.Hkv, w.D, w.NB, w.bs, w.scale, out.data_ptr(),
                                           None, stream)
    assert st == 0, lib.pkv_last_error()
    return out


def _close(a, b):
    x = a.float().cpu().numpy()
    y = b.float().cpu().numpy()
    assert np.isfinite(x).all()
    err = np.abs(x - y)
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (err.max(), err.mean())


def test_noalloc_matches_regular_entry_point_twice_in_a_row(lib):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # two different steps: a long-context GQA-4 batch, then the small tiny-config one
    steps = [
        wl.make_workload("a", B=12, Hq=16, Hkv=4, D=128, bs=16,
                         context_lens=[1, 7, 16, 33, 100, 257, 600, 1024, 1500, 2048, 3001, 4096],
                         rng=np.random.default_rng(21)),
        wl.config_workload(0),
    ]
    for w in steps:
        d = _dev(w)
        got = _noalloc(lib, w, d, stream)
        ref = _regular(lib, w, d, stream)
        torch.cuda.synchronize()
        _close(got, ref)
