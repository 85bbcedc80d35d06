"""The bounded pipeline wait reports a timeout and returns (no hang, no fault).

Every mbarrier wait in the decode and prefill kernels gives up after a time
limit, ORs PKV_FLAG_TIMEOUT into err_flag and returns.  The production
kernels never run into that limit on valid inputs, so this test drives the
same wait helper through pkv_selftest_bounded_wait: one warp waits about a
millisecond on a barrier that nothing completes (no copy is in flight), and
the test checks that the flag comes back, that the call returned within the
limit, and that the device still runs a decode step correctly afterwards.
"""

import ctypes
import time

import numpy as np
import pytest

import oracle
from paged_kv_cache_85_gb300 import workload as wl

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

FLAG_TIMEOUT = 0x8


@pytest.fixture(scope="module")
def lib(cuda_lib_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = ctypes.CDLL(cuda_lib_path)
    lib.pkv_selftest_bounded_wait.restype = ctypes.c_int
    lib.pkv_selftest_bounded_wait.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p]
    lib.pkv_last_error.restype = ctypes.c_char_p
    return lib


def _wait(lib, limit_ns, arrive):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = lib.pkv_selftest_bounded_wait(limit_ns, arrive, err.data_ptr(), waited.data_ptr(), stream)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert st == 0, lib.pkv_last_error()
    return int(err.item()), int(waited.item()), dt


def test_wait_that_nothing_completes_times_out_and_returns(lib):
    limit = 1_000_000  # 1 ms
    flags, waited, dt = _wait(lib, limit, arrive=0)
    assert flags & FLAG_TIMEOUT
    assert limit <= waited < 50 * limit
    assert dt < 1.0  # the call returned; nothing hung


def test_completed_wait_sets_no_flag(lib):
    flags, waited, _ = _wait(lib, 1_000_000, arrive=1)
    assert flags == 0
    assert waited < 1_000_000


def test_device_is_usable_after_a_timeout(lib):
    import paged_kv_cache_85_gb300 as pkv

    _wait(lib, 2_000_000, arrive=0)
    pkv.load_library()
    w = wl.config_workload(0)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()

    q, kc, vc = bf(w.q), bf(w.k_cache), bf(w.v_cache)
    out = torch.empty_like(q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.store_kvcache(bf(w.k_new), bf(w.v_new), kc, vc, torch.from_numpy(w.slot_mapping).cuda(),
                      err_flag=err)
    pkv.paged_attn_decode(q, kc, vc, torch.from_numpy(w.block_tables).cuda(),
                          torch.from_numpy(w.context_lens).cuda(), w.scale, out, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    okc, ovc, _ = oracle.store_kvcache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    ref = oracle.paged_attn_decode(w.q, okc, ovc, w.block_tables, w.context_lens, w.scale)
    d = np.abs(out.float().cpu().numpy() - ref)
    assert d.max() <= 1e-2 and d.mean() <= 1e-3
