"""The attention calls write their result into pinned host memory.

`out` of paged_attn_decode, paged_attn_decode_fp8 and paged_prefill may be
page-locked host memory that the device addresses directly; the kernels then
write the result over the host link.  The result must be bit-identical to the
one written into device memory (which the parity tests compare with the
oracle), and memory the device cannot address must be refused.
"""

import numpy as np
import pytest

from paged_kv_cache_85_gb300 import workload as wl

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv(cuda_lib_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_85_gb300 as m

    m.load_library()
    return m


def bf16_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def bits(t):
    return t.view(torch.int16).cpu().numpy()


def decode_inputs(w):
    return dict(q=bf16_dev(w.q), kc=bf16_dev(w.k_cache), vc=bf16_dev(w.v_cache),
                tables=torch.from_numpy(w.block_tables).cuda(),
                lens=torch.from_numpy(w.context_lens).cuda())


@pytest.mark.parametrize("idx", [1, 3])
def test_decode_into_pinned_host_memory_is_bit_identical(pkv, idx):
    w = wl.config_workload(idx)
    d = decode_inputs(w)
    out_d = torch.empty_like(d["q"])
    out_h = torch.full(tuple(d["q"].shape), float("nan"), dtype=torch.bfloat16).pin_memory()
    for o in (out_d, out_h):
        pkv.paged_attn_decode(d["q"], d["kc"], d["vc"], d["tables"], d["lens"], w.scale, o)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out_d), bits(out_h))


def test_fp8_decode_into_pinned_host_memory_is_bit_identical(pkv):
    w = wl.config_workload(1)
    d = decode_inputs(w)
    k8 = torch.empty(d["kc"].shape, dtype=torch.uint8, device="cuda")
    v8 = torch.empty_like(k8)
    NB, bs, Hkv, D = d["kc"].shape
    # every cached token through the quantizing store, slot i = token i
    kflat, vflat = d["kc"].reshape(-1, Hkv, D), d["vc"].reshape(-1, Hkv, D)
    slots = torch.arange(kflat.shape[0], dtype=torch.int64, device="cuda")
    k_scale = float(kflat.float().abs().max()) / 448.0
    v_scale = float(vflat.float().abs().max()) / 448.0
    pkv.store_kvcache_fp8(kflat, vflat, k8, v8, slots, k_scale, v_scale)
    out_d = torch.empty_like(d["q"])
    out_h = torch.full(tuple(d["q"].shape), float("nan"), dtype=torch.bfloat16).pin_memory()
    for o in (out_d, out_h):
        pkv.paged_attn_decode_fp8(d["q"], k8, v8, d["tables"], d["lens"], w.scale, k_scale,
                                  v_scale, o)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out_d), bits(out_h))


@pytest.mark.parametrize("idx", [0, 2])
def test_prefill_into_pinned_host_memory_is_bit_identical(pkv, idx):
    w = wl.prefill_config_workload(idx)
    q, kc, vc = bf16_dev(w.q), bf16_dev(w.k_cache), bf16_dev(w.v_cache)
    pkv.store_kvcache(bf16_dev(w.k_new), bf16_dev(w.v_new), kc, vc,
                      torch.from_numpy(w.slot_mapping).cuda())
    tables = torch.from_numpy(w.block_tables).cuda()
    cu_q, cu_k = torch.from_numpy(w.cu_seqlens_q).cuda(), torch.from_numpy(w.cu_seqlens_k).cuda()
    out_d = torch.zeros_like(q)
    out_h = torch.zeros(tuple(q.shape), dtype=torch.bfloat16).pin_memory()
    for o in (out_d, out_h):
        pkv.paged_prefill(q, kc, vc, tables, cu_q, cu_k, w.max_seqlen_q, w.scale, o)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out_d), bits(out_h))


def test_unpinned_host_memory_is_refused(pkv):
    w = wl.config_workload(0)
    d = decode_inputs(w)
    with pytest.raises(ValueError):
        pkv.paged_attn_decode(d["q"], d["kc"], d["vc"], d["tables"], d["lens"], w.scale,
                              torch.empty(tuple(d["q"].shape), dtype=torch.bfloat16))
    # inputs stay device-only: a pinned q is refused
    with pytest.raises(ValueError):
        pkv.paged_attn_decode(d["q"].cpu().pin_memory(), d["kc"], d["vc"], d["tables"], d["lens"],
                              w.scale, torch.empty_like(d["q"]))
