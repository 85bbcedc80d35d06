"""A decode step driven by the host block allocator, against the oracle.

The allocator hands out the blocks (with shared prompt prefixes), the step
appends one token per sequence, and store_kvcache + paged_attn_decode run on
the tables and slots it builds.
"""

import numpy as np
import pytest

import oracle
from paged_kv_cache_85_gb300 import workload as wl
from paged_kv_cache_85_gb300.block_manager import BlockManager

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bs", [16, 256])
def test_allocator_driven_decode_step(cuda_lib_path, bs):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_85_gb300 as pkv

    rng = np.random.default_rng(bs)
    B, Hq, Hkv, D, NB = 24, 8, 2, 128, 400
    bm = BlockManager(NB, bs)
    shared = list(rng.integers(0, 50, 2 * bs))
    for sid in range(B):
        n = int(rng.integers(1, 3 * bs))
        prompt = shared[:n] if sid % 3 == 0 else list(rng.integers(0, 50, n))
        bm.allocate(sid, prompt)
    # the step: every sequence gains one token
    slots = np.array([bm.append(sid, int(rng.integers(0, 50))) for sid in range(B)], np.int64)
    MBS = max(len(bm.block_table(s)) for s in range(B))
    tables, lens, slots2 = bm.decode_batch(list(range(B)), MBS)
    np.testing.assert_array_equal(slots, slots2)
    kc = wl.f32_to_bf16_bits(rng.standard_normal((NB, bs, Hkv, D), dtype=np.float32))
    vc = wl.f32_to_bf16_bits(rng.standard_normal((NB, bs, Hkv, D), dtype=np.float32))
    q = wl.f32_to_bf16_bits(rng.standard_normal((B, Hq, D), dtype=np.float32))
    kn = wl.f32_to_bf16_bits(rng.standard_normal((B, Hkv, D), dtype=np.float32))
    vn = wl.f32_to_bf16_bits(rng.standard_normal((B, Hkv, D), dtype=np.float32))
    scale = float(np.float32(D ** -0.5))
    okc, ovc, bad = oracle.store_kvcache(kn, vn, kc, vc, slots)
    assert bad == 0
    ref = oracle.paged_attn_decode(q, okc, ovc, tables, lens, scale)

    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    dkc, dvc = bf(kc), bf(vc)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    pkv.store_kvcache(bf(kn), bf(vn), dkc, dvc, torch.from_numpy(slots).cuda())
    pkv.paged_attn_decode(bf(q), dkc, dvc, torch.from_numpy(tables).cuda(),
                          torch.from_numpy(lens).cuda(), scale, out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(dkc.view(torch.int16).cpu().numpy().view(np.uint16), okc)
    got = out.float().cpu().numpy()
    err = np.abs(got - ref.astype(np.float32))
    assert err.max() <= 1e-2 and err.mean() <= 1e-3, (err.max(), err.mean())
