"""Host-side checks of the seeded input generator (no GPU, no oracle math)."""

import numpy as np
import pytest
import torch

from paged_kv_cache_85_gb300 import workload as wl


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(-6, 6, 100000),
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 65504.0], np.float32)])
    x = x.astype(np.float32)
    ours = wl.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    back = wl.bf16_bits_to_f32(ours)
    np.testing.assert_array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_decode_slot_matches_append_example():
    """MinivLLM guide §4.5: token 257 with bs=256 opens a new block; it lands at its offset 0."""
    table = np.array([11, 42], np.int32)  # block 42 was just appended for token 257
    assert wl.decode_slot(table, 257, 256) == 42 * 256
    assert wl.decode_slot(table[:1], 256, 256) == 11 * 256 + 255
    assert wl.decode_slot(np.array([5], np.int32), 1, 16) == 5 * 16


def test_config_tiny_shapes_and_determinism():
    a = wl.config_workload(0)
    b = wl.config_workload(0)
    for f in ("q", "k_cache", "v_cache", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))
    assert a.NB == 64 and a.bs == 16 and a.D == 64 and (a.Hq, a.Hkv) == (4, 2)
    assert list(a.context_lens) == [1, 17, 40, 300]
    assert a.MBS == 19
    used = a.block_tables[a.block_tables >= 0]
    assert len(used) == 1 + 2 + 3 + 19 and len(set(used.tolist())) == len(used)


def test_every_slot_is_the_last_context_token():
    w = wl.config_workload(0)
    for b in range(w.B):
        n = int(w.context_lens[b])
        t = n - 1
        assert w.slot_mapping[b] == w.block_tables[b, t // w.bs] * w.bs + t % w.bs


@pytest.mark.parametrize("idx", [1, 2, 3])
def test_full_configs_index_structure(idx, monkeypatch):
    # skip drawing GB-sized caches: only the index structure is checked here
    monkeypatch.setattr(wl, "_randn_bf16", lambda rng, shape: np.zeros(shape, np.uint16))
    w = wl.config_workload(idx)
    nblk = (w.context_lens.astype(np.int64) + w.bs - 1) // w.bs
    assert w.NB == int(np.ceil(1.25 * nblk.sum()))
    used = w.block_tables[w.block_tables >= 0]
    assert len(set(used.tolist())) == len(used) == nblk.sum()
    assert (w.block_tables[:, :].max() < w.NB)
    if idx == 1:
        assert w.B == 64 and w.context_lens.min() >= 128 and w.context_lens.max() <= 4096
    if idx == 2:
        assert w.B == 256 and w.bs == 16 and w.context_lens.max() <= 2048
    if idx == 3:
        assert w.B == 512 and int((w.slot_mapping == -1).sum()) == 26
        assert w.context_lens.min() >= 16 and w.context_lens.max() <= 4096


def test_shared_prefix_config(monkeypatch):
    monkeypatch.setattr(wl, "_randn_bf16", lambda rng, shape: np.zeros(shape, np.uint16))
    w = wl.config_workload(4)
    assert w.B == 8 and (w.context_lens == 32768).all() and w.MBS == 128
    for b in range(1, 8):
        np.testing.assert_array_equal(w.block_tables[b, :32], w.block_tables[0, :32])
    own = w.block_tables[:, 32:].reshape(-1)
    assert len(set(own.tolist())) == own.size
    assert w.unique_kv_bytes() < w.kv_bytes()
