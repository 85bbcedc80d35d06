"""Decode steps replayed from CUDA graphs at padded batch sizes."""

import numpy as np
import pytest

import oracle
from paged_kv_cache_85_gb300 import workload as wl
from paged_kv_cache_85_gb300.graph_runner import graph_batch_sizes

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_graph_batch_sizes_follow_the_guide():
    assert graph_batch_sizes(64) == [1, 2, 4, 8, 16, 32, 48, 64]
    assert graph_batch_sizes(5) == [1, 2, 4, 5]


@pytest.mark.parametrize("bs", [1, 3, 5, 16, 20])
def test_padded_graph_replay_matches_oracle(cuda_lib_path, bs):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_85_gb300.graph_runner import DecodeGraphRunner

    rng = np.random.default_rng(bs)
    Hq, Hkv, D, blk = 8, 2, 128, 16
    lens = rng.integers(1, 300, bs)
    w = wl.make_workload("g", B=bs, Hq=Hq, Hkv=Hkv, D=D, bs=blk, context_lens=lens, NB=512, rng=rng)
    kc, vc, _ = oracle.store_kvcache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    ref = oracle.paged_attn_decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)

    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    dkc, dvc = bf(w.k_cache), bf(w.v_cache)
    MBS = 24
    runner = DecodeGraphRunner(dkc, dvc, Hq, max_bs=32, max_blocks_per_seq=MBS, scale=w.scale)
    tables = np.full((bs, MBS), -1, np.int32)
    tables[:, : w.MBS] = w.block_tables
    out = runner.step(bf(w.q), bf(w.k_new), bf(w.v_new), torch.from_numpy(w.slot_mapping).cuda(),
                      torch.from_numpy(tables).cuda(), torch.from_numpy(w.context_lens).cuda())
    torch.cuda.synchronize()
    got = out.float().cpu().numpy()
    err = np.abs(got - ref.astype(np.float32))
    assert err.max() <= 1e-2 and err.mean() <= 1e-3, (err.max(), err.mean())
    np.testing.assert_array_equal(dkc.view(torch.int16).cpu().numpy().view(np.uint16), kc)
    gb = runner.graph_size(bs)
    if gb > bs:  # padded rows: zero-length contexts give zeros
        assert (runner.out[bs:gb].float() == 0).all()


def test_replay_twice_with_new_inputs(cuda_lib_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_85_gb300.graph_runner import DecodeGraphRunner

    w = wl.config_workload(0)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    dkc, dvc = bf(w.k_cache), bf(w.v_cache)
    runner = DecodeGraphRunner(dkc, dvc, w.Hq, max_bs=8, max_blocks_per_seq=w.MBS, scale=w.scale)
    kc, vc, _ = oracle.store_kvcache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    for trial in range(2):
        q = w.q if trial == 0 else wl.f32_to_bf16_bits(
            np.random.default_rng(5).standard_normal(w.q.shape, dtype=np.float32))
        v = runner.inputs(w.B)
        v["q"].copy_(bf(q))
        v["k_new"].copy_(bf(w.k_new))
        v["v_new"].copy_(bf(w.v_new))
        v["slot_mapping"].copy_(torch.from_numpy(w.slot_mapping))
        v["block_tables"].copy_(torch.from_numpy(w.block_tables))
        v["context_lens"].copy_(torch.from_numpy(w.context_lens))
        out = runner.replay(w.B)
        torch.cuda.synchronize()
        ref = oracle.paged_attn_decode(q, kc, vc, w.block_tables, w.context_lens, w.scale)
        err = np.abs(out.float().cpu().numpy() - ref.astype(np.float32))
        assert err.max() <= 1e-2 and err.mean() <= 1e-3
