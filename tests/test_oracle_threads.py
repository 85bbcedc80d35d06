"""Splitting the oracle's (row, head) pairs over host threads changes no bit.

The multi-core CPU baseline and the full-size prefill parity test run the
oracle's pair routines on a thread pool; each pair is computed on its own, so
the results must equal the single-threaded call exactly.
"""

import numpy as np

import oracle
from paged_kv_cache_85_gb300 import workload as wl


def test_threaded_decode_pairs_are_bit_identical():
    w = wl.make_workload("t", B=5, Hq=8, Hkv=2, D=64, bs=16, context_lens=[1, 30, 77, 200, 513],
                         rng=np.random.default_rng(3))
    pairs = np.array([(b, h) for b in range(w.B) for h in range(w.Hq)], np.int32)[::-1].copy()
    one = oracle.paged_attn_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                   w.scale, pairs=pairs)
    many = oracle.paged_attn_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                    w.scale, pairs=pairs, threads=4)
    assert np.array_equal(one, many)
    full = oracle.paged_attn_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                    w.scale)
    assert np.array_equal(full.reshape(-1, w.D)[::-1], many)


def test_threaded_prefill_is_bit_identical():
    p = wl.prefill_config_workload(0)
    kc, vc, _ = oracle.store_kvcache(p.k_new, p.v_new, p.k_cache, p.v_cache, p.slot_mapping)
    args = (p.q, kc, vc, p.block_tables, p.cu_seqlens_q, p.cu_seqlens_k, p.scale)
    assert np.array_equal(oracle.paged_prefill(*args), oracle.paged_prefill(*args, threads=3))
