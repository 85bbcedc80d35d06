"""Pins of the prefill oracle against what the pages and the mathematics fix.

The oracle computes each (query row, head) of a prefill step as attention
over the row's first position + 1 tokens of its sequence, read through the
block table.  It is checked against:
  * the pages' cu_seqlens example and a worked causal example (golden files);
  * an independently written dense causal routine over contiguous K/V;
  * a numpy brute force (explicit score matrix, triangular mask, np.exp);
  * closed forms: the first token of a fresh sequence returns its own V, and
    identical keys give the running mean of V;
  * invariance under permuting the physical blocks.
"""

import math
import os

import numpy as np
import pytest

import oracle
from paged_kv_cache_85_gb300 import workload as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fields(name):
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            k, *v = line.split()
            out[k] = [float(x) for x in v]
    return out


def bf(x):
    return wl.f32_to_bf16_bits(np.asarray(x, np.float32))


def stored(w):
    """Caches after the step's store (a plain bit copy through slot_mapping)."""
    kc, vc, bad = oracle.store_kvcache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    assert bad == 0
    return kc, vc


def gather(cache, table, n, bs):
    pos = np.arange(n)
    return cache[table[pos // bs], pos % bs]


def test_cu_seqlens_match_the_pages_example():
    g = _fields("prefill_cu_seqlens.txt")
    got = wl.cu_seqlens([int(x) for x in g["lengths"]])
    assert got.tolist() == [int(x) for x in g["cu_seqlens"]]


def test_worked_causal_example():
    g = _fields("prefill_causal_two_queries.txt")
    D, bs, NB = 2, 16, 4
    blk = int(g["block"][0])
    kc = np.zeros((NB, bs, 1, D), np.uint16)
    vc = np.zeros((NB, bs, 1, D), np.uint16)
    kc[blk, :3, 0] = bf(np.array(g["k"]).reshape(3, D))
    vc[blk, :3, 0] = bf(np.array(g["v"]).reshape(3, D))
    q = bf(np.array(g["q"]).reshape(2, 1, D))
    tables = np.array([[blk]], np.int32)
    scale = float(np.float32(math.log(g["scale_ln"][0])))
    out = oracle.paged_prefill(q, kc, vc, tables, [0, 2], [0, 3], scale)
    np.testing.assert_allclose(out.reshape(-1), g["out"], rtol=0, atol=1e-6)


def _random(rng, G, D, bs, q_lens, cached):
    Hkv = 2
    return wl.make_prefill_workload("rand", Hq=G * Hkv, Hkv=Hkv, D=D, bs=bs, q_lens=q_lens,
                                    cached_lens=cached, rng=rng)


@pytest.mark.parametrize("G,D,bs", [(1, 16, 16), (2, 32, 16), (4, 16, 32), (8, 8, 16)])
def test_paged_prefill_equals_dense_causal(G, D, bs):
    rng = np.random.default_rng(40 + G + D + bs)
    w = _random(rng, G, D, bs, q_lens=[1, 7, 20, 33], cached=[0, bs, 2 * bs, 0])
    kc, vc = stored(w)
    got = oracle.paged_prefill(w.q, kc, vc, w.block_tables, w.cu_seqlens_q, w.cu_seqlens_k,
                               w.scale)
    for b in range(w.B):
        k = gather(kc, w.block_tables[b], int(w.k_lens[b]), w.bs)
        v = gather(vc, w.block_tables[b], int(w.k_lens[b]), w.bs)
        q = w.q[w.cu_seqlens_q[b] : w.cu_seqlens_q[b + 1]]
        ref = oracle.dense_causal_attn(q, k, v, w.scale)
        np.testing.assert_allclose(got[w.cu_seqlens_q[b] : w.cu_seqlens_q[b + 1]], ref,
                                   rtol=0, atol=1e-12)


def test_paged_prefill_matches_numpy_brute_force():
    rng = np.random.default_rng(41)
    w = _random(rng, 2, 16, 16, q_lens=[3, 12, 1], cached=[16, 0, 32])
    kc, vc = stored(w)
    got = oracle.paged_prefill(w.q, kc, vc, w.block_tables, w.cu_seqlens_q, w.cu_seqlens_k,
                               w.scale)
    f64 = lambda a: wl.bf16_bits_to_f32(a).astype(np.float64)
    for b in range(w.B):
        ql, kl = int(w.q_lens[b]), int(w.k_lens[b])
        Q = f64(w.q[w.cu_seqlens_q[b] : w.cu_seqlens_q[b + 1]])            # [ql, Hq, D]
        K = f64(gather(kc, w.block_tables[b], kl, w.bs))                     # [kl, Hkv, D]
        V = f64(gather(vc, w.block_tables[b], kl, w.bs))
        Kh = np.repeat(K, w.G, axis=1)                                       # [kl, Hq, D]
        Vh = np.repeat(V, w.G, axis=1)
        S = np.einsum("ihd,jhd->hij", Q, Kh) * w.scale                       # [Hq, ql, kl]
        allowed = np.arange(kl)[None, :] <= (kl - ql + np.arange(ql))[:, None]
        S = np.where(allowed[None], S, -np.inf)
        P = np.exp(S - S.max(-1, keepdims=True))
        P /= P.sum(-1, keepdims=True)
        ref = np.einsum("hij,jhd->ihd", P, Vh)
        np.testing.assert_allclose(got[w.cu_seqlens_q[b] : w.cu_seqlens_q[b + 1]], ref,
                                   rtol=0, atol=1e-12)


def test_first_token_of_a_fresh_sequence_returns_its_own_v():
    rng = np.random.default_rng(42)
    w = _random(rng, 4, 32, 16, q_lens=[9, 5], cached=[0, 0])
    kc, vc = stored(w)
    got = oracle.paged_prefill(w.q, kc, vc, w.block_tables, w.cu_seqlens_q, w.cu_seqlens_k,
                               w.scale)
    for b in range(w.B):
        r = int(w.cu_seqlens_q[b])
        v0 = wl.bf16_bits_to_f32(gather(vc, w.block_tables[b], 1, w.bs)[0]).astype(np.float64)
        for h in range(w.Hq):
            np.testing.assert_array_equal(got[r, h], v0[h // w.G])


def test_identical_keys_give_the_running_mean_of_v():
    rng = np.random.default_rng(43)
    w = _random(rng, 2, 16, 16, q_lens=[6, 11], cached=[16, 0])
    kc, vc = stored(w)
    for b in range(w.B):
        t0 = w.block_tables[b, 0]
        for pos in range(int(w.k_lens[b])):
            kc[w.block_tables[b, pos // w.bs], pos % w.bs] = kc[t0, 0]
    got = oracle.paged_prefill(w.q, kc, vc, w.block_tables, w.cu_seqlens_q, w.cu_seqlens_k,
                               w.scale)
    for b in range(w.B):
        ql, kl = int(w.q_lens[b]), int(w.k_lens[b])
        V = wl.bf16_bits_to_f32(gather(vc, w.block_tables[b], kl, w.bs)).astype(np.float64)
        for i in range(ql):
            pos = kl - ql + i
            mean = V[: pos + 1].mean(0)
            for h in range(w.Hq):
                np.testing.assert_allclose(got[w.cu_seqlens_q[b] + i, h], mean[h // w.G],
                                           rtol=0, atol=1e-12)


def test_block_permutation_leaves_prefill_unchanged():
    rng = np.random.default_rng(44)
    w = _random(rng, 2, 16, 16, q_lens=[4, 20, 9], cached=[32, 0, 16])
    kc, vc = stored(w)
    a = oracle.paged_prefill(w.q, kc, vc, w.block_tables, w.cu_seqlens_q, w.cu_seqlens_k,
                             w.scale)
    pi = rng.permutation(w.NB)
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[pi], vc2[pi] = kc, vc
    tables = np.where(w.block_tables >= 0, pi[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    b = oracle.paged_prefill(w.q, kc2, vc2, tables, w.cu_seqlens_q, w.cu_seqlens_k, w.scale)
    np.testing.assert_array_equal(a, b)


def test_one_token_prefill_is_the_decode_step():
    """A prefill of one new token is the decode of that token (same definition)."""
    rng = np.random.default_rng(45)
    w = _random(rng, 4, 32, 16, q_lens=[1, 1, 1], cached=[0, 32, 48])
    kc, vc = stored(w)
    got = oracle.paged_prefill(w.q, kc, vc, w.block_tables, w.cu_seqlens_q, w.cu_seqlens_k,
                               w.scale)
    dec = oracle.paged_attn_decode(w.q, kc, vc, w.block_tables, w.k_lens, w.scale)
    np.testing.assert_array_equal(got, dec)


def test_sampled_pairs_equal_the_full_result():
    rng = np.random.default_rng(46)
    w = _random(rng, 2, 16, 16, q_lens=[5, 17], cached=[16, 0])
    kc, vc = stored(w)
    full = oracle.paged_prefill(w.q, kc, vc, w.block_tables, w.cu_seqlens_q, w.cu_seqlens_k,
                                w.scale)
    pairs = np.array([[0, 3], [21, 0], [5, 1], [6, 2]], np.int32)
    part = oracle.paged_prefill(w.q, kc, vc, w.block_tables, w.cu_seqlens_q, w.cu_seqlens_k,
                                w.scale, pairs=pairs)
    for i, (r, h) in enumerate(pairs):
        np.testing.assert_array_equal(part[i], full[r, h])


def test_prefill_workload_layout():
    w = wl.prefill_config_workload(3)
    # a prefix-cache hit: every table starts with the same physical blocks
    n_shared = 2048 // w.bs
    assert (w.block_tables[:, :n_shared] == w.block_tables[0, :n_shared]).all()
    # new tokens get distinct slots in each sequence's own blocks, after the prefix
    assert len(np.unique(w.slot_mapping)) == w.Tq
    for b in range(w.B):
        s = w.slot_mapping[w.cu_seqlens_q[b] : w.cu_seqlens_q[b + 1]]
        pos = np.arange(int(w.k_lens[b]) - int(w.q_lens[b]), int(w.k_lens[b]))
        assert (s == w.block_tables[b, pos // w.bs].astype(np.int64) * w.bs + pos % w.bs).all()
    assert w.Tq == 16384 and int(w.k_lens.max()) <= 4096
