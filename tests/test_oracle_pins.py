"""Pins for the CPU oracle: facts fixed by the pages or by mathematics.

Each test here checks the oracle against something other than itself: a
hand-derived worked example, a closed form, an invariant the definition
implies, a special case that reduces to a library routine, or an
independent brute force.  Each is chosen so that a plausible slip in the
oracle (a dropped term, a wrong sign, a wrong head or block index, a
transposed layout) fails at least one of them.
"""

import math
import os

import numpy as np
import pytest

import oracle
from paged_kv_cache_85_gb300 import workload as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _read_fixture(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rows[key] = vals
    return rows


def _bits(vals):
    return np.array([int(x, 0) for x in vals], dtype=np.uint16)


def _bf16(x):
    return wl.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _tiny(rng, B=3, Hq=4, Hkv=2, D=8, bs=4, ctx=(1, 5, 11), NB=12, values="normal"):
    """A small paged problem with a random block placement."""
    ctx = np.asarray(ctx, dtype=np.int32)
    nblk = (ctx + bs - 1) // bs
    MBS = int(nblk.max())
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.full((B, MBS), -1, dtype=np.int32)
    cur = 0
    for b in range(B):
        tables[b, : nblk[b]] = perm[cur : cur + nblk[b]]
        cur += nblk[b]
    if values == "normal":
        q = _bf16(rng.standard_normal((B, Hq, D)))
        kc = _bf16(rng.standard_normal((NB, bs, Hkv, D)))
        vc = _bf16(rng.standard_normal((NB, bs, Hkv, D)))
    else:  # small integers: every sum below is exact
        q = _bf16(rng.integers(-3, 4, (B, Hq, D)))
        kc = _bf16(rng.integers(-3, 4, (NB, bs, Hkv, D)))
        vc = _bf16(rng.integers(-3, 4, (NB, bs, Hkv, D)))
    return q, kc, vc, tables, ctx


def _f(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------- store


def test_store_golden_layout():
    fx = _read_fixture("store_layout_tiny.txt")
    shp = dict(kv.split("=") for kv in fx["shape"])
    NB, bs, Hkv, D = (int(shp[k]) for k in ("NB", "bs", "Hkv", "D"))
    slots = np.array([int(s) for s in fx["slots"]], dtype=np.int64)
    k = _bits(fx["k"]).reshape(-1, Hkv, D)
    v = _bits(fx["v"]).reshape(-1, Hkv, D)
    z = np.zeros((NB, bs, Hkv, D), dtype=np.uint16)
    kc, vc, bad = oracle.store_kvcache(k, v, z, z, slots)
    assert bad == 0
    np.testing.assert_array_equal(kc.reshape(-1), _bits(fx["k_cache"]))
    np.testing.assert_array_equal(vc.reshape(-1), _bits(fx["v_cache"]))


def test_store_matches_fancy_index_and_skips_padding():
    rng = np.random.default_rng(1)
    NB, bs, Hkv, D, N = 7, 16, 3, 16, 40
    kc0 = rng.integers(0, 1 << 16, (NB, bs, Hkv, D), dtype=np.uint16)
    vc0 = rng.integers(0, 1 << 16, (NB, bs, Hkv, D), dtype=np.uint16)
    k = rng.integers(0, 1 << 16, (N, Hkv, D), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, (N, Hkv, D), dtype=np.uint16)
    slots = rng.choice(NB * bs, size=N, replace=False).astype(np.int64)
    slots[::7] = -1
    kc, vc, bad = oracle.store_kvcache(k, v, kc0, vc0, slots)
    assert bad == 0
    ek, ev = kc0.copy().reshape(NB * bs, Hkv, D), vc0.copy().reshape(NB * bs, Hkv, D)
    m = slots >= 0
    ek[slots[m]] = k[m]
    ev[slots[m]] = v[m]
    np.testing.assert_array_equal(kc.reshape(NB * bs, Hkv, D), ek)
    np.testing.assert_array_equal(vc.reshape(NB * bs, Hkv, D), ev)


def test_store_out_of_range_is_counted_and_skipped():
    NB, bs, Hkv, D = 2, 16, 1, 8
    z = np.zeros((NB, bs, Hkv, D), dtype=np.uint16)
    k = np.full((3, Hkv, D), 0x3F80, dtype=np.uint16)
    slots = np.array([NB * bs, -5, 3], dtype=np.int64)
    kc, vc, bad = oracle.store_kvcache(k, k, z, z, slots)
    assert bad == 2
    assert (kc.reshape(-1, D)[3] == 0x3F80).all()
    assert int((kc != 0).sum()) == D


# ------------------------------------------------------------- decode


def test_attn_two_token_closed_form():
    fx = _read_fixture("attn_two_token.txt")
    q = _bf16([float(x) for x in fx["q"]]).reshape(1, 1, 2)
    kk = _bf16([float(x) for x in fx["k"]]).reshape(2, 1, 2)
    vv = _bf16([float(x) for x in fx["v"]]).reshape(2, 1, 2)
    scale = float(np.float32(math.log(float(fx["scale_ln"][0]))))
    blk = int(fx["block"][0])
    NB, bs = 4, 16
    kc = np.zeros((NB, bs, 1, 2), dtype=np.uint16)
    vc = np.zeros_like(kc)
    kc[blk, :2] = kk
    vc[blk, :2] = vv
    out = oracle.paged_attn_decode(q, kc, vc, np.array([[blk]], np.int32),
                                   np.array([2], np.int32), scale)
    expect = np.array([float(x) for x in fx["out"]])
    np.testing.assert_allclose(out[0, 0], expect, rtol=0, atol=1e-6)


def test_brute_force_tiny():
    """Independent explicit score matrix / softmax / weighted sum in numpy."""
    rng = np.random.default_rng(2)
    for trial in range(4):
        B, Hq, Hkv, D, bs = 3, 6, 2, 8, 4
        ctx = rng.integers(1, 14, B)
        NB = int(((ctx + bs - 1) // bs).sum()) + 3
        q, kc, vc, tables, ctx = _tiny(rng, B, Hq, Hkv, D, bs, ctx, NB)
        scale = float(np.float32(0.37))
        got = oracle.paged_attn_decode(q, kc, vc, tables, ctx, scale)
        G = Hq // Hkv
        for b in range(B):
            n = int(ctx[b])
            toks = [(tables[b, t // bs], t % bs) for t in range(n)]
            for h in range(Hq):
                K = np.stack([_f(kc[p, o, h // G]) for p, o in toks])
                V = np.stack([_f(vc[p, o, h // G]) for p, o in toks])
                s = scale * (K @ _f(q[b, h]))
                w = np.exp(s - s.max())
                ref = (w[:, None] * V).sum(0) / w.sum()
                np.testing.assert_allclose(got[b, h], ref, rtol=1e-12, atol=1e-13)


def test_ctx1_returns_v_exactly():
    rng = np.random.default_rng(3)
    q, kc, vc, tables, ctx = _tiny(rng, ctx=(1, 1, 1))
    out = oracle.paged_attn_decode(q, kc, vc, tables, ctx, 0.5)
    G = 2
    for b in range(3):
        for h in range(4):
            np.testing.assert_array_equal(out[b, h], _f(vc[tables[b, 0], 0, h // G]))


def test_ctx0_gives_zeros():
    rng = np.random.default_rng(4)
    q, kc, vc, tables, ctx = _tiny(rng, ctx=(3, 5, 2))
    ctx = np.array([0, 5, 0], np.int32)
    out = oracle.paged_attn_decode(q, kc, vc, tables, ctx, 0.5)
    assert (out[0] == 0).all() and (out[2] == 0).all()
    assert np.abs(out[1]).sum() > 0


def test_identical_keys_give_mean_of_v():
    rng = np.random.default_rng(5)
    q, kc, vc, tables, ctx = _tiny(rng, ctx=(4, 9, 13))
    bs = kc.shape[1]
    G = 2
    for b in range(3):  # every context token of a sequence gets the same key
        for t in range(int(ctx[b])):
            kc[tables[b, t // bs], t % bs] = kc[tables[b, 0], 0]
    out = oracle.paged_attn_decode(q, kc, vc, tables, ctx, 0.7)
    for b in range(3):
        n = int(ctx[b])
        for h in range(4):
            V = np.stack([_f(vc[tables[b, t // bs], t % bs, h // G]) for t in range(n)])
            np.testing.assert_allclose(out[b, h], V.mean(0), rtol=1e-13, atol=1e-14)


def test_hard_attention_limit_picks_argmax_key():
    """A huge scale turns softmax into a one-hot on the largest score."""
    rng = np.random.default_rng(6)
    q, kc, vc, tables, ctx = _tiny(rng, ctx=(7, 12, 5), D=16)
    bs, G = kc.shape[1], 2
    out = oracle.paged_attn_decode(q, kc, vc, tables, ctx, 1.0e6)
    for b in range(3):
        n = int(ctx[b])
        for h in range(4):
            K = np.stack([_f(kc[tables[b, t // bs], t % bs, h // G]) for t in range(n)])
            dots = K @ _f(q[b, h])
            order = np.sort(dots)
            if n > 1 and order[-1] - order[-2] < 1e-3:
                continue  # near tie: the limit is not one-hot at this scale
            t = int(np.argmax(dots))
            np.testing.assert_allclose(out[b, h], _f(vc[tables[b, t // bs], t % bs, h // G]),
                                       rtol=0, atol=1e-12)


def test_gqa_head_mapping():
    """Query head h reads KV head h // (Hq/Hkv): give each KV head a constant V."""
    rng = np.random.default_rng(7)
    Hq, Hkv = 8, 2
    q, kc, vc, tables, ctx = _tiny(rng, Hq=Hq, Hkv=Hkv, ctx=(3, 9, 6))
    for j in range(Hkv):
        vc[:, :, j, :] = _bf16(np.full(vc.shape[-1], float(j + 1)))
    out = oracle.paged_attn_decode(q, kc, vc, tables, ctx, 0.3)
    for h in range(Hq):
        np.testing.assert_allclose(out[:, h], float(h // (Hq // Hkv) + 1), rtol=1e-14)


def test_block_permutation_invariance_bitwise():
    rng = np.random.default_rng(8)
    q, kc, vc, tables, ctx = _tiny(rng, ctx=(6, 13, 9), NB=16)
    out = oracle.paged_attn_decode(q, kc, vc, tables, ctx, 0.25)
    NB = kc.shape[0]
    pi = rng.permutation(NB)
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[pi] = kc
    vc2[pi] = vc
    t2 = np.where(tables >= 0, pi[np.maximum(tables, 0)], -1).astype(np.int32)
    out2 = oracle.paged_attn_decode(q, kc2, vc2, t2, ctx, 0.25)
    np.testing.assert_array_equal(out, out2)


def test_equals_dense_attention_over_gathered_kv():
    rng = np.random.default_rng(9)
    q, kc, vc, tables, ctx = _tiny(rng, ctx=(6, 13, 9), NB=16)
    bs = kc.shape[1]
    out = oracle.paged_attn_decode(q, kc, vc, tables, ctx, 0.25)
    for b in range(3):
        n = int(ctx[b])
        idx = np.arange(n)
        K = kc[tables[b, idx // bs], idx % bs]
        V = vc[tables[b, idx // bs], idx % bs]
        dense = oracle.dense_attn(q[b], K, V, 0.25)
        np.testing.assert_array_equal(out[b], dense)


def test_unread_slots_do_not_matter():
    """NaN in every slot past the context (and -1 past the used table) changes nothing."""
    rng = np.random.default_rng(10)
    q, kc, vc, tables, ctx = _tiny(rng, ctx=(6, 13, 9), NB=16)
    out = oracle.paged_attn_decode(q, kc, vc, tables, ctx, 0.25)
    kc2, vc2 = kc.copy(), vc.copy()
    wl.poison_unused_slots(kc2, vc2, tables, ctx, kc.shape[1])
    assert (kc2 == wl.BF16_NAN).sum() > 0
    out2 = oracle.paged_attn_decode(q, kc2, vc2, tables, ctx, 0.25)
    assert np.isfinite(out2).all()
    np.testing.assert_array_equal(out, out2)


def test_shift_of_all_keys_along_a_fixed_vector_changes_nothing():
    """Adding c to every key adds scale*q.c to every score: softmax is unchanged."""
    rng = np.random.default_rng(11)
    q, kc, vc, tables, ctx = _tiny(rng, ctx=(6, 13, 9), NB=16, values="int")
    out = oracle.paged_attn_decode(q, kc, vc, tables, ctx, 0.125)
    c = rng.integers(-2, 3, kc.shape[-1]).astype(np.float32)
    kc2 = _bf16(wl.bf16_bits_to_f32(kc) + c)
    out2 = oracle.paged_attn_decode(q, kc2, vc, tables, ctx, 0.125)
    np.testing.assert_allclose(out, out2, rtol=1e-12, atol=1e-13)


def test_affine_in_v():
    """Weights sum to one: out(2V + 1) = 2 out(V) + 1."""
    rng = np.random.default_rng(12)
    q, kc, vc, tables, ctx = _tiny(rng, ctx=(6, 13, 9), NB=16, values="int")
    out = oracle.paged_attn_decode(q, kc, vc, tables, ctx, 0.125)
    vc2 = _bf16(2.0 * wl.bf16_bits_to_f32(vc) + 1.0)
    out2 = oracle.paged_attn_decode(q, kc, vc2, tables, ctx, 0.125)
    np.testing.assert_allclose(out2, 2 * out + 1, rtol=1e-12, atol=1e-12)


def test_pairs_subset_matches_full():
    rng = np.random.default_rng(13)
    q, kc, vc, tables, ctx = _tiny(rng, ctx=(6, 13, 9), NB=16)
    full = oracle.paged_attn_decode(q, kc, vc, tables, ctx, 0.25)
    pairs = np.array([[2, 3], [0, 1], [1, 0]], np.int32)
    sub = oracle.paged_attn_decode(q, kc, vc, tables, ctx, 0.25, pairs=pairs)
    for i, (b, h) in enumerate(pairs):
        np.testing.assert_array_equal(sub[i], full[b, h])


def test_invalid_table_entry_reported():
    rng = np.random.default_rng(14)
    q, kc, vc, tables, ctx = _tiny(rng, ctx=(6, 13, 9), NB=16)
    t2 = tables.copy()
    t2[1, 1] = 99  # past NB
    out = oracle.paged_attn_decode(q, kc, vc, t2, ctx, 0.25)
    assert (out[1] == 0).all()


def test_inplace_store_matches_functional_store():
    rng = np.random.default_rng(15)
    NB, bs, Hkv, D, N = 5, 16, 2, 8, 9
    kc0 = rng.integers(0, 1 << 16, (NB, bs, Hkv, D), dtype=np.uint16)
    vc0 = rng.integers(0, 1 << 16, (NB, bs, Hkv, D), dtype=np.uint16)
    k = rng.integers(0, 1 << 16, (N, Hkv, D), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, (N, Hkv, D), dtype=np.uint16)
    slots = rng.choice(NB * bs, size=N, replace=False).astype(np.int64)
    slots[3] = -1
    kc, vc, bad = oracle.store_kvcache(k, v, kc0, vc0, slots)
    kc2, vc2 = kc0.copy(), vc0.copy()
    assert oracle.store_kvcache_(k, v, kc2, vc2, slots) == bad == 0
    np.testing.assert_array_equal(kc, kc2)
    np.testing.assert_array_equal(vc, vc2)
