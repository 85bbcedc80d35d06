"""Pins for the FP8 (E4M3) cache path of the oracle.

E4M3 per the OCP FP8 format ("e4m3fn"): 1 sign, 4 exponent (bias 7) and 3
mantissa bits, subnormals at exponent field 0, no infinities, S.1111.111 is
NaN, largest finite 448.  Quantization: nearest, ties to even, saturating.
The page ("VLLM-0.7.3 源码" §5.3) asks only for FP8 storage with higher-
precision compute; the per-tensor scale convention is this build's reading.
"""

import math

import numpy as np
import pytest

import oracle
from paged_kv_cache_85_gb300 import workload as wl


@pytest.mark.parametrize("x,code", [
    (0.0, 0x00), (-0.0, 0x80), (1.0, 0x38), (-1.0, 0xB8), (448.0, 0x7E), (-448.0, 0xFE),
    (0.875, 0x36), (3.0, 0x44), (2.0 ** -9, 0x01), (2.0 ** -6, 0x08), (7 * 2.0 ** -9, 0x07),
    (1.0625, 0x38),    # halfway 1.0 / 1.125 -> even mantissa (1.0)
    (1.1875, 0x3A),    # halfway 1.125 / 1.25 -> even mantissa (1.25)
    (2.0 ** -10, 0x00),  # halfway 0 / 2^-9 -> even (0)
    (3 * 2.0 ** -10, 0x02),  # halfway 2^-9 / 2^-8 -> even (2 * 2^-9)
    (464.0, 0x7E), (1000.0, 0x7E), (float("inf"), 0x7E), (float("-inf"), 0xFE),
])
def test_e4m3_encode_known_values(x, code):
    assert oracle.e4m3_encode(x) == code


def test_e4m3_decode_table_and_round_trip():
    finite = [c for c in range(256) if (c & 0x7F) != 0x7F]
    for c in finite:
        v = oracle.e4m3_decode(c)
        assert math.isfinite(v)
        assert oracle.e4m3_encode(v) == c or (v == 0 and c in (0x00, 0x80))
    pos = [oracle.e4m3_decode(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))  # strictly increasing magnitudes
    assert pos[-1] == 448.0 and pos[1] == 2.0 ** -9
    assert math.isnan(oracle.e4m3_decode(0x7F)) and math.isnan(oracle.e4m3_decode(0xFF))
    assert math.isnan(oracle.e4m3_decode(0x7F))


def test_e4m3_encode_is_nearest():
    rng = np.random.default_rng(0)
    table = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])
    for x in rng.standard_normal(400) * 10.0 ** rng.integers(-3, 3, 400):
        c = oracle.e4m3_encode(x)
        v = abs(oracle.e4m3_decode(c))
        err = np.abs(table - min(abs(x), 448.0)).min()
        assert abs(v - min(abs(x), 448.0)) == pytest.approx(err, abs=0, rel=0) or abs(x) >= 448
        assert (c & 0x80) == (0x80 if np.signbit(x) else 0)


def test_store_fp8_quantizes_into_the_same_slots():
    rng = np.random.default_rng(1)
    NB, bs, Hkv, D, N = 6, 16, 2, 8, 9
    k = wl.f32_to_bf16_bits(rng.standard_normal((N, Hkv, D), dtype=np.float32))
    v = wl.f32_to_bf16_bits(rng.standard_normal((N, Hkv, D), dtype=np.float32))
    slots = rng.choice(NB * bs, size=N, replace=False).astype(np.int64)
    slots[4] = -1
    z = np.zeros((NB, bs, Hkv, D), np.uint8)
    ks, vs = 0.05, 0.02
    kc, vc, bad = oracle.store_kvcache_fp8(k, v, z, z, slots, ks, vs)
    assert bad == 0
    flat_k, flat_v = kc.reshape(NB * bs, Hkv * D), vc.reshape(NB * bs, Hkv * D)
    kinv, vinv = np.float32(1.0) / np.float32(ks), np.float32(1.0) / np.float32(vs)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        kx = wl.bf16_bits_to_f32(k[i]).reshape(-1) * kinv
        vx = wl.bf16_bits_to_f32(v[i]).reshape(-1) * vinv
        assert list(flat_k[s]) == [oracle.e4m3_encode(x) for x in kx]
        assert list(flat_v[s]) == [oracle.e4m3_encode(x) for x in vx]
    written = set(int(s) for s in slots if s >= 0)
    for s in range(NB * bs):
        if s not in written:
            assert (flat_k[s] == 0).all() and (flat_v[s] == 0).all()


def test_fp8_decode_equals_bf16_decode_on_representable_values():
    """With scale 1 and E4M3-representable K/V, both oracles see the same numbers."""
    rng = np.random.default_rng(2)
    B, Hq, Hkv, D, bs, NB = 3, 4, 2, 16, 16, 8
    codes_k = rng.integers(0, 0x7F, (NB, bs, Hkv, D)).astype(np.uint8) | (rng.integers(0, 2, (NB, bs, Hkv, D)).astype(np.uint8) << 7)
    codes_v = rng.integers(0, 0x7F, (NB, bs, Hkv, D)).astype(np.uint8) | (rng.integers(0, 2, (NB, bs, Hkv, D)).astype(np.uint8) << 7)
    codes_k = np.where(codes_k & 0x7F == 0x7F, 0, codes_k).astype(np.uint8)
    codes_v = np.where(codes_v & 0x7F == 0x7F, 0, codes_v).astype(np.uint8)
    kb = wl.f32_to_bf16_bits(oracle.dequant_fp8(codes_k, 1.0).astype(np.float32))
    vb = wl.f32_to_bf16_bits(oracle.dequant_fp8(codes_v, 1.0).astype(np.float32))
    q = wl.f32_to_bf16_bits(rng.standard_normal((B, Hq, D), dtype=np.float32) * 0.01)
    tables = np.array([[0, 1], [2, 3], [5, 4]], np.int32)
    lens = np.array([20, 32, 7], np.int32)
    a = oracle.paged_attn_decode_fp8(q, codes_k, codes_v, tables, lens, 0.25, 1.0, 1.0)
    b = oracle.paged_attn_decode(q, kb, vb, tables, lens, 0.25)
    np.testing.assert_array_equal(a, b)


def test_fp8_decode_scales_are_applied():
    """V scaled by s scales the output by s; K scaled by s scales the scores by s."""
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 0x70, (4, 16, 1, 8)).astype(np.uint8)
    q = wl.f32_to_bf16_bits(rng.standard_normal((1, 1, 8), dtype=np.float32))
    tables, lens = np.array([[0, 1]], np.int32), np.array([30], np.int32)
    base = oracle.paged_attn_decode_fp8(q, codes, codes, tables, lens, 0.5, 1.0, 1.0)
    vs = oracle.paged_attn_decode_fp8(q, codes, codes, tables, lens, 0.5, 1.0, 0.25)
    np.testing.assert_allclose(vs, 0.25 * base, rtol=1e-14)
    ks = oracle.paged_attn_decode_fp8(q, codes, codes, tables, lens, 0.25, 2.0, 1.0)
    np.testing.assert_allclose(ks, base, rtol=1e-13)  # scale 0.25 * k_scale 2 == scale 0.5


def test_table_quantizer_equals_the_plain_store():
    """The memoised quantizer gives the plain store's codes for every input."""
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 65536, size=(40, 2, 64)).astype(np.uint16)
    slots = np.arange(40, dtype=np.int64)
    cache = np.zeros((10, 4, 2, 64), np.uint8)
    for scale in (1.0, 0.0137, 3.7):
        kc, vc, bad = oracle.store_kvcache_fp8(bits, bits, cache, cache, slots, scale, scale)
        assert bad == 0
        np.testing.assert_array_equal(oracle.quantize_bf16(bits, scale), kc.reshape(40, 2, 64))
