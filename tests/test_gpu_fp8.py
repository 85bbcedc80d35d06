"""GPU parity of the FP8 (E4M3) KV cache against the CPU oracle, through the C ABI.

The store is byte work: its codes must equal the oracle's bit for bit (NaN
inputs: both sides must write a NaN code; E4M3 has one NaN magnitude, and the
sign of a NaN carries nothing).  Decode is compared with the fp64 oracle run
over the same dequantized caches, so quantization error is common to both
sides; the bar is max-abs <= 1e-2 + 2^-8 |exact| (the extra term is the bf16
rounding of the output, since code * v_scale is in general not a bf16 value)
and mean-abs <= 1e-3.  Per-tensor scales follow amax / 448 (448 being the
largest E4M3 value) over the bf16 caches and the step's new rows.
"""

import numpy as np
import pytest

import oracle
from paged_kv_cache_85_gb300 import workload as wl

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-2
REL = 2.0 ** -8
MEAN_ABS = 1e-3


@pytest.fixture(scope="module")
def pkv(cuda_lib_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_kv_cache_85_gb300 as m

    m.load_library()
    return m


def bf16_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def u8_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits_host(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def amax_scale(*arrays):
    m = max(float(np.abs(wl.bf16_bits_to_f32(a)).max()) if a.size else 0.0 for a in arrays)
    return float(np.float32(max(m, 1e-6) / 448.0))


class Fp8Case:
    """A bf16 workload with its caches quantized on the host by the oracle."""

    def __init__(self, w, with_store=True):
        self.w = w
        self.k_scale = amax_scale(w.k_cache, w.k_new)
        self.v_scale = amax_scale(w.v_cache, w.v_new)
        self.kc = oracle.quantize_bf16(w.k_cache, self.k_scale)
        self.vc = oracle.quantize_bf16(w.v_cache, self.v_scale)
        slots = w.slot_mapping if with_store else np.full_like(w.slot_mapping, -1)
        self.slots = slots
        self.kc2, self.vc2, bad = oracle.store_kvcache_fp8(w.k_new, w.v_new, self.kc, self.vc,
                                                          slots, self.k_scale, self.v_scale)
        assert bad == 0

    def reference(self, pairs=None):
        w = self.w
        return oracle.paged_attn_decode_fp8(w.q, self.kc2, self.vc2, w.block_tables,
                                            w.context_lens, w.scale, self.k_scale, self.v_scale,
                                            pairs=pairs)

    def device(self):
        w = self.w
        return dict(q=bf16_dev(w.q), kc=u8_dev(self.kc), vc=u8_dev(self.vc),
                    k_new=bf16_dev(w.k_new), v_new=bf16_dev(w.v_new),
                    slots=torch.from_numpy(self.slots).cuda(),
                    tables=torch.from_numpy(w.block_tables).cuda(),
                    lens=torch.from_numpy(w.context_lens).cuda())


def run_step(pkv, c, d, max_ctas=0, err=None):
    pkv.store_kvcache_fp8(d["k_new"], d["v_new"], d["kc"], d["vc"], d["slots"], c.k_scale,
                          c.v_scale, err_flag=err)
    out = torch.empty_like(d["q"])
    pkv.paged_attn_decode_fp8(d["q"], d["kc"], d["vc"], d["tables"], d["lens"], c.w.scale,
                              c.k_scale, c.v_scale, out, max_ctas=max_ctas, err_flag=err)
    torch.cuda.synchronize()
    return out


def compare(out, ref, what=""):
    got = wl.bf16_bits_to_f32(bits_host(out)).astype(np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = MAX_ABS + REL * np.abs(ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), f"{what}: err {err[worst]:.3e} > {bound[worst]:.3e} at {worst}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean-abs {err.mean():.3e}"
    return float(err.max()), float(err.mean())


# ---------------------------------------------------------------- quantizer


@pytest.mark.parametrize("scale", [1.0, 0.0137, 3.7, 2.0 ** -6, 1e-30])
def test_store_quantizer_every_bf16_pattern(pkv, scale):
    """All 65536 bf16 inputs (K) and the same reversed (V) through the store."""
    Hkv, D, bs = 8, 128, 16
    x = np.arange(65536, dtype=np.uint16).reshape(64, Hkv, D)
    y = x[::-1].reshape(64, Hkv, D).copy()
    slots = np.arange(64, dtype=np.int64)
    zero = np.zeros((4, bs, Hkv, D), np.uint8)
    kc, vc, bad = oracle.store_kvcache_fp8(x, y, zero, zero, slots, scale, scale)
    assert bad == 0
    dk, dv = u8_dev(zero), u8_dev(zero)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.store_kvcache_fp8(bf16_dev(x), bf16_dev(y), dk, dv, torch.from_numpy(slots).cuda(),
                          scale, scale, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for got, exp, src in ((dk.cpu().numpy(), kc, x), (dv.cpu().numpy(), vc, y)):
        got, exp = got.reshape(-1), exp.reshape(-1)
        srcf = wl.bf16_bits_to_f32(src.reshape(-1))
        nan = np.isnan(srcf)
        np.testing.assert_array_equal(got[~nan], exp[~nan])
        assert ((got[nan] & 0x7F) == 0x7F).all() and ((exp[nan] & 0x7F) == 0x7F).all()


def test_store_fp8_skips_padding_and_flags_bad_slots(pkv):
    rng = np.random.default_rng(21)
    w = wl.make_workload("rand", B=3, Hq=4, Hkv=2, D=64, bs=16, context_lens=[5, 40, 300], rng=rng)
    c = Fp8Case(w)
    d = c.device()
    before = d["kc"].cpu().numpy().copy()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    d["slots"] = torch.tensor([-1, w.NB * w.bs, -5], dtype=torch.int64, device="cuda")
    pkv.store_kvcache_fp8(d["k_new"], d["v_new"], d["kc"], d["vc"], d["slots"], c.k_scale,
                          c.v_scale, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.FLAG_BAD_SLOT
    np.testing.assert_array_equal(d["kc"].cpu().numpy(), before)


# ---------------------------------------------------------------- decode

_cache = {}


def config_case(idx):
    if idx not in _cache:
        _cache.clear()
        c = Fp8Case(wl.config_workload(idx))
        _cache[idx] = (c, c.reference())
    return _cache[idx]


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_config_store_bitexact_and_decode_parity(pkv, idx):
    c, ref = config_case(idx)
    d = c.device()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_step(pkv, c, d, err=err)
    assert int(err.item()) == 0
    np.testing.assert_array_equal(d["kc"].cpu().numpy(), c.kc2)
    np.testing.assert_array_equal(d["vc"].cpu().numpy(), c.vc2)
    compare(out, ref, c.w.name)


@pytest.mark.parametrize("ctas", [1, 2, 3, 5, 0])
def test_grid_size_invariance_tiny(pkv, ctas):
    c, ref = config_case(0)
    out = run_step(pkv, c, c.device(), max_ctas=ctas)
    compare(out, ref, f"max_ctas={ctas}")


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [16, 32, 48, 256])
def test_group_dim_block_variants(pkv, G, D, bs):
    rng = np.random.default_rng(300 + G * 7 + D + bs)
    lens = [1, 15, 16, 17, 63, 64, 65, 257, 700][: 5 + G // 2]
    w = wl.make_workload("rand", B=len(lens), Hq=G * 2, Hkv=2, D=D, bs=bs, context_lens=lens,
                         rng=rng)
    c = Fp8Case(w)
    ref = c.reference()
    for ctas in (0, 1, 3):
        out = run_step(pkv, c, c.device(), max_ctas=ctas)
        compare(out, ref, f"G={G} D={D} bs={bs} max_ctas={ctas}")


@pytest.mark.parametrize("bs", [16, 256])
def test_context_len_one_returns_dequantized_v(pkv, bs):
    rng = np.random.default_rng(22)
    w = wl.make_workload("rand", B=6, Hq=8, Hkv=2, D=128, bs=bs, context_lens=[1] * 6, rng=rng)
    c = Fp8Case(w)
    out = wl.bf16_bits_to_f32(bits_host(run_step(pkv, c, c.device()))).astype(np.float64)
    for b in range(6):
        blk = w.block_tables[b, 0]
        for h in range(8):
            v = oracle.dequant_fp8(c.vc2[blk, 0, h // 4], c.v_scale)
            assert (np.abs(out[b, h] - v) <= REL * np.abs(v)).all()


@pytest.mark.parametrize("bs", [16, 32, 256])
def test_nan_codes_in_unread_slots_change_nothing(pkv, bs):
    # G = 4 at D = 128: 32-token boxes where bs allows
    rng = np.random.default_rng(23)
    lens = [1, 17, 40, 300, 33, 5, 48]
    w = wl.make_workload("rand", B=7, Hq=8, Hkv=2, D=128, bs=bs, context_lens=lens, rng=rng)
    c = Fp8Case(w)
    clean = bits_host(run_step(pkv, c, c.device(), max_ctas=2))
    # mark every slot no sequence reads with the E4M3 NaN code
    kc, vc = c.kc2.copy(), c.vc2.copy()
    used = np.zeros((w.NB, w.bs), bool)
    for b in range(w.B):
        for t in range(int(w.context_lens[b])):
            used[w.block_tables[b, t // w.bs], t % w.bs] = True
    kc[~used], vc[~used] = 0x7F, 0xFF
    c.kc, c.vc, c.slots = kc, vc, np.full_like(w.slot_mapping, -1)
    out = bits_host(run_step(pkv, c, c.device(), max_ctas=2))
    assert np.isfinite(wl.bf16_bits_to_f32(out)).all()
    np.testing.assert_array_equal(out, clean)


@pytest.mark.parametrize("bs", [32, 64])
@pytest.mark.parametrize("D,G,B", [(128, 4, 18), (64, 8, 4000)])
def test_box_tails_of_32_token_boxes(pkv, D, G, B, bs):
    """Where three CTAs per SM hold fewer than four stages of 16-token boxes
    and the block size is a multiple of 32, the kernel takes 32-token boxes
    (two 16-token MMA tiles each).  G = 4 at D = 128 is such a shape; at
    D = 64 it takes B in the thousands (the per-sequence arrays share the
    CTA's shared memory).  Every tail length of a box, including a second
    half with no valid token, and slices cut at odd box positions."""
    rng = np.random.default_rng(400 + D + bs)
    tails = [1, 2, 15, 16, 17, 31, 32, 33, 47, 48, 49, 63, 64, 65, 95, 96, 97, 130]
    lens = [tails[i % len(tails)] for i in range(B)]
    w = wl.make_workload("rand", B=B, Hq=2 * G, Hkv=2, D=D, bs=bs, context_lens=lens, rng=rng)
    c = Fp8Case(w)
    ref = c.reference()
    for ctas in (0, 1, 2, 7):
        out = run_step(pkv, c, c.device(), max_ctas=ctas)
        compare(out, ref, f"D={D} G={G} B={B} bs={bs} max_ctas={ctas}")


@pytest.mark.parametrize("bs", [16, 32])
def test_bad_block_drops_only_its_tokens(pkv, bs):
    """A bad block id in a table drops that block's tokens from the softmax
    and flags PKV_FLAG_BAD_BLOCK (G = 4, D = 128: 16-token boxes at bs = 16,
    32-token boxes at bs = 32).  Decode attention does not depend on token
    order, so the expected result is the oracle's over the table without
    that block."""
    rng = np.random.default_rng(500 + bs)
    lens = [100, 37, 260, 9, 100, 64]
    w = wl.make_workload("rand", B=len(lens), Hq=8, Hkv=2, D=128, bs=bs, context_lens=lens,
                         rng=rng)
    c = Fp8Case(w)
    ref = c.reference()
    bad_b, bad_j = 4, 2  # a full block in the middle of a 100-token context
    tables = w.block_tables.copy()
    tables[bad_b, bad_j:-1] = w.block_tables[bad_b, bad_j + 1:]
    tables[bad_b, -1] = -1
    lens2 = w.context_lens.copy()
    lens2[bad_b] -= bs
    ref[bad_b] = oracle.paged_attn_decode_fp8(w.q, c.kc2, c.vc2, tables, lens2, w.scale, c.k_scale,
                                              c.v_scale)[bad_b]
    for ctas in (0, 3):
        d = c.device()
        bad = d["tables"].clone()
        bad[bad_b, bad_j] = w.NB + 11
        d["tables"] = bad
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = run_step(pkv, c, d, max_ctas=ctas, err=err)
        assert int(err.item()) & pkv.FLAG_BAD_BLOCK
        compare(out, ref, f"bs={bs} max_ctas={ctas}")


def test_fp8_dtype_caches_are_accepted(pkv):
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    c, ref = config_case(0)
    d = c.device()
    d["kc"], d["vc"] = d["kc"].view(torch.float8_e4m3fn), d["vc"].view(torch.float8_e4m3fn)
    compare(run_step(pkv, c, d), ref, "float8_e4m3fn views")


def test_cuda_graph_capture_and_replay(pkv):
    c, ref = config_case(0)
    d = c.device()
    out = torch.empty_like(d["q"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run_step(pkv, c, d)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pkv.store_kvcache_fp8(d["k_new"], d["v_new"], d["kc"], d["vc"], d["slots"],
                                  c.k_scale, c.v_scale)
            pkv.paged_attn_decode_fp8(d["q"], d["kc"], d["vc"], d["tables"], d["lens"],
                                      c.w.scale, c.k_scale, c.v_scale, out)
    for _ in range(3):
        out.zero_()
        g.replay()
    torch.cuda.synchronize()
    compare(out, ref, "graph replay")
