"""GPU parity of the paged prefill against the CPU oracle, through the C ABI.

The step is store_kvcache (bit-exact over the whole cache) then
paged_prefill.  Attention must match the fp64 oracle to max-abs <= 1e-2 and
mean-abs <= 1e-3 (bf16 in and out) over every output of every step, the
16k-token steps included: the oracle runs all their (token row, head) pairs,
split over the host's cores (each pair is computed on its own, so the split
changes no bit).
"""

import numpy as np
import pytest

import oracle
from paged_kv_cache_85_gb300 import workload as wl

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-2
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


def bits_host(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def to_dev(w):
    return dict(
        q=bf16_dev(w.q), k_cache=bf16_dev(w.k_cache), v_cache=bf16_dev(w.v_cache),
        k_new=bf16_dev(w.k_new), v_new=bf16_dev(w.v_new),
        slots=torch.from_numpy(w.slot_mapping).cuda(),
        tables=torch.from_numpy(w.block_tables).cuda(),
        cu_q=torch.from_numpy(w.cu_seqlens_q).cuda(), cu_k=torch.from_numpy(w.cu_seqlens_k).cuda(),
    )


def run_step(pkv, w, d, err=None, out=None, store=True):
    if store:
        pkv.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slots"],
                          err_flag=err)
    if out is None:
        out = torch.empty_like(d["q"])
    pkv.paged_prefill(d["q"], d["k_cache"], d["v_cache"], d["tables"], d["cu_q"], d["cu_k"],
                      w.max_seqlen_q, w.scale, out, err_flag=err)
    torch.cuda.synchronize()
    return out


def stored(w):
    kc, vc, bad = oracle.store_kvcache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    assert bad == 0
    return kc, vc


def compare(got, ref, what=""):
    got = wl.bf16_bits_to_f32(got).astype(np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= MAX_ABS, f"{what}: max-abs {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean-abs {err.mean():.3e}"
    return float(err.max()), float(err.mean())


_cache = {}


def config(idx):
    """Workload idx with its stored caches and the oracle's full [Tq, Hq, D]
    output (every row and head)."""
    if idx not in _cache:
        _cache.clear()
        w = wl.prefill_config_workload(idx)
        kc, vc = stored(w)
        ref = oracle.paged_prefill(w.q, kc, vc, w.block_tables, w.cu_seqlens_q, w.cu_seqlens_k,
                                   w.scale, threads=oracle.host_cores())
        _cache[idx] = (w, kc, vc, ref, None)
    return _cache[idx]


@pytest.mark.parametrize("idx", [0, 1, 2, 3])
def test_config_store_bitexact_and_prefill_parity(pkv, idx):
    w, kc, vc, ref, pairs = config(idx)
    d = to_dev(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_step(pkv, w, d, err=err)
    assert int(err.item()) == 0
    np.testing.assert_array_equal(bits_host(d["k_cache"]), kc)
    np.testing.assert_array_equal(bits_host(d["v_cache"]), vc)
    o = bits_host(out)
    assert np.isfinite(wl.bf16_bits_to_f32(o)).all()
    assert ref.shape == o.shape  # every output of the step
    compare(o, ref, w.name)


def _random(rng, G, D, bs, q_lens, cached, NB=None, Hkv=2, poison=False):
    return wl.make_prefill_workload("rand", Hq=G * Hkv, Hkv=Hkv, D=D, bs=bs, q_lens=q_lens,
                                    cached_lens=cached, NB=NB, rng=rng, poison_unused=poison)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [16, 32, 256])
def test_group_dim_block_variants(pkv, G, D, bs):
    rng = np.random.default_rng(500 + 7 * G + D + bs)
    q_lens = [1, 15, 16, 17, 63, 64, 65, 130, 200][: 4 + G // 2]
    cached = [bs * int(c) for c in rng.integers(0, 3, size=len(q_lens))]
    w = _random(rng, G, D, bs, q_lens, cached)
    kc, vc = stored(w)
    ref = oracle.paged_prefill(w.q, kc, vc, w.block_tables, w.cu_seqlens_q, w.cu_seqlens_k,
                               w.scale)
    compare(bits_host(run_step(pkv, w, to_dev(w))), ref, f"G={G} D={D} bs={bs}")


@pytest.mark.parametrize("n_seqs", [256, 300])
def test_many_sequences_every_tile_once(pkv, n_seqs):
    """Up to 256 sequences the CTAs take tiles longest first (ranked in the
    kernel); beyond that the launch order is used.  Both must cover every
    (sequence, head, tile) exactly once."""
    rng = np.random.default_rng(520 + n_seqs)
    q_lens = [int(x) for x in rng.integers(1, 90, size=n_seqs)]
    cached = [16 * int(c) for c in rng.integers(0, 5, size=n_seqs)]
    w = _random(rng, 2, 64, 16, q_lens, cached)
    kc, vc = stored(w)
    ref = oracle.paged_prefill(w.q, kc, vc, w.block_tables, w.cu_seqlens_q, w.cu_seqlens_k,
                               w.scale)
    compare(bits_host(run_step(pkv, w, to_dev(w))), ref, f"{n_seqs} sequences")


@pytest.mark.parametrize("n_seqs", [5, 300])
def test_loose_max_seqlen_q_gives_the_same_bits(pkv, n_seqs):
    """max_seqlen_q only bounds the work space: a bound far above every query
    length leaves most work positions empty, and the persistent CTAs must
    skip or stop at them and still produce every row, bit for bit."""
    rng = np.random.default_rng(530 + n_seqs)
    q_lens = [int(x) for x in rng.integers(1, 70, size=n_seqs)]
    cached = [16 * int(c) for c in rng.integers(0, 4, size=n_seqs)]
    w = _random(rng, 2, 64, 16, q_lens, cached)
    d = to_dev(w)
    tight = bits_host(run_step(pkv, w, d))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(d["q"])
    pkv.paged_prefill(d["q"], d["k_cache"], d["v_cache"], d["tables"], d["cu_q"], d["cu_k"],
                      8 * w.max_seqlen_q, w.scale, out, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    np.testing.assert_array_equal(bits_host(out), tight)


def test_long_context_rows_across_many_tiles(pkv):
    """One long sequence (cached 1024 + 700 new) at G = 2: many K tiles and query tiles."""
    rng = np.random.default_rng(510)
    w = _random(rng, 2, 128, 256, [700, 3], [1024, 256])
    kc, vc = stored(w)
    ref = oracle.paged_prefill(w.q, kc, vc, w.block_tables, w.cu_seqlens_q, w.cu_seqlens_k,
                               w.scale)
    compare(bits_host(run_step(pkv, w, to_dev(w))), ref, "long")


def f16_rounded(bits):
    """bf16 bits of V as the kernel's P.V sees it: rounded to f16 (exact for
    |v| >= 2^-17, where f16 holds every bf16 value), back in bf16 bits."""
    v = wl.bf16_bits_to_f32(bits).astype(np.float16).astype(np.float32)
    return wl.f32_to_bf16_bits(v)


def test_first_token_of_a_fresh_sequence_returns_its_v_bitexact(pkv):
    rng = np.random.default_rng(511)
    w = _random(rng, 4, 128, 16, [5, 40, 1], [0, 0, 0])
    kc, vc = stored(w)
    out = bits_host(run_step(pkv, w, to_dev(w)))
    for b in range(w.B):
        r = int(w.cu_seqlens_q[b])
        blk = w.block_tables[b, 0]
        for h in range(w.Hq):
            v = vc[blk, 0, h // w.G]
            np.testing.assert_array_equal(out[r, h], f16_rounded(v))
            assert np.array_equal(f16_rounded(v), v)  # N(0,1) data: every value exact in f16


def test_tiny_v_values_round_to_f16_subnormals(pkv):
    """V scaled by 2^-20 (magnitudes around 1e-6, below f16's normal range):
    the output matches the oracle over V rounded to f16, relative to the
    scale, and differs from the exact oracle by at most 2^-25 per value."""
    rng = np.random.default_rng(517)
    w = _random(rng, 2, 128, 16, [3, 40, 70], [16, 0, 32])
    for name in ("v_cache", "v_new"):
        x = wl.bf16_bits_to_f32(getattr(w, name)) * np.float32(2.0 ** -20)
        setattr(w, name, wl.f32_to_bf16_bits(x))
    kc, vc = stored(w)
    got = wl.bf16_bits_to_f32(bits_host(run_step(pkv, w, to_dev(w)))).astype(np.float64)
    ref16 = oracle.paged_prefill(w.q, kc, f16_rounded(vc), w.block_tables, w.cu_seqlens_q,
                                 w.cu_seqlens_k, w.scale)
    ref = oracle.paged_prefill(w.q, kc, vc, w.block_tables, w.cu_seqlens_q, w.cu_seqlens_k,
                               w.scale)
    err = np.abs(got - ref16) * 2.0 ** 20
    assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (err.max(), err.mean())
    assert np.abs(ref16 - ref).max() <= 2.0 ** -25 * (1 + 1e-6)


def test_v_beyond_f16_range_is_clamped_and_flagged(pkv):
    """65280 (the largest bf16 value within f16's range) passes unflagged; a
    value of 65536 or more in a row that is read sets PKV_FLAG_V_RANGE and
    the output stays finite."""
    rng = np.random.default_rng(518)
    w = _random(rng, 2, 64, 16, [9, 20], [16, 0])
    b, t = 1, 3  # sequence 1, token 3: read by its own and later queries
    slot = int(w.slot_mapping[int(w.cu_seqlens_q[b]) + t])
    for val, flagged in ((65280.0, False), (65536.0, True), (1.0e6, True)):
        kc, vc = stored(w)
        vc = vc.copy()
        vc[slot // w.bs, slot % w.bs, 0, 5] = wl.f32_to_bf16_bits(np.float32([val]))[0]
        d = to_dev(w)
        d["k_cache"], d["v_cache"] = bf16_dev(kc), bf16_dev(vc)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = run_step(pkv, w, d, err=err, store=False)
        assert bool(int(err.item()) & pkv.FLAG_V_RANGE) == flagged, (val, int(err.item()))
        assert torch.isfinite(out.float()).all()


def test_nan_in_unread_slots_changes_nothing(pkv):
    rng = np.random.default_rng(512)
    q_lens, cached = [3, 17, 40, 1], [16, 0, 32, 48]
    w = _random(rng, 4, 128, 16, q_lens, cached)
    clean = bits_host(run_step(pkv, w, to_dev(w)))
    kc, vc = stored(w)
    wl.poison_unused_slots(kc, vc, w.block_tables, w.k_lens, w.bs)
    d = to_dev(w)
    d["k_cache"], d["v_cache"] = bf16_dev(kc), bf16_dev(vc)
    out = bits_host(run_step(pkv, w, d, store=False))
    assert np.isfinite(wl.bf16_bits_to_f32(out)).all()
    np.testing.assert_array_equal(out, clean)


def test_block_permutation_gives_identical_output(pkv):
    rng = np.random.default_rng(513)
    w = _random(rng, 2, 128, 16, [20, 77, 5], [32, 0, 64], NB=64)
    kc, vc = stored(w)
    d = to_dev(w)
    d["k_cache"], d["v_cache"] = bf16_dev(kc), bf16_dev(vc)
    a = bits_host(run_step(pkv, w, d, store=False))
    pi = rng.permutation(w.NB)
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[pi], vc2[pi] = kc, vc
    d["k_cache"], d["v_cache"] = bf16_dev(kc2), bf16_dev(vc2)
    d["tables"] = torch.from_numpy(
        np.where(w.block_tables >= 0, pi[np.maximum(w.block_tables, 0)], -1).astype(np.int32)).cuda()
    b = bits_host(run_step(pkv, w, d, store=False))
    np.testing.assert_array_equal(a, b)


def test_rows_outside_the_sequences_are_untouched(pkv):
    rng = np.random.default_rng(514)
    w = _random(rng, 2, 64, 16, [9, 4], [0, 16])
    d = to_dev(w)
    Tq = w.Tq
    big = torch.zeros((Tq + 5, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    big[:Tq] = d["q"]
    d["q"] = big
    out = torch.full_like(big, 7.0)
    run_step(pkv, w, d, out=out)
    assert (out[Tq:] == 7.0).all()
    assert torch.isfinite(out[:Tq].float()).all() and not (out[:Tq] == 7.0).all()


def test_error_flags(pkv):
    rng = np.random.default_rng(515)
    w = _random(rng, 2, 64, 16, [9, 20], [16, 0])
    d = to_dev(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tables = d["tables"].clone()
    tables[1, 0] = w.NB + 3
    d["tables"] = tables
    out = run_step(pkv, w, d, err=err)
    assert int(err.item()) & pkv.FLAG_BAD_BLOCK
    assert torch.isfinite(out.float()).all()
    err.zero_()
    d = to_dev(w)
    d["cu_k"] = torch.tensor([0, 5, 25], dtype=torch.int32, device="cuda")  # k_len 5 < q_len 9
    run_step(pkv, w, d, err=err, store=False)
    assert int(err.item()) & pkv.FLAG_BAD_CONTEXT_LEN
    err.zero_()
    d = to_dev(w)
    out = torch.empty_like(d["q"])
    pkv.paged_prefill(d["q"], d["k_cache"], d["v_cache"], d["tables"], d["cu_q"], d["cu_k"],
                      8, w.scale, out, err_flag=err)  # max_seqlen_q below q_len 9
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.FLAG_BAD_CONTEXT_LEN


def test_cuda_graph_capture_and_replay(pkv):
    w, kc, vc, ref, _ = config(0)
    d = to_dev(w)
    out = torch.empty_like(d["q"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run_step(pkv, w, d)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pkv.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slots"])
            pkv.paged_prefill(d["q"], d["k_cache"], d["v_cache"], d["tables"], d["cu_q"],
                              d["cu_k"], w.max_seqlen_q, w.scale, out)
    for _ in range(3):
        out.zero_()
        g.replay()
    torch.cuda.synchronize()
    compare(bits_host(out), ref, "graph replay")


@pytest.mark.parametrize("scale", [-0.09, 0.0, 0.3])
def test_negative_zero_and_large_scales(pkv, scale):
    rng = np.random.default_rng(516)
    w = _random(rng, 2, 128, 16, [1, 30, 70], [0, 16, 32])
    w.scale = scale
    kc, vc = stored(w)
    ref = oracle.paged_prefill(w.q, kc, vc, w.block_tables, w.cu_seqlens_q, w.cu_seqlens_k, scale)
    compare(bits_host(run_step(pkv, w, to_dev(w))), ref, f"scale={scale}")


def test_repeated_full_size_runs_are_bit_identical(pkv):
    """The kernel has no atomics or order-dependent sums across CTAs, so every
    run of a step gives the same bits; a race between its warps would not."""
    w = wl.prefill_config_workload(1)
    d = to_dev(w)
    pkv.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slots"])
    first = bits_host(run_step(pkv, w, d, store=False))
    out = torch.empty_like(d["q"])
    for _ in range(12):
        out.zero_()
        np.testing.assert_array_equal(bits_host(run_step(pkv, w, d, out=out, store=False)), first)
