"""GPU parity: the CUDA path against the CPU oracle, through the C ABI.

store_kvcache must be bit-exact over the whole cache.  Attention must match
the fp64 oracle (cast to fp32) to max-abs <= 1e-2 and mean-abs <= 1e-3 over
all outputs (bf16 in and out).
"""

import math

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
        lens=torch.from_numpy(w.context_lens).cuda(),
    )


def run_step(pkv, w, d, max_ctas=0, err=None):
    pkv.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slots"], err_flag=err)
    out = torch.empty_like(d["q"])
    pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["tables"], d["lens"], w.scale, out,
                          max_ctas=max_ctas, err_flag=err)
    torch.cuda.synchronize()
    return out


def oracle_step(w):
    kc, vc, bad = oracle.store_kvcache(w.k_new, w.v_new, w.k_cache, w.v_cache, w.slot_mapping)
    assert bad == 0
    ref = oracle.paged_attn_decode(w.q, kc, vc, w.block_tables, w.context_lens, w.scale)
    return kc, vc, ref


def compare(out, ref, what=""):
    got = wl.bf16_bits_to_f32(bits_host(out)).astype(np.float32)
    exp = ref.astype(np.float32)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - exp)
    assert err.max() <= MAX_ABS, f"{what}: max-abs {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean-abs {err.mean():.3e}"
    return float(err.max()), float(err.mean())


_cache = {}


def config(idx):
    if idx not in _cache:
        w = wl.config_workload(idx)
        _cache.clear()
        _cache[idx] = (w, oracle_step(w))
    return _cache[idx]


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_config_store_bitexact_and_decode_parity(pkv, idx):
    w, (kc, vc, ref) = config(idx)
    d = to_dev(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_step(pkv, w, d, err=err)
    assert int(err.item()) == 0
    np.testing.assert_array_equal(bits_host(d["k_cache"]), kc)
    np.testing.assert_array_equal(bits_host(d["v_cache"]), vc)
    compare(out, ref, w.name)


@pytest.mark.parametrize("ctas", [1, 2, 3, 5, 7, 0])
def test_grid_size_invariance_tiny(pkv, ctas):
    """Fewer CTAs move the slice boundaries (and so the merges) elsewhere."""
    w, (kc, vc, ref) = config(0)
    d = to_dev(w)
    out = run_step(pkv, w, d, max_ctas=ctas)
    compare(out, ref, f"max_ctas={ctas}")


def test_grid_sizes_agree_qwen3_shape(pkv):
    w, (kc, vc, ref) = config(1)
    d = to_dev(w)
    outs = [run_step(pkv, w, d, max_ctas=s) for s in (1, 13, 77, 0)]
    for o in outs:
        compare(o, ref)
    a = wl.bf16_bits_to_f32(bits_host(outs[0]))
    for o in outs[1:]:
        b = wl.bf16_bits_to_f32(bits_host(o))
        assert np.abs(a - b).max() <= 2 * MAX_ABS


def _random_problem(rng, B, Hq, Hkv, D, bs, lens, NB=None, poison=False):
    return wl.make_workload("rand", B=B, Hq=Hq, Hkv=Hkv, D=D, bs=bs, context_lens=lens, NB=NB,
                            rng=rng, poison_unused=poison)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("bs", [16, 48, 256])
def test_group_dim_block_variants(pkv, G, D, bs):
    rng = np.random.default_rng(100 + G * 7 + D + bs)
    Hkv = 2
    lens = [1, 15, 16, 17, 63, 64, 65, 257, 700][: 5 + G // 2]
    w = _random_problem(rng, len(lens), G * Hkv, Hkv, D, bs, lens)
    kc, vc, ref = oracle_step(w)
    d = to_dev(w)
    for ctas in (0, 1, 3):
        out = run_step(pkv, w, d, max_ctas=ctas)
        compare(out, ref, f"G={G} D={D} bs={bs} max_ctas={ctas}")


def test_context_len_one_returns_v_bitexact(pkv):
    rng = np.random.default_rng(7)
    w = _random_problem(rng, 6, 8, 2, 128, 16, [1] * 6)
    kc, vc, ref = oracle_step(w)
    d = to_dev(w)
    out = bits_host(run_step(pkv, w, d))
    G = 4
    for b in range(6):
        blk = w.block_tables[b, 0]
        for h in range(8):
            np.testing.assert_array_equal(out[b, h], vc[blk, 0, h // G])


def test_identical_keys_give_mean_of_v(pkv):
    rng = np.random.default_rng(8)
    w = _random_problem(rng, 3, 4, 2, 64, 16, [5, 40, 300])
    kc, vc, _ = oracle_step(w)
    for b in range(3):
        for t in range(int(w.context_lens[b])):
            kc[w.block_tables[b, t // 16], t % 16] = kc[w.block_tables[b, 0], 0]
    w.k_cache, w.v_cache = kc, vc
    w.slot_mapping = np.full_like(w.slot_mapping, -1)  # caches already hold the step's tokens
    d = to_dev(w)
    out = wl.bf16_bits_to_f32(bits_host(run_step(pkv, w, d)))
    for b in range(3):
        n = int(w.context_lens[b])
        for h in range(4):
            V = np.stack([wl.bf16_bits_to_f32(vc[w.block_tables[b, t // 16], t % 16, h // 2]) for t in range(n)])
            np.testing.assert_allclose(out[b, h], V.astype(np.float64).mean(0), atol=MAX_ABS, rtol=0)


def test_nan_in_unread_slots_changes_nothing(pkv):
    rng = np.random.default_rng(9)
    lens = [1, 17, 40, 300, 33]
    w = _random_problem(rng, 5, 8, 2, 128, 16, lens)
    d = to_dev(w)
    clean = bits_host(run_step(pkv, w, d, max_ctas=2))
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    # store first on the host so poisoning leaves the new tokens intact
    kc, vc, _ = oracle.store_kvcache(w.k_new, w.v_new, kc, vc, w.slot_mapping)
    wl.poison_unused_slots(kc, vc, w.block_tables, w.context_lens, w.bs)
    d2 = to_dev(w)
    d2["k_cache"], d2["v_cache"] = bf16_dev(kc), bf16_dev(vc)
    d2["slots"] = torch.full_like(d2["slots"], -1)
    out = bits_host(run_step(pkv, w, d2, max_ctas=2))
    assert np.isfinite(wl.bf16_bits_to_f32(out)).all()
    np.testing.assert_array_equal(out, clean)


def test_block_permutation_gives_identical_output(pkv):
    rng = np.random.default_rng(10)
    w = _random_problem(rng, 4, 8, 2, 128, 16, [20, 77, 130, 5], NB=64)
    d = to_dev(w)
    a = bits_host(run_step(pkv, w, d))
    pi = rng.permutation(w.NB)
    kc2, vc2 = np.empty_like(w.k_cache), np.empty_like(w.v_cache)
    kc2[pi], vc2[pi] = w.k_cache, w.v_cache
    w.block_tables = np.where(w.block_tables >= 0, pi[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    w.slot_mapping = np.array([wl.decode_slot(w.block_tables[b], int(w.context_lens[b]), w.bs)
                               for b in range(w.B)], np.int64)
    w.k_cache, w.v_cache = kc2, vc2
    b = bits_host(run_step(pkv, w, to_dev(w)))
    np.testing.assert_array_equal(a, b)


def test_zero_context_gives_zeros(pkv):
    rng = np.random.default_rng(11)
    w = _random_problem(rng, 3, 4, 2, 64, 16, [5, 9, 300])
    d = to_dev(w)
    d["lens"] = torch.tensor([0, 9, 0], dtype=torch.int32, device="cuda")
    out = bits_host(run_step(pkv, w, d, max_ctas=4))
    assert (out[0] == 0).all() and (out[2] == 0).all()
    assert (out[1] != 0).any()


def test_error_flags_and_skips(pkv):
    rng = np.random.default_rng(12)
    w = _random_problem(rng, 3, 4, 2, 64, 16, [5, 40, 300])
    d = to_dev(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = bits_host(d["k_cache"]).copy()
    d["slots"] = torch.tensor([-1, w.NB * w.bs + 3, -7], dtype=torch.int64, device="cuda")
    pkv.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slots"], err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.FLAG_BAD_SLOT
    np.testing.assert_array_equal(bits_host(d["k_cache"]), before)
    err.zero_()
    tables = d["tables"].clone()
    tables[2, 3] = w.NB + 5
    out = torch.empty_like(d["q"])
    pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], tables, d["lens"], w.scale, out, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.FLAG_BAD_BLOCK
    assert torch.isfinite(out.float()).all()
    err.zero_()
    lens = d["lens"].clone()
    lens[0] = 10 ** 6
    pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["tables"], lens, w.scale, out, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pkv.FLAG_BAD_CONTEXT_LEN


def test_empty_batch_is_a_no_op(pkv):
    """B = 0 decode and N = 0 store succeed and touch nothing; a store whose
    slots are all padding (-1) leaves the cache bit-identical."""
    rng = np.random.default_rng(13)
    w = _random_problem(rng, 3, 4, 2, 64, 16, [5, 40, 300])
    d = to_dev(w)
    kc0, vc0 = bits_host(d["k_cache"]).copy(), bits_host(d["v_cache"]).copy()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.store_kvcache(d["k_new"][:0], d["v_new"][:0], d["k_cache"], d["v_cache"], d["slots"][:0],
                      err_flag=err)
    q0 = d["q"][:0]
    out0 = torch.empty_like(q0)
    pkv.paged_attn_decode(q0, d["k_cache"], d["v_cache"], d["tables"][:0], d["lens"][:0], w.scale,
                          out0, err_flag=err)
    pad = torch.full_like(d["slots"], -1)
    pkv.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], pad, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    np.testing.assert_array_equal(bits_host(d["k_cache"]), kc0)
    np.testing.assert_array_equal(bits_host(d["v_cache"]), vc0)


def test_maximum_batch_parity_and_one_past_it_is_rejected(pkv):
    """8192 sequences (the most one call takes: their box prefix sums live in
    shared memory) match the oracle; 8193 are refused before any launch."""
    rng = np.random.default_rng(14)
    B = 8192
    lens = rng.integers(1, 41, size=B)
    w = _random_problem(rng, B, 2, 1, 64, 16, lens)
    kc, vc, ref = oracle_step(w)
    d = to_dev(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_step(pkv, w, d, err=err)
    assert int(err.item()) == 0
    np.testing.assert_array_equal(bits_host(d["k_cache"]), kc)
    compare(out, ref, "B=8192")
    q1 = torch.zeros((B + 1, 2, 64), dtype=torch.bfloat16, device="cuda")
    tables1 = torch.zeros((B + 1, d["tables"].shape[1]), dtype=torch.int32, device="cuda")
    lens1 = torch.ones(B + 1, dtype=torch.int32, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_attn_decode(q1, d["k_cache"], d["v_cache"], tables1, lens1, w.scale,
                              torch.empty_like(q1), workspace=torch.zeros(16, dtype=torch.uint8,
                                                                            device="cuda"))
    assert e.value.status == 2  # PKV_ERR_UNSUPPORTED


def test_workspace_too_small_is_rejected(pkv):
    w, _ = config(0)
    d = to_dev(w)
    out = torch.empty_like(d["q"])
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError):
        pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["tables"], d["lens"], w.scale,
                              out, workspace=small)


def test_cuda_graph_capture_and_replay(pkv):
    w, (kc, vc, ref) = config(0)
    d = to_dev(w)
    out = torch.empty_like(d["q"])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run_step(pkv, w, d)  # warm-up: allocates the workspace outside capture
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            pkv.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slots"])
            pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["tables"], d["lens"],
                                  w.scale, out)
    for _ in range(3):
        out.zero_()
        g.replay()
    torch.cuda.synchronize()
    compare(out, ref, "graph replay")


def test_back_to_back_steps_on_one_stream(pkv):
    """Programmatic dependent launches chain store -> decode -> merge across steps."""
    w, (kc, vc, ref) = config(0)
    d = to_dev(w)
    out = torch.empty_like(d["q"])
    for _ in range(20):
        pkv.store_kvcache(d["k_new"], d["v_new"], d["k_cache"], d["v_cache"], d["slots"])
        pkv.paged_attn_decode(d["q"], d["k_cache"], d["v_cache"], d["tables"], d["lens"], w.scale,
                              out, max_ctas=3)
    torch.cuda.synchronize()
    compare(out, ref, "20 steps")
