"""Host block allocator (C++ via the C ABI) against the pages' rules.

Pins come from the MinivLLM guide, sections 3.2-3.3 and 4.5 (worked example
of the 257th token, ref_count 1 on allocation, chained prefix hashes, the
token-id collision guard); a randomised comparison against the plain Python
restatement in oracle/block_manager.py checks every block id, slot, length
and reference count bit for bit.
"""

import numpy as np
import pytest

from oracle.block_manager import RefBlockManager
from paged_kv_cache_85_gb300.block_manager import BlockManager
from paged_kv_cache_85_gb300 import PkvError


@pytest.fixture(autouse=True)
def _lib(cuda_lib_path):
    return cuda_lib_path


def test_257th_token_opens_a_new_block_at_its_offset_0():
    """MinivLLM §4.5: 256 % 256 == 0 finalises block 0; 257 % 256 == 1 allocates the next free block."""
    bm = BlockManager(num_blocks=4, block_size=256)
    assert bm.allocate(7, np.arange(256)) == 0
    assert list(bm.block_table(7)) == [0]
    slot = bm.append(7, 1000)  # token 257
    assert list(bm.block_table(7)) == [0, 1]
    assert slot == 1 * 256 + 1 - 1
    assert bm.seq_len(7) == 257
    # token 258 goes to offset 1 of the same block
    assert bm.append(7, 1001) == 256 + 1


def test_fresh_blocks_have_ref_count_one_and_free_at_zero():
    bm = BlockManager(num_blocks=6, block_size=4)
    bm.allocate(1, [1, 2, 3, 4, 5])
    t = bm.block_table(1)
    assert [bm.ref_count(b) for b in t] == [1, 1]
    assert bm.num_free_blocks == 4
    bm.deallocate(1)
    assert [bm.ref_count(b) for b in t] == [0, 0]
    assert bm.num_free_blocks == 6


def test_prefix_sharing_reuses_full_blocks_and_counts_references():
    bm = BlockManager(num_blocks=16, block_size=4)
    a = [1, 2, 3, 4, 5, 6, 7, 8, 9]
    b = [1, 2, 3, 4, 5, 6, 7, 8, 42, 43]
    assert bm.allocate(0, a) == 0
    assert bm.allocate(1, b) == 8  # two full blocks found cached
    ta, tb = bm.block_table(0), bm.block_table(1)
    assert list(ta[:2]) == list(tb[:2]) and ta[2] != tb[2]
    assert [bm.ref_count(x) for x in ta[:2]] == [2, 2]
    bm.deallocate(0)
    assert [bm.ref_count(x) for x in tb[:2]] == [1, 1]


def test_same_tokens_under_a_different_prefix_do_not_hit():
    """The hash chains the prefix: [p1][x] and [p2][x] are different blocks."""
    bm = BlockManager(num_blocks=16, block_size=2)
    bm.allocate(0, [1, 2, 9, 9])
    assert bm.allocate(1, [3, 4, 9, 9]) == 0
    assert bm.block_table(0)[1] != bm.block_table(1)[1]


def test_cached_block_survives_release_until_reused():
    bm = BlockManager(num_blocks=3, block_size=2)
    bm.allocate(0, [5, 6, 7])
    blk = bm.block_table(0)[0]
    bm.deallocate(0)
    assert bm.ref_count(blk) == 0
    assert bm.allocate(1, [5, 6, 1]) == 2  # still registered: a hit on a free block
    assert bm.block_table(1)[0] == blk and bm.ref_count(blk) == 1


def test_append_hashes_a_block_when_it_fills():
    bm = BlockManager(num_blocks=8, block_size=2)
    bm.allocate(0, [1])
    bm.append(0, 2)  # block 0 is now full: [1, 2]
    assert bm.allocate(1, [1, 2, 3]) == 2


def test_errors_and_capacity():
    bm = BlockManager(num_blocks=2, block_size=4)
    assert bm.can_allocate(8) and not bm.can_allocate(9)
    with pytest.raises(PkvError):
        bm.allocate(0, np.arange(9))
    assert bm.num_free_blocks == 2  # a failed allocation changes nothing
    bm.allocate(0, np.arange(8))
    with pytest.raises(PkvError):
        bm.allocate(0, [1])  # id in use
    assert not bm.can_append(0)  # token 9 needs a block and none is free
    with pytest.raises(PkvError):
        bm.append(0, 9)
    with pytest.raises(PkvError):
        bm.deallocate(99)


def test_decode_batch_matches_prepare_decode_formula():
    bm = BlockManager(num_blocks=32, block_size=4)
    for sid, n in [(10, 1), (11, 4), (12, 5), (13, 13)]:
        bm.allocate(sid, np.arange(n) + 100 * sid)
    tables, lens, slots = bm.decode_batch([13, 10, 12, 11], MBS=5)
    assert list(lens) == [13, 1, 5, 4]
    for i, sid in enumerate([13, 10, 12, 11]):
        t = bm.block_table(sid)
        assert list(tables[i, : len(t)]) == list(t) and (tables[i, len(t):] == -1).all()
        n = lens[i]
        last_block_num_tokens = n - (len(t) - 1) * 4
        assert slots[i] == t[-1] * 4 + last_block_num_tokens - 1
        assert slots[i] == bm.slots(sid, n - 1, n)[0]


@pytest.mark.parametrize("seed", range(6))
def test_random_operations_match_reference(seed):
    rng = np.random.default_rng(seed)
    bs = int(rng.choice([1, 2, 3, 4, 16]))
    nb = int(rng.integers(8, 64))
    ours, ref = BlockManager(nb, bs), RefBlockManager(nb, bs)
    live = []
    next_id = 0
    vocab = 5  # a small vocabulary makes shared prefixes common
    for step in range(400):
        op = rng.integers(0, 10)
        if op < 3:
            n = int(rng.integers(1, 4 * bs + 2))
            base = live[rng.integers(len(live))] if live and rng.random() < 0.5 else None
            if base is not None:  # start from an existing sequence's prompt to hit the cache
                toks = list(ref.seqs[base][0][:n])
                toks += list(rng.integers(0, vocab, n - len(toks)))
            else:
                toks = list(rng.integers(0, vocab, n))
            if ours.can_allocate(n) != ref.can_allocate(n):
                raise AssertionError("can_allocate differs")
            if not ref.can_allocate(n):
                continue
            c1 = ours.allocate(next_id, toks)
            c2 = ref.allocate(next_id, toks)
            assert c1 == c2
            live.append(next_id)
            next_id += 1
        elif op < 8 and live:
            sid = live[rng.integers(len(live))]
            tok = int(rng.integers(0, vocab))
            ok = ours.can_append(sid)
            need = len(ref.seqs[sid][0]) % bs == 0
            assert ok == (not need or len(ref.free) > 0)
            if not ok:
                continue
            assert ours.append(sid, tok) == ref.append(sid, tok)
        elif live:
            sid = live.pop(rng.integers(len(live)))
            ours.deallocate(sid)
            ref.deallocate(sid)
        assert ours.num_free_blocks == len(ref.free)
        for sid in live:
            assert list(ours.block_table(sid)) == ref.seqs[sid][1]
            assert ours.seq_len(sid) == len(ref.seqs[sid][0])
        for b in range(nb):
            assert ours.ref_count(b) == ref.blocks[b].ref_count


def test_reference_collision_guard_compares_token_ids(monkeypatch):
    """MinivLLM §3.2: a hash hit whose stored tokens differ is a miss."""
    monkeypatch.setattr(RefBlockManager, "compute_hash", staticmethod(lambda toks, prefix: 12345))
    ref = RefBlockManager(8, 2)
    ref.allocate(0, [1, 2])
    assert ref.allocate(1, [3, 4]) == 0  # same (forced) hash, different tokens
    assert ref.seqs[0][1] != ref.seqs[1][1]
    assert ref.allocate(2, [3, 4]) == 2  # genuine hit


def test_append_batch_is_all_or_nothing_and_matches_single_appends():
    a, b = BlockManager(10, 4), BlockManager(10, 4)
    for bm in (a, b):
        for sid, n in [(0, 4), (1, 3), (2, 8)]:
            bm.allocate(sid, np.arange(n) + 10 * sid)
    slots = a.append_batch([0, 1, 2], [7, 8, 9])
    assert list(slots) == [b.append(0, 7), b.append(1, 8), b.append(2, 9)]
    tight = BlockManager(3, 4)
    tight.allocate(0, np.arange(4))
    tight.allocate(1, np.arange(8))  # both full, 0 free blocks left
    with pytest.raises(PkvError):
        tight.append_batch([0, 1], [1, 1])
    assert tight.seq_len(0) == 4 and tight.seq_len(1) == 8


def test_prefix_hits_on_freed_blocks_scale_to_a_large_cache():
    """A prefix-cache hit on a freed block takes it out of the middle of the
    free pool; with ~100k blocks that must not cost a scan of the pool per
    hit.  500 sequences of 3000 tokens fill ~94k blocks of 16 tokens, are
    released (their full blocks stay cached in the pool), then come back:
    every full block is a hit on a freed block."""
    import time

    bs, n_seq, n_tok = 16, 500, 3000
    bm = BlockManager(num_blocks=100_000, block_size=bs)
    rng = np.random.default_rng(40)
    prompts = [rng.integers(0, 50_000, size=n_tok) for _ in range(n_seq)]
    first = []
    for s, p in enumerate(prompts):
        assert bm.allocate(s, p) == 0
        first.append(list(bm.block_table(s)))
    for s in range(n_seq):
        bm.deallocate(s)
    assert bm.num_free_blocks == 100_000
    t0 = time.perf_counter()
    for s, p in enumerate(prompts):
        assert bm.allocate(1000 + s, p) == (n_tok // bs) * bs  # every full block cached
    dt = time.perf_counter() - t0
    for s in range(n_seq):
        # the full blocks come back as they were; the partial last block is fresh
        assert list(bm.block_table(1000 + s))[: n_tok // bs] == first[s][: n_tok // bs]
    assert bm.num_free_blocks == 100_000 - n_seq * -(-n_tok // bs)
    assert dt < 5.0, f"{dt:.2f} s for {n_seq * (n_tok // bs)} hits on freed blocks"


def test_free_pool_order_after_hits_matches_the_restatement():
    """Blocks taken out of the middle of the pool by cache hits leave the rest
    in FIFO order: the next fresh allocations agree with the Python
    restatement block for block."""
    bs = 4
    bm, ref = BlockManager(num_blocks=64, block_size=bs), RefBlockManager(64, bs)
    rng = np.random.default_rng(41)
    prompts = [rng.integers(0, 100, size=int(rng.integers(5, 30))) for _ in range(6)]
    for s, p in enumerate(prompts):
        assert bm.allocate(s, p) == ref.allocate(s, p)
    for s in (1, 3, 4):
        bm.deallocate(s)
        ref.deallocate(s)
    for s, p in [(10, prompts[3]), (11, rng.integers(0, 100, size=17)), (12, prompts[1][:9])]:
        assert bm.allocate(s, p) == ref.allocate(s, p)
        assert list(bm.block_table(s)) == ref.seqs[s][1]
    assert bm.num_free_blocks == len(ref.free)
