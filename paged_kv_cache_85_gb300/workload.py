"""Seeded synthetic inputs for paged decode and prefill attention.

This module only *draws* inputs: context lengths, block placement, block
tables, slot mappings and bf16 tensors.  It holds none of the arithmetic of
the method (no scatter, no scores, no softmax); both the CUDA path and the
CPU oracle consume what it returns.

Shapes follow the serving settings the pages describe:

* nano-vllm ``Config``: ``max_num_seqs=512``, ``max_model_len=4096``,
  ``kvcache_block_size=256`` ("Nano-vLLM 源码学习(2)", §2 Config).
* vLLM 0.7.3 parameter table: ``block_size=16``, ``max_num_seqs=256``
  ("VLLM-0.7.3 源码", §3.3).
* A sequence's KV lives in fixed-size physical blocks named by its
  ``block_table``; a new decode token is written at
  ``block_table[-1] * block_size + last_block_num_tokens - 1``
  (MinivLLM guide, §4.5 ``prepare_decode``).

All arrays are numpy.  bf16 tensors are ``uint16`` arrays holding the raw
bf16 bit patterns (fp32 N(0,1) rounded to nearest-even), so host and device
see identical bits.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

BF16_NAN = np.uint16(0x7FC0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); return bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _randn_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    step = 1 << 24  # bounded temporaries for GB-sized caches
    for s in range(0, n, step):
        e = min(n, s + step)
        out[s:e] = f32_to_bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


@dataclasses.dataclass
class Workload:
    """One decode step's inputs (store first, then attend)."""

    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    bs: int
    NB: int
    MBS: int
    scale: float
    context_lens: np.ndarray  # int32 [B]; includes the new token
    block_tables: np.ndarray  # int32 [B, MBS]; -1 past the used blocks
    q: np.ndarray  # u16 bf16 [B, Hq, D]
    k_cache: np.ndarray  # u16 bf16 [NB, bs, Hkv, D]
    v_cache: np.ndarray  # u16 bf16 [NB, bs, Hkv, D]
    k_new: np.ndarray  # u16 bf16 [N, Hkv, D]
    v_new: np.ndarray  # u16 bf16 [N, Hkv, D]
    slot_mapping: np.ndarray  # int64 [N]; -1 = padding, skipped
    recipe: str = ""
    ctx_dist: str = ""  # how context_lens were drawn, e.g. "uniform [128, 4096]"

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def context_lens_summary(self) -> dict:
        """The drawn context lengths: distribution and realised statistics."""
        c = self.context_lens.astype(np.int64)
        return {"dist": self.ctx_dist or "given", "min": int(c.min()), "max": int(c.max()),
                "mean": round(float(c.mean()), 1), "total_tokens": int(c.sum())}

    @property
    def N(self) -> int:
        return int(self.slot_mapping.shape[0])

    def kv_bytes(self, elem_bytes: int = 2) -> int:
        """K and V bytes over every sequence's context (logical); 1 byte per
        element for an FP8 cache."""
        return int(self.context_lens.astype(np.int64).sum()) * self.Hkv * self.D * elem_bytes * 2

    def unique_kv_bytes(self) -> int:
        """K and V bytes of the distinct physical blocks the step reads."""
        seen = set()
        tok = 0
        for b in range(self.B):
            n = int(self.context_lens[b])
            for j in range((n + self.bs - 1) // self.bs):
                p = int(self.block_tables[b, j])
                if p in seen:
                    continue
                seen.add(p)
                tok += min(self.bs, n - j * self.bs)
        return tok * self.Hkv * self.D * 2 * 2

    def decode_bytes(self, kv_elem_bytes: int = 2) -> int:
        """Algorithmic bytes of one decode: K/V over context + q + out + table + lens."""
        tables = sum((int(n) + self.bs - 1) // self.bs for n in self.context_lens) * 4
        return self.kv_bytes(kv_elem_bytes) + 2 * self.B * self.Hq * self.D * 2 + tables + 4 * self.B

    def store_bytes(self, kv_elem_bytes: int = 2) -> int:
        """Algorithmic bytes of one store: valid bf16 rows read, cache rows
        written (kv_elem_bytes per element), plus slots."""
        nv = int((self.slot_mapping >= 0).sum())
        return nv * self.Hkv * self.D * (2 + kv_elem_bytes) * 2 + 8 * self.N


def decode_slot(block_table_row: np.ndarray, ctx: int, bs: int) -> int:
    """Slot of a sequence's newest token, as ``prepare_decode`` forms it.

    ``block_table[-1] * block_size + last_block_num_tokens - 1`` where the
    table holds exactly the used blocks (MinivLLM guide, §4.5).
    """
    nblocks = (ctx + bs - 1) // bs
    last_block_num_tokens = ctx - (nblocks - 1) * bs
    return int(block_table_row[nblocks - 1]) * bs + last_block_num_tokens - 1


def make_workload(
    name: str,
    B: int,
    Hq: int,
    Hkv: int,
    D: int,
    bs: int,
    context_lens,
    NB: int | None = None,
    seed: int = 0,
    shared_prefix_tokens: int = 0,
    pad_frac: float = 0.0,
    poison_unused: bool = False,
    recipe: str = "",
    rng: np.random.Generator | None = None,
    ctx_dist: str = "",
) -> Workload:
    """Draw one step's inputs.

    Draw order: (context_lens come in) -> block permutation -> q -> k_cache
    -> v_cache -> new k -> new v -> padding mask.  Physical blocks are a
    seeded permutation of ``[0, NB)`` handed out in sequence order, so block
    placement is fully fragmented.  With ``shared_prefix_tokens`` the first
    blocks of every table are the same physical ids (prefix sharing).
    """
    if rng is None:
        rng = np.random.default_rng(seed)
    ctx = np.asarray(context_lens, dtype=np.int32).reshape(B)
    assert (ctx >= 1).all(), "every running sequence holds at least its new token"
    nblk = (ctx.astype(np.int64) + bs - 1) // bs
    MBS = int(nblk.max())
    n_shared = shared_prefix_tokens // bs
    assert shared_prefix_tokens % bs == 0
    own = nblk - n_shared
    assert (own >= 1).all(), "the new token must land in a sequence's own block"
    need = n_shared + int(own.sum())
    if NB is None:
        NB = int(math.ceil(1.25 * need))
    assert NB >= need
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.full((B, MBS), -1, dtype=np.int32)
    cur = 0
    shared_ids = perm[:n_shared]
    cur = n_shared
    for b in range(B):
        tables[b, :n_shared] = shared_ids
        k = int(own[b])
        tables[b, n_shared : n_shared + k] = perm[cur : cur + k]
        cur += k
    q = _randn_bf16(rng, (B, Hq, D))
    k_cache = _randn_bf16(rng, (NB, bs, Hkv, D))
    v_cache = _randn_bf16(rng, (NB, bs, Hkv, D))
    k_new = _randn_bf16(rng, (B, Hkv, D))
    v_new = _randn_bf16(rng, (B, Hkv, D))
    slots = np.array([decode_slot(tables[b], int(ctx[b]), bs) for b in range(B)], dtype=np.int64)
    if pad_frac > 0:
        npad = int(math.floor(pad_frac * B + 0.5))
        idx = rng.choice(B, size=npad, replace=False)
        slots[idx] = -1
    if poison_unused:
        poison_unused_slots(k_cache, v_cache, tables, ctx, bs)
    return Workload(
        name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, bs=bs, NB=NB, MBS=MBS,
        scale=float(np.float32(1.0 / math.sqrt(D))),
        context_lens=ctx, block_tables=tables, q=q, k_cache=k_cache, v_cache=v_cache,
        k_new=k_new, v_new=v_new, slot_mapping=slots, recipe=recipe, ctx_dist=ctx_dist,
    )


def poison_unused_slots(k_cache, v_cache, tables, ctx, bs) -> None:
    """Fill every cache slot no sequence reads (unassigned blocks, tail slots) with NaN."""
    NB = k_cache.shape[0]
    used = np.zeros((NB, bs), dtype=bool)
    for b in range(tables.shape[0]):
        n = int(ctx[b])
        for j in range((n + bs - 1) // bs):
            lo = j * bs
            used[tables[b, j], : min(bs, n - lo)] = True
    k_cache[~used] = BF16_NAN
    v_cache[~used] = BF16_NAN


# Serving-shaped configurations.  Index 0 is the small case the oracle
# finishes instantly; 1..4 are the full-size steps.
CONFIG_NAMES = [
    "tiny_paged_decode",
    "qwen3_0p6b_decode",
    "vllm_bs16_8b_heads",
    "max_concurrency",
    "long_context_shared_prefix",
]


def config_workload(idx: int, seed: int = 0, poison_unused: bool = False) -> Workload:
    """The five serving-shaped steps (seeded with ``SeedSequence([seed, idx])``)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, idx]))
    name = CONFIG_NAMES[idx]
    if idx == 0:
        return make_workload(
            name, B=4, Hq=4, Hkv=2, D=64, bs=16, context_lens=[1, 17, 40, 300], NB=64,
            rng=rng, poison_unused=poison_unused, ctx_dist="fixed {1, 17, 40, 300}",
            recipe="4 seqs, ctx {1,17,40,300}, bs16, 4Q/2KV, D64, NB=64 permuted, N(0,1) bf16",
        )
    if idx == 1:
        ctx = rng.integers(128, 4096, size=64, endpoint=True)
        return make_workload(
            name, B=64, Hq=16, Hkv=8, D=128, bs=256, context_lens=ctx, rng=rng,
            poison_unused=poison_unused, ctx_dist="uniform integers [128, 4096]",
            recipe="64 seqs, ctx U[128,4096], bs256, 16Q/8KV, D128, NB=ceil(1.25*used), N(0,1) bf16",
        )
    if idx == 2:
        ctx = rng.integers(1, 2048, size=256, endpoint=True)
        return make_workload(
            name, B=256, Hq=32, Hkv=8, D=128, bs=16, context_lens=ctx, rng=rng,
            poison_unused=poison_unused, ctx_dist="uniform integers [1, 2048]",
            recipe="256 seqs, ctx U[1,2048], bs16, 32Q/8KV, D128, NB=ceil(1.25*used), N(0,1) bf16",
        )
    if idx == 3:
        ctx = np.rint(np.exp(rng.uniform(math.log(16), math.log(4096), size=512))).astype(np.int64)
        return make_workload(
            name, B=512, Hq=16, Hkv=8, D=128, bs=256, context_lens=ctx, rng=rng, pad_frac=0.05,
            poison_unused=poison_unused, ctx_dist="round(exp(uniform [ln 16, ln 4096]))",
            recipe="512 seqs, ctx logU[16,4096], bs256, 16Q/8KV, D128, 26 slots=-1, N(0,1) bf16",
        )
    if idx == 4:
        return make_workload(
            name, B=8, Hq=32, Hkv=8, D=128, bs=256, context_lens=[32768] * 8,
            shared_prefix_tokens=8192, rng=rng, poison_unused=poison_unused,
            ctx_dist="fixed 32768, first 8192 tokens' blocks shared by all tables",
            recipe="8 seqs x 32768, bs256, 32Q/8KV, D128, first 8192 tokens' blocks shared",
        )
    raise ValueError(f"no config {idx}")


# ---------------------------------------------------------------- prefill


@dataclasses.dataclass
class PrefillWorkload:
    """One prefill step's inputs: the new tokens of B sequences, flattened.

    Sequence b has ``q_lens[b]`` new tokens after a cached prefix of
    ``k_lens[b] - q_lens[b]`` tokens (whole blocks, as prefix caching keeps
    them).  The step stores the new tokens' K/V through ``slot_mapping``
    (only uncached tokens get slots) and then attends through
    ``block_tables`` (MinivLLM guide, §4.5 ``prepare_prefill``).
    """

    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    bs: int
    NB: int
    MBS: int
    scale: float
    q_lens: np.ndarray  # int32 [B]
    k_lens: np.ndarray  # int32 [B]; cached prefix + new tokens
    cu_seqlens_q: np.ndarray  # int32 [B + 1]
    cu_seqlens_k: np.ndarray  # int32 [B + 1]
    block_tables: np.ndarray  # int32 [B, MBS]; -1 past the used blocks
    q: np.ndarray  # u16 bf16 [Tq, Hq, D]
    k_cache: np.ndarray  # u16 bf16 [NB, bs, Hkv, D]
    v_cache: np.ndarray  # u16 bf16 [NB, bs, Hkv, D]
    k_new: np.ndarray  # u16 bf16 [Tq, Hkv, D]
    v_new: np.ndarray  # u16 bf16 [Tq, Hkv, D]
    slot_mapping: np.ndarray  # int64 [Tq]
    recipe: str = ""

    @property
    def Tq(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def max_seqlen_q(self) -> int:
        return int(self.q_lens.max())

    def attended_keys(self) -> int:
        """Sum over query tokens of the keys each one sees (causal)."""
        tot = 0
        for ql, kl in zip(self.q_lens.tolist(), self.k_lens.tolist()):
            # query i sees kl - ql + i + 1 keys
            tot += ql * (kl - ql) + ql * (ql + 1) // 2
        return tot

    def flops(self) -> int:
        """Algorithmic FLOPs: 2 per multiply-add of q.K and of P.V, causal keys only."""
        return 4 * self.attended_keys() * self.Hq * self.D

    def kv_bytes(self) -> int:
        """K and V bytes of every sequence's context, read once."""
        return int(self.k_lens.astype(np.int64).sum()) * self.Hkv * self.D * 2 * 2

    def io_bytes(self) -> int:
        """K/V once + q + out + tables + cu_seqlens."""
        tables = sum((int(n) + self.bs - 1) // self.bs for n in self.k_lens) * 4
        return self.kv_bytes() + 2 * self.Tq * self.Hq * self.D * 2 + tables + 8 * (self.B + 1)


def cu_seqlens(lengths) -> np.ndarray:
    """[0, l0, l0 + l1, ...] as int32: the boundaries of flattened sequences."""
    out = np.zeros(len(lengths) + 1, dtype=np.int32)
    out[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return out


def make_prefill_workload(
    name: str,
    Hq: int,
    Hkv: int,
    D: int,
    bs: int,
    q_lens,
    cached_lens,
    NB: int | None = None,
    shared_prefix_tokens: int = 0,
    poison_unused: bool = False,
    recipe: str = "",
    rng: np.random.Generator | None = None,
    seed: int = 0,
) -> PrefillWorkload:
    """Draw one prefill step's inputs.

    Draw order: block permutation -> q -> k_cache -> v_cache -> new k -> new v.
    Cached prefixes are whole blocks.  With ``shared_prefix_tokens`` the first
    blocks of every table are the same physical ids (a prefix-cache hit shared
    by all sequences); the rest of each table is the sequence's own blocks,
    taken from a seeded permutation of ``[0, NB)``.
    """
    if rng is None:
        rng = np.random.default_rng(seed)
    ql = np.asarray(q_lens, dtype=np.int32)
    cl = np.asarray(cached_lens, dtype=np.int32)
    B = int(ql.shape[0])
    assert cl.shape == ql.shape and (ql >= 1).all() and (cl >= 0).all()
    assert (cl % bs == 0).all(), "prefix caching keeps whole blocks"
    assert shared_prefix_tokens % bs == 0 and (cl >= shared_prefix_tokens).all()
    kl = cl + ql
    nblk = (kl.astype(np.int64) + bs - 1) // bs
    MBS = int(nblk.max())
    n_shared = shared_prefix_tokens // bs
    own = nblk - n_shared
    need = n_shared + int(own.sum())
    if NB is None:
        NB = int(math.ceil(1.25 * need))
    assert NB >= need
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.full((B, MBS), -1, dtype=np.int32)
    cur = n_shared
    for b in range(B):
        tables[b, :n_shared] = perm[:n_shared]
        k = int(own[b])
        tables[b, n_shared : n_shared + k] = perm[cur : cur + k]
        cur += k
    cq = cu_seqlens(ql)
    Tq = int(cq[-1])
    q = _randn_bf16(rng, (Tq, Hq, D))
    k_cache = _randn_bf16(rng, (NB, bs, Hkv, D))
    v_cache = _randn_bf16(rng, (NB, bs, Hkv, D))
    k_new = _randn_bf16(rng, (Tq, Hkv, D))
    v_new = _randn_bf16(rng, (Tq, Hkv, D))
    slots = np.empty(Tq, dtype=np.int64)
    for b in range(B):
        pos = np.arange(int(cl[b]), int(kl[b]), dtype=np.int64)
        slots[cq[b] : cq[b + 1]] = tables[b, pos // bs].astype(np.int64) * bs + pos % bs
    if poison_unused:
        poison_unused_slots(k_cache, v_cache, tables, kl, bs)
    return PrefillWorkload(
        name=name, B=B, Hq=Hq, Hkv=Hkv, D=D, bs=bs, NB=NB, MBS=MBS,
        scale=float(np.float32(1.0 / math.sqrt(D))), q_lens=ql, k_lens=kl.astype(np.int32),
        cu_seqlens_q=cq, cu_seqlens_k=cu_seqlens(kl), block_tables=tables, q=q,
        k_cache=k_cache, v_cache=v_cache, k_new=k_new, v_new=v_new, slot_mapping=slots,
        recipe=recipe,
    )


# Prefill steps shaped like the pages' settings: a token budget of
# max_num_batched_tokens = 16384 per step and max_model_len = 4096
# ("Nano-vLLM 源码学习(2)", §2 Config), block sizes 256 (nano-vllm) and 16
# (vLLM 0.7.3), cached prefixes from prefix caching.  Index 0 is tiny.
PREFILL_CONFIG_NAMES = [
    "tiny_paged_prefill",
    "qwen3_prefill_16k",
    "vllm_bs16_prefill_ragged",
    "shared_prefix_prefill",
]


def prefill_config_workload(idx: int, seed: int = 0, poison_unused: bool = False) -> PrefillWorkload:
    """The prefill steps (seeded with ``SeedSequence([seed, 100 + idx])``)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 100 + idx]))
    name = PREFILL_CONFIG_NAMES[idx]
    if idx == 0:
        return make_prefill_workload(
            name, Hq=4, Hkv=2, D=64, bs=16, q_lens=[1, 5, 17, 40], cached_lens=[0, 16, 32, 0],
            NB=64, rng=rng, poison_unused=poison_unused,
            recipe="4 seqs, new {1,5,17,40} after cached {0,16,32,0}, bs16, 4Q/2KV, D64, NB=64",
        )
    if idx == 1:
        return make_prefill_workload(
            name, Hq=16, Hkv=8, D=128, bs=256, q_lens=[2048] * 8,
            cached_lens=[0, 0, 0, 0, 256, 512, 1024, 2048], rng=rng, poison_unused=poison_unused,
            recipe="8 seqs x 2048 new tokens (16384), cached {0,0,0,0,256,512,1024,2048}, "
                   "bs256, 16Q/8KV, D128",
        )
    if idx == 2:
        ql = rng.integers(1, 1023, size=32, endpoint=True)
        cl = 16 * rng.integers(0, 64, size=32, endpoint=True)
        return make_prefill_workload(
            name, Hq=32, Hkv=8, D=128, bs=16, q_lens=ql, cached_lens=cl, rng=rng,
            poison_unused=poison_unused,
            recipe="32 seqs, new U[1,1023], cached 16*U[0,64], bs16, 32Q/8KV, D128",
        )
    if idx == 3:
        return make_prefill_workload(
            name, Hq=16, Hkv=8, D=128, bs=256, q_lens=[1024] * 16, cached_lens=[2048] * 16,
            shared_prefix_tokens=2048, rng=rng, poison_unused=poison_unused,
            recipe="16 seqs x 1024 new tokens after one shared cached 2048-token prefix, "
                   "bs256, 16Q/8KV, D128",
        )
    raise ValueError(f"no prefill config {idx}")
