"""CUDA-graph replay of decode steps at padded batch sizes.

Following the MinivLLM guide (sections 4.6 and 4.7): decode steps have a fixed
shape (one token per sequence), so whole steps are captured once per batch
size in [1, 2, 4, 8] + range(16, max_bs + 1, 16), largest first, over static
input buffers; a step of ``bs`` sequences replays the smallest graph that
holds it, with the unused rows padded by sentinels -- slot -1 (the store
skips it) and context length 0 (attention writes zeros and reads nothing).
Replaying removes the per-launch host cost, which dominates small batches.

A step is store_kvcache followed by paged_attn_decode, exactly as the eager
calls; only the launches are recorded.  The caches, block-table width (MBS)
and softmax scale are fixed per runner.
"""

from __future__ import annotations

from . import decode_workspace_bytes, paged_attn_decode, store_kvcache


def graph_batch_sizes(max_bs: int) -> list[int]:
    """[1, 2, 4, 8] + multiples of 16 up to max_bs (and max_bs itself)."""
    sizes = [b for b in (1, 2, 4, 8) if b <= max_bs] + list(range(16, max_bs + 1, 16))
    if not sizes or sizes[-1] != max_bs:
        sizes.append(max_bs)
    return sorted(set(sizes))


class DecodeGraphRunner:
    """Captured decode steps over fixed caches; ``step`` replays one."""

    def __init__(self, k_cache, v_cache, num_q_heads: int, max_bs: int, max_blocks_per_seq: int,
                 scale: float, batch_sizes=None, stream=None):
        import torch

        self.torch = torch
        self.k_cache, self.v_cache = k_cache, v_cache
        NB, bs, Hkv, D = k_cache.shape
        dev = k_cache.device
        self.Hq, self.Hkv, self.D, self.MBS = num_q_heads, Hkv, D, max_blocks_per_seq
        self.scale = float(scale)
        self.max_bs = max_bs
        bf = torch.bfloat16
        self.q = torch.zeros((max_bs, num_q_heads, D), dtype=bf, device=dev)
        self.k_new = torch.zeros((max_bs, Hkv, D), dtype=bf, device=dev)
        self.v_new = torch.zeros((max_bs, Hkv, D), dtype=bf, device=dev)
        self.slots = torch.full((max_bs,), -1, dtype=torch.int64, device=dev)
        self.tables = torch.full((max_bs, max_blocks_per_seq), -1, dtype=torch.int32, device=dev)
        self.lens = torch.zeros((max_bs,), dtype=torch.int32, device=dev)
        self.out = torch.zeros((max_bs, num_q_heads, D), dtype=bf, device=dev)
        self.sizes = sorted(batch_sizes or graph_batch_sizes(max_bs))
        ws_bytes = max(decode_workspace_bytes(b, num_q_heads, Hkv, D, max_blocks_per_seq, bs)
                       for b in self.sizes)
        self.ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        self.stream = stream or torch.cuda.Stream(dev)
        self.graphs = {}
        with torch.cuda.stream(self.stream):
            for b in reversed(self.sizes):  # largest first, as the guide captures
                self._run(b)  # warm-up outside capture (library set-up, cached descriptors)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=self.stream):
                    self._run(b)
                self.graphs[b] = g
        torch.cuda.synchronize(dev)

    def _run(self, b: int):
        store_kvcache(self.k_new[:b], self.v_new[:b], self.k_cache, self.v_cache, self.slots[:b])
        paged_attn_decode(self.q[:b], self.k_cache, self.v_cache, self.tables[:b], self.lens[:b],
                          self.scale, self.out[:b], workspace=self.ws)

    def graph_size(self, bs: int) -> int:
        for b in self.sizes:
            if b >= bs:
                return b
        raise ValueError(f"batch of {bs} exceeds the largest captured size {self.sizes[-1]}")

    def inputs(self, bs: int) -> dict:
        """Views of the static input buffers for a step of ``bs`` sequences.

        Fill them in place (q, k_new, v_new, slot_mapping, block_tables,
        context_lens) and call ``replay(bs)``: no copy launches in between.
        """
        return dict(q=self.q[:bs], k_new=self.k_new[:bs], v_new=self.v_new[:bs],
                    slot_mapping=self.slots[:bs], block_tables=self.tables[:bs],
                    context_lens=self.lens[:bs])

    def replay(self, bs: int):
        """Pad rows bs.. of the chosen graph with sentinels and replay it on the
        current stream; returns ``out[:bs]``."""
        gb = self.graph_size(bs)
        if gb > bs:
            self.slots[bs:gb].fill_(-1)
            self.lens[bs:gb].zero_()
        self.graphs[gb].replay()
        return self.out[:bs]

    def step(self, q, k_new, v_new, slot_mapping, block_tables, context_lens):
        """Copy a step's inputs into the static buffers and replay, all on the
        current stream; returns ``out[:bs]`` (a view).  Writing the inputs
        straight into ``inputs(bs)`` and calling ``replay`` avoids the copies."""
        bs = q.shape[0]
        mbs = block_tables.shape[1]
        if mbs > self.MBS:
            raise ValueError("block_tables wider than the runner's max_blocks_per_seq")
        self.q[:bs].copy_(q)
        self.k_new[:bs].copy_(k_new)
        self.v_new[:bs].copy_(v_new)
        self.slots[:bs].copy_(slot_mapping)
        self.tables[:bs, :mbs].copy_(block_tables)
        if mbs < self.MBS:
            self.tables[:bs, mbs:].fill_(-1)
        self.lens[:bs].copy_(context_lens)
        return self.replay(bs)
