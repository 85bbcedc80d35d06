"""Reference block allocator (test infrastructure): the pages' rules, plainly.

MinivLLM guide "HowToApproachvLLM", sections 3.1-3.3 and 4.5:
  * a block has a reference count (1 when handed out) and, once full, a
    content hash chained with the previous block's hash, plus its token ids
    (compared on lookup to guard against hash collisions);
  * free block ids wait in a queue; allocation takes the first one;
  * a prompt reuses cached full blocks until the first miss, then allocates;
  * appending the token that makes num_tokens % block_size == 1 opens a new
    block; num_tokens % block_size == 0 means the last block is full and
    gets hashed; the new token's slot is
    block_table[-1] * block_size + last_block_num_tokens - 1;
  * releasing a sequence drops one reference per block; blocks at 0 return
    to the back of the queue.
The hash is any fixed function of (previous hash, token ids); Python's tuple
hash is used here, so block ids can differ from another implementation only
if two different contents collide, which the token comparison rules out.
"""

from __future__ import annotations

from collections import deque


class Block:
    def __init__(self, block_id):
        self.block_id = block_id
        self.ref_count = 0
        self.hash = None
        self.token_ids = []

    def reset(self):
        self.ref_count = 1
        self.hash = None
        self.token_ids = []


class RefBlockManager:
    def __init__(self, num_blocks, block_size):
        self.block_size = block_size
        self.blocks = [Block(i) for i in range(num_blocks)]
        self.free = deque(range(num_blocks))
        self.hash_to_block = {}
        self.seqs = {}  # seq_id -> (token_ids list, block_table list)

    @staticmethod
    def compute_hash(token_ids, prefix):
        return hash((prefix, tuple(token_ids)))

    def _allocate_block(self, block_id):
        self.free.remove(block_id)
        self.blocks[block_id].reset()
        return self.blocks[block_id]

    def _release(self, block_id):
        b = self.blocks[block_id]
        b.ref_count -= 1
        if b.ref_count == 0:
            self.free.append(block_id)

    def can_allocate(self, num_tokens):
        return len(self.free) >= -(-num_tokens // self.block_size)

    def allocate(self, seq_id, tokens):
        assert seq_id not in self.seqs
        bs = self.block_size
        tokens = list(tokens)
        table = []
        h = None
        cache_miss = False
        cached = 0
        nblocks = -(-len(tokens) // bs)
        for i in range(nblocks):
            chunk = tokens[i * bs:(i + 1) * bs]
            h = self.compute_hash(chunk, h) if len(chunk) == bs else None
            block_id = self.hash_to_block.get(h, -1) if h is not None else -1
            if block_id == -1 or self.blocks[block_id].token_ids != chunk:
                cache_miss = True
            if cache_miss:
                block = self._allocate_block(self.free[0])
            else:
                cached += bs
                block = self.blocks[block_id]
                if block.ref_count > 0:
                    block.ref_count += 1
                else:
                    self.free.remove(block_id)
                    block.ref_count = 1
            if h is not None:
                block.hash = h
                block.token_ids = chunk
                self.hash_to_block[h] = block.block_id
            table.append(block.block_id)
        self.seqs[seq_id] = (tokens, table)
        return cached

    def append(self, seq_id, token):
        tokens, table = self.seqs[seq_id]
        bs = self.block_size
        tokens.append(token)
        n = len(tokens)
        if n % bs == 1 or bs == 1:
            table.append(self._allocate_block(self.free[0]).block_id)
        if n % bs == 0:
            last = self.blocks[table[-1]]
            prefix = self.blocks[table[-2]].hash if len(table) > 1 else None
            last.hash = self.compute_hash(tokens[-bs:], prefix)
            last.token_ids = tokens[-bs:]
            self.hash_to_block[last.hash] = last.block_id
        last_block_num_tokens = n - (len(table) - 1) * bs
        return table[-1] * bs + last_block_num_tokens - 1

    def deallocate(self, seq_id):
        tokens, table = self.seqs.pop(seq_id)
        for block_id in reversed(table):
            self._release(block_id)
