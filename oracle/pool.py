"""Plain-Python model of the KV block pool (test infrastructure only).

Follows the Paged KV Cache of the mini-infer README ("项目概述": BlockTable +
free-block pool; "架构设计": KVCacheManager) and the allocate sketch of the
nxmr.cn article, §2.1 "KV缓存的内存革命" (pages_needed = ceil(seq_len /
PAGE_SIZE), popped from the end of the free list), with the pool fixed in size
(no fallback allocation when the list is empty: the request fails and nothing
changes).

Conventions (the same ones the library documents in its public header):
  * a Python list is the free stack; ``pop()`` takes from its end;
  * at creation the stack is arranged so that successive pops return
    ``initial_order[0], initial_order[1], ...`` (or 0, 1, 2, ... when no order
    is given);
  * growing a sequence to n tokens appends ceil(n/16) - len(table) popped
    blocks to its table, in pop order;
  * freeing a sequence pushes its table entries in table order, so the next pop
    returns its last block.
Status codes mirror the library's: 0 ok, 1 invalid argument, 2 out of blocks,
3 unknown sequence.
"""
from __future__ import annotations

import numpy as np

BLOCK = 16
OK, INVALID_ARG, OUT_OF_BLOCKS, UNKNOWN_SEQ = 0, 1, 2, 3


class PoolModel:
    def __init__(self, num_blocks, max_seqs, max_blocks_per_seq, initial_order=None):
        order = list(range(num_blocks)) if initial_order is None else [int(x) for x in initial_order]
        assert sorted(order) == list(range(num_blocks))
        self.free_stack = order[::-1]          # pop() returns order[0] first
        self.max_seqs = max_seqs
        self.num_blocks = num_blocks
        self.max_blocks_per_seq = max_blocks_per_seq
        self.tables = {}                       # seq id -> list of block ids
        self.tokens = {}                       # seq id -> token count

    def num_free(self):
        return len(self.free_stack)

    def admission(self, running_decodes, hard_bp=None, soft_bp=None):
        """Brake level for a new prefill request (oracle.admission)."""
        from oracle import admission as A
        return A.admission(len(self.free_stack), self.num_blocks, running_decodes,
                           A.HARD_BP if hard_bp is None else hard_bp, A.SOFT_BP if soft_bp is None else soft_bp)

    def alloc(self, seq, num_tokens):
        if not (0 <= seq < self.max_seqs) or num_tokens < 0:
            return INVALID_ARG
        have = self.tables.get(seq, [])
        if num_tokens < self.tokens.get(seq, 0):
            return INVALID_ARG
        need = -(-num_tokens // BLOCK)
        if need > self.max_blocks_per_seq:
            return INVALID_ARG
        extra = need - len(have)
        if extra > len(self.free_stack):
            return OUT_OF_BLOCKS
        table = list(have)
        for _ in range(max(extra, 0)):
            table.append(self.free_stack.pop())
        self.tables[seq] = table
        self.tokens[seq] = num_tokens
        return OK

    def free(self, seq):
        if seq not in self.tables:
            return UNKNOWN_SEQ
        for blk in self.tables.pop(seq):
            self.free_stack.append(blk)
        del self.tokens[seq]
        return OK

    def batch_meta(self, seq_ids):
        """block_tables [B][max_blocks_per_seq] (pad -1), context_lens [B], slot of the last token [B]."""
        B = len(seq_ids)
        bt = np.full((B, self.max_blocks_per_seq), -1, np.int32)
        cl = np.zeros(B, np.int32)
        sl = np.full(B, -1, np.int32)
        for i, s in enumerate(seq_ids):
            t = self.tables[s]
            bt[i, :len(t)] = t
            n = self.tokens[s]
            cl[i] = n
            if n > 0:
                sl[i] = t[(n - 1) // BLOCK] * BLOCK + (n - 1) % BLOCK
        return bt, cl, sl

    def token_slots(self, seq, first, count):
        """Slots of tokens first .. first+count-1 of a sequence (must be held)."""
        t = self.tables[seq]
        return np.array([t[(i) // BLOCK] * BLOCK + i % BLOCK for i in range(first, first + count)], np.int32)
