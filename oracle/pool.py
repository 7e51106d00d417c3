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
        self.tables = {}                       # seq id -> list of block ids (resident sequences)
        self.tokens = {}                       # seq id -> token count (resident or swapped out)
        self.swapped = set()                   # sequences whose blocks are swapped out
        self.clock = 0                         # use counter for LRU eviction
        self.last_use = {}                     # resident seq id -> clock of its last use

    def num_free(self):
        return len(self.free_stack)

    def admission(self, running_decodes, hard_bp=None, soft_bp=None):
        """Brake level for a new prefill request (oracle.admission)."""
        from oracle import admission as A
        return A.admission(len(self.free_stack), self.num_blocks, running_decodes,
                           A.HARD_BP if hard_bp is None else hard_bp, A.SOFT_BP if soft_bp is None else soft_bp)

    def alloc(self, seq, num_tokens):
        if not (0 <= seq < self.max_seqs) or num_tokens < 0 or seq in self.swapped:
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
        self._use([seq])
        return OK

    def free(self, seq):
        if seq in self.swapped:
            self.swapped.discard(seq)
            del self.tokens[seq]
            return OK
        if seq not in self.tables:
            return UNKNOWN_SEQ
        for blk in self.tables.pop(seq):
            self.free_stack.append(blk)
        del self.tokens[seq]
        self.last_use.pop(seq, None)
        return OK

    # ---- swap to host memory with LRU eviction (NJU course brief, optional
    # task 3 "KV Cache Offloading": inactive KV blocks go to CPU memory and come
    # back when needed, under an eviction policy such as LRU)

    def _use(self, seqs):
        self.clock += 1
        for s in seqs:
            self.last_use[s] = self.clock

    def touch(self, seqs):
        """Mark resident sequences as used now (one clock tick for the call)."""
        if any(s not in self.tables for s in seqs):
            return UNKNOWN_SEQ
        self._use(seqs)
        return OK

    def lru_victim(self, exclude=()):
        """Least recently used resident sequence holding a block, not in
        exclude (ties: lower id); -1 when there is none."""
        cand = [(self.last_use.get(s, 0), s) for s, t in self.tables.items() if t and s not in set(exclude)]
        return min(cand)[1] if cand else -1

    def swap_out(self, seq):
        """Release a resident sequence's blocks (pushed as free() pushes them)
        and keep its token count; returns (status, its former table)."""
        if seq not in self.tables:
            return UNKNOWN_SEQ, []
        table = self.tables.pop(seq)
        for blk in table:
            self.free_stack.append(blk)
        self.swapped.add(seq)
        self.last_use.pop(seq, None)
        return OK, table

    def swap_in(self, seq):
        """Give a swapped-out sequence ceil(tokens/16) fresh blocks in pop
        order; returns (status, its new table). Out of blocks: unchanged."""
        if seq not in self.swapped:
            return UNKNOWN_SEQ, []
        need = -(-self.tokens[seq] // BLOCK)
        if need > len(self.free_stack):
            return OUT_OF_BLOCKS, []
        table = [self.free_stack.pop() for _ in range(need)]
        self.tables[seq] = table
        self.swapped.discard(seq)
        self._use([seq])
        return OK, list(table)

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
