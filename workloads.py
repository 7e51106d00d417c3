"""Seeded synthetic workloads for the paged-KV decode step.

This module only makes inputs: shapes, context lengths, pool operation
sequences and random bf16 values. It holds none of the method's arithmetic (no
RoPE, no slot arithmetic, no attention) and imports neither the product package
nor the oracle, so both sides can be fed from it.

The five workloads follow the shapes the pages work with: Qwen3-1.7B / Qwen3-8B
layers (NJU course brief "端侧大模型推理框架", §2.1 and §2.2), Qwen2.5-7B at
mini-infer's batch 8 with 128 new tokens (mini-infer README, "性能数据"), 16-token
KV blocks in a fixed pool (mini-infer README, "项目概述"), plus a tiny case and a
skewed long-context batch.

Values are N(0,1) drawn with numpy's PCG64 (stream-stable across platforms)
and rounded to bf16 by torch (round to nearest even). The big serving workload
fills its caches on the device with torch's seeded CUDA generator instead; the
tests copy back the blocks they check.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

BLOCK = 16
CANARY_BF16 = 0x7FA5  # a NaN pattern: slots no request owns, and block tails


@dataclass(frozen=True)
class Workload:
    name: str
    index: int                  # 1-based position in the workload list (seed = 1000 + index)
    layers: int
    B: int
    Hq: int
    Hkv: int
    head_dim: int
    num_blocks: int             # physical blocks per layer
    max_seqs: int
    theta: float = 1.0e6
    ctx_kind: str = "fixed"     # fixed | uniform | loguniform | skewed | sweep
    ctx_args: tuple = ()
    permuted_pool: bool = True  # pool handed out in a seeded random order
    churn: bool = False         # fragment the pool first (serving workload)
    sweep_steps: int = 1        # decode steps in one pass (128 for the sweep)
    device_fill: bool = False   # caches filled on the device

    @property
    def G(self):
        return self.Hq // self.Hkv

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def seed(self):
        return 1000 + self.index

    def max_context(self):
        """Largest post-append length any request reaches in one pass."""
        if self.ctx_kind == "fixed":
            return max(self.ctx_args) + 1
        if self.ctx_kind in ("uniform", "loguniform"):
            return self.ctx_args[1] + 1
        if self.ctx_kind == "skewed":
            return self.ctx_args[0] + 1
        if self.ctx_kind == "sweep":
            return self.ctx_args[0] + self.sweep_steps
        raise ValueError(self.ctx_kind)

    @property
    def max_blocks_per_seq(self):
        return -(-self.max_context() // BLOCK)

    @property
    def max_pos(self):
        return self.max_context()


WORKLOADS = {
    "tiny": Workload("tiny", 1, layers=1, B=2, Hq=4, Hkv=2, head_dim=64, num_blocks=64,
                     max_seqs=2, ctx_kind="fixed", ctx_args=(17, 40)),
    "qwen3_1p7b": Workload("qwen3_1p7b", 2, layers=1, B=8, Hq=16, Hkv=8, head_dim=128,
                           num_blocks=1024, max_seqs=8, ctx_kind="uniform", ctx_args=(128, 2048)),
    "qwen25_7b_sweep": Workload("qwen25_7b_sweep", 3, layers=28, B=8, Hq=28, Hkv=4, head_dim=128,
                                num_blocks=4096, max_seqs=8, ctx_kind="sweep", ctx_args=(128,),
                                sweep_steps=128),
    "qwen3_8b": Workload("qwen3_8b", 4, layers=36, B=64, Hq=32, Hkv=8, head_dim=128,
                         num_blocks=24576, max_seqs=4096, ctx_kind="loguniform",
                         ctx_args=(512, 8192), permuted_pool=False, churn=True, device_fill=True),
    "skewed": Workload("skewed", 5, layers=1, B=256, Hq=32, Hkv=8, head_dim=128, num_blocks=16384,
                       max_seqs=256, ctx_kind="skewed", ctx_args=(32768, 16, 1024)),
}


def rng_for(w: Workload, stream: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([w.seed, stream]))


def context_lengths(w: Workload) -> np.ndarray:
    """Tokens already cached per request before the first appended token."""
    r = rng_for(w, 1)
    if w.ctx_kind == "fixed":
        c = np.array(w.ctx_args, np.int64)
    elif w.ctx_kind == "uniform":
        c = r.integers(w.ctx_args[0], w.ctx_args[1] + 1, size=w.B)
    elif w.ctx_kind == "loguniform":
        lo, hi = w.ctx_args
        c = np.floor(np.exp(r.uniform(math.log(lo), math.log(hi), size=w.B))).astype(np.int64)
        c = np.clip(c, lo, hi)
    elif w.ctx_kind == "skewed":
        long_len, lo, hi = w.ctx_args
        c = r.integers(lo, hi + 1, size=w.B)
        c[int(r.integers(0, w.B))] = long_len
    elif w.ctx_kind == "sweep":
        c = np.full(w.B, w.ctx_args[0], np.int64)
    else:
        raise ValueError(w.ctx_kind)
    return c.astype(np.int32)


def initial_free_order(w: Workload):
    """Pop order of a fresh pool: a seeded permutation, or None for 0, 1, 2, ..."""
    if not w.permuted_pool:
        return None
    return rng_for(w, 2).permutation(w.num_blocks).astype(np.int32)


def churn(w: Workload, pool, first_dummy_id: int) -> int:
    """Fragment the free pool with allocate/free rounds of dummy sequences.

    Eight rounds of: allocate dummies of U{1..256} blocks until fewer than half
    the blocks are free, then free each live dummy with probability 1/2. Then
    free random dummies until at most 8192 dummy blocks remain. ``pool`` needs
    alloc(seq, tokens) -> status, free(seq) -> status and num_free().
    Returns the number of dummy blocks left allocated.
    """
    r = rng_for(w, 3)
    live = {}  # dummy id -> blocks
    nxt = first_dummy_id
    for _ in range(8):
        while pool.num_free() >= w.num_blocks // 2:
            nb = int(r.integers(1, 257))
            if nb > pool.num_free():
                break
            assert pool.alloc(nxt, nb * BLOCK) == 0
            live[nxt] = nb
            nxt += 1
            assert nxt < w.max_seqs
        for s in sorted(live):
            if r.random() < 0.5:
                assert pool.free(s) == 0
                del live[s]
    while sum(live.values()) > 8192:
        ids = sorted(live)
        s = ids[int(r.integers(0, len(ids)))]
        assert pool.free(s) == 0
        del live[s]
    return sum(live.values())


def setup_pool(w: Workload, pool, ctx: np.ndarray) -> None:
    """Run the workload's pool history on ``pool``: churn (if any), then give
    request b (sequence id b) ``ctx[b]`` tokens."""
    if w.churn:
        churn(w, pool, first_dummy_id=w.B)
    for b in range(w.B):
        st = pool.alloc(b, int(ctx[b]))
        assert st == 0, f"request {b} does not fit the pool (status {st})"


# --------------------------------------------------------------- values ------

def bf16_normal(r: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) values rounded to bf16, returned as uint16 bit patterns."""
    import torch
    x = r.standard_normal(size=shape, dtype=np.float32)
    t = torch.from_numpy(x).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def new_token_values(w: Workload, layer: int, step: int = 0):
    """q [B][Hq][d], k [B][Hkv][d], v [B][Hkv][d] (bf16 bits) for one layer and step."""
    r = np.random.Generator(np.random.PCG64([w.seed, 100, step, layer]))
    q = bf16_normal(r, (w.B, w.Hq, w.head_dim))
    k = bf16_normal(r, (w.B, w.Hkv, w.head_dim))
    v = bf16_normal(r, (w.B, w.Hkv, w.head_dim))
    return q, k, v


def history_cache(w: Workload, layer: int, block_tables: np.ndarray, ctx: np.ndarray):
    """Host K/V caches [num_blocks][Hkv][16][d] (bf16 bits) for one layer: the
    slots of tokens 0..ctx[b]-1 of every request hold N(0,1) values (taken as
    already rotated keys), every other slot holds the NaN canary."""
    r = np.random.Generator(np.random.PCG64([w.seed, 200, layer]))
    shape = (w.num_blocks, w.Hkv, BLOCK, w.head_dim)
    kc = np.full(shape, CANARY_BF16, np.uint16)
    vc = np.full(shape, CANARY_BF16, np.uint16)
    for b in range(w.B):
        n = int(ctx[b])
        if n <= 0:
            continue
        nblk = -(-n // BLOCK)
        blks = block_tables[b, :nblk].astype(np.int64)
        kv = bf16_normal(r, (2, nblk, w.Hkv, BLOCK, w.head_dim))
        full = n // BLOCK
        kc[blks[:full]] = kv[0, :full]
        vc[blks[:full]] = kv[1, :full]
        rem = n - full * BLOCK
        if rem:
            kc[blks[full], :, :rem] = kv[0, full, :, :rem]
            vc[blks[full], :, :rem] = kv[1, full, :, :rem]
    return kc, vc


def device_fill_cache(w: Workload, layer: int, k_cache, v_cache) -> None:
    """Fill a layer's device caches (torch bf16 tensors) with N(0,1) values
    from torch's seeded CUDA generator (every slot, no canary)."""
    import torch
    g = torch.Generator(device=k_cache.device)
    g.manual_seed(w.seed * 1000 + layer)
    for t in (k_cache, v_cache):
        flat = t.view(-1)
        chunk = 1 << 28
        for s in range(0, flat.numel(), chunk):
            e = min(flat.numel(), s + chunk)
            flat[s:e].copy_(torch.randn(e - s, generator=g, device=t.device, dtype=torch.float32))


# ------------------------------------------------------------- prefill -------

@dataclass(frozen=True)
class PrefillWorkload:
    """A prefill / chunked-prefill batch of one layer: request r holds
    history[r] cached tokens and appends new[r] tokens at positions
    history[r] .. history[r] + new[r] - 1 (NJU course brief §2.1, the prefill
    stage; mini-infer README "项目概述", prefill as its own pass).

    kind "explicit": ``args`` = (history tuple, new tuple).
    kind "mixed": ``args`` = (fresh, fresh_lo, fresh_hi, cont, cont_lo, cont_hi,
    chunk): ``fresh`` whole prompts of U[fresh_lo, fresh_hi] tokens with no
    history, then ``cont`` continuations with log-uniform [cont_lo, cont_hi]
    history and a ``chunk``-token chunk each."""
    name: str
    index: int
    Hq: int
    Hkv: int
    head_dim: int
    num_blocks: int
    kind: str
    args: tuple
    theta: float = 1.0e6
    layers: int = 1

    @property
    def G(self):
        return self.Hq // self.Hkv

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def seed(self):
        return 1000 + self.index

    @property
    def B(self):
        return len(self.lengths()[0])

    def lengths(self):
        """(history, new) int32 arrays, one entry per request."""
        if self.kind == "explicit":
            h, n = self.args
            return np.array(h, np.int32), np.array(n, np.int32)
        if self.kind == "mixed":
            fresh, flo, fhi, cont, clo, chi, chunk = self.args
            r = np.random.Generator(np.random.PCG64([self.seed, 1]))
            fn = r.integers(flo, fhi + 1, size=fresh)
            ch = np.floor(np.exp(r.uniform(math.log(clo), math.log(chi), size=cont))).astype(np.int64)
            h = np.concatenate([np.zeros(fresh, np.int64), np.clip(ch, clo, chi)])
            n = np.concatenate([fn, np.full(cont, chunk, np.int64)])
            return h.astype(np.int32), n.astype(np.int32)
        raise ValueError(self.kind)

    def max_context(self):
        h, n = self.lengths()
        return int((h + n).max())

    @property
    def max_blocks_per_seq(self):
        return -(-self.max_context() // BLOCK)

    @property
    def max_pos(self):
        return self.max_context()

    @property
    def max_seqs(self):
        return self.B


PREFILL_WORKLOADS = {
    # small enough for the oracle to check every row: several tiles, ragged
    # tails, a one-token request, a request with no history
    "prefill_small": PrefillWorkload("prefill_small", 6, Hq=8, Hkv=2, head_dim=128, num_blocks=256,
                                     kind="explicit",
                                     args=((0, 0, 37, 100, 300, 16), (1, 70, 16, 129, 33, 47))),
    # Qwen3-8B layer shape (Hq 32, Hkv 8, d 128): 8 fresh prompts of 512..2048
    # tokens and 8 chunked continuations (512-token chunks over 1k..8k history)
    "qwen3_8b_prefill": PrefillWorkload("qwen3_8b_prefill", 7, Hq=32, Hkv=8, head_dim=128,
                                        num_blocks=4096, kind="mixed",
                                        args=(8, 512, 2048, 8, 1024, 8192, 512)),
    # the same kind of request mix at the Qwen2.5-7B layer shape (Hq 28, Hkv 4: G = 7,
    # which does not divide a 128-row tile)
    "qwen25_7b_prefill": PrefillWorkload("qwen25_7b_prefill", 8, Hq=28, Hkv=4, head_dim=128,
                                         num_blocks=4096, kind="mixed",
                                         args=(8, 512, 2048, 8, 1024, 8192, 512)),
}


def device_int8_cache(w: Workload, layer: int, device):
    """INT8 caches of one layer on the device, as a decode over INT8 caches
    sees them: codes round(N(0,1) * 127 / 4) clamped to [-127, 127], and for
    every block and KV head a group maximum uniform in [3.5, 4.5] (what a
    64-token group of N(0,1) values gives), in arrays of num_blocks * Hkv
    floats. Seeded torch CUDA generator.
    Returns (k_codes, v_codes, k_amax, v_amax)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(w.seed * 1000 + 500 + layer)
    shape = (w.num_blocks, w.Hkv, BLOCK, w.head_dim)
    n_amax = w.num_blocks * w.Hkv
    out = []
    for _ in range(2):
        c = torch.empty(shape, dtype=torch.int8, device=device)
        flat = c.view(-1)
        chunk = 1 << 28
        for s0 in range(0, flat.numel(), chunk):
            e = min(flat.numel(), s0 + chunk)
            x = torch.randn(e - s0, generator=g, device=device) * (127.0 / 4.0)
            flat[s0:e].copy_(x.round_().clamp_(-127, 127).to(torch.int8))
        out.append(c)
    for _ in range(2):
        out.append(3.5 + torch.rand(n_amax, generator=g, device=device))
    return tuple(out)


def prefill_setup_pool(w: PrefillWorkload, pool) -> None:
    """Give request r (sequence id r) history[r] + new[r] tokens, in order."""
    h, n = w.lengths()
    for r in range(w.B):
        st = pool.alloc(r, int(h[r] + n[r]))
        assert st == 0, f"request {r} does not fit the pool (status {st})"


def prefill_new_values(w: PrefillWorkload, layer: int = 0):
    """q [T][Hq][d], k [T][Hkv][d], v [T][Hkv][d] (bf16 bits) of the new
    tokens, request after request."""
    T = int(w.lengths()[1].sum())
    r = np.random.Generator(np.random.PCG64([w.seed, 300, layer]))
    q = bf16_normal(r, (T, w.Hq, w.head_dim))
    k = bf16_normal(r, (T, w.Hkv, w.head_dim))
    v = bf16_normal(r, (T, w.Hkv, w.head_dim))
    return q, k, v


# ------------------------------------------------- continuous batching -------

def serving_churn(pool, steps: int, seed: int, use_brakes: bool = True, arrival_max: int = 4,
                  prompt=(64, 1024), gen=(16, 512), max_seqs: int = 4096, hard_bp=None, soft_bp=None):
    """Drive a pool through a continuous-batching schedule (mini-infer README
    "项目概述": every step admits what it can and decodes the running batch)
    and return the trace of pool events.

    Each step: 0..arrival_max new requests arrive (prompt U[prompt], output
    U[gen] tokens, seeded); waiting requests are admitted in arrival order
    while ``pool.admission(len(running))`` says proceed (or always, when
    use_brakes is False) and their prompt fits; every running request then
    grows by one token, and one that finds no free block is preempted (freed,
    back to the head of the queue, its tokens to be recomputed); finished
    requests are freed. ``pool`` needs alloc, free, num_free and admission.
    Returns a list of per-step tuples (admitted ids, preempted ids, finished
    ids, free blocks after the step)."""
    r = np.random.Generator(np.random.PCG64([seed, 400]))
    waiting, running, trace = [], [], []
    target = {}  # request -> (prompt tokens, total tokens)
    held = {}    # running request -> tokens in the pool
    nxt = 0
    kw = {} if hard_bp is None else {"hard_bp": hard_bp, "soft_bp": soft_bp}
    for _ in range(steps):
        for _ in range(int(r.integers(0, arrival_max + 1))):
            if nxt < max_seqs:
                p_len = int(r.integers(prompt[0], prompt[1] + 1))
                target[nxt] = (p_len, p_len + int(r.integers(gen[0], gen[1] + 1)))
                waiting.append(nxt)
                nxt += 1
        admitted, preempted, finished = [], [], []
        while waiting:
            if use_brakes and pool.admission(len(running), **kw) != 0:
                break
            s = waiting[0]
            if pool.alloc(s, target[s][0]) != 0:
                break
            waiting.pop(0)
            running.append(s)
            held[s] = target[s][0]
            admitted.append(s)
        for s in list(running):
            n = held[s] + 1
            if pool.alloc(s, n) != 0:
                assert pool.free(s) == 0
                running.remove(s)
                del held[s]
                waiting.insert(0, s)
                preempted.append(s)
                continue
            held[s] = n
            if n >= target[s][1]:
                assert pool.free(s) == 0
                running.remove(s)
                del held[s]
                finished.append(s)
        trace.append((tuple(admitted), tuple(preempted), tuple(finished), pool.num_free()))
    return trace
