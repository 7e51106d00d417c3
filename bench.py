"""Benchmark of the paged-KV decode step on one GB300 (or N replicas).

One step = the whole hot path over one decode batch of the Qwen3-8B-shaped
serving workload: for each of 36 layers, RoPE append of the new token
(mi_paged_kv_append) and paged GQA decode attention (mi_paged_decode_attention)
over 64 requests with log-uniform contexts in [512, 8192] whose blocks come
from a churned 24,576-block pool. Every layer reads its own 727 MB of K/V, far
more than the 129 MB L2, so no flush is needed between steps.

Printed: one JSON line (rank 0). ``value`` = algorithmic bytes of the step (K/V
of valid tokens, q, out, live table entries, lengths, append traffic) over the
device-timed step, inputs resident in HBM. ``e2e`` = the same metric for real
decode steps driven through the C ABI from host buffers: host pool growth and
metadata, H2D of metadata and new q/k/v from pinned memory, 36 layers, D2H of
the outputs. ``roofline`` = the attention call (split-KV kernel + LSE combine)
against the measured HBM copy bandwidth (one kernel per layer: the log-sum-exp
combine of split units runs inside it). ``cpu_baseline`` = the fp64 oracle on
the host cores on a bounded sample. The default run adds ``per_config`` (the
Qwen3-1.7B layer, the Qwen2.5-7B 128-step sweep and the skewed batch, each
with the oracle on the host cores) and ``per_variant`` records: ``fp8``
(the same step over e4m3 caches, run as ``--kv fp8`` in a child process) and
``prefill`` (the Qwen3-8B-shaped prefill step on the default prefill kernel,
run as ``--workload qwen3_8b_prefill`` in a child process).

``--impl reference`` times the oracle alone (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import (BLOCK, PREFILL_WORKLOADS, WORKLOADS, context_lengths, device_fill_cache,  # noqa: E402
                       device_int8_cache,
                       history_cache, initial_free_order, new_token_values, prefill_new_values,
                       prefill_setup_pool, setup_pool)

METRIC = "paged decode-attention KV GB/s"
PREFILL_METRIC = "paged prefill-attention TFLOP/s"
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------- bytes ----

def attention_bytes(w, lens, kvb=2):
    """Algorithmic bytes of one attention call (one layer); kvb = bytes per
    cached element (2 for bf16, 1 for e4m3)."""
    lens = np.maximum(np.asarray(lens, np.int64), 0)
    kv = int(lens.sum()) * w.Hkv * w.head_dim * kvb * 2
    qo = 2 * w.B * w.Hq * w.head_dim * 2
    tables = 4 * int(np.sum(-(-lens // BLOCK))) + 4 * w.B
    return kv + qo + tables


def append_bytes(w, kvb=2):
    """Algorithmic bytes of one append call (one layer): new q, k, v read;
    q_out and the cache rows (kvb bytes per element) written; table rows,
    positions and slots read."""
    new = w.B * (w.Hq + 2 * w.Hkv) * w.head_dim * 2
    written = w.B * w.Hq * w.head_dim * 2 + w.B * 2 * w.Hkv * w.head_dim * kvb
    rope_rows = w.B * (w.head_dim // 2) * 8
    return new + written + rope_rows + 8 * w.B


def int8_extra_attention_bytes(w, lens):
    """The INT8 attention's bytes beyond its one-byte K/V tiles: the K and V
    group maxima of every block and KV head it reads (4 bytes each)."""
    lens = np.maximum(np.asarray(lens, np.int64), 0)
    return 8 * int(np.sum(-(-lens // BLOCK))) * w.Hkv


def int8_extra_append_bytes(w):
    """The INT8 append's bytes beyond append_bytes(w, 1): the new k and v rows
    also written in bf16 to the open-group buffer, the group maxima read and
    written, the open slots read. (When a new row raises its group's maximum,
    the group's earlier rows are read back and quantised again: data
    dependent, not counted.)"""
    return w.B * 2 * w.Hkv * w.head_dim * 2 + w.B * 2 * w.Hkv * 8 + 4 * w.B


def step_kv_bytes(w, lens, kv):
    """Algorithmic bytes of one layer of the decode step (append + attention)
    for KV cache type kv ("bf16", "fp8", "int8")."""
    kvb = 2 if kv == "bf16" else 1
    b = attention_bytes(w, lens, kvb) + append_bytes(w, kvb)
    if kv == "int8":
        b += int8_extra_attention_bytes(w, lens) + int8_extra_append_bytes(w)
    return b


def fp8_scales(w):
    """Per-KV-head e4m3 scales: about 3..6 standard deviations of the N(0,1)
    values at e4m3's largest finite value, 448 (seeded)."""
    r = np.random.Generator(np.random.PCG64([w.seed, 500]))
    return (((3.0 + 3.0 * r.random(w.Hkv)) / 448.0).astype(np.float32),
            ((3.0 + 3.0 * r.random(w.Hkv)) / 448.0).astype(np.float32))


def device_fill_fp8(w, layer, k_cache, v_cache, ks, vs):
    """e4m3 caches (uint8 tensors) of N(0,1) values over the per-head scales,
    clamped to +-448 (torch's e4m3 cast turns overflow into NaN)."""
    import torch
    g = torch.Generator(device=k_cache.device)
    g.manual_seed(w.seed * 1000 + layer)
    for t, sc in ((k_cache, ks), (v_cache, vs)):
        inv = torch.from_numpy(1.0 / sc).to(t.device)
        for blk in range(0, t.shape[0], 4096):
            e = min(t.shape[0], blk + 4096)
            x = torch.randn((e - blk,) + tuple(t.shape[1:]), generator=g, device=t.device)
            x.mul_(inv[None, :, None, None]).clamp_(-448.0, 448.0)
            t[blk:e].copy_(x.to(torch.float8_e4m3fn).view(torch.uint8))


def describe(w):
    return {"workload": w.name, "layers": w.layers, "batch": w.B, "Hq": w.Hq, "Hkv": w.Hkv,
            "head_dim": w.head_dim, "block_size": BLOCK, "pool_blocks_per_layer": w.num_blocks,
            "contexts": "log-uniform [512, 8192] + 1 appended" if w.ctx_kind == "loguniform" else w.ctx_kind,
            "pool": "fragmented by seeded alloc/free churn" if w.churn else "seeded permutation",
            "l2": "no flush: every layer reads its own K/V (> L2) once per step",
            "parallelism": "replicas"}


def kv_variant_record(args, kv):
    """The same serving step over one-byte caches (kv "fp8": the fused e4m3
    decode step; "int8": the INT8 append and attention), run as `bench.py
    --kv <kv>` in a child process with this run's steps and warm-up; its
    headline figures, for the default line."""
    cmd = [sys.executable, os.path.abspath(__file__), "--kv", kv, "--steps", str(args.steps), "--warmup",
           str(args.warmup), "--no-cpu-baseline", "--e2e-steps", "3"]
    try:
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
        line = [x for x in r.stdout.splitlines() if x.startswith("{")][-1]
        d = json.loads(line)
    except Exception as e:  # reported, not fatal: the bf16 line stands on its own
        return {"unavailable": ("%s: %s" % (type(e).__name__, e))[:200]}
    rf = d["roofline"]
    return {"metric": d["metric"], "value": d["value"], "unit": d["unit"], "ms_per_step": d["ms_per_step"],
            "steps_per_s": d["steps_per_s"], "dtype": d["dtype"], "kv_cache": d["config"]["kv_cache"],
            "roofline": {k: rf[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic", "kernel",
                                            "avg_launch_ms", "avg_launch_source")},
            "per_layer_ms": d["per_layer_ms"], "e2e": d["e2e"], "clocks": d["clocks"],
            "command": " ".join(["python", "bench.py"] + cmd[2:])}


def prefill_variant_record(args):
    """The Qwen3-8B-shaped prefill step (36 layers of chunked append + causal
    prefill attention on the default kernel), run as `bench.py --workload
    qwen3_8b_prefill` in a child process; its headline figures, for the
    default line."""
    cmd = [sys.executable, os.path.abspath(__file__), "--workload", "qwen3_8b_prefill", "--steps",
           str(min(args.steps, 20)), "--warmup", str(args.warmup), "--no-cpu-baseline", "--e2e-steps", "1"]
    try:
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
        line = [x for x in r.stdout.splitlines() if x.startswith("{")][-1]
        d = json.loads(line)
    except Exception as e:  # reported, not fatal: the decode line stands on its own
        return {"unavailable": ("%s: %s" % (type(e).__name__, e))[:200]}
    rf = d["roofline"]
    return {"metric": d["metric"], "value": d["value"], "unit": d["unit"], "ms_per_step": d["ms_per_step"],
            "dtype": d["dtype"], "workload": d["config"]["workload"],
            "roofline": {k: rf[k] for k in ("bound", "achieved", "peak", "unit", "frac", "peak_kind", "kernel",
                                            "algorithmic_flops_per_launch", "avg_launch_ms")},
            "e2e": d["e2e"], "clocks": d["clocks"], "command": " ".join(["python", "bench.py"] + cmd[2:])}


def arm_config(w, args):
    """The `config` object of a decode line; the GPU arm and the reference
    arm print the same one."""
    if args.kv == "fp8":
        return dict(describe(w), variant="fp8 tensor-core tile", kv_cache="e4m3, per-KV-head fp32 scales")
    if args.kv == "int8":
        return dict(describe(w), variant="int8 tensor-core tile",
                    kv_cache="int8, symmetric per 64-token group and KV head (group maxima per block)")
    return dict(describe(w), variant=args.variant, kv_cache="bf16")


def measured_peak(key="hbm_gbs"):
    fallback = {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)[key]), "measured"
    except Exception:
        return fallback[key], "fallback"


def prefill_flops(w, hist, new):
    """Algorithmic FLOPs of one prefill attention call: new token i of request
    r at position hist[r] + i attends to hist[r] + i + 1 keys; per key and query
    head, 2*d for q.k and 2*d for p*v."""
    h = np.asarray(hist, np.float64)
    m = np.asarray(new, np.float64)
    keys = float(np.sum(m * h + m * (m + 1) / 2))
    return 4.0 * w.head_dim * w.Hq * keys


def kernel_source_hash():
    """Hash of the attention kernel's sources (decode.cu and the headers it
    includes) with comments and whitespace removed, so that a recorded traffic figure stays valid across comment
    edits and is dropped as soon as any code changes."""
    h = hashlib.sha256()
    for f in ("decode.cu", "common.cuh", "tma.cuh", "rope.cuh"):
        with open(os.path.join(ROOT, "paged_kv_decode_25_gb300", "csrc", f), encoding="utf-8") as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per attention launch from the committed ncu summary, when it
    was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "attention_traffic.txt")
    try:
        lines = open(path).read().splitlines()
    except Exception:
        return None
    for line in lines:
        kv = dict(tok.split("=", 1) for tok in line.split() if "=" in tok)
        if kv.get("source") == kernel_source_hash() and kv.get("workload") == workload:
            return float(kv["dram_bytes_per_launch"])
    return None


# ---------------------------------------------------------------- clocks ---

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------- oracle timing --

def oracle_sample(w, nthreads, rank_seed=0):
    """Host inputs for one layer of the step, and a callable that runs the
    oracle's append + attention on them (test infrastructure only)."""
    import oracle
    from oracle.pool import PoolModel
    ctx = context_lengths(w)
    model = PoolModel(w.num_blocks, w.max_seqs, w.max_blocks_per_seq, initial_free_order(w))
    setup_pool(w, model, ctx)
    bt_hist, _, _ = model.batch_meta(range(w.B))
    for b in range(w.B):
        assert model.alloc(b, int(ctx[b]) + 1) == 0
    bt, cl, sl = model.batch_meta(range(w.B))
    kc, vc = history_cache(w, 0, bt_hist, ctx)
    q, k, v = new_token_values(w, 0)
    table = oracle.rope_table(w.theta, w.head_dim, w.max_pos)
    pos = (cl - 1).astype(np.int32)

    def run(nt=nthreads):
        q_out, _ = oracle.append(q, k, v, pos, sl, table, kc, vc)
        oracle.paged_attention(q_out, kc, vc, bt, cl, w.scale, nthreads=nt)
        return oracle.paged_attention.threads_used

    return run, attention_bytes(w, cl) + append_bytes(w)


def time_oracle(w, budget_s=12.0):
    nthreads = os.cpu_count() or 1
    run, nbytes = oracle_sample(w, nthreads)
    t0 = time.perf_counter()
    used = run()
    n = 1
    while time.perf_counter() - t0 < budget_s and n < 50:
        run()
        n += 1
    dt = (time.perf_counter() - t0) / n
    # the same layer on one thread (rows are independent, so the threads do
    # not change the results, only the time)
    t1 = time.perf_counter()
    run(1)
    dt1 = time.perf_counter() - t1
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": int(used), "kind": "oracle",
            "sample": f"one layer of the step (append + attention, all {w.B} requests, {w.Hq} heads), "
                      f"repeated {n}x, fp64 C on {used} POSIX threads; seconds per layer {dt:.3f}",
            "s_per_layer": dt, "single_thread": {"s_per_layer": dt1, "value": nbytes / dt1 / 1e9}}


def prefill_oracle_sample(w, nthreads, rows_per_request=2):
    """Host inputs for a bounded sample of one prefill layer (the first and a
    random new token of every request, each as a one-token request over its
    causal prefix) and a callable running the oracle's chunked append of all
    new tokens plus causal attention of the sampled rows (test infrastructure
    only). Returns (run, flops of the sampled rows)."""
    import oracle
    from oracle.pool import PoolModel
    model = PoolModel(w.num_blocks, w.max_seqs, w.max_blocks_per_seq, None)
    prefill_setup_pool(w, model)
    bt, _, _ = model.batch_meta(range(w.B))
    h, m = w.lengths()
    kc, vc = history_cache(w, 0, bt, h)
    q, k, v = prefill_new_values(w, 0)
    table = oracle.rope_table(w.theta, w.head_dim, w.max_pos)
    pos = np.concatenate([np.arange(h[r], h[r] + m[r]) for r in range(w.B)]).astype(np.int32)
    slots = np.concatenate([model.token_slots(r, int(h[r]), int(m[r])) for r in range(w.B)])
    qs = np.concatenate([[0], np.cumsum(m)]).astype(np.int64)
    rng = np.random.Generator(np.random.PCG64(5))
    rows, lens, tabs = [], [], []
    for r in range(w.B):
        for i in [0] + [int(rng.integers(0, m[r])) for _ in range(rows_per_request - 1)]:
            rows.append(int(qs[r]) + i)
            lens.append(int(h[r]) + i + 1)
            tabs.append(bt[r])
    rows = np.array(rows)
    lens = np.array(lens, np.int32)
    tabs = np.stack(tabs)
    qs1 = np.arange(len(rows) + 1, dtype=np.int32)
    flops = 4.0 * w.head_dim * w.Hq * float(lens.sum())

    def run():
        # the append writes the same values to the same slots on every call
        q_out, _ = oracle.append(q, k, v, pos, slots, table, kc, vc)
        oracle.paged_prefill_attention(q_out[rows], kc, vc, tabs, lens, qs1, w.scale, nthreads=nthreads)
        return nthreads

    return run, flops, len(rows)


# ----------------------------------------------------- the other configs ----

def l2_flush_buffer(device):
    """A device buffer of twice the L2 size: writing it evicts whatever a step
    left in L2, so the next step starts cold."""
    import torch
    l2 = int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0)) or (129 << 20)
    return torch.empty(2 * l2 // 4, dtype=torch.float32, device=device)


def _median_event_ms(fn, stream, reps, warm, flush=None):
    """Median device time of fn() over `reps` runs after `warm` untimed ones,
    events on `stream` around each run; with `flush`, the buffer is written
    before every run, outside the events."""
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for e0, e1 in evs:
        if flush is not None:
            flush.zero_()
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)


def _time_oracle_layer(run, budget_s):
    """Runs the oracle sample `run` (returns the threads it used) until
    budget_s has passed (at least once); returns (seconds per run, runs, threads)."""
    t0 = time.perf_counter()
    used = run()
    n = 1
    while time.perf_counter() - t0 < budget_s and n < 20:
        run()
        n += 1
    return (time.perf_counter() - t0) / n, n, int(used)


def measure_one_layer_config(mi, device, stream, w, peak, flush, reps, warm, oracle_budget_s):
    """One decode layer of workload w (pool history, one appended token per
    request): the fused step and the two calls (append, attention), each the
    median of `reps` event-timed launches; with `flush`, L2 is flushed before
    every launch. The oracle's append + attention of the same layer is timed on
    the host cores over the same blocks (copied back from the device)."""
    import torch
    import oracle
    ctx = context_lengths(w)
    pool = mi.Pool(w.num_blocks, w.max_seqs, w.max_blocks_per_seq, initial_free_order(w))
    setup_pool(w, pool, ctx)
    for b in range(w.B):
        mi.check(pool.alloc(b, int(ctx[b]) + 1), "alloc")
    bt, cl, sl = pool.batch_meta(range(w.B))
    pos = (cl - 1).astype(np.int32)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    shape = (w.num_blocks, w.Hkv, BLOCK, w.head_dim)
    kc = torch.empty(shape, dtype=torch.bfloat16, device=device)
    vc = torch.empty_like(kc)
    device_fill_cache(w, 0, kc, vc)
    q, k, v = new_token_values(w, 0)
    u16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)  # noqa: E731
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(device)  # noqa: E731
    q_d, k_d, v_d = u16(q), u16(k), u16(v)
    qo_d, out_d = torch.empty_like(q_d), torch.empty_like(q_d)
    bt_d, cl_d, sl_d, pos_d = i32(bt), i32(cl), i32(sl), i32(pos)
    st, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos)
    mi.check(st, "rope table")
    rope = torch.from_numpy(table).to(device)
    ws = torch.empty(mi.mi_paged_decode_workspace_bytes(d) // 4 + 4, dtype=torch.float32, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)

    def fused():
        mi.check(mi.mi_paged_decode_step(d, q_d, k_d, v_d, rope, w.max_pos, bt_d, cl_d, w.scale, qo_d, kc, vc,
                                         out_d, ws, dev_err=err, stream=stream), "decode step")

    def two_calls():
        mi.check(mi.mi_paged_kv_append(d, q_d, k_d, v_d, pos_d, sl_d, rope, w.max_pos, qo_d, kc, vc, err, stream),
                 "append")
        mi.check(mi.mi_paged_decode_attention(d, qo_d, kc, vc, bt_d, cl_d, w.scale, out_d, ws, dev_err=err,
                                              stream=stream), "attention")

    t_fused = _median_event_ms(fused, stream, reps, warm, flush)
    t_two = _median_event_ms(two_calls, stream, reps, warm, flush)
    assert int(err.item()) == 0, "device error word %#x" % int(err.item())
    nbytes = attention_bytes(w, cl) + append_bytes(w)
    gbs = nbytes / (t_fused * 1e-3) / 1e9
    rec = {"workload": w.name, "layers": 1, "batch": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.head_dim,
           "path": "fused step (mi_paged_decode_step)", "median_ms": t_fused, "steps_per_s": 1e3 / t_fused,
           "gbs": gbs, "frac": gbs / peak, "algorithmic_bytes_per_step": nbytes,
           "two_calls": {"median_ms": t_two, "gbs": nbytes / (t_two * 1e-3) / 1e9},
           "launches_per_step": 1, "reps": reps,
           "l2": ("flushed before every step (2x L2 written), flush outside the events; launch-bound: the "
                  "step's bytes fit in L2 and take a few microseconds at HBM speed")
           if flush is not None else "no flush: the layer's K/V are larger than L2"}
    # the oracle on the host cores: the same layer over the same blocks
    kc_s, vc_s, bt_s, _ = gather_blocks_to_host(kc, vc, bt, cl)
    table_ref = oracle.rope_table(w.theta, w.head_dim, w.max_pos)
    sl_s = oracle.slot_mapping(bt_s, pos)
    nthreads = os.cpu_count() or 1

    def run():
        q_ref, _ = oracle.append(q, k, v, pos, sl_s, table_ref, kc_s, vc_s)
        oracle.paged_attention(q_ref, kc_s, vc_s, bt_s, cl, w.scale, nthreads=nthreads)
        return oracle.paged_attention.threads_used

    dt, n, used = _time_oracle_layer(run, oracle_budget_s)
    rec["cpu_baseline"] = {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": used, "kind": "oracle",
                           "sample": f"the whole layer (append + attention, all {w.B} requests, {w.Hq} heads), "
                                     f"fp64 C, repeated {n}x; seconds per layer {dt:.4f}"}
    return rec


def measure_sweep_config(mi, device, stream, w, peak, flush, oracle_budget_s):
    """The decode sweep of workload w: from a history of ctx tokens per
    request, w.sweep_steps decode steps over w.layers layers. Each step grows
    the host pool by one token per request, builds the block tables and
    lengths (mi_kv_pool_batch_meta) into pinned buffers, copies them and the
    new q/k/v of every layer to the device, and replays a CUDA graph of the
    layers' fused steps. Timed twice: with L2 flushed before every step (the
    flush outside each step's events; steps/s = steps / the summed step
    times) and back to back without a flush (steps / the whole sweep)."""
    import torch
    import oracle
    from oracle.pool import PoolModel
    ctx = context_lengths(w)
    B, L, S = w.B, w.layers, w.sweep_steps
    seqs = list(range(B))
    d = mi.dims(B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    shape = (w.num_blocks, w.Hkv, BLOCK, w.head_dim)
    caches = []
    for layer in range(L):
        kc = torch.empty(shape, dtype=torch.bfloat16, device=device)
        vc = torch.empty_like(kc)
        device_fill_cache(w, layer, kc, vc)
        caches.append((kc, vc))
    st, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos)
    mi.check(st, "rope table")
    rope = torch.from_numpy(table).to(device)
    u16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)  # noqa: E731
    vals = [new_token_values(w, layer) for layer in range(L)]
    h_q = torch.stack([u16(x[0]) for x in vals]).pin_memory()
    h_k = torch.stack([u16(x[1]) for x in vals]).pin_memory()
    h_v = torch.stack([u16(x[2]) for x in vals]).pin_memory()
    q_all, k_all, v_all = h_q.to(device), h_k.to(device), h_v.to(device)
    qo_all, out_all = torch.empty_like(q_all), torch.empty_like(q_all)
    bt_d = torch.empty((B, w.max_blocks_per_seq), dtype=torch.int32, device=device)
    cl_d = torch.empty(B, dtype=torch.int32, device=device)
    # two sets of pinned metadata buffers, each reused only once the copies
    # out of it have run (an event per set)
    meta = [(torch.empty((B, w.max_blocks_per_seq), dtype=torch.int32).pin_memory(),
             torch.empty(B, dtype=torch.int32).pin_memory(), np.empty(B, np.int32), torch.cuda.Event())
            for _ in range(2)]
    # two workspaces in turn: consecutive layers start early (MI_STEP_EARLY_START)
    ws = [torch.empty(mi.mi_paged_decode_workspace_bytes(d) // 4 + 4, dtype=torch.float32, device=device)
          for _ in range(2)]
    err = torch.zeros(1, dtype=torch.int32, device=device)

    def layers(st_):
        for layer in range(L):
            kc, vc = caches[layer]
            mi.check(mi.mi_paged_decode_step(d, q_all[layer], k_all[layer], v_all[layer], rope, w.max_pos, bt_d,
                                             cl_d, w.scale, qo_all[layer], kc, vc, out_all[layer], ws[layer % 2],
                                             dev_err=err, stream=st_, flags=mi.MI_STEP_EARLY_START),
                     "decode step")

    def host_step(pool, s, buf):
        h_bt, h_cl, h_sl, ev = meta[buf]
        ev.synchronize()  # the copies out of this set (two steps ago) have run
        for b in seqs:
            mi.check(pool.alloc(b, int(ctx[b]) + s + 1), "alloc")
        st_, _, _, _ = mi.mi_kv_pool_batch_meta(pool.handle, seqs, w.max_blocks_per_seq, h_bt.numpy(),
                                                h_cl.numpy(), h_sl)
        mi.check(st_, "batch_meta")
        bt_d.copy_(h_bt, non_blocking=True)
        cl_d.copy_(h_cl, non_blocking=True)
        ev.record(stream)
        q_all.copy_(h_q, non_blocking=True)
        k_all.copy_(h_k, non_blocking=True)
        v_all.copy_(h_v, non_blocking=True)
        return L * (attention_bytes(w, h_cl.numpy()) + append_bytes(w))

    def fresh_pool():
        pool = mi.Pool(w.num_blocks, w.max_seqs, w.max_blocks_per_seq, initial_free_order(w))
        setup_pool(w, pool, ctx)
        return pool

    # first step eagerly (kernel attributes, tensor maps), then capture the layers
    pool = fresh_pool()
    host_step(pool, 0, 0)
    layers(stream)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layers(torch.cuda.current_stream(device))
    torch.cuda.synchronize()

    def sweep(flushed):
        pool = fresh_pool()
        nbytes = 0
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(S)]
        for s in range(S):
            if flushed:
                flush.zero_()
            evs[s][0].record(stream)
            nbytes += host_step(pool, s, s & 1)
            g.replay()
            evs[s][1].record(stream)
        torch.cuda.synchronize()
        per = [e0.elapsed_time(e1) for e0, e1 in evs]
        return nbytes, sum(per), evs[0][0].elapsed_time(evs[-1][1])

    sweep(True)  # warm-up sweep
    runs = [sweep(True) for _ in range(3)]
    warm_runs = [sweep(False) for _ in range(3)]
    # the device side alone: the graph of the layers replayed on the last
    # step's inputs, back to back (no host work, no copies)
    ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ga.record(stream)
    for _ in range(20):
        g.replay()
    gb.record(stream)
    torch.cuda.synchronize()
    graph_ms = ga.elapsed_time(gb) / 20
    assert int(err.item()) == 0, "device error word %#x" % int(err.item())
    nbytes = runs[0][0]
    t_flushed = statistics.median(r[1] for r in runs)
    t_warm = statistics.median(r[2] for r in warm_runs)
    gbs = nbytes / (t_flushed * 1e-3) / 1e9
    rec = {"workload": w.name, "layers": L, "batch": B, "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.head_dim,
           "sweep_steps": S, "contexts": f"{int(ctx[0]) + 1} -> {int(ctx[0]) + S} tokens per request",
           "path": ("per step: host pool growth + mi_kv_pool_batch_meta, H2D of tables, lengths and every "
                    "layer's new q/k/v from pinned memory, then a CUDA graph of the layers' fused steps"),
           "sweep_ms": t_flushed, "steps_per_s": S / (t_flushed * 1e-3), "median_ms": t_flushed / S,
           "gbs": gbs, "frac": gbs / peak, "algorithmic_bytes_per_sweep": nbytes,
           "l2_warm": {"sweep_ms": t_warm, "steps_per_s": S / (t_warm * 1e-3),
                       "note": "steps back to back without a flush: a step's K/V (about 91 MB) stay in L2"},
           "graph_only_ms_per_step": graph_ms,
           "launches_per_step": L, "sweeps_timed": len(runs),
           "l2": ("flushed before every step (2x L2 written), flush outside the step's events; launch-bound: "
                  "each layer's K/V is a few MB")}
    # the oracle on the host cores: layer 0 followed through the whole sweep
    # (its own pool model, append and attention), extrapolated to all layers
    kc_h = caches[0][0].view(torch.int16).cpu().numpy().view(np.uint16).copy()
    vc_h = caches[0][1].view(torch.int16).cpu().numpy().view(np.uint16).copy()
    q0, k0, v0 = vals[0]
    table_ref = oracle.rope_table(w.theta, w.head_dim, w.max_pos)
    nthreads = os.cpu_count() or 1

    def run():
        model = PoolModel(w.num_blocks, w.max_seqs, w.max_blocks_per_seq, initial_free_order(w))
        setup_pool(w, model, ctx)
        for s in range(S):
            for b in seqs:
                assert model.alloc(b, int(ctx[b]) + s + 1) == 0
            bt_m, cl_m, sl_m = model.batch_meta(seqs)
            q_ref, _ = oracle.append(q0, k0, v0, (cl_m - 1).astype(np.int32), sl_m, table_ref, kc_h, vc_h)
            oracle.paged_attention(q_ref, kc_h, vc_h, bt_m, cl_m, w.scale, nthreads=nthreads)
        return oracle.paged_attention.threads_used

    dt, n, used = _time_oracle_layer(run, oracle_budget_s)
    rec["cpu_baseline"] = {"value": S / (dt * L), "unit": "steps/s", "cores": used, "kind": "oracle",
                           "gbs": nbytes / (dt * L) / 1e9, "extrapolated": True,
                           "sample": f"layer 0 through all {S} steps (pool model, append, attention), fp64 C, "
                                     f"repeated {n}x, {dt:.3f} s per pass; x{L} layers for a sweep"}
    return rec


def gather_blocks_to_host(kc_d, vc_d, bt, cl):
    """Host copies of the blocks the requests use, renumbered 0..n-1, with
    their tables rewritten to the new numbers (data movement only)."""
    import torch
    live = [bt[b, :-(-max(int(cl[b]), 0) // BLOCK)] for b in range(len(cl))]
    used = sorted({int(x) for row in live for x in row})
    remap = np.full(max(used) + 1, -1, np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    idx = torch.tensor(used, dtype=torch.int64, device=kc_d.device)
    kc = kc_d[idx].view(torch.int16).cpu().numpy().view(np.uint16)
    vc = vc_d[idx].view(torch.int16).cpu().numpy().view(np.uint16)
    bt_s = np.full(bt.shape, -1, np.int32)
    for i, row in enumerate(live):
        bt_s[i, :len(row)] = remap[row]
    return kc, vc, bt_s, used


def measure_configs(mi, device, peak, oracle_budget_s=3.0):
    """The workloads other than the headline, one GPU: the Qwen3-1.7B-shaped
    layer and the Qwen2.5-7B-shaped 128-step sweep (both L2-flushed before
    every step), and the skewed batch of one 32k and 255 short contexts."""
    import torch
    stream = torch.cuda.current_stream(device)
    flush = l2_flush_buffer(device)
    out = {}
    out["qwen3_1p7b"] = measure_one_layer_config(mi, device, stream, WORKLOADS["qwen3_1p7b"], peak, flush,
                                                 reps=50, warm=5, oracle_budget_s=oracle_budget_s)
    out["qwen25_7b_sweep"] = measure_sweep_config(mi, device, stream, WORKLOADS["qwen25_7b_sweep"], peak, flush,
                                                  oracle_budget_s=oracle_budget_s)
    del flush
    torch.cuda.empty_cache()
    out["skewed"] = measure_one_layer_config(mi, device, stream, WORKLOADS["skewed"], peak, None,
                                             reps=50, warm=5, oracle_budget_s=oracle_budget_s)
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------ reference ----

def run_reference(args, w, rank, world):
    """The reference arm: the oracle as it stands, on the host cores, one
    layer of the step (append + attention, every request and head) per timed
    step; ms_per_step is that layer's time x the step's layers (an
    extrapolation, said so in the line)."""
    if rank != 0:
        return
    nthreads = os.cpu_count() or 1
    run, nbytes = oracle_sample(w, nthreads)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    used = nthreads
    for _ in range(args.steps):
        used = run()
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    val = nbytes / dt / 1e9
    sample = (f"one of the {w.layers} layers per step (append + attention, all {w.B} requests, {w.Hq} heads), "
              f"fp64 C; the step time is {w.layers} x the layer's")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 * w.layers,
            "extrapolated": True, "ms_per_layer": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": arm_config(w, args),
            "steps_per_s": 1.0 / (dt * w.layers),
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": int(used), "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def run_prefill(args, w, rank, world):
    """Prefill step: for each layer, the chunked append of every new token
    (RoPE, scatter through mi_kv_pool_token_slots slots) and the causal paged
    prefill attention. Prints one JSON line on rank 0."""
    import dataclasses
    layers = args.layers if args.layers is not None else 36
    w = dataclasses.replace(w, layers=layers)
    h, m = w.lengths()
    n = (h + m).astype(np.int32)
    R, T = w.B, int(m.sum())
    if args.impl == "reference":
        if rank != 0:
            return
        run, flops, nrows = prefill_oracle_sample(w, os.cpu_count() or 1)
        for _ in range(args.warmup):
            run()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            used = run()
        dt = (time.perf_counter() - t0) / args.steps
        val = flops / dt / 1e12
        cores = min(int(used), nrows * w.Hq)
        sample = f"append of all {T} new tokens + causal attention of {nrows} sampled new tokens, one layer"
        print(json.dumps({
            "impl": "reference", "metric": PREFILL_METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "requests": R, "new_tokens": T, "Hq": w.Hq, "Hkv": w.Hkv,
                       "head_dim": w.head_dim, "sample": sample},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}), flush=True)
        return

    import torch
    import paged_kv_decode_25_gb300 as mi
    mi.load()
    device = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    pool = mi.Pool(w.num_blocks, w.max_seqs, w.max_blocks_per_seq, None)
    prefill_setup_pool(w, pool)
    bt, _, _ = pool.batch_meta(range(R))
    slots = np.concatenate([pool.token_slots(r, int(h[r]), int(m[r])) for r in range(R)]).astype(np.int32)
    pos = np.concatenate([np.arange(h[r], h[r] + m[r]) for r in range(R)]).astype(np.int32)
    qs = np.concatenate([[0], np.cumsum(m)]).astype(np.int32)
    d_app = mi.dims(T, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    d_att = mi.dims(R, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    shape = (w.num_blocks, w.Hkv, BLOCK, w.head_dim)
    caches = []
    for layer in range(layers):
        kc = torch.empty(shape, dtype=torch.bfloat16, device=device)
        vc = torch.empty_like(kc)
        device_fill_cache(w, layer + 1000 * rank, kc, vc)
        caches.append((kc, vc))
    st, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos)
    mi.check(st, "rope table")
    rope = torch.from_numpy(table).to(device)

    def u16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)

    q_h, k_h, v_h = (u16(a) for a in prefill_new_values(w, 0))  # one set of new-token values, every layer
    q_d, k_d, v_d = q_h.to(device), k_h.to(device), v_h.to(device)
    qo_d, out_d = torch.empty_like(q_d), torch.empty_like(q_d)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(device)  # noqa: E731
    bt_d, n_d, qs_d, sl_d, pos_d = i32(bt), i32(n), i32(qs), i32(slots), i32(pos)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    max_q = int(m.max())
    pvar = {"mma": mi.MI_PREFILL_MMA, "single": mi.MI_PREFILL_TCGEN05,
            "pair": mi.MI_PREFILL_TCGEN05_PAIR}.get(args.variant, mi.MI_PREFILL_DEFAULT)
    kernel_name = {"mma": "paged prefill attention (mma.sync m16n8k16 bf16), per layer",
                   "single": "paged prefill attention (tcgen05.mma, one Q tile per CTA, two CTAs per SM), per layer"
                   }.get(args.variant, "paged prefill attention (tcgen05.mma, two Q tiles per CTA sharing 128-key "
                                       "stages, 16 softmax warps), per layer")

    def step(ev=None):
        for layer in range(layers):
            kc, vc = caches[layer]
            mi.check(mi.mi_paged_kv_append(d_app, q_d, k_d, v_d, pos_d, sl_d, rope, w.max_pos, qo_d, kc, vc,
                                           err, stream), "append")
            if ev is not None:
                ev[layer][0].record(stream)
            mi.check(mi.mi_paged_prefill_attention_variant(d_att, T, max_q, qo_d, kc, vc, bt_d, n_d, qs_d, w.scale,
                                                           out_d, variant=pvar, dev_err=err, stream=stream),
                     "prefill attention")
            if ev is not None:
                ev[layer][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(layers)]
           for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(device.index)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_start.record(stream)
    for s_ in range(args.steps):
        step(evs[s_])
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    assert int(err.item()) == 0, "device error word %#x" % int(err.item())
    step_ms = max_over_ranks(t_start.elapsed_time(t_end) / args.steps, world, device)
    attn_ms = [evs[s_][l_][0].elapsed_time(evs[s_][l_][1]) for s_ in range(args.steps) for l_ in range(layers)]
    attn_avg_ms = sum(attn_ms) / len(attn_ms)
    fl = prefill_flops(w, h, m)
    value = world * layers * fl / (step_ms * 1e-3) / 1e12
    peak, peak_kind = measured_peak("bf16_tflops_sustained")
    achieved = fl / (attn_avg_ms * 1e-3) / 1e12

    # end to end: new-token values and metadata from pinned host memory, outputs back
    e2e_steps = args.e2e_steps if args.e2e_steps is not None else max(3, min(args.steps, 10))
    pin = lambda t: t.clone().pin_memory()  # noqa: E731
    hq, hk, hv = pin(q_h), pin(k_h), pin(v_h)
    meta = [(pin(torch.from_numpy(np.ascontiguousarray(a, np.int32))), dst)
            for a, dst in ((bt, bt_d), (n, n_d), (qs, qs_d), (slots, sl_d), (pos, pos_d))]
    h_out = torch.empty(out_d.shape, dtype=torch.bfloat16).pin_memory()

    def e2e_step():
        for src, dst in meta + [(hq, q_d), (hk, k_d), (hv, v_d)]:
            dst.copy_(src, non_blocking=True)
        step()
        h_out.copy_(out_d, non_blocking=True)
        torch.cuda.synchronize()

    e2e_step()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, device) / e2e_steps
    h2d = sum(t.numel() * t.element_size() for t, _ in meta) + sum(
        t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = h_out.numel() * h_out.element_size()
    if rank != 0:
        barrier(world)
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        run, flops, nrows = prefill_oracle_sample(w, os.cpu_count() or 1)
        t0 = time.perf_counter()
        run()
        reps = 1
        while time.perf_counter() - t0 < 12.0 and reps < 20:
            run()
            reps += 1
        dt = (time.perf_counter() - t0) / reps
        cpu = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": min(os.cpu_count() or 1, nrows * w.Hq),
               "kind": "oracle",
               "sample": f"append of all {T} new tokens + causal attention of {nrows} sampled new tokens "
                         f"(one layer), fp64 C, repeated {reps}x; seconds per sample {dt:.3f}"}
    line = {
        "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "layers": layers, "requests": R, "new_tokens": T,
                   "history": "8 fresh prompts U[512, 2048]; 8 chunks of 512 over log-uniform [1024, 8192]",
                   "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.head_dim, "block_size": BLOCK,
                   "l2": "no flush: every layer reads its own caches", "parallelism": "replicas"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None, "peak_kind": peak_kind + " (sustained bf16)",
                     "kernel": kernel_name,
                     "algorithmic_flops_per_launch": fl, "avg_launch_ms": attn_avg_ms},
        "cpu_baseline": cpu,
        "e2e": {"value": world * layers * fl / e2e_s / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": e2e_s * 1e3},
        "gpu_launches": args.steps * layers * 2,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    barrier(world)


def run_swap(args, rank, world):
    """KV swap step on the Qwen3-8B serving pool (one layer's caches): the 16
    least recently used sequences are swapped out to a pinned host cache and
    back in, each direction one mi_kv_copy_blocks launch. Prints one
    JSON line on rank 0; the reference rate is a contiguous pinned
    cudaMemcpyAsync of the same bytes, each direction, timed in the same run."""
    import torch
    import paged_kv_decode_25_gb300 as mi
    w = WORKLOADS["qwen3_8b"]
    name = "qwen3_8b_swap"
    if args.impl == "reference":
        if rank != 0:
            return
        import oracle.swap as osw
        r = np.random.Generator(np.random.PCG64(1))
        nb = 4096
        src = r.integers(0, 1 << 16, size=(nb, w.Hkv, BLOCK, w.head_dim), dtype=np.uint16)
        dst = np.zeros((nb, w.Hkv, BLOCK, w.head_dim), np.uint16)
        ids = r.permutation(nb)
        for _ in range(args.warmup):
            osw.copy_blocks(src, ids, dst, np.arange(nb))
        t0 = time.perf_counter()
        for _ in range(args.steps):
            osw.copy_blocks(src, ids, dst, np.arange(nb))
        dt = (time.perf_counter() - t0) / args.steps
        val = 2 * src.nbytes / dt / 1e9  # K and V counted as in the GPU arm: one cache copied twice
        sample = f"{nb} scattered blocks of one cache copied block by block with numpy, one thread"
        print(json.dumps({
            "impl": "reference", "metric": "KV swap GB/s", "value": val, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u16", "data": "synthetic",
            "config": {"workload": name, "sample": sample},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}), flush=True)
        return
    mi.load()
    device = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(device)
    ctx = context_lengths(w)
    pool = mi.Pool(w.num_blocks, w.max_seqs, w.max_blocks_per_seq, initial_free_order(w))
    setup_pool(w, pool, ctx)
    seqs = list(range(w.B))
    assert pool.touch(seqs[16:]) == 0  # the batch's last 48 requests were just used
    victims = []  # LRU order: idle sequences left by the churn first, then requests 0..15
    for _ in range(16):
        v = pool.lru_victim(victims)
        victims.append(v)
    host = mi.Pool(w.num_blocks, w.max_seqs, w.max_blocks_per_seq)
    src_blocks, host_blocks = [], []
    for v in victims:
        st, blocks = pool.swap_out(v)
        mi.check(st, "swap_out")
        mi.check(host.alloc(v, len(blocks) * BLOCK), "host alloc")
        src_blocks += blocks
        host_blocks += [int(x) for x in mi.mi_kv_pool_seq_blocks(host.handle, v)]
    back_blocks = []
    for v in victims:
        st, blocks = pool.swap_in(v)
        mi.check(st, "swap_in")
        back_blocks += blocks
    n = len(src_blocks)
    shape = (w.num_blocks, w.Hkv, BLOCK, w.head_dim)
    kc = torch.empty(shape, dtype=torch.bfloat16, device=device)
    vc = torch.empty_like(kc)
    device_fill_cache(w, 0, kc, vc)
    nh = max(host_blocks) + 1
    hk = torch.empty((nh,) + shape[1:], dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(device)  # noqa: E731
    s_d, h_d, b_d = i32(src_blocks), i32(host_blocks), i32(back_blocks)
    dims = mi.dims(1, w.Hkv, w.Hkv, w.head_dim, 1, 1)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    block_bytes = w.Hkv * BLOCK * w.head_dim * 2
    moved = 2 * 2 * n * block_bytes  # K and V, out and back

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        mi.check(mi.mi_kv_copy_blocks(dims, kc, vc, w.num_blocks, s_d, hk, hv, nh, h_d, n, err, stream), "out")
        if ev is not None:
            ev[1].record(stream)
        mi.check(mi.mi_kv_copy_blocks(dims, hk, hv, nh, h_d, kc, vc, w.num_blocks, b_d, n, err, stream), "in")
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(device.index)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    for e in evs:
        step(e)
    torch.cuda.synchronize()
    clk = clocks.stop()
    assert int(err.item()) == 0, "device error word %#x" % int(err.item())
    out_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    in_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps
    step_ms = out_ms + in_ms
    # reference: the same bytes as one contiguous pinned copy per direction and cache
    half = n * block_bytes
    dflat = kc.view(-1)[: half // 2]
    hflat = hk.view(-1)[: half // 2]
    ce = []
    for _ in range(3 + args.steps):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record(stream)
        hflat.copy_(dflat, non_blocking=True)
        hflat.copy_(dflat, non_blocking=True)
        e[1].record(stream)
        dflat.copy_(hflat, non_blocking=True)
        dflat.copy_(hflat, non_blocking=True)
        e[2].record(stream)
        ce.append(e)
    torch.cuda.synchronize()
    ce = ce[3:]
    ce_out = sum(e[0].elapsed_time(e[1]) for e in ce) / len(ce)
    ce_in = sum(e[1].elapsed_time(e[2]) for e in ce) / len(ce)
    gbs = lambda ms: 2 * half / (ms * 1e-3) / 1e9  # noqa: E731
    value = moved / (step_ms * 1e-3) / 1e9
    peak = moved / ((ce_out + ce_in) * 1e-3) / 1e9
    line = {
        "metric": "KV swap GB/s", "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, "victims": 16, "blocks": n, "bytes_per_direction": 2 * half,
                   "from": "qwen3_8b pool after churn: the 16 least recently used sequences, one layer",
                   "host": "pinned (cudaHostAlloc through torch), read and written in place by the kernel"},
        "swap_out_gbs": gbs(out_ms), "swap_in_gbs": gbs(in_ms),
        "roofline": {"bound": "link", "achieved": value, "peak": peak, "unit": "GB/s", "frac": value / peak,
                     "traffic": None, "peak_kind": "measured in this run: contiguous pinned cudaMemcpyAsync "
                                                  "of the same bytes, each direction",
                     "peak_out_gbs": gbs(ce_out), "peak_in_gbs": gbs(ce_in)},
        "cpu_baseline": None,
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": moved // 2, "d2h_bytes_per_step": moved // 2,
                "note": "the swap is itself host<->device traffic"},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- main -----

def dist_setup(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_rate(units_per_rank, seconds_max, world):
    """Whole-job throughput of `world` replicas that each process
    units_per_rank units, timed as the slowest rank's seconds."""
    return world * units_per_rank / seconds_max


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--workload", default="qwen3_8b",
                    choices=list(WORKLOADS) + list(PREFILL_WORKLOADS) + ["qwen3_8b_swap"])
    ap.add_argument("--variant", default="default", choices=["default", "mma", "fma", "pair", "single"],
                    help="decode: attention tile (mma, fma); prefill: mma (mma.sync), single (tcgen05, one Q tile "
                         "per CTA) or pair (the default: two Q tiles per CTA)")
    ap.add_argument("--unfused", action="store_true",
                    help="decode: time append and attention as two calls instead of the fused step")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8", "int8"],
                    help="KV cache element type of the decode step (fp8: e4m3 with per-head scales; int8: "
                         "symmetric 64-token groups)")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--layers", type=int, default=None,
                    help="layers per step (default: the workload's); fewer only for small profiling runs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-early-start", action="store_true",
                    help="fused steps wait for the layer before them before planning (no MI_STEP_EARLY_START)")
    ap.add_argument("--no-per-variant", action="store_true",
                    help="skip the e4m3-cache run of the same step in the default line")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other workloads' records (Qwen3-1.7B layer, Qwen2.5-7B sweep, skewed batch)")
    args = ap.parse_args()
    assert args.warmup >= 0 and args.steps >= 1
    rank, world, local = dist_setup(args)
    if args.workload in PREFILL_WORKLOADS:
        run_prefill(args, PREFILL_WORKLOADS[args.workload], rank, world)
        return
    if args.workload == "qwen3_8b_swap":
        run_swap(args, rank, world)
        return
    w = WORKLOADS[args.workload]
    if args.layers is not None:
        import dataclasses
        w = dataclasses.replace(w, layers=args.layers)
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    import torch
    import paged_kv_decode_25_gb300 as mi
    mi.load()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    variant = {"default": mi.MI_ATTN_DEFAULT, "mma": mi.MI_ATTN_MMA, "fma": mi.MI_ATTN_FMA}[args.variant]
    fp8, int8 = args.kv == "fp8", args.kv == "int8"
    kvb = 1 if (fp8 or int8) else 2
    if (fp8 or int8) and not w.device_fill:
        raise SystemExit("--kv %s is measured on the device-filled serving workload" % args.kv)

    # ---- workload: pool history, caches, new-token values (one replica per rank)
    ctx = context_lengths(w)
    pool = mi.Pool(w.num_blocks, w.max_seqs, w.max_blocks_per_seq, initial_free_order(w))
    setup_pool(w, pool, ctx)
    seqs = list(range(w.B))
    for b in seqs:
        mi.check(pool.alloc(b, int(ctx[b]) + 1), "alloc")
    bt, cl, sl = pool.batch_meta(seqs)
    pos = (cl - 1).astype(np.int32)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    shape = (w.num_blocks, w.Hkv, BLOCK, w.head_dim)
    caches = []
    ks_h, vs_h = fp8_scales(w)
    ks_d, vs_d = torch.from_numpy(ks_h).to(device), torch.from_numpy(vs_h).to(device)
    for layer in range(w.layers):
        if int8:
            # codes, group maxima and each sequence's open-group rows (slot b)
            k8, v8, ka, va = device_int8_cache(w, layer + 1000 * rank, device)
            ko = torch.zeros((w.B, w.Hkv, 64, w.head_dim), dtype=torch.bfloat16, device=device)
            caches.append((k8, v8, ka, va, ko, torch.zeros_like(ko)))
            continue
        kc = torch.empty(shape, dtype=torch.uint8 if fp8 else torch.bfloat16, device=device)
        vc = torch.empty_like(kc)
        if fp8:
            device_fill_fp8(w, layer + 1000 * rank, kc, vc, ks_h, vs_h)
        elif w.device_fill:
            device_fill_cache(w, layer + 1000 * rank, kc, vc)
        else:
            hk, hv = history_cache(w, layer, bt, ctx)
            kc.copy_(torch.from_numpy(hk.view(np.int16)).view(torch.bfloat16))
            vc.copy_(torch.from_numpy(hv.view(np.int16)).view(torch.bfloat16))
        caches.append((kc, vc))
    st, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos + 4096)
    mi.check(st, "rope table")
    rope = torch.from_numpy(table).to(device)
    max_pos = table.shape[0]

    def u16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)

    qkv_host = [new_token_values(w, layer) for layer in range(w.layers)]
    q_all = torch.stack([u16(x[0]) for x in qkv_host]).to(device)   # [L][B][Hq][d]
    k_all = torch.stack([u16(x[1]) for x in qkv_host]).to(device)
    v_all = torch.stack([u16(x[2]) for x in qkv_host]).to(device)
    qo_all = torch.empty_like(q_all)
    out_all = torch.empty_like(q_all)
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(device)  # noqa: E731
    bt_d, cl_d, sl_d, pos_d = i32(bt), i32(cl), i32(sl), i32(pos)
    open_slots_d = i32(np.arange(w.B))
    dev_bufs = (q_all, k_all, v_all, qo_all, out_all, bt_d, cl_d, sl_d, pos_d)
    ws = torch.empty(mi.mi_paged_decode_workspace_bytes(d) // 4 + 4, dtype=torch.float32, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    stream = stream0 = torch.cuda.current_stream(device)
    # fused steps start early (each layer's plan and first copies overlap the
    # layer before): no layer writes another's inputs, and two workspaces in
    # turn keep each step's plan entries away from the step before it
    early = not args.no_early_start
    step_flags = mi.MI_STEP_EARLY_START if early else 0
    ws_step = (ws, torch.empty_like(ws)) if early else (ws, ws)

    # the fused step (append + attention in one launch per layer; bf16 caches
    # on the MMA tile, or e4m3 caches) is the timed path; the two calls are
    # timed after it to report append and attention separately
    fused = (fp8 or variant in (mi.MI_ATTN_DEFAULT, mi.MI_ATTN_MMA)) and not args.unfused and not int8

    def step(ev=None, fuse=False, st=None, bufs=None):
        stream = st if st is not None else stream0
        q_all, k_all, v_all, qo_all, out_all, bt_d, cl_d, sl_d, pos_d = bufs if bufs is not None else dev_bufs
        for layer in range(w.layers):
            kc, vc = caches[layer][:2]
            if fuse:
                if ev is not None:
                    ev[layer][0].record(stream)
                wsl = ws_step[layer % 2]
                if fp8:
                    mi.check(mi.mi_paged_decode_step_fp8(d, q_all[layer], k_all[layer], v_all[layer], rope, max_pos,
                                                         bt_d, cl_d, ks_d, vs_d, w.scale, qo_all[layer], kc, vc,
                                                         out_all[layer], wsl, dev_err=err, stream=stream,
                                                         flags=step_flags), "decode step (e4m3)")
                else:
                    mi.check(mi.mi_paged_decode_step(d, q_all[layer], k_all[layer], v_all[layer], rope, max_pos,
                                                     bt_d, cl_d, w.scale, qo_all[layer], kc, vc, out_all[layer], wsl,
                                                     dev_err=err, stream=stream, flags=step_flags), "decode step")
                if ev is not None:
                    ev[layer][1].record(stream)
                continue
            if int8:
                _, _, ka, va, ko, vo = caches[layer]
                mi.check(mi.mi_paged_kv_append_int8(d, q_all[layer], k_all[layer], v_all[layer], rope, max_pos,
                                                    bt_d, cl_d, open_slots_d, qo_all[layer], kc, vc, ka, va, ko, vo,
                                                    err, stream), "append (int8)")
            elif fp8:
                mi.check(mi.mi_paged_kv_append_fp8(d, q_all[layer], k_all[layer], v_all[layer], pos_d, sl_d, rope,
                                                   max_pos, qo_all[layer], kc, vc, ks_d, vs_d, err, stream),
                         "append")
            else:
                mi.check(mi.mi_paged_kv_append(d, q_all[layer], k_all[layer], v_all[layer], pos_d, sl_d, rope,
                                               max_pos, qo_all[layer], kc, vc, err, stream), "append")
            if ev is not None:
                ev[layer][0].record(stream)
            if int8:
                mi.check(mi.mi_paged_decode_attention_int8(d, qo_all[layer], kc, vc, ka, va, bt_d, cl_d, w.scale,
                                                           out_all[layer], ws, dev_err=err, stream=stream),
                         "attention (int8)")
            elif fp8:
                mi.check(mi.mi_paged_decode_attention_fp8(d, qo_all[layer], kc, vc, ks_d, vs_d, bt_d, cl_d, w.scale,
                                                          out_all[layer], ws, dev_err=err, stream=stream),
                         "attention")
            else:
                mi.check(mi.mi_paged_decode_attention_variant(d, qo_all[layer], kc, vc, bt_d, cl_d, w.scale,
                                                              out_all[layer], ws, variant=variant, dev_err=err,
                                                              stream=stream), "attention")
            if ev is not None:
                ev[layer][1].record(stream)

    # ---- device-timed steps (fixed step replayed; inputs resident). Every
    # step rewrites the same new-token rows, so replays see the same inputs.
    # The timed region replays K times a CUDA graph that holds one step (the
    # launches a serving loop captures once), with a CUDA event between the
    # replays (the per-step times give the median). Events between the
    # kernels would serialise the graph's launches, so per-kernel times come
    # from separate passes after it: the steps as a graph with an event
    # captured around every timed kernel, and launched on the stream.
    def new_events(n, **kw):
        return [[[torch.cuda.Event(enable_timing=True, **kw) for _ in range(2)] for _ in range(w.layers)]
                for _ in range(n)]

    def capture(n, evs=None):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cap = torch.cuda.current_stream(device)
            for s in range(n):
                step(None if evs is None else evs[s], fuse=fused, st=cap)
        return g

    step(fuse=fused)  # first launches (kernel attributes, tensor maps) happen outside any capture
    torch.cuda.synchronize()
    try:
        g_step = capture(1)
        launch_mode = "cuda graph of one step, replayed K times"
    except RuntimeError as e:  # capture refused: time stream launches instead
        g_step = None
        launch_mode = "stream launches (%s)" % str(e).splitlines()[0][:120]
    if fused and early:
        launch_mode += "; fused steps start early (MI_STEP_EARLY_START, two workspaces in turn)"
    evs_t = new_events(args.steps) if g_step is None else None
    for _ in range(args.warmup):
        if g_step is not None:
            g_step.replay()
        else:
            step(fuse=fused)
    torch.cuda.synchronize()
    t_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
    clocks = ClockSampler(int(vis[local]) if len(vis) > local and vis[local].isdigit() else local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_ev[0].record(stream)
    for s in range(args.steps):
        if g_step is not None:
            g_step.replay()
        else:
            step(evs_t[s], fuse=fused)
        t_ev[s + 1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    assert int(err.item()) == 0, "device error word %#x" % int(err.item())
    step_ms_local = t_ev[0].elapsed_time(t_ev[args.steps]) / args.steps
    step_ms = max_over_ranks(step_ms_local, world, device)
    median_step_ms = statistics.median(t_ev[s].elapsed_time(t_ev[s + 1]) for s in range(args.steps))

    def kernel_avg(evs, n):
        return sum(evs[s][layer][0].elapsed_time(evs[s][layer][1]) for s in range(n)
                   for layer in range(w.layers)) / (n * w.layers)

    # per-kernel events: the steps as a graph with events around every timed
    # kernel (where this torch records events inside graphs), and on the stream
    ev_steps = max(3, min(args.steps, 10))
    try:
        evs_g = new_events(ev_steps, external=True)
        g_ev = capture(ev_steps, evs_g)
        g_ev.replay()
        torch.cuda.synchronize()
        del g_ev
        graph_events = {"ms_per_timed_kernel": kernel_avg(evs_g, ev_steps), "steps": ev_steps}
    except (TypeError, RuntimeError) as e:
        evs_g, graph_events = None, {"unavailable": str(e).splitlines()[0][:120]}
    evs_s = new_events(ev_steps)
    tsa, tsb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tsa.record(stream)
    for s in range(ev_steps):
        step(evs_s[s], fuse=fused)
    tsb.record(stream)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, "device error word %#x" % int(err.item())
    stream_launch = {"ms_per_step": tsa.elapsed_time(tsb) / ev_steps, "steps": ev_steps,
                     "ms_per_timed_kernel": kernel_avg(evs_s, ev_steps)}
    # the dominant kernel's average launch: the fused step is the only launch
    # of a layer, so the timed region per launch bounds it from above (gaps
    # between launches included); otherwise the attention launch's events
    if evs_t is not None:
        kern_avg_ms, kern_src = kernel_avg(evs_t, args.steps), "events around each launch in the timed region"
    elif fused:
        kern_avg_ms = step_ms / w.layers
        kern_src = "timed region / launches (one launch per layer; gaps between launches included)"
    elif evs_g is not None:
        kern_avg_ms, kern_src = graph_events["ms_per_timed_kernel"], "events around each launch, captured in a graph"
    else:
        kern_avg_ms, kern_src = stream_launch["ms_per_timed_kernel"], "events around each stream launch"
    a_bytes = attention_bytes(w, cl, kvb) + (int8_extra_attention_bytes(w, cl) if int8 else 0)
    ap_bytes = append_bytes(w, kvb) + (int8_extra_append_bytes(w) if int8 else 0)
    step_bytes = w.layers * step_kv_bytes(w, cl, args.kv)
    value = whole_job_rate(step_bytes, step_ms * 1e-3, world) / 1e9
    peak, peak_kind = measured_peak()
    # the dominant kernel: the fused step (its bytes include the append's), or the attention
    k_bytes = a_bytes + (ap_bytes if fused else 0)
    achieved = k_bytes / (kern_avg_ms * 1e-3) / 1e9
    traffic = recorded_traffic(w.name + ("_fp8" if fp8 else "_int8" if int8 else "") + ("_step" if fused else ""))

    # append and attention timed separately (the two calls), for the split
    if fused:
        split_steps = ev_steps
        evs2 = new_events(split_steps)
        for _ in range(2):
            step()
        t2a, t2b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t2a.record(stream)
        for s in range(split_steps):
            step(evs2[s])
        t2b.record(stream)
        torch.cuda.synchronize()
        two_call_step_ms = t2a.elapsed_time(t2b) / split_steps
    else:
        split_steps = ev_steps if evs_t is None else args.steps
        evs2 = evs_t if evs_t is not None else (evs_g if evs_g is not None else evs_s)
        two_call_step_ms = step_ms
    attn_avg_ms = kernel_avg(evs2, split_steps)
    # append of layer l runs between the end of layer l-1's attention and its own start event
    app_ms = [evs2[s][layer - 1][1].elapsed_time(evs2[s][layer][0]) for s in range(split_steps)
              for layer in range(1, w.layers)]
    app_avg_ms = sum(app_ms) / len(app_ms) if app_ms else None
    assert int(err.item()) == 0, "device error word %#x" % int(err.item())


    # ---- end to end: real decode steps from host buffers through the C ABI
    e2e_steps = args.e2e_steps if args.e2e_steps is not None else max(3, min(args.steps, 20))
    e2e_warm = min(args.warmup, 2)
    # each e2e step grows every context by one token: stay within the tables
    headroom = int(w.max_blocks_per_seq * BLOCK - int(np.max(cl)))
    e2e_steps = max(1, min(e2e_steps, headroom - e2e_warm))
    e2e_warm = min(e2e_warm, headroom - e2e_steps)
    ctx_now = cl.copy()
    seq_arr = np.asarray(seqs, np.int32)
    # Two sets, each with pinned host buffers (tables, lengths, the step's
    # result) and device buffers (tables, lengths, every layer's new rows and
    # outputs) and its own captured one-step graph: step s uses set s % 2.
    # Copies in run on one stream, the steps on another, copies out on a
    # third, so step s + 1's inputs go in and step s - 1's result comes out
    # while step s computes; the host fills a set once its step two back is
    # done (copies and result).
    def dev_set():
        return tuple(torch.empty_like(t) for t in dev_bufs)

    sets = [dict(bt=torch.empty((w.B, w.max_blocks_per_seq), dtype=torch.int32).pin_memory(),
                 cl=torch.empty(w.B, dtype=torch.int32).pin_memory(),
                 sl=torch.empty(w.B, dtype=torch.int32).pin_memory(),
                 pos=torch.empty(w.B, dtype=torch.int32).pin_memory(),
                 out=torch.empty(out_all.shape, dtype=torch.bfloat16).pin_memory(),
                 dev=dev_set(), done=torch.cuda.Event(), inp=torch.cuda.Event(), comp=torch.cuda.Event())
            for _ in range(2)]
    h_q = torch.stack([u16(x[0]) for x in qkv_host]).pin_memory()
    h_k = torch.stack([u16(x[1]) for x in qkv_host]).pin_memory()
    h_v = torch.stack([u16(x[2]) for x in qkv_host]).pin_memory()
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    for hs in sets:  # the sets' device buffers start from the resident step's contents
        for dst, src in zip(hs["dev"], dev_bufs):
            dst.copy_(src)
    torch.cuda.synchronize()
    e2e_graphs = None
    if g_step is not None:
        e2e_graphs = []
        for hs in sets:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(fuse=fused, st=torch.cuda.current_stream(device), bufs=hs["dev"])
            e2e_graphs.append(g)
    e2e_bytes = 0.0
    e2e_no = 0

    def e2e_step():
        nonlocal ctx_now, e2e_bytes, e2e_no
        k = e2e_no & 1
        hs = sets[k]
        e2e_no += 1
        hs["done"].synchronize()  # the step two back (same set): copies done, result read
        ctx_now = ctx_now + 1
        mi.check(pool.alloc_batch(seq_arr, ctx_now.astype(np.int32)), "alloc_batch")
        st_, _, _, _ = mi.mi_kv_pool_batch_meta(pool.handle, seqs, w.max_blocks_per_seq, hs["bt"].numpy(),
                                                hs["cl"].numpy(), hs["sl"].numpy())
        mi.check(st_, "batch_meta")
        hs["pos"].numpy()[:] = hs["cl"].numpy() - 1
        q_d, k_d, v_d, qo_d, out_d, bt_e, cl_e, sl_e, pos_e = hs["dev"]
        copies = ((hs["bt"], bt_e), (hs["cl"], cl_e)) + (() if fused or int8 else ((hs["sl"], sl_e), (hs["pos"], pos_e))) + \
            ((h_q, q_d), (h_k, k_d), (h_v, v_d))
        with torch.cuda.stream(s_in):
            s_in.wait_event(hs["comp"])  # the set's step two back has read its inputs
            for src, dst in copies:
                dst.copy_(src, non_blocking=True)
            hs["inp"].record(s_in)
        stream.wait_event(hs["inp"])
        if e2e_graphs is not None:
            e2e_graphs[k].replay()
        else:
            step(fuse=fused, bufs=hs["dev"])
        hs["comp"].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(hs["comp"])
            hs["out"].copy_(out_d, non_blocking=True)
            hs["done"].record(s_out)
        e2e_bytes += w.layers * step_kv_bytes(w, hs["cl"].numpy(), args.kv)

    for _ in range(e2e_warm):
        e2e_step()
    torch.cuda.synchronize()
    e2e_bytes = 0.0
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    torch.cuda.synchronize()  # the last step's result is on the host
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, device)
    assert int(err.item()) == 0, "device error word %#x" % int(err.item())
    # the pipeline read back what the step computed: the same step again,
    # eagerly, over the last set's inputs (it rewrites the same new rows)
    # gives the host copy's bits
    last = sets[(e2e_no - 1) & 1]
    check_out = torch.empty_like(last["dev"][4])
    step(fuse=fused, bufs=last["dev"][:4] + (check_out,) + last["dev"][5:])
    torch.cuda.synchronize()
    assert torch.equal(check_out.cpu().view(torch.int16), last["out"].view(torch.int16)), \
        "end-to-end result differs from the step recomputed on its inputs"
    del g_step
    hs = sets[0]
    h2d = sum(t.numel() * t.element_size() for t in (hs["bt"], hs["cl"], h_q, h_k, h_v)) + \
        (0 if fused or int8 else sum(t.numel() * t.element_size() for t in (hs["sl"], hs["pos"])))
    d2h = hs["out"].numel() * hs["out"].element_size()
    e2e_val = world * (e2e_bytes / e2e_steps) / (e2e_s / e2e_steps) / 1e9

    if rank != 0:
        barrier(world)
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = time_oracle(w)
    per_config = None
    if world == 1 and w.name == "qwen3_8b" and args.kv == "bf16" and not args.no_per_config:
        per_config = measure_configs(mi, device, peak)
    per_variant = None
    if world == 1 and w.name == "qwen3_8b" and args.kv == "bf16" and not args.no_per_variant:
        per_variant = {"fp8": kv_variant_record(args, "fp8"), "int8": kv_variant_record(args, "int8"),
                       "prefill": prefill_variant_record(args)}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "median_ms_per_step": median_step_ms,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": ("fp8e4m3 KV, bf16 q/out" if fp8 else "int8 KV, bf16 q/out" if int8 else "bf16"),
        "data": "synthetic",
        "config": arm_config(w, args),
        "steps_per_s": 1e3 / step_ms * world,
        "hbm_frac_step": value / world / peak,
        "per_layer_ms": {"step": step_ms / w.layers, "fused_step_kernel": kern_avg_ms if fused else None,
                         "append": app_avg_ms, "attention": attn_avg_ms,
                         "append+attention (two calls)": two_call_step_ms / w.layers,
                         "append_bytes": ap_bytes, "attention_bytes": a_bytes},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": ("fused decode step (RoPE + cache write of the new token%s, split-KV attention, "
                                "LSE combine), per layer" % (" quantised to e4m3" if fp8 else "") if fused else
                                "paged decode attention%s (split-KV kernel with the LSE combine of cut units fused), "
                                "per layer" % (" over INT8 caches (group maxima staged with each block)" if int8
                                               else "")),
                     "algorithmic_bytes_per_launch": k_bytes, "avg_launch_ms": kern_avg_ms,
                     "avg_launch_source": kern_src},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "ms_per_step": e2e_s / e2e_steps * 1e3,
                "path": ("per step: host pool growth (mi_kv_pool_alloc_batch) and mi_kv_pool_batch_meta into one "
                         "of two pinned buffer sets, H2D of tables, lengths and every layer's new q/k/v from "
                         "pinned memory, "
                         + ("a captured one-step CUDA graph" if launch_mode.startswith("cuda graph")
                            else "stream launches") + ", D2H of every layer's output; two sets of host and "
                         "device buffers (a graph each), copies in and out on their own streams, so step s + 1's "
                         "inputs go in and step s - 1's result comes out while step s computes, and the host "
                         "prepares a set once its step two back is done; timed from the first step's host work to "
                         "the last step's result on the host")},
        "per_config": per_config,
        "per_variant": per_variant,
        "gpu_launches": args.steps * w.layers * (1 if fused else 2),  # fused step, or append + attention
        "launch": launch_mode,
        "graph_with_kernel_events": graph_events,
        "stream_launch": stream_launch,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    barrier(world)


if __name__ == "__main__":
    main()
