"""Oracle for the paged-KV decode step (fp64, CPU).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers. The product library does
not import, link or execute anything under ``oracle/``, and nothing here imports
the product package.

``oracle.c`` holds the arithmetic (bf16 conversion, RoPE table and rotation,
append, paged decode, causal paged prefill and contiguous attention); this module compiles it with gcc into
``oracle/_build/liboracle.so`` and wraps it with ctypes over numpy arrays.
``pool.py`` is a plain-Python model of the block pool. Sources of each function
are cited in ``oracle.c`` and ``pool.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (no fast-math, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.or_double_from_bf16.argtypes = [ctypes.c_uint16]
            lib.or_double_from_bf16.restype = f64
            lib.or_bf16_from_double.argtypes = [f64]
            lib.or_bf16_from_double.restype = ctypes.c_uint16
            lib.or_bf16_from_double_array.argtypes = [P, i64, P]
            lib.or_double_from_bf16_array.argtypes = [P, i64, P]
            lib.or_rope_table.argtypes = [f64, i32, i32, P]
            lib.or_rope_rotate.argtypes = [P, i32, i32, P, i32, P]
            lib.or_slot_mapping.argtypes = [i32, P, i32, P, P]
            lib.or_slot_mapping.restype = i32
            lib.or_append.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, i32, P, P, P]
            lib.or_append.restype = i32
            lib.or_paged_attention.argtypes = [i32, i32, i32, i32, P, P, P, P, i32, P, f64, P, i32]
            lib.or_paged_attention.restype = i32
            lib.or_contiguous_attention.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, f64, P]
            lib.or_paged_prefill_attention.argtypes = [i32, i32, i32, i32, P, P, P, P, i32, P, P, f64, P, i32]
            lib.or_paged_prefill_attention.restype = i32
            lib.or_e4m3_from_double_array.argtypes = [P, ctypes.c_int64, P]
            lib.or_double_from_e4m3_array.argtypes = [P, ctypes.c_int64, P]
            lib.or_append_fp8.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P, i32, P, P, P, P, P]
            lib.or_append_fp8.restype = i32
            lib.or_paged_attention_fp8.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, i32, P, f64, P, i32]
            lib.or_paged_attention_fp8.restype = i32
            lib.or_int8_quantize.argtypes = [P, i64, P]
            lib.or_int8_quantize.restype = ctypes.c_float
            lib.or_int8_from_bf16_cache.argtypes = [i32, i32, i32, i32, P, P, P, i32, P, P, i32, P, P, P, P, P, P]
            lib.or_int8_from_bf16_cache.restype = i32
            lib.or_append_int8.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, i32, P, i32, P, P, i32,
                                           P, P, P, P, P, P, P]
            lib.or_append_int8.restype = i32
            lib.or_paged_attention_int8.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, i32, P, f64, P, i32]
            lib.or_paged_attention_int8.restype = i32
            _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


# --------------------------------------------------------------- bf16 ------

def bf16_to_f64(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exact."""
    h = _c(h, np.uint16)
    out = np.empty(h.shape, np.float64)
    _load().or_double_from_bf16_array(_p(h), h.size, _p(out))
    return out


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns, one rounding to nearest-even."""
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().or_bf16_from_double_array(_p(x), x.size, _p(out))
    return out


def bf16_from_double_scalar(x: float) -> int:
    return int(_load().or_bf16_from_double(float(x)))


# --------------------------------------------------------------- RoPE ------

def rope_table(theta: float, head_dim: int, max_pos: int) -> np.ndarray:
    """float32 [max_pos][head_dim/2][2] of (cos, sin)."""
    out = np.empty((max_pos, head_dim // 2, 2), np.float32)
    _load().or_rope_table(float(theta), head_dim, max_pos, _p(out))
    return out


def rope_rotate(x: np.ndarray, table: np.ndarray, pos: int) -> np.ndarray:
    """Rotate bf16 vectors x[..., d] (uint16 bits), all at position pos."""
    x = _c(x, np.uint16)
    d = x.shape[-1]
    table = _c(table, np.float32)
    assert 0 <= pos < table.shape[0] and table.shape[1] * 2 == d
    y = np.empty_like(x)
    _load().or_rope_rotate(_p(x), x.size // d, d, _p(table), int(pos), _p(y))
    return y


# ------------------------------------------------------ slots / append ------

def slot_mapping(block_tables: np.ndarray, positions: np.ndarray) -> np.ndarray:
    bt = _c(block_tables, np.int32)
    pos = _c(positions, np.int32)
    out = np.empty(pos.shape, np.int32)
    _load().or_slot_mapping(pos.shape[0], _p(bt), bt.shape[1], _p(pos), _p(out))
    return out


def append(q, k, v, positions, slot_mapping_, table, k_cache, v_cache):
    """Returns q_out; writes k_cache / v_cache (uint16 arrays [nb][Hkv][16][d]) in place."""
    q = _c(q, np.uint16); k = _c(k, np.uint16); v = _c(v, np.uint16)
    B, Hq, d = q.shape
    Hkv = k.shape[1]
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16
    pos = _c(positions, np.int32); sm = _c(slot_mapping_, np.int32)
    table = _c(table, np.float32)
    q_out = np.empty_like(q)
    st = _load().or_append(B, Hq, Hkv, d, k_cache.shape[0], _p(q), _p(k), _p(v), _p(pos), _p(sm),
                           _p(table), table.shape[0], _p(q_out), _p(k_cache), _p(v_cache))
    return q_out, st


# ---------------------------------------------------------- attention ------

def paged_attention(q, k_cache, v_cache, block_tables, context_lens, scale, nthreads=1):
    """q uint16 [B][Hq][d]; caches uint16 [nb][Hkv][16][d]; returns float64 [B][Hq][d]."""
    q = _c(q, np.uint16)
    B, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    kc = _c(k_cache, np.uint16); vc = _c(v_cache, np.uint16)
    bt = _c(block_tables, np.int32); cl = _c(context_lens, np.int32)
    out = np.empty((B, Hq, d), np.float64)
    used = _load().or_paged_attention(B, Hq, Hkv, d, _p(q), _p(kc), _p(vc), _p(bt), bt.shape[1],
                                      _p(cl), float(scale), _p(out), int(nthreads))
    paged_attention.threads_used = used
    return out


def contiguous_attention(q, K, V, lens, scale):
    """q uint16 [B][Hq][d]; K, V uint16 [B][Hkv][n_max][d]; returns float64 [B][Hq][d]."""
    q = _c(q, np.uint16); K = _c(K, np.uint16); V = _c(V, np.uint16)
    B, Hq, d = q.shape
    Hkv, n_max = K.shape[1], K.shape[2]
    ln = _c(lens, np.int32)
    out = np.empty((B, Hq, d), np.float64)
    _load().or_contiguous_attention(B, Hq, Hkv, d, n_max, _p(q), _p(K), _p(V), _p(ln), float(scale),
                                    _p(out))
    return out


def paged_prefill_attention(q, k_cache, v_cache, block_tables, context_lens, query_start, scale, nthreads=1):
    """Causal attention of each request's new tokens (rows query_start[r] ..
    query_start[r+1]-1 of q uint16 [T][Hq][d]); returns float64 [T][Hq][d]."""
    q = _c(q, np.uint16)
    T, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    kc = _c(k_cache, np.uint16); vc = _c(v_cache, np.uint16)
    bt = _c(block_tables, np.int32); cl = _c(context_lens, np.int32); qs = _c(query_start, np.int32)
    R = cl.shape[0]
    assert qs.shape == (R + 1,) and qs[R] == T
    out = np.empty((T, Hq, d), np.float64)
    _load().or_paged_prefill_attention(R, Hq, Hkv, d, _p(q), _p(kc), _p(vc), _p(bt), bt.shape[1], _p(cl), _p(qs),
                                       float(scale), _p(out), int(nthreads))
    return out


# ------------------------------------------------------------- FP8 KV ------

def e4m3_from_f64(x: np.ndarray) -> np.ndarray:
    """float64 -> e4m3 codes (uint8): nearest-even, saturating to +-448."""
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint8)
    _load().or_e4m3_from_double_array(_p(x), x.size, _p(out))
    return out


def e4m3_to_f64(c: np.ndarray) -> np.ndarray:
    """e4m3 codes (uint8) -> float64, exact."""
    c = _c(c, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().or_double_from_e4m3_array(_p(c), c.size, _p(out))
    return out


def append_fp8(q, k, v, positions, slot_mapping_, table, k_scale, v_scale, k_cache, v_cache):
    """As append, into uint8 e4m3 caches with fp32 per-KV-head scales.
    Returns (q_out, status)."""
    q = _c(q, np.uint16); k = _c(k, np.uint16); v = _c(v, np.uint16)
    B, Hq, d = q.shape
    Hkv = k.shape[1]
    assert k_cache.dtype == np.uint8 and k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    pos = _c(positions, np.int32); sm = _c(slot_mapping_, np.int32)
    table = _c(table, np.float32)
    ks = _c(k_scale, np.float32); vs = _c(v_scale, np.float32)
    q_out = np.empty_like(q)
    st = _load().or_append_fp8(B, Hq, Hkv, d, k_cache.shape[0], _p(q), _p(k), _p(v), _p(pos), _p(sm),
                               _p(table), table.shape[0], _p(ks), _p(vs), _p(q_out), _p(k_cache), _p(v_cache))
    return q_out, st


def paged_attention_fp8(q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, scale, nthreads=1):
    """q uint16 [B][Hq][d]; caches uint8 e4m3 [nb][Hkv][16][d]; per-KV-head
    fp32 scales; returns float64 [B][Hq][d]."""
    q = _c(q, np.uint16)
    B, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    kc = _c(k_cache, np.uint8); vc = _c(v_cache, np.uint8)
    ks = _c(k_scale, np.float32); vs = _c(v_scale, np.float32)
    bt = _c(block_tables, np.int32); cl = _c(context_lens, np.int32)
    out = np.empty((B, Hq, d), np.float64)
    used = _load().or_paged_attention_fp8(B, Hq, Hkv, d, _p(q), _p(kc), _p(vc), _p(ks), _p(vs), _p(bt),
                                          bt.shape[1], _p(cl), float(scale), _p(out), int(nthreads))
    paged_attention_fp8.threads_used = used
    return out


# ------------------------------------------------------------ INT8 KV ------

GROUP = 64  # tokens per quantisation group


def int8_quantize(x) -> tuple:
    """One group of bf16 values (uint16 bits, any shape) -> (int8 codes of
    the same shape, m = max |x| as a float)."""
    x = _c(x, np.uint16)
    codes = np.empty(x.shape, np.int8)
    m = _load().or_int8_quantize(_p(x), x.size, _p(codes))
    return codes, float(m)


def int8_state(num_blocks: int, Hkv: int, d: int, num_slots: int) -> dict:
    """Zeroed INT8 cache state: int8 caches [nb][Hkv][16][d], fp32 group
    maxima [nb][Hkv], bf16 open-group buffers [slots][Hkv][64][d]."""
    return {
        "k8": np.zeros((num_blocks, Hkv, 16, d), np.int8), "v8": np.zeros((num_blocks, Hkv, 16, d), np.int8),
        "k_amax": np.zeros((num_blocks, Hkv), np.float32), "v_amax": np.zeros((num_blocks, Hkv), np.float32),
        "k_open": np.zeros((num_slots, Hkv, GROUP, d), np.uint16),
        "v_open": np.zeros((num_slots, Hkv, GROUP, d), np.uint16),
    }


def _state_args(st):
    for key in ("k8", "v8", "k_amax", "v_amax", "k_open", "v_open"):
        assert st[key].flags.c_contiguous
    return (_p(st["k8"]), _p(st["v8"]), _p(st["k_amax"]), _p(st["v_amax"]), _p(st["k_open"]), _p(st["v_open"]))


def int8_from_bf16_cache(k_cache, v_cache, block_tables, context_lens, open_slots, st) -> int:
    """Fill the INT8 state `st` (from int8_state) from the first
    context_lens[b] tokens of each request held in bf16 caches (uint16
    [nb][Hkv][16][d]) at the same slots. Returns the status."""
    kc = _c(k_cache, np.uint16); vc = _c(v_cache, np.uint16)
    nb, Hkv, _, d = kc.shape
    bt = _c(block_tables, np.int32); cl = _c(context_lens, np.int32); sl = _c(open_slots, np.int32)
    return _load().or_int8_from_bf16_cache(cl.shape[0], Hkv, d, nb, _p(kc), _p(vc), _p(bt), bt.shape[1], _p(cl),
                                           _p(sl), st["k_open"].shape[0], *_state_args(st))


def append_int8(q, k, v, table, block_tables, context_lens, open_slots, st):
    """Append one token per request (position context_lens[b] - 1) into the
    INT8 state `st`, in place. Returns (q_out, status)."""
    q = _c(q, np.uint16); k = _c(k, np.uint16); v = _c(v, np.uint16)
    B, Hq, d = q.shape
    Hkv = k.shape[1]
    table = _c(table, np.float32)
    bt = _c(block_tables, np.int32); cl = _c(context_lens, np.int32); sl = _c(open_slots, np.int32)
    q_out = np.zeros_like(q)
    status = _load().or_append_int8(B, Hq, Hkv, d, st["k8"].shape[0], _p(q), _p(k), _p(v), _p(table), table.shape[0],
                                    _p(bt), bt.shape[1], _p(cl), _p(sl), st["k_open"].shape[0], _p(q_out),
                                    *_state_args(st))
    return q_out, status


def append_int8_tokens(q, k, v, table, block_tables, context_lens, query_start, open_slots, st):
    """Many new tokens per request: request r's rows query_start[r] ..
    query_start[r+1]-1 of q [T][Hq][d], k and v [T][Hkv][d], at positions
    n_r - m_r .. n_r - 1, appended one token at a time with append_int8 (the
    definition). Returns (q_out [T][Hq][d], status)."""
    q = _c(q, np.uint16); k = _c(k, np.uint16); v = _c(v, np.uint16)
    qs = _c(query_start, np.int32); cl = _c(context_lens, np.int32)
    R = cl.shape[0]
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    m = qs[1:] - qs[:-1]
    q_out = np.zeros_like(q)
    status = 0
    for i in range(int(m.max()) if R else 0):
        live = m > i
        cl_i = np.where(live, cl - m + i + 1, 0).astype(np.int32)
        rows = np.where(live, qs[:-1] + i, 0)
        qo, st_i = append_int8(q[rows], k[rows], v[rows], table, block_tables, cl_i, open_slots, st)
        status = min(status, st_i)
        q_out[rows[live]] = qo[live]
    return q_out, status


def paged_attention_int8(q, k8, v8, k_amax, v_amax, block_tables, context_lens, scale, nthreads=1):
    """q uint16 [B][Hq][d]; int8 caches [nb][Hkv][16][d]; fp32 group maxima
    [nb][Hkv]; returns float64 [B][Hq][d]."""
    q = _c(q, np.uint16)
    B, Hq, d = q.shape
    Hkv = k8.shape[1]
    kc = _c(k8, np.int8); vc = _c(v8, np.int8)
    ka = _c(k_amax, np.float32); va = _c(v_amax, np.float32)
    bt = _c(block_tables, np.int32); cl = _c(context_lens, np.int32)
    out = np.empty((B, Hq, d), np.float64)
    used = _load().or_paged_attention_int8(B, Hq, Hkv, d, _p(q), _p(kc), _p(vc), _p(ka), _p(va), _p(bt),
                                           bt.shape[1], _p(cl), float(scale), _p(out), int(nthreads))
    paged_attention_int8.threads_used = used
    return out
