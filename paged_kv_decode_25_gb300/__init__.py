"""Python binding of the paged-KV decode library (libmi.so).

Argument marshalling only: every function here forwards to the C ABI of
include/mi.h with the same name, passing device pointers of torch tensors (or
host numpy buffers for the pool) and the current CUDA stream. All arithmetic of
the decode step runs in the library's CUDA kernels; nothing here computes a
result. The library must have been built (``build.build()``); calling any entry
point without it raises RuntimeError.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmi.so")
_lock = threading.Lock()
_lib = None

MI_OK, MI_ERR_INVALID_ARG, MI_ERR_OUT_OF_BLOCKS, MI_ERR_UNKNOWN_SEQ = 0, 1, 2, 3
MI_ERR_UNSUPPORTED, MI_ERR_CUDA, MI_ERR_DEVICE_BOUNDS, MI_ERR_TIMEOUT = 4, 5, 6, 7
MI_DEVERR_BAD_BLOCK, MI_DEVERR_BAD_SLOT, MI_DEVERR_BAD_POS = 0x1, 0x2, 0x4
MI_DEVERR_BAD_CONTEXT, MI_DEVERR_TIMEOUT, MI_DEVERR_BAD_QUERY, MI_DEVERR_BAD_SCALE = 0x8, 0x10, 0x20, 0x40
MI_ATTN_DEFAULT, MI_ATTN_MMA, MI_ATTN_FMA = 0, 1, 2
MI_ADMIT_PROCEED, MI_ADMIT_SOFT_BRAKE, MI_ADMIT_HARD_BRAKE = 0, 1, 2
MI_ADMIT_HARD_BP_DEFAULT, MI_ADMIT_SOFT_BP_DEFAULT = 1000, 3000
MI_PREFILL_DEFAULT, MI_PREFILL_MMA, MI_PREFILL_TCGEN05, MI_PREFILL_TCGEN05_PAIR = 0, 1, 2, 3
MI_DEVERR_INTERNAL = 0x80
MI_STEP_EARLY_START = 0x1

# every symbol include/mi.h declares
EXPORTS = (
    "mi_status_string", "mi_kv_pool_create", "mi_kv_pool_destroy", "mi_kv_pool_alloc", "mi_kv_pool_alloc_batch",
    "mi_kv_pool_free", "mi_kv_pool_num_free", "mi_kv_pool_batch_meta", "mi_kv_pool_token_slots",
    "mi_kv_pool_admission", "mi_kv_pool_touch", "mi_kv_pool_lru_victim", "mi_kv_pool_swap_out",
    "mi_kv_pool_swap_in", "mi_kv_copy_blocks", "mi_kv_copy_rows",
    "mi_kv_pool_seq_blocks",
    "mi_rope_table", "mi_paged_kv_append", "mi_paged_decode_workspace_bytes",
    "mi_paged_decode_attention", "mi_paged_decode_attention_variant",
    "mi_paged_kv_append_fp8", "mi_paged_decode_attention_fp8",
    "mi_paged_kv_append_int8", "mi_paged_decode_attention_int8", "mi_paged_kv_append_int8_tokens",
    "mi_paged_prefill_attention", "mi_paged_prefill_attention_variant", "mi_paged_decode_attention_noalloc",
    "mi_paged_decode_step", "mi_paged_decode_step_fp8", "mi_test_set_wait_limit", "mi_test_withhold_copy",
)
MI_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


class MiDims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("B", "Hq", "Hkv", "head_dim", "block_size", "num_blocks", "max_blocks_per_seq")]


class MIError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, status_string(status), status))


def load():
    """Load libmi.so (raises RuntimeError when it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmi.so is not built at %s; run paged_kv_decode_25_gb300/build.py"
                               % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        P, i32, f32, f64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_double
        dims_p = ctypes.POINTER(MiDims)
        sig = {
            "mi_status_string": ([i32], ctypes.c_char_p),
            "mi_kv_pool_create": ([i32, i32, i32, i32, P, ctypes.POINTER(P)], i32),
            "mi_kv_pool_destroy": ([P], None),
            "mi_kv_pool_alloc": ([P, i32, i32], i32),
            "mi_kv_pool_alloc_batch": ([P, P, P, i32], i32),
            "mi_kv_pool_free": ([P, i32], i32),
            "mi_kv_pool_num_free": ([P], i32),
            "mi_kv_pool_batch_meta": ([P, P, i32, P, P, P], i32),
            "mi_kv_pool_token_slots": ([P, i32, i32, i32, P], i32),
            "mi_kv_pool_admission": ([P, i32, i32, i32, P], i32),
            "mi_kv_pool_touch": ([P, P, i32], i32),
            "mi_kv_pool_lru_victim": ([P, P, i32], i32),
            "mi_kv_pool_swap_out": ([P, i32, P, i32, P], i32),
            "mi_kv_pool_swap_in": ([P, i32, P, i32, P], i32),
            "mi_kv_copy_blocks": ([dims_p, P, P, i32, P, P, P, i32, P, i32, P, P], i32),
            "mi_kv_pool_seq_blocks": ([P, i32, P, i32], i32),
            "mi_rope_table": ([f64, i32, i32, P], i32),
            "mi_paged_kv_append": ([dims_p, P, P, P, P, P, P, i32, P, P, P, P, P], i32),
            "mi_paged_decode_workspace_bytes": ([dims_p], ctypes.c_size_t),
            "mi_paged_decode_attention": ([dims_p, P, P, P, P, P, f32, P, P, ctypes.c_size_t, P, P], i32),
            "mi_paged_decode_attention_variant": (
                [dims_p, P, P, P, P, P, f32, P, P, ctypes.c_size_t, P, P, i32, i32], i32),
            "mi_paged_prefill_attention": ([dims_p, i32, i32, P, P, P, P, P, P, f32, P, P, P], i32),
            "mi_paged_prefill_attention_variant": ([dims_p, i32, i32, P, P, P, P, P, P, f32, P, P, P, i32], i32),
            "mi_paged_kv_append_fp8": ([dims_p, P, P, P, P, P, P, i32, P, P, P, P, P, P, P], i32),
            "mi_paged_decode_attention_fp8": (
                [dims_p, P, P, P, P, P, P, P, f32, P, P, ctypes.c_size_t, P, P], i32),
            "mi_paged_decode_attention_noalloc": ([dims_p, P, P, P, P, P, f32, P, P, P], i32),
            "mi_kv_copy_rows": ([P, ctypes.c_int64, P, P, ctypes.c_int64, P, i32, ctypes.c_int64, P, P], i32),
            "mi_paged_kv_append_int8": (
                [dims_p, P, P, P, P, i32, P, P, P, i32, P, P, P, P, P, P, P, P, P], i32),
            "mi_paged_kv_append_int8_tokens": (
                [dims_p, i32, P, P, P, P, i32, P, P, P, P, i32, P, P, P, P, P, P, P, P, P], i32),
            "mi_paged_decode_attention_int8": (
                [dims_p, P, P, P, P, P, P, P, f32, P, P, ctypes.c_size_t, P, P], i32),
            "mi_paged_decode_step": (
                [dims_p, P, P, P, P, i32, P, P, f32, P, P, P, P, P, ctypes.c_size_t, P, P, ctypes.c_uint32], i32),
            "mi_paged_decode_step_fp8": (
                [dims_p, P, P, P, P, i32, P, P, P, P, f32, P, P, P, P, P, ctypes.c_size_t, P, P, ctypes.c_uint32],
                i32),
            "mi_test_set_wait_limit": ([ctypes.c_int64], i32),
            "mi_test_withhold_copy": ([i32], i32),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def status_string(s: int) -> str:
    return load().mi_status_string(int(s)).decode()


def check(status: int, what: str = "mi call") -> None:
    if status != MI_OK:
        raise MIError(status, what)


# ------------------------------------------------------------ marshalling --

def _ptr(x):
    """Device/host address of a torch tensor or numpy array (None -> NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        assert x.flags.c_contiguous
        return x.ctypes.data
    assert x.is_contiguous(), "tensors must be contiguous"
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def dims(B, Hq, Hkv, head_dim, num_blocks, max_blocks_per_seq, block_size=16) -> MiDims:
    return MiDims(B, Hq, Hkv, head_dim, block_size, num_blocks, max_blocks_per_seq)


# ------------------------------------------------------------------ pool ---

def mi_kv_pool_create(num_blocks, block_size, max_seqs, max_blocks_per_seq, initial_free_order=None):
    """Returns (status, handle)."""
    order = None
    if initial_free_order is not None:
        order = np.ascontiguousarray(initial_free_order, dtype=np.int32)
        assert order.shape == (num_blocks,)
    h = ctypes.c_void_p()
    st = load().mi_kv_pool_create(num_blocks, block_size, max_seqs, max_blocks_per_seq,
                                  _ptr(order), ctypes.byref(h))
    return st, h.value


def mi_kv_pool_destroy(handle):
    load().mi_kv_pool_destroy(handle)


def mi_kv_pool_alloc(handle, seq_id, num_tokens):
    return load().mi_kv_pool_alloc(handle, int(seq_id), int(num_tokens))


def mi_kv_pool_alloc_batch(handle, seq_ids, num_tokens):
    """seq_ids, num_tokens: sequences of ints of equal length (host)."""
    sids = np.ascontiguousarray(seq_ids, dtype=np.int32)
    ntok = np.ascontiguousarray(num_tokens, dtype=np.int32)
    assert sids.shape == ntok.shape and sids.ndim == 1
    return load().mi_kv_pool_alloc_batch(handle, _ptr(sids), _ptr(ntok), int(sids.size))


def mi_kv_pool_free(handle, seq_id):
    return load().mi_kv_pool_free(handle, int(seq_id))


def mi_kv_pool_num_free(handle):
    return load().mi_kv_pool_num_free(handle)


def mi_kv_pool_batch_meta(handle, seq_ids, max_blocks_per_seq, block_tables=None, context_lens=None,
                          slot_mapping=None):
    """Fills (or allocates) host int32 outputs; returns (status, block_tables, context_lens, slot_mapping)."""
    ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
    B = ids.shape[0]
    bt = np.empty((B, max_blocks_per_seq), np.int32) if block_tables is None else block_tables
    cl = np.empty(B, np.int32) if context_lens is None else context_lens
    sl = np.empty(B, np.int32) if slot_mapping is None else slot_mapping
    st = load().mi_kv_pool_batch_meta(handle, _ptr(ids), B, _ptr(bt), _ptr(cl), _ptr(sl))
    return st, bt, cl, sl


def mi_kv_pool_token_slots(handle, seq_id, first_token, count):
    """Returns (status, int32 [count] host array of slots)."""
    out = np.empty(max(int(count), 1), np.int32)
    st = load().mi_kv_pool_token_slots(handle, int(seq_id), int(first_token), int(count), _ptr(out))
    return st, out[:max(int(count), 0)]


def mi_kv_pool_admission(handle, running_decodes, hard_bp=MI_ADMIT_HARD_BP_DEFAULT,
                         soft_bp=MI_ADMIT_SOFT_BP_DEFAULT):
    """Returns (status, decision)."""
    out = ctypes.c_int32(-1)
    st = load().mi_kv_pool_admission(handle, int(running_decodes), int(hard_bp), int(soft_bp),
                                     ctypes.byref(out))
    return st, int(out.value)


def mi_kv_pool_touch(handle, seq_ids):
    ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
    return load().mi_kv_pool_touch(handle, _ptr(ids), int(ids.shape[0]))


def mi_kv_pool_lru_victim(handle, exclude=()):
    ex = np.ascontiguousarray(exclude, dtype=np.int32)
    return int(load().mi_kv_pool_lru_victim(handle, _ptr(ex) if ex.size else None, int(ex.size)))


def _swap(fn, handle, seq_id, max_out):
    out = np.empty(max(int(max_out), 1), np.int32)
    n = ctypes.c_int32(0)
    st = fn(handle, int(seq_id), _ptr(out), int(max_out), ctypes.byref(n))
    return st, out[:n.value].copy()


def mi_kv_pool_swap_out(handle, seq_id, max_out=1 << 20):
    """Returns (status, the sequence's former blocks)."""
    return _swap(load().mi_kv_pool_swap_out, handle, seq_id, max_out)


def mi_kv_pool_swap_in(handle, seq_id, max_out=1 << 20):
    """Returns (status, the sequence's new blocks)."""
    return _swap(load().mi_kv_pool_swap_in, handle, seq_id, max_out)


def mi_kv_pool_seq_blocks(handle, seq_id, max_out=1 << 20):
    n = load().mi_kv_pool_seq_blocks(handle, int(seq_id), None, 0)
    if n < 0:
        return None
    out = np.empty(max(n, 1), np.int32)
    load().mi_kv_pool_seq_blocks(handle, int(seq_id), _ptr(out), n)
    return out[:n]


class Pool:
    """Owner of a library pool handle, with the alloc/free/num_free/batch_meta
    calls the workloads expect (each returns the library's status)."""

    def __init__(self, num_blocks, max_seqs, max_blocks_per_seq, initial_order=None, block_size=16):
        st, self.handle = mi_kv_pool_create(num_blocks, block_size, max_seqs, max_blocks_per_seq,
                                            initial_order)
        check(st, "mi_kv_pool_create")
        self.max_blocks_per_seq = max_blocks_per_seq

    def alloc(self, seq, num_tokens):
        return mi_kv_pool_alloc(self.handle, seq, num_tokens)

    def alloc_batch(self, seqs, num_tokens):
        return mi_kv_pool_alloc_batch(self.handle, seqs, num_tokens)

    def free(self, seq):
        return mi_kv_pool_free(self.handle, seq)

    def num_free(self):
        return mi_kv_pool_num_free(self.handle)

    def token_slots(self, seq, first_token, count):
        st, slots = mi_kv_pool_token_slots(self.handle, seq, first_token, count)
        check(st, "mi_kv_pool_token_slots")
        return slots

    def admission(self, running_decodes, hard_bp=MI_ADMIT_HARD_BP_DEFAULT, soft_bp=MI_ADMIT_SOFT_BP_DEFAULT):
        st, dec = mi_kv_pool_admission(self.handle, running_decodes, hard_bp, soft_bp)
        check(st, "mi_kv_pool_admission")
        return dec

    def touch(self, seq_ids):
        return mi_kv_pool_touch(self.handle, seq_ids)

    def lru_victim(self, exclude=()):
        return mi_kv_pool_lru_victim(self.handle, exclude)

    def swap_out(self, seq):
        st, blocks = mi_kv_pool_swap_out(self.handle, seq)
        return st, [int(b) for b in blocks]

    def swap_in(self, seq):
        st, blocks = mi_kv_pool_swap_in(self.handle, seq)
        return st, [int(b) for b in blocks]

    def batch_meta(self, seq_ids):
        st, bt, cl, sl = mi_kv_pool_batch_meta(self.handle, seq_ids, self.max_blocks_per_seq)
        check(st, "mi_kv_pool_batch_meta")
        return bt, cl, sl

    def close(self):
        if self.handle:
            mi_kv_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ------------------------------------------------------------ device ops ---

def mi_rope_table(theta, head_dim, max_pos):
    """Returns (status, float32 [max_pos][head_dim/2][2] host array)."""
    out = np.empty((max_pos, head_dim // 2, 2), np.float32)
    st = load().mi_rope_table(float(theta), int(head_dim), int(max_pos), _ptr(out))
    return st, out


def mi_paged_kv_append(d: MiDims, q, k, v, positions, slot_mapping, rope_cos_sin, max_pos, q_out,
                       k_cache, v_cache, dev_err=None, stream=None):
    return load().mi_paged_kv_append(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(positions),
                                     _ptr(slot_mapping), _ptr(rope_cos_sin), int(max_pos), _ptr(q_out),
                                     _ptr(k_cache), _ptr(v_cache), _ptr(dev_err), _stream(stream))


def mi_paged_decode_workspace_bytes(d: MiDims) -> int:
    return int(load().mi_paged_decode_workspace_bytes(ctypes.byref(d)))


def mi_paged_decode_attention(d: MiDims, q, k_cache, v_cache, block_tables, context_lens, scale, out,
                              workspace, workspace_bytes=None, dev_err=None, stream=None):
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    return load().mi_paged_decode_attention(ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                            _ptr(block_tables), _ptr(context_lens), float(scale),
                                            _ptr(out), _ptr(workspace), int(wb), _ptr(dev_err),
                                            _stream(stream))


def mi_paged_decode_attention_variant(d: MiDims, q, k_cache, v_cache, block_tables, context_lens, scale,
                                      out, workspace, variant=MI_ATTN_DEFAULT, ctas=0,
                                      workspace_bytes=None, dev_err=None, stream=None):
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    return load().mi_paged_decode_attention_variant(
        ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        float(scale), _ptr(out), _ptr(workspace), int(wb), _ptr(dev_err), _stream(stream),
        int(variant), int(ctas))


def mi_paged_decode_step(d: MiDims, q, k, v, rope_cos_sin, max_pos, block_tables, context_lens, scale, q_out,
                         k_cache, v_cache, out, workspace, workspace_bytes=None, dev_err=None, stream=None,
                         flags=0):
    """flags: 0 or MI_STEP_EARLY_START (the step plans and issues its first
    KV copies before the kernel ahead of it on the stream ends; the caller
    keeps the contract of include/mi.h, e.g. two workspaces in turn for
    consecutive early-start calls)."""
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    return load().mi_paged_decode_step(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(rope_cos_sin),
                                       int(max_pos), _ptr(block_tables), _ptr(context_lens), float(scale),
                                       _ptr(q_out), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(workspace),
                                       int(wb), _ptr(dev_err), _stream(stream), int(flags))


def mi_paged_kv_append_fp8(d: MiDims, q, k, v, positions, slot_mapping, rope_cos_sin, max_pos, q_out,
                           k_cache, v_cache, k_scale, v_scale, dev_err=None, stream=None):
    return load().mi_paged_kv_append_fp8(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(positions),
                                         _ptr(slot_mapping), _ptr(rope_cos_sin), int(max_pos), _ptr(q_out),
                                         _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                         _ptr(dev_err), _stream(stream))


def mi_paged_decode_attention_fp8(d: MiDims, q, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens,
                                  scale, out, workspace, workspace_bytes=None, dev_err=None, stream=None):
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    return load().mi_paged_decode_attention_fp8(ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                                _ptr(k_scale), _ptr(v_scale), _ptr(block_tables),
                                                _ptr(context_lens), float(scale), _ptr(out), _ptr(workspace),
                                                int(wb), _ptr(dev_err), _stream(stream))


def mi_paged_kv_append_int8(d: MiDims, q, k, v, rope_cos_sin, max_pos, block_tables, context_lens, open_slots,
                            q_out, k_cache, v_cache, k_amax, v_amax, k_open, v_open, dev_err=None, stream=None):
    """The INT8 decode append; the open buffers' first dimension is the number
    of open-group slots."""
    return load().mi_paged_kv_append_int8(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(rope_cos_sin),
                                          int(max_pos), _ptr(block_tables), _ptr(context_lens), _ptr(open_slots),
                                          int(k_open.shape[0]), _ptr(q_out), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(k_amax), _ptr(v_amax), _ptr(k_open), _ptr(v_open), _ptr(dev_err),
                                          _stream(stream))


def mi_paged_kv_append_int8_tokens(d: MiDims, total_tokens, q, k, v, rope_cos_sin, max_pos, block_tables,
                                   context_lens, query_start, open_slots, q_out, k_cache, v_cache, k_amax, v_amax,
                                   k_open, v_open, dev_err=None, stream=None):
    """The INT8 append of many new tokens per request (rows query_start[r] ..
    query_start[r+1]-1); the open buffers' first dimension is the number of
    open-group slots."""
    return load().mi_paged_kv_append_int8_tokens(
        ctypes.byref(d), int(total_tokens), _ptr(q), _ptr(k), _ptr(v), _ptr(rope_cos_sin), int(max_pos),
        _ptr(block_tables), _ptr(context_lens), _ptr(query_start), _ptr(open_slots), int(k_open.shape[0]),
        _ptr(q_out), _ptr(k_cache), _ptr(v_cache), _ptr(k_amax), _ptr(v_amax), _ptr(k_open), _ptr(v_open),
        _ptr(dev_err), _stream(stream))


def mi_paged_decode_attention_int8(d: MiDims, q, k_cache, v_cache, k_amax, v_amax, block_tables, context_lens,
                                   scale, out, workspace, workspace_bytes=None, dev_err=None, stream=None):
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    return load().mi_paged_decode_attention_int8(ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                                 _ptr(k_amax), _ptr(v_amax), _ptr(block_tables),
                                                 _ptr(context_lens), float(scale), _ptr(out), _ptr(workspace),
                                                 int(wb), _ptr(dev_err), _stream(stream))


def mi_kv_copy_rows(src, src_count, src_ids, dst, dst_count, dst_ids, n, row_bytes, dev_err=None, stream=None):
    """Copy n rows of row_bytes: src row src_ids[i] to dst row dst_ids[i]."""
    return load().mi_kv_copy_rows(_ptr(src), int(src_count), _ptr(src_ids), _ptr(dst), int(dst_count),
                                  _ptr(dst_ids), int(n), int(row_bytes), _ptr(dev_err), _stream(stream))


def amax_floats(num_blocks: int, Hkv: int) -> int:
    """Floats of a group-maxima array: one per block and KV head."""
    return num_blocks * Hkv


def mi_paged_prefill_attention(d: MiDims, total_q, max_query_len, q, k_cache, v_cache, block_tables,
                               context_lens, query_start, scale, out, dev_err=None, stream=None):
    return load().mi_paged_prefill_attention(ctypes.byref(d), int(total_q), int(max_query_len), _ptr(q),
                                             _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                             _ptr(context_lens), _ptr(query_start), float(scale), _ptr(out),
                                             _ptr(dev_err), _stream(stream))


def mi_kv_copy_blocks(d: MiDims, src_k, src_v, src_num_blocks, src_blocks, dst_k, dst_v, dst_num_blocks,
                      dst_blocks, n, dev_err=None, stream=None):
    return load().mi_kv_copy_blocks(ctypes.byref(d), _ptr(src_k), _ptr(src_v), int(src_num_blocks),
                                    _ptr(src_blocks), _ptr(dst_k), _ptr(dst_v), int(dst_num_blocks),
                                    _ptr(dst_blocks), int(n), _ptr(dev_err), _stream(stream))


def mi_paged_prefill_attention_variant(d: MiDims, total_q, max_query_len, q, k_cache, v_cache, block_tables,
                                       context_lens, query_start, scale, out, variant=MI_PREFILL_DEFAULT,
                                       dev_err=None, stream=None):
    return load().mi_paged_prefill_attention_variant(ctypes.byref(d), int(total_q), int(max_query_len), _ptr(q),
                                                     _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                                     _ptr(context_lens), _ptr(query_start), float(scale),
                                                     _ptr(out), _ptr(dev_err), _stream(stream), int(variant))


def mi_paged_decode_attention_noalloc(d: MiDims, q, k_cache, v_cache, block_tables, context_lens, scale, out,
                                      dev_err=None, stream=None):
    """Attention with the library's own fixed scratch array (no workspace
    argument, no allocation). See include/mi.h for the sharing rules."""
    return load().mi_paged_decode_attention_noalloc(ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                                    _ptr(block_tables), _ptr(context_lens), float(scale),
                                                    _ptr(out), _ptr(dev_err), _stream(stream))


def mi_paged_decode_step_fp8(d: MiDims, q, k, v, rope_cos_sin, max_pos, block_tables, context_lens, k_scale,
                             v_scale, scale, q_out, k_cache, v_cache, out, workspace, workspace_bytes=None,
                             dev_err=None, stream=None, flags=0):
    """flags as for mi_paged_decode_step."""
    wb = workspace.numel() * workspace.element_size() if workspace_bytes is None else workspace_bytes
    return load().mi_paged_decode_step_fp8(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(rope_cos_sin),
                                           int(max_pos), _ptr(block_tables), _ptr(context_lens), _ptr(k_scale),
                                           _ptr(v_scale), float(scale), _ptr(q_out), _ptr(k_cache), _ptr(v_cache),
                                           _ptr(out), _ptr(workspace), int(wb), _ptr(dev_err), _stream(stream),
                                           int(flags))


def mi_test_set_wait_limit(ns):
    """Bound on each device wait of later launches (ns; 0 = the 2 s default)."""
    return load().mi_test_set_wait_limit(int(ns))


def mi_test_withhold_copy(enable):
    """Failure-detection test hook: later attention launches withhold one
    staged copy, so a bounded wait runs out (see include/mi.h)."""
    return load().mi_test_withhold_copy(1 if enable else 0)
