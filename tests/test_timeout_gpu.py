"""Failure detection on the GPU without a fault: every mbarrier wait in the
attention kernels is bounded, and a wait that runs out sets
MI_DEVERR_TIMEOUT and lets the kernel return.

A test hook (mi_test_withhold_copy) makes one producer neither copy nor
announce a staged block, so a consumer's wait on it can never be satisfied
and no copy is left in flight; mi_test_set_wait_limit shortens every wait of
the launch to 1 ms. Each test checks that the error bit is set, that the call
comes back promptly (well inside the default 2 s limit), and that the next
call on the same, re-zeroed workspace matches the oracle. The hooks are reset
whatever happens."""
import time

import numpy as np
import pytest

import oracle
from helpers import assert_attention_close, from_dev_u16, to_dev_i32, to_dev_u16
from workloads import BLOCK, PREFILL_WORKLOADS, bf16_normal

pytestmark = pytest.mark.gpu

LIMIT_NS = 1_000_000  # 1 ms


def _mi():
    import paged_kv_decode_25_gb300 as mi
    return mi


class _Withheld:
    """The hooks on for the body of a with-statement, reset on exit."""

    def __enter__(self):
        mi = _mi()
        assert mi.mi_test_set_wait_limit(LIMIT_NS) == mi.MI_OK
        assert mi.mi_test_withhold_copy(1) == mi.MI_OK
        return self

    def __exit__(self, *exc):
        mi = _mi()
        mi.mi_test_withhold_copy(0)
        mi.mi_test_set_wait_limit(0)
        return False


def _paged_case(seed, B=12, Hq=16, Hkv=4, d=128):
    r = np.random.Generator(np.random.PCG64(seed))
    lens = r.integers(40, 3000, size=B).astype(np.int32)
    nblk = [-(-int(n) // BLOCK) for n in lens]
    nb = sum(nblk) + 5
    mbps = max(nblk)
    perm = r.permutation(nb)
    bt = np.full((B, mbps), -1, np.int32)
    kc = bf16_normal(r, (nb, Hkv, BLOCK, d))
    vc = bf16_normal(r, (nb, Hkv, BLOCK, d))
    i = 0
    for b in range(B):
        bt[b, :nblk[b]] = perm[i:i + nblk[b]]
        i += nblk[b]
    q, k, v = bf16_normal(r, (B, Hq, d)), bf16_normal(r, (B, Hkv, d)), bf16_normal(r, (B, Hkv, d))
    return q, k, v, kc, vc, bt, lens, nb, mbps


def test_hook_arguments_checked():
    mi = _mi()
    assert mi.mi_test_set_wait_limit(-1) == mi.MI_ERR_INVALID_ARG
    assert mi.mi_test_set_wait_limit(3_000_000_000) == mi.MI_ERR_INVALID_ARG
    assert mi.mi_test_set_wait_limit(0) == mi.MI_OK


@pytest.mark.parametrize("kind", ["attention", "fp8", "int8", "step"])
def test_decode_wait_runs_out_then_recovers(cuda_device, kind):
    """A decode launch whose first staged block never arrives sets the timeout
    bit and returns within milliseconds; after the workspace is zeroed the
    next call (hooks off) on the same workspace is correct."""
    import torch
    mi = _mi()
    q, k, v, kc, vc, bt, lens, nb, mbps = _paged_case(5)
    B, Hq, d = q.shape
    Hkv = kc.shape[1]
    dims = mi.dims(B, Hq, Hkv, d, nb, mbps)
    scale = 1.0 / np.sqrt(d)
    ws = torch.empty(mi.mi_paged_decode_workspace_bytes(dims) // 4 + 4, dtype=torch.float32, device=cuda_device)
    bt_d, cl_d = to_dev_i32(bt, cuda_device), to_dev_i32(lens, cuda_device)
    _, table = mi.mi_rope_table(1e6, d, 4096)
    rope_d = torch.from_numpy(table).to(cuda_device)
    ks = np.full(Hkv, 4.0 / 448.0, np.float32)
    ks_d = torch.from_numpy(ks).to(cuda_device)
    if kind == "fp8":
        # e4m3 caches and the oracle's view of them (exact dequantised values)
        kc8 = oracle.e4m3_from_f64(oracle.bf16_to_f64(kc) / ks[None, :, None, None].astype(np.float64))
        vc8 = oracle.e4m3_from_f64(oracle.bf16_to_f64(vc) / ks[None, :, None, None].astype(np.float64))
        kc_d = torch.from_numpy(kc8).to(cuda_device)
        vc_d = torch.from_numpy(vc8).to(cuda_device)
    elif kind == "int8":
        # INT8 codes and group maxima of the same history (the oracle's quantiser)
        st8 = oracle.int8_state(nb, Hkv, d, B)
        assert oracle.int8_from_bf16_cache(kc, vc, bt, lens, np.arange(B, dtype=np.int32), st8) == 0
        kc_d, vc_d = torch.from_numpy(st8["k8"]).to(cuda_device), torch.from_numpy(st8["v8"]).to(cuda_device)
        ka_d = torch.from_numpy(st8["k_amax"].ravel()).to(cuda_device)
        va_d = torch.from_numpy(st8["v_amax"].ravel()).to(cuda_device)
    else:
        kc_d, vc_d = to_dev_u16(kc, cuda_device), to_dev_u16(vc, cuda_device)
    q_d, k_d, v_d = (to_dev_u16(a, cuda_device) for a in (q, k, v))

    def call(out, qo, err):
        if kind == "attention":
            return mi.mi_paged_decode_attention(dims, q_d, kc_d, vc_d, bt_d, cl_d, scale, out, ws, dev_err=err)
        if kind == "fp8":
            return mi.mi_paged_decode_attention_fp8(dims, q_d, kc_d, vc_d, ks_d, ks_d, bt_d, cl_d, scale, out, ws,
                                                    dev_err=err)
        if kind == "int8":
            return mi.mi_paged_decode_attention_int8(dims, q_d, kc_d, vc_d, ka_d, va_d, bt_d, cl_d, scale, out, ws,
                                                     dev_err=err)
        return mi.mi_paged_decode_step(dims, q_d, k_d, v_d, rope_d, 4096, bt_d, cl_d, scale, qo, kc_d, vc_d, out,
                                       ws, dev_err=err)

    call(torch.empty_like(q_d), torch.empty_like(q_d), None)  # first launch outside the timing
    torch.cuda.synchronize()
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    with _Withheld():
        t0 = time.perf_counter()
        assert call(torch.empty_like(q_d), torch.empty_like(q_d), err) == mi.MI_OK
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    assert int(err.item()) & mi.MI_DEVERR_TIMEOUT
    assert dt < 1.0, dt  # a few wait limits plus drains, far inside the 2 s default

    # recovery on the same workspace, zeroed as the library asks after a timeout
    ws.zero_()
    err.zero_()
    out, qo = torch.full_like(q_d, float("nan")), torch.full_like(q_d, float("nan"))
    assert call(out, qo, err) == mi.MI_OK
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    if kind == "step":
        pos = (lens - 1).astype(np.int32)
        kc_h, vc_h = kc.copy(), vc.copy()
        q_ref, st = oracle.append(q, k, v, pos, oracle.slot_mapping(bt, pos), oracle.rope_table(1e6, d, 4096),
                                  kc_h, vc_h)
        assert st == 0
        assert np.array_equal(from_dev_u16(qo), q_ref)
        ref = oracle.paged_attention(q_ref, kc_h, vc_h, bt, lens, scale, nthreads=8)
    elif kind == "fp8":
        ref = oracle.paged_attention_fp8(q, kc8, vc8, ks, ks, bt, lens, scale, nthreads=8)
    elif kind == "int8":
        ref = oracle.paged_attention_int8(q, st8["k8"], st8["v8"], st8["k_amax"], st8["v_amax"], bt, lens, scale,
                                          nthreads=8)
    else:
        ref = oracle.paged_attention(q, kc, vc, bt, lens, scale, nthreads=8)
    assert_attention_close(from_dev_u16(out), ref, f"{kind} after a timed-out launch")


@pytest.mark.parametrize("variant", [2, 3])  # MI_PREFILL_TCGEN05, MI_PREFILL_TCGEN05_PAIR
def test_prefill_wait_runs_out_then_recovers(cuda_device, variant):
    """The tcgen05 prefill kernels: every CTA's first K stage is withheld, so
    its MMA, softmax and P.V waits run out; no MMA is left running and the
    tensor memory is released (the next launch allocates it again); the next
    call is correct."""
    import torch
    from test_prefill_gpu import _run_prefill
    mi = _mi()
    w = PREFILL_WORKLOADS["prefill_small"]
    x = _run_prefill(w, cuda_device, order_seed=3, variant=variant)
    R = w.B
    d_att = mi.dims(R, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    bt_d, n_d, qs_d = (to_dev_i32(a, cuda_device) for a in (x["bt"], x["n"], x["qs"]))
    max_q = int(x["m"].max())
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    with _Withheld():
        t0 = time.perf_counter()
        assert mi.mi_paged_prefill_attention_variant(d_att, x["T"], max_q, x["qo_d"], x["kc_d"], x["vc_d"], bt_d,
                                                     n_d, qs_d, w.scale, torch.empty_like(x["qo_d"]),
                                                     variant=variant, dev_err=err) == mi.MI_OK
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    assert int(err.item()) & mi.MI_DEVERR_TIMEOUT
    assert dt < 1.0, dt
    err.zero_()
    out = torch.full_like(x["qo_d"], float("nan"))
    assert mi.mi_paged_prefill_attention_variant(d_att, x["T"], max_q, x["qo_d"], x["kc_d"], x["vc_d"], bt_d, n_d,
                                                 qs_d, w.scale, out, variant=variant,
                                                 dev_err=err) == mi.MI_OK
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.paged_prefill_attention(x["q_ref"], x["kc"], x["vc"], x["bt"], x["n"], x["qs"], w.scale,
                                         nthreads=8)
    assert_attention_close(from_dev_u16(out), ref, "prefill after a timed-out launch")
