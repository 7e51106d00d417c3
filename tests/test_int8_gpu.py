"""GPU parity of the INT8 KV path (64-token groups, symmetric, truncating
cast) against the oracle: mi_paged_kv_append_int8 bit-exact (q_out, both
code caches, both group-maxima arrays and the open-group buffers, every other
byte untouched) after one step on three workloads and over 70 steps that
cross group boundaries and grow group maxima; mi_paged_decode_attention_int8
within the attention tolerance of the fp64 oracle over the dequantised
caches on those workloads, on a full-size serving layer (every request and
head), on edge lengths, bitwise invariant to where blocks sit, and across
group maxima that span four orders of magnitude; the append's error bits."""
import numpy as np
import pytest

import oracle
from helpers import assert_attention_close, from_dev_u16, grow, pools_for, to_dev_i32, to_dev_u16
from workloads import BLOCK, WORKLOADS, bf16_normal, device_int8_cache, history_cache, new_token_values

pytestmark = pytest.mark.gpu

GRP = 64


def _mi():
    import paged_kv_decode_25_gb300 as mi
    return mi


def _workspace(mi, d, device):
    import torch
    n = mi.mi_paged_decode_workspace_bytes(d)
    assert n > 0
    return torch.empty(n // 4 + 4, dtype=torch.float32, device=device)


class DevState:
    """Device copies of an oracle INT8 state (oracle.int8_state layout)."""

    def __init__(self, st, device):
        import torch
        mi = _mi()
        nb, Hkv = st["k_amax"].shape
        self.nb, self.Hkv = nb, Hkv
        self.k8 = torch.from_numpy(st["k8"]).to(device)
        self.v8 = torch.from_numpy(st["v8"]).to(device)
        n = mi.amax_floats(nb, Hkv)
        self.k_amax = torch.zeros(n, dtype=torch.float32, device=device)
        self.v_amax = torch.zeros(n, dtype=torch.float32, device=device)
        self.k_amax[: nb * Hkv] = torch.from_numpy(st["k_amax"].ravel()).to(device)
        self.v_amax[: nb * Hkv] = torch.from_numpy(st["v_amax"].ravel()).to(device)
        self.k_open = to_dev_u16(st["k_open"], device)
        self.v_open = to_dev_u16(st["v_open"], device)

    def host(self):
        n = self.nb * self.Hkv
        return {
            "k8": self.k8.cpu().numpy(), "v8": self.v8.cpu().numpy(),
            "k_amax": self.k_amax[:n].cpu().numpy().reshape(self.nb, self.Hkv),
            "v_amax": self.v_amax[:n].cpu().numpy().reshape(self.nb, self.Hkv),
            "k_open": from_dev_u16(self.k_open), "v_open": from_dev_u16(self.v_open),
        }


def _assert_state_equal(got, want, what=""):
    for key in ("k8", "v8", "k_amax", "v_amax", "k_open", "v_open"):
        assert np.array_equal(got[key], want[key]), f"{what}: {key} differs"


def _gpu_append(mi, d, ds, q, k, v, table, max_pos, bt, cl, slots, device):
    import torch
    q_d = to_dev_u16(q, device)
    qo_d = torch.zeros_like(q_d)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    st = mi.mi_paged_kv_append_int8(d, q_d, to_dev_u16(k, device), to_dev_u16(v, device),
                                    torch.from_numpy(table).to(device), max_pos, to_dev_i32(bt, device),
                                    to_dev_i32(cl, device), to_dev_i32(slots, device), qo_d, ds.k8, ds.v8,
                                    ds.k_amax, ds.v_amax, ds.k_open, ds.v_open, err)
    assert st == 0, mi.status_string(st)
    torch.cuda.synchronize()
    return from_dev_u16(qo_d), int(err.item())


def _gpu_attend(mi, d, q, ds, bt, cl, scale, device, k8=None, v8=None, k_amax=None, v_amax=None):
    import torch
    q_d = to_dev_u16(q, device)
    out = torch.full(q_d.shape, float("nan"), dtype=torch.bfloat16, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    st = mi.mi_paged_decode_attention_int8(d, q_d, ds.k8 if k8 is None else k8, ds.v8 if v8 is None else v8,
                                           ds.k_amax if k_amax is None else k_amax,
                                           ds.v_amax if v_amax is None else v_amax, to_dev_i32(bt, device),
                                           to_dev_i32(cl, device), scale, out, _workspace(mi, d, device),
                                           dev_err=err)
    assert st == 0, mi.status_string(st)
    torch.cuda.synchronize()
    return from_dev_u16(out), int(err.item())


@pytest.mark.parametrize("name", ["tiny", "qwen3_1p7b", "skewed"])
def test_int8_append_bit_exact_and_attention_matches_oracle(cuda_device, name):
    mi = _mi()
    w = WORKLOADS[name]
    lib, model, ctx = pools_for(w)
    bt_hist, _, _ = lib.batch_meta(range(w.B))
    grow(lib, w.B, ctx + 1)
    bt, cl, _ = lib.batch_meta(range(w.B))
    kc16, vc16 = history_cache(w, 0, bt_hist, ctx)
    slots = np.arange(w.B, dtype=np.int32)[::-1].copy()           # any one-to-one slot map
    st = oracle.int8_state(w.num_blocks, w.Hkv, w.head_dim, w.B)
    assert oracle.int8_from_bf16_cache(kc16, vc16, bt_hist, ctx, slots, st) == 0
    del kc16, vc16
    ds = DevState(st, cuda_device)
    q, k, v = new_token_values(w, 0)
    table = oracle.rope_table(w.theta, w.head_dim, w.max_pos)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    q_gpu, err = _gpu_append(mi, d, ds, q, k, v, table, w.max_pos, bt, cl, slots, cuda_device)
    assert err == 0
    q_ref, s = oracle.append_int8(q, k, v, table, bt, cl, slots, st)
    assert s == 0
    assert np.array_equal(q_gpu, q_ref)
    _assert_state_equal(ds.host(), st, name)
    ref = oracle.paged_attention_int8(q_ref, st["k8"], st["v8"], st["k_amax"], st["v_amax"], bt, cl, w.scale,
                                      nthreads=8)
    out, err = _gpu_attend(mi, d, q_ref, ds, bt, cl, w.scale, cuda_device)
    assert err == 0
    assert_attention_close(out, ref, f"int8 {name}")


@pytest.mark.parametrize("d_head,Hq,Hkv", [(64, 4, 2), (128, 8, 1)])
def test_int8_append_many_steps_crossing_groups(cuda_device, d_head, Hq, Hkv):
    """70 decode steps from histories of every phase of a group (0, 1, 15,
    63, 64, 100 tokens); each step's k and v rows are drawn at one of several
    magnitudes (zero rows included), so group maxima grow, stay and restart;
    the whole INT8 state after every 10 steps, and the attention at the end."""
    mi = _mi()
    r = np.random.Generator(np.random.PCG64(40 + d_head + Hq))
    hist = np.array([0, 1, 15, 63, 64, 100], np.int32)
    B, steps, max_pos = len(hist), 70, 256
    nblk = [-(-(int(n) + steps) // BLOCK) for n in hist]
    nb = sum(nblk) + 5
    perm = r.permutation(nb)
    mbps = max(nblk) + 1
    bt = np.full((B, mbps), -1, np.int32)
    i = 0
    for b in range(B):
        bt[b, :nblk[b]] = perm[i:i + nblk[b]]
        i += nblk[b]
    kc16 = np.zeros((nb, Hkv, BLOCK, d_head), np.uint16)
    vc16 = np.zeros_like(kc16)
    for b in range(B):
        for t in range(int(hist[b])):
            kc16[bt[b, t // BLOCK], :, t % BLOCK] = bf16_normal(r, (Hkv, d_head))
            vc16[bt[b, t // BLOCK], :, t % BLOCK] = bf16_normal(r, (Hkv, d_head))
    slots = r.permutation(B + 3)[:B].astype(np.int32)
    st = oracle.int8_state(nb, Hkv, d_head, B + 3)
    assert oracle.int8_from_bf16_cache(kc16, vc16, bt, hist, slots, st) == 0
    ds = DevState(st, cuda_device)
    table = oracle.rope_table(1e6, d_head, max_pos)
    d = mi.dims(B, Hq, Hkv, d_head, nb, mbps)
    lens = hist.copy()
    for s in range(steps):
        lens = lens + 1
        q = bf16_normal(r, (B, Hq, d_head))
        mag = r.choice([0.0, 0.25, 1.0, 3.0, 10.0], size=(2, B, Hkv, 1), p=[0.1, 0.2, 0.4, 0.2, 0.1])
        k = oracle.f64_to_bf16(oracle.bf16_to_f64(bf16_normal(r, (B, Hkv, d_head))) * mag[0])
        v = oracle.f64_to_bf16(oracle.bf16_to_f64(bf16_normal(r, (B, Hkv, d_head))) * mag[1])
        q_gpu, err = _gpu_append(mi, d, ds, q, k, v, table, max_pos, bt, lens, slots, cuda_device)
        q_ref, sref = oracle.append_int8(q, k, v, table, bt, lens, slots, st)
        assert err == 0 and sref == 0
        assert np.array_equal(q_gpu, q_ref), s
        if s % 10 == 9 or s == steps - 1:
            _assert_state_equal(ds.host(), st, f"step {s}")
    ref = oracle.paged_attention_int8(q_ref, st["k8"], st["v8"], st["k_amax"], st["v_amax"], bt, lens, 0.1)
    out, err = _gpu_attend(mi, d, q_ref, ds, bt, lens, 0.1, cuda_device)
    assert err == 0
    # V values reach ~10x N(0,1) here: the tolerance scales with the largest |V|
    vmax = float(st["v_amax"].max())
    got = oracle.bf16_to_f64(out)
    assert np.all(np.isfinite(got))
    assert np.abs(got - ref).max() <= 1e-2 * max(1.0, vmax / 4)


def test_int8_full_size_serving_layer(cuda_device):
    """Qwen3-8B-shaped layer at full size (INT8 caches and group maxima filled
    on the device), persistent grid: every request and head against the
    oracle over the blocks the requests use (copied back and renumbered)."""
    import os
    import torch
    mi = _mi()
    w = WORKLOADS["qwen3_8b"]
    lib, model, ctx = pools_for(w)
    grow(lib, w.B, ctx + 1)
    bt, cl, _ = lib.batch_meta(range(w.B))
    k8, v8, ka, va = device_int8_cache(w, 0, cuda_device)
    q, _, _ = new_token_values(w, 0)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)

    class _S:
        pass
    ds = _S()
    ds.k8, ds.v8, ds.k_amax, ds.v_amax = k8, v8, ka, va
    out, err = _gpu_attend(mi, d, q, ds, bt, cl, w.scale, cuda_device)
    assert err == 0
    live = [bt[b, :-(-int(cl[b]) // BLOCK)] for b in range(w.B)]
    used = sorted({int(x) for row in live for x in row})
    remap = {blk: i for i, blk in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.int64, device=cuda_device)
    bt_s = np.full(bt.shape, -1, np.int32)
    for i, row in enumerate(live):
        bt_s[i, :len(row)] = [remap[int(x)] for x in row]
    n = w.num_blocks * w.Hkv
    ka_s = ka[:n].view(w.num_blocks, w.Hkv)[idx].cpu().numpy()
    va_s = va[:n].view(w.num_blocks, w.Hkv)[idx].cpu().numpy()
    ref = oracle.paged_attention_int8(q, k8[idx].cpu().numpy(), v8[idx].cpu().numpy(), ka_s, va_s, bt_s, cl,
                                      w.scale, nthreads=os.cpu_count() or 8)
    assert_attention_close(out, ref, "int8 qwen3_8b")


def _random_int8_case(r, B, Hq, Hkv, d_head, lens, amax_lo=3.5, amax_hi=4.5):
    nblk = [-(-int(n) // BLOCK) for n in lens]
    nb = sum(nblk) + 3
    perm = r.permutation(nb)
    mbps = max(max(nblk), 1) + 1
    bt = np.full((B, mbps), -1, np.int32)
    i = 0
    for b in range(B):
        bt[b, :nblk[b]] = perm[i:i + nblk[b]]
        i += nblk[b]
    k8 = np.clip(np.round(r.standard_normal((nb, Hkv, BLOCK, d_head)) * 32), -127, 127).astype(np.int8)
    v8 = np.clip(np.round(r.standard_normal((nb, Hkv, BLOCK, d_head)) * 32), -127, 127).astype(np.int8)
    ka = r.uniform(amax_lo, amax_hi, (nb, Hkv)).astype(np.float32)
    va = r.uniform(amax_lo, amax_hi, (nb, Hkv)).astype(np.float32)
    q = bf16_normal(r, (B, Hq, d_head))
    return q, k8, v8, ka, va, bt, np.array(lens, np.int32)


def _dev_case(k8, v8, ka, va, device):
    import torch
    mi = _mi()
    nb, Hkv = ka.shape

    class _S:
        pass
    ds = _S()
    ds.k8, ds.v8 = torch.from_numpy(k8).to(device), torch.from_numpy(v8).to(device)
    n = mi.amax_floats(nb, Hkv)
    ds.k_amax = torch.zeros(n, dtype=torch.float32, device=device)
    ds.v_amax = torch.zeros(n, dtype=torch.float32, device=device)
    ds.k_amax[: nb * Hkv] = torch.from_numpy(ka.ravel()).to(device)
    ds.v_amax[: nb * Hkv] = torch.from_numpy(va.ravel()).to(device)
    return ds


@pytest.mark.parametrize("d_head,Hq,Hkv", [(64, 8, 2), (128, 16, 2), (128, 32, 8), (64, 7, 7), (128, 7, 1)])
def test_int8_edge_lengths_and_paging_invariance(cuda_device, d_head, Hq, Hkv):
    mi = _mi()
    r = np.random.Generator(np.random.PCG64(50 + d_head + Hq + Hkv))
    lens = [0, 1, 15, 16, 17, 63, 64, 65, 200, 1000, 4097]
    B = len(lens)
    q, k8, v8, ka, va, bt, cl = _random_int8_case(r, B, Hq, Hkv, d_head, lens)
    nb = ka.shape[0]
    d = mi.dims(B, Hq, Hkv, d_head, nb, bt.shape[1])
    ds = _dev_case(k8, v8, ka, va, cuda_device)
    out, err = _gpu_attend(mi, d, q, ds, bt, cl, 0.09, cuda_device)
    assert err == 0
    ref = oracle.paged_attention_int8(q, k8, v8, ka, va, bt, cl, 0.09, nthreads=8)
    assert_attention_close(out, ref, f"int8 edges {d_head}/{Hq}/{Hkv}")
    assert not oracle.bf16_to_f64(out[0]).any()                       # a context of 0 gives zeros
    # the same data at other physical blocks (maxima moved with them): the same bits
    perm = r.permutation(nb)
    inv = np.argsort(perm)
    bt2 = np.where(bt >= 0, inv[np.maximum(bt, 0)], -1).astype(np.int32)
    ds2 = _dev_case(k8[perm], v8[perm], ka[perm], va[perm], cuda_device)
    out2, err2 = _gpu_attend(mi, d, q, ds2, bt2, cl, 0.09, cuda_device)
    assert err2 == 0 and np.array_equal(out, out2)


def test_int8_attention_across_group_maxima_ranges(cuda_device):
    """Group maxima from 1e-2 to 1e2 within one request (the V reference
    factor rises and O is rescaled), zero groups, and a request whose first
    blocks are zero groups: within a tolerance relative to the largest |V|."""
    mi = _mi()
    r = np.random.Generator(np.random.PCG64(61))
    B, Hq, Hkv, dh = 4, 8, 2, 128
    lens = [300, 513, 64, 700]
    q, k8, v8, ka, va, bt, cl = _random_int8_case(r, B, Hq, Hkv, dh, lens)
    ka = (10.0 ** r.uniform(-2, 2, ka.shape)).astype(np.float32)
    va = (10.0 ** r.uniform(-2, 2, va.shape)).astype(np.float32)
    va[r.random(va.shape) < 0.15] = 0.0
    ka[r.random(ka.shape) < 0.10] = 0.0
    for j in range(4):                                                 # request 3: first four blocks zero in V
        va[bt[3, j]] = 0.0
    k8[ka == 0] = 0
    v8[va == 0] = 0
    q = oracle.f64_to_bf16(oracle.bf16_to_f64(q) * 0.05)               # keep scores moderate (K up to 100)
    d = mi.dims(B, Hq, Hkv, dh, ka.shape[0], bt.shape[1])
    ds = _dev_case(k8, v8, ka, va, cuda_device)
    out, err = _gpu_attend(mi, d, q, ds, bt, cl, 0.09, cuda_device)
    assert err == 0
    ref = oracle.paged_attention_int8(q, k8, v8, ka, va, bt, cl, 0.09)
    got = oracle.bf16_to_f64(out)
    assert np.all(np.isfinite(got))
    G = Hq // Hkv
    for b in range(B):
        blks = bt[b, :-(-lens[b] // BLOCK)]
        for j in range(Hq):
            vmax = float(va[blks, j // G].max())
            assert np.abs(got[b, j] - ref[b, j]).max() <= 1e-2 * max(vmax, 1e-3), (b, j)


def test_int8_append_errors(cuda_device):
    """A bad position skips the request (q_out too), a bad slot or a bad block
    id of the group skips its cache writes; the other requests append."""
    mi = _mi()
    r = np.random.Generator(np.random.PCG64(70))
    B, Hq, Hkv, dh, nb = 4, 4, 2, 64, 12
    q, k, v = (bf16_normal(r, (B, H, dh)) for H in (Hq, Hkv, Hkv))
    table = oracle.rope_table(1e6, dh, 40)
    bt = np.array([[0, 1, 2, -1], [3, 4, 5, 6], [7, 99, -1, -1], [8, 9, -1, -1]], np.int32)
    cl = np.array([5, 50, 20, 30], np.int32)        # request 1: position 49 >= max_pos 40
    slots = np.array([0, 1, 2, 9], np.int32)        # request 3: slot 9 outside [0, 4)
    st = oracle.int8_state(nb, Hkv, dh, 4)
    ds = DevState(st, cuda_device)
    d = mi.dims(B, Hq, Hkv, dh, nb, 4)
    q_gpu, err = _gpu_append(mi, d, ds, q, k, v, table, 40, bt, cl, slots, cuda_device)
    assert err & mi.MI_DEVERR_BAD_POS and err & mi.MI_DEVERR_BAD_BLOCK and err & mi.MI_DEVERR_BAD_SLOT
    q_ref, s = oracle.append_int8(q, k, v, table, bt, cl, slots, st)
    assert s == -1
    assert np.array_equal(q_gpu, q_ref)
    _assert_state_equal(ds.host(), st, "errors")
    got = ds.host()
    assert got["k8"][0, :, 4].any() and not got["k8"][3:].any()        # only request 0 wrote codes


def _tokens_case(seed, hist, m, Hq, Hkv, d_head, spare=4):
    r = np.random.Generator(np.random.PCG64(seed))
    final = [h + c for h, c in zip(hist, m)]
    B = len(hist)
    nblk = [max(-(-f // BLOCK), 1) for f in final]
    nb = sum(nblk) + spare
    perm = r.permutation(nb)
    bt = np.full((B, max(nblk) + 1), -1, np.int32)
    i = 0
    for b in range(B):
        bt[b, :nblk[b]] = perm[i:i + nblk[b]]
        i += nblk[b]
    kc16 = np.zeros((nb, Hkv, BLOCK, d_head), np.uint16)
    vc16 = np.zeros_like(kc16)
    for b in range(B):
        for t in range(hist[b]):
            kc16[bt[b, t // BLOCK], :, t % BLOCK] = bf16_normal(r, (Hkv, d_head))
            vc16[bt[b, t // BLOCK], :, t % BLOCK] = bf16_normal(r, (Hkv, d_head))
    slots = r.permutation(B + 2)[:B].astype(np.int32)
    st = oracle.int8_state(nb, Hkv, d_head, B + 2)
    assert oracle.int8_from_bf16_cache(kc16, vc16, bt, np.array(hist, np.int32), slots, st) == 0
    qs = np.concatenate([[0], np.cumsum(m)]).astype(np.int32)
    T = int(qs[-1])
    q = bf16_normal(r, (T, Hq, d_head))
    # rows at several magnitudes (zero rows included): group maxima grow, stay and restart
    mag = r.choice([0.0, 0.5, 1.0, 4.0], size=(2, T, Hkv, 1), p=[0.05, 0.25, 0.5, 0.2])
    k = oracle.f64_to_bf16(oracle.bf16_to_f64(bf16_normal(r, (T, Hkv, d_head))) * mag[0])
    v = oracle.f64_to_bf16(oracle.bf16_to_f64(bf16_normal(r, (T, Hkv, d_head))) * mag[1])
    return st, bt, np.array(final, np.int32), qs, slots, q, k, v


def _assert_tokens_state_equal(got, want, cl, slots, what=""):
    """Codes and maxima everywhere; of the open-group buffers, the live rows
    of each request's last group (rows past them are unspecified after a
    many-token append: the token-by-token definition leaves an earlier full
    group's rows there, the kernel leaves the slot's earlier contents)."""
    for key in ("k8", "v8", "k_amax", "v_amax"):
        assert np.array_equal(got[key], want[key]), f"{what}: {key} differs"
    for b, n in enumerate(cl):
        if n > 0:
            o = (int(n) - 1) % GRP + 1
            for key in ("k_open", "v_open"):
                assert np.array_equal(got[key][slots[b], :, :o], want[key][slots[b], :, :o]), (what, key, b)


def _gpu_append_tokens(mi, d, ds, q, k, v, table, max_pos, bt, cl, qs, slots, device):
    import torch
    qo_d = torch.zeros((q.shape[0],) + q.shape[1:], dtype=torch.bfloat16, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    st = mi.mi_paged_kv_append_int8_tokens(d, q.shape[0], to_dev_u16(q, device), to_dev_u16(k, device),
                                           to_dev_u16(v, device), torch.from_numpy(table).to(device), max_pos,
                                           to_dev_i32(bt, device), to_dev_i32(cl, device), to_dev_i32(qs, device),
                                           to_dev_i32(slots, device), qo_d, ds.k8, ds.v8, ds.k_amax, ds.v_amax,
                                           ds.k_open, ds.v_open, err)
    assert st == 0, mi.status_string(st)
    torch.cuda.synchronize()
    return from_dev_u16(qo_d), int(err.item())


@pytest.mark.parametrize("d_head,Hq,Hkv", [(128, 8, 2), (64, 4, 4), (128, 7, 1)])
def test_int8_append_tokens_equals_sequential_appends(cuda_device, d_head, Hq, Hkv):
    """Prompts and chunks (1 to 300 new tokens, from histories at every phase
    of a group) through mi_paged_kv_append_int8_tokens: q_out and the whole
    INT8 state bit for bit as the oracle's token-by-token appends, then the
    attention over the result within the tolerance."""
    mi = _mi()
    hist = [0, 1, 15, 63, 64, 100, 500, 10]
    m = [300, 1, 70, 2, 129, 28, 64, 0]
    st, bt, cl, qs, slots, q, k, v = _tokens_case(70 + d_head + Hq, hist, m, Hq, Hkv, d_head)
    table = oracle.rope_table(1e6, d_head, 1024)
    d = mi.dims(len(hist), Hq, Hkv, d_head, st["k8"].shape[0], bt.shape[1])
    ds = DevState(st, cuda_device)
    q_gpu, err = _gpu_append_tokens(mi, d, ds, q, k, v, table, 1024, bt, cl, qs, slots, cuda_device)
    assert err == 0
    q_ref, s = oracle.append_int8_tokens(q, k, v, table, bt, cl, qs, slots, st)
    assert s == 0
    assert np.array_equal(q_gpu, q_ref)
    _assert_tokens_state_equal(ds.host(), st, cl, slots, "tokens")
    # decode attention over the appended state (the last token's q of each request)
    last = np.maximum(qs[1:] - 1, 0)
    qd = q_ref[last]
    live = cl > 0
    ref = oracle.paged_attention_int8(qd, st["k8"], st["v8"], st["k_amax"], st["v_amax"], bt, cl, 0.1)
    out, err = _gpu_attend(mi, d, qd, ds, bt, cl, 0.1, cuda_device)
    assert err == 0
    got = oracle.bf16_to_f64(out)
    vmax = float(st["v_amax"].max())
    assert np.abs(got[live] - ref[live]).max() <= 1e-2 * max(1.0, vmax / 4)


def test_int8_append_tokens_errors(cuda_device):
    """query_start out of order, more new tokens than the context, a position
    past max_pos, a bad slot and a bad block id each set their bit and skip
    what they name; a good request in the same call appends."""
    mi = _mi()
    hist = [10, 20, 30, 40, 50, 60]
    m = [5, 5, 5, 5, 5, 5]
    st, bt, cl, qs, slots, q, k, v = _tokens_case(80, hist, m, 4, 2, 64)
    table = oracle.rope_table(1e6, 64, 66)
    cl = cl.copy(); qs = qs.copy(); slots = slots.copy(); bt = bt.copy()
    cl[1] = 3                      # 5 new tokens in a context of 3: bad query
    slots[2] = 99                  # bad slot
    bt[3, 2] = 10_000              # bad block in the touched group
    cl[4] = 70                     # last position 69 >= max_pos 66 (request 5 ends at 64)
    d = mi.dims(len(hist), 4, 2, 64, st["k8"].shape[0], bt.shape[1])
    ds = DevState(st, cuda_device)
    q_gpu, err = _gpu_append_tokens(mi, d, ds, q, k, v, table, 66, bt, cl, qs, slots, cuda_device)
    for bit in (mi.MI_DEVERR_BAD_QUERY, mi.MI_DEVERR_BAD_SLOT, mi.MI_DEVERR_BAD_BLOCK, mi.MI_DEVERR_BAD_POS):
        assert err & bit, bit
    got = ds.host()
    # requests 0 and 5 appended like the oracle's token-by-token appends
    ref_st = {key: val.copy() for key, val in st.items()}
    keep = np.array([0, 5])
    sub_qs = np.array([0, 5, 10], np.int32)
    rows = np.concatenate([np.arange(qs[b], qs[b + 1]) for b in keep])
    q_ref, s = oracle.append_int8_tokens(q[rows], k[rows], v[rows], table, bt[keep], cl[keep], sub_qs, slots[keep],
                                         ref_st)
    assert s == 0
    _assert_tokens_state_equal(got, ref_st, cl[keep], slots[keep], "errors")
    assert np.array_equal(q_gpu[rows], q_ref)
    assert not q_gpu[qs[4]:qs[5]].any() and not q_gpu[qs[1]:qs[2]].any()   # skipped requests: no q_out
