"""GPU parity of the prefill path against the oracle: a chunked append of every
new token (mi_paged_kv_append with one row per token, slots from
mi_kv_pool_token_slots) bit-exact, then mi_paged_prefill_attention within the
attention tolerance of the fp64 causal oracle. Full-size rows are checked on a
sample, each as a one-token request over the same table (the oracle's
definition of a single row's causal prefix); error bits and edge cases use
small inputs."""
import numpy as np
import pytest

import oracle
from helpers import assert_attention_close, from_dev_u16, to_dev_i32, to_dev_u16
from oracle.pool import PoolModel
from workloads import (BLOCK, PREFILL_WORKLOADS, bf16_normal, history_cache,
                       prefill_new_values, prefill_setup_pool)

pytestmark = pytest.mark.gpu

VARIANTS = [1, 2, 3]  # MI_PREFILL_MMA (mma.sync tiles), MI_PREFILL_TCGEN05 (tcgen05 + tensor memory), MI_PREFILL_TCGEN05_PAIR


def _mi():
    import paged_kv_decode_25_gb300 as mi
    return mi


def _run_prefill(w, device, layer=0, order_seed=None, variant=0):
    """Chunked append + prefill attention on the device; returns everything the
    checks need (host copies of the oracle's inputs and the device outputs)."""
    import torch
    mi = _mi()
    order = None if order_seed is None else \
        np.random.Generator(np.random.PCG64(order_seed)).permutation(w.num_blocks).astype(np.int32)
    lib = mi.Pool(w.num_blocks, w.max_seqs, w.max_blocks_per_seq, order)
    model = PoolModel(w.num_blocks, w.max_seqs, w.max_blocks_per_seq, order)
    prefill_setup_pool(w, lib)
    prefill_setup_pool(w, model)
    R = w.B
    bt, _, _ = lib.batch_meta(range(R))
    assert np.array_equal(bt, model.batch_meta(range(R))[0])
    h, m = w.lengths()
    n = (h + m).astype(np.int32)
    slots = np.concatenate([lib.token_slots(r, int(h[r]), int(m[r])) for r in range(R)]).astype(np.int32)
    slots_m = np.concatenate([model.token_slots(r, int(h[r]), int(m[r])) for r in range(R)])
    assert np.array_equal(slots, slots_m)
    pos = np.concatenate([np.arange(h[r], h[r] + m[r]) for r in range(R)]).astype(np.int32)
    qs = np.concatenate([[0], np.cumsum(m)]).astype(np.int32)
    T = int(qs[-1])

    kc, vc = history_cache(w, layer, bt, h)
    q, k, v = prefill_new_values(w, layer)
    st, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos)
    assert st == 0
    d_app = mi.dims(T, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    d_att = mi.dims(R, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    kc_d, vc_d = to_dev_u16(kc, device), to_dev_u16(vc, device)
    q_d, k_d, v_d = (to_dev_u16(a, device) for a in (q, k, v))
    qo_d = torch.empty_like(q_d)
    out_d = torch.empty_like(q_d)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    rope_d = torch.from_numpy(table).to(device)
    assert mi.mi_paged_kv_append(d_app, q_d, k_d, v_d, to_dev_i32(pos, device), to_dev_i32(slots, device),
                                 rope_d, w.max_pos, qo_d, kc_d, vc_d, err) == 0
    bt_d, n_d, qs_d = (to_dev_i32(a, device) for a in (bt, n, qs))
    assert mi.mi_paged_prefill_attention_variant(d_att, T, int(m.max()), qo_d, kc_d, vc_d, bt_d, n_d, qs_d,
                                                 w.scale, out_d, variant=variant, dev_err=err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # the oracle's append on the host copies
    q_ref, st = oracle.append(q, k, v, pos, slots_m, oracle.rope_table(w.theta, w.head_dim, w.max_pos),
                              kc, vc)
    assert st == 0
    return dict(bt=bt, n=n, h=h, m=m, qs=qs, T=T, kc=kc, vc=vc, q_ref=q_ref, qo_d=qo_d, kc_d=kc_d,
                vc_d=vc_d, out_d=out_d, v_new=v)


@pytest.mark.parametrize("variant", VARIANTS)
def test_prefill_small_full_parity(cuda_device, variant):
    w = PREFILL_WORKLOADS["prefill_small"]
    x = _run_prefill(w, cuda_device, order_seed=3, variant=variant)
    assert np.array_equal(from_dev_u16(x["qo_d"]), x["q_ref"])
    assert np.array_equal(from_dev_u16(x["kc_d"]), x["kc"])
    assert np.array_equal(from_dev_u16(x["vc_d"]), x["vc"])
    ref = oracle.paged_prefill_attention(x["q_ref"], x["kc"], x["vc"], x["bt"], x["n"], x["qs"], w.scale,
                                         nthreads=8)
    got = from_dev_u16(x["out_d"])
    assert_attention_close(got, ref, "prefill_small")
    # request 0 is one token at position 0: softmax over one key returns its V exactly
    G = w.G
    for j in range(w.Hq):
        assert np.array_equal(got[0, j], x["v_new"][0, j // G])


@pytest.mark.parametrize("name", ["qwen3_8b_prefill", "qwen25_7b_prefill"])
@pytest.mark.parametrize("variant", VARIANTS)
def test_prefill_full_size_sampled(cuda_device, variant, name):
    w = PREFILL_WORKLOADS[name]
    x = _run_prefill(w, cuda_device, variant=variant)
    # append: the new tokens' rows and slots, bit-exact
    assert np.array_equal(from_dev_u16(x["qo_d"]), x["q_ref"])
    kc_got, vc_got = from_dev_u16(x["kc_d"]), from_dev_u16(x["vc_d"])
    assert np.array_equal(kc_got, x["kc"]) and np.array_equal(vc_got, x["vc"])
    # attention: first, last and two random new tokens of every request
    r = np.random.Generator(np.random.PCG64(17))
    rows, lens, tabs = [], [], []
    for b in range(w.B):
        mb = int(x["m"][b])
        for i in sorted({0, mb - 1, int(r.integers(0, mb)), int(r.integers(0, mb))}):
            rows.append(int(x["qs"][b]) + i)
            lens.append(int(x["n"][b]) - mb + i + 1)  # the row's causal prefix as a one-token request
            tabs.append(x["bt"][b])
    rows = np.array(rows)
    qs1 = np.arange(len(rows) + 1, dtype=np.int32)
    ref = oracle.paged_prefill_attention(x["q_ref"][rows], x["kc"], x["vc"], np.stack(tabs),
                                         np.array(lens, np.int32), qs1, w.scale, nthreads=16)
    got = from_dev_u16(x["out_d"])[rows]
    assert_attention_close(got, ref, f"{name} sampled rows")
    assert np.all(np.isfinite(oracle.bf16_to_f64(from_dev_u16(x["out_d"]))))


def _random_case(seed, Hq, Hkv, d, hist, new, nb_extra=5):
    """Paged caches with every context token (history and new) already in
    place, plus q rows for the new tokens: the attention alone."""
    r = np.random.Generator(np.random.PCG64(seed))
    hist, new = np.asarray(hist, np.int32), np.asarray(new, np.int32)
    n = hist + new
    R = len(n)
    nblk = [-(-int(x) // BLOCK) for x in n]
    nb = sum(nblk) + nb_extra
    perm = r.permutation(nb)
    mbps = max(max(nblk), 1)
    bt = np.full((R, mbps), -1, np.int32)
    kc = np.full((nb, Hkv, BLOCK, d), 0x7FA5, np.uint16)  # NaN canary outside the contexts
    vc = kc.copy()
    i = 0
    for b in range(R):
        kv = bf16_normal(r, (2, Hkv, max(int(n[b]), 1), d))
        for j in range(nblk[b]):
            blk = int(perm[i]); i += 1
            bt[b, j] = blk
            c = min(BLOCK, int(n[b]) - j * BLOCK)
            kc[blk, :, :c] = kv[0, :, j * BLOCK: j * BLOCK + c]
            vc[blk, :, :c] = kv[1, :, j * BLOCK: j * BLOCK + c]
    qs = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    q = bf16_normal(r, (int(qs[-1]), Hq, d))
    return q, kc, vc, bt, n.astype(np.int32), qs


def _attend(device, q, kc, vc, bt, n, qs, scale, max_q=None, variant=0):
    import torch
    mi = _mi()
    T, Hq, d = q.shape
    nb, Hkv = kc.shape[0], kc.shape[1]
    dm = mi.dims(len(n), Hq, Hkv, d, nb, bt.shape[1])
    out = torch.full((max(T, 1), Hq, d), 7.0, dtype=torch.bfloat16, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    mq = int(np.diff(qs).max()) if max_q is None else max_q
    st = mi.mi_paged_prefill_attention_variant(dm, T, mq, to_dev_u16(q, device), to_dev_u16(kc, device),
                                               to_dev_u16(vc, device), to_dev_i32(bt, device), to_dev_i32(n, device),
                                               to_dev_i32(qs, device), scale, out, variant=variant, dev_err=err)
    assert st == 0
    torch.cuda.synchronize()
    return from_dev_u16(out)[:T], int(err.item())


@pytest.mark.parametrize("Hq,Hkv,d", [(4, 4, 64), (8, 4, 128), (8, 2, 64), (16, 2, 128), (32, 8, 128),
                                       (28, 4, 128), (12, 4, 64), (24, 4, 128), (20, 4, 128)])
@pytest.mark.parametrize("variant", VARIANTS)
def test_prefill_group_and_head_dim(cuda_device, Hq, Hkv, d, variant):
    hist = [0, 5, 64, 200, 31, 0]
    new = [3, 64, 1, 77, 130, 16]
    q, kc, vc, bt, n, qs = _random_case(Hq * 100 + d, Hq, Hkv, d, hist, new)
    scale = 1.0 / np.sqrt(d)
    got, err = _attend(cuda_device, q, kc, vc, bt, n, qs, scale, variant=variant)
    assert err == 0
    ref = oracle.paged_prefill_attention(q, kc, vc, bt, n, qs, scale, nthreads=8)
    assert_attention_close(got, ref, f"G={Hq // Hkv} d={d}")


@pytest.mark.parametrize("variant", VARIANTS)
def test_prefill_one_token_requests_match_decode_oracle(cuda_device, variant):
    # m = 1 everywhere: the prefill kernel computes decode attention
    q, kc, vc, bt, n, qs = _random_case(5, 8, 2, 128, [0, 15, 16, 17, 500, 1023], [1] * 6)
    got, err = _attend(cuda_device, q, kc, vc, bt, n, qs, 0.09, variant=variant)
    assert err == 0
    ref = oracle.paged_attention(q, kc, vc, bt, n, 0.09)
    assert_attention_close(got, ref, "one-token prefill")


@pytest.mark.parametrize("variant", VARIANTS)
def test_prefill_paging_invariance_bitwise(cuda_device, variant):
    hist, new = [40, 0, 123], [50, 97, 33]
    q, kc, vc, bt, n, qs = _random_case(9, 8, 2, 128, hist, new)
    a, _ = _attend(cuda_device, q, kc, vc, bt, n, qs, 0.1, variant=variant)
    # move every block to another physical id
    r = np.random.Generator(np.random.PCG64(10))
    perm = r.permutation(kc.shape[0])
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    b, _ = _attend(cuda_device, q, kc2, vc2, bt2, n, qs, 0.1, variant=variant)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("variant", VARIANTS)
def test_prefill_edge_lengths(cuda_device, variant):
    # zero-token requests, block-aligned and ragged contexts, one long chunk
    hist = [0, 16, 0, 1, 47, 0, 255]
    new = [0, 16, 32, 0, 1, 65, 1]
    q, kc, vc, bt, n, qs = _random_case(12, 8, 4, 64, hist, new)
    got, err = _attend(cuda_device, q, kc, vc, bt, n, qs, 0.125, variant=variant)
    assert err == 0
    ref = oracle.paged_prefill_attention(q, kc, vc, bt, n, qs, 0.125)
    assert_attention_close(got, ref, "edge lengths")


@pytest.mark.parametrize("scale", [0.0, -0.09])
@pytest.mark.parametrize("variant", VARIANTS)
def test_prefill_nonpositive_scale(cuda_device, scale, variant):
    """A scale of zero or below takes the softmax path that scales every
    score before the row max (the fast path folds a positive scale into the
    exponent); with scale 0 every row is the mean of V over its causal
    window."""
    hist, new = [0, 37, 300], [70, 140, 9]
    q, kc, vc, bt, n, qs = _random_case(21, 16, 4, 128, hist, new)
    got, err = _attend(cuda_device, q, kc, vc, bt, n, qs, scale, variant=variant)
    assert err == 0
    ref = oracle.paged_prefill_attention(q, kc, vc, bt, n, qs, scale, nthreads=8)
    assert_attention_close(got, ref, f"scale {scale}")


@pytest.mark.parametrize("variant", VARIANTS)
def test_prefill_growing_scores_rescale(cuda_device, variant):
    """Keys whose magnitude grows along the context (block j of every request
    scaled by 1 + j / 2) push each row's running max up by far more than 2^8
    (base 2) many times over: the kernels' lazy rescaling of O and l has to
    give the oracle's result."""
    hist, new = [400, 900], [64, 130]
    q, kc, vc, bt, n, qs = _random_case(22, 8, 2, 128, hist, new)
    k64 = oracle.bf16_to_f64(kc)
    for b in range(len(n)):
        for j in range(-(-int(n[b]) // BLOCK)):
            k64[bt[b, j]] *= 1.0 + j / 2.0
    kc = oracle.f64_to_bf16(k64)
    scale = 1.0 / np.sqrt(128)
    got, err = _attend(cuda_device, q, kc, vc, bt, n, qs, scale, variant=variant)
    assert err == 0
    ref = oracle.paged_prefill_attention(q, kc, vc, bt, n, qs, scale, nthreads=8)
    # the input does what it is for: for the last new token of request 1
    # (query head 0, KV head 0) the running max of its base-2 scores over
    # 128-key stages grows by more than 8 at least three times
    b, row = 1, int(qs[2]) - 1
    keys = np.stack([oracle.bf16_to_f64(kc[bt[b, t // BLOCK], 0, t % BLOCK]) for t in range(int(n[b]))])
    s2 = keys @ oracle.bf16_to_f64(q[row, 0]) * scale * np.log2(np.e)
    stage_max = np.maximum.accumulate([s2[i:i + 128].max() for i in range(0, len(s2), 128)])
    assert int(np.sum(np.diff(stage_max) > 8.0)) >= 3
    # Rows here are nearly one-hot, so outputs are about as large as V (up to
    # ~4) and the fixed absolute tolerance of the other tests does not apply.
    # The kernels round each weight p_i to bf16 for the P.V product (relative
    # error <= 2^-9) and the output to bf16 (<= 2^-9 |o|); scores, sums and
    # O are fp32. So per element |got - ref| <= 2^-9 (sum_i p_i |v_i| + |ref|),
    # checked with a factor 2 of margin; sum_i p_i |v_i| is the oracle's
    # attention over |V|.
    vabs = np.where(np.isnan(oracle.bf16_to_f64(vc)), vc, vc & np.uint16(0x7FFF)).astype(np.uint16)
    ref_abs = oracle.paged_prefill_attention(q, kc, vabs, bt, n, qs, scale, nthreads=8)
    g = oracle.bf16_to_f64(got)
    assert np.all(np.isfinite(g))
    bound = 2.0 ** -8 * (ref_abs + np.abs(ref))
    worst = float(np.max(np.abs(g - ref) / bound))
    assert worst <= 1.0, f"growing scores: error {worst:.2f} x the bound"


@pytest.mark.parametrize("variant", VARIANTS)
def test_prefill_error_bits(cuda_device, variant):
    mi = _mi()
    q, kc, vc, bt, n, qs = _random_case(13, 4, 2, 64, [10, 20], [6, 12])
    # more new tokens than context: rows at negative positions are zero
    n_bad = n.copy()
    n_bad[0] = 4  # 6 new tokens, context 4: tokens 0, 1 at positions -2, -1
    got, err = _attend(cuda_device, q, kc, vc, bt, n_bad, qs, 0.125, variant=variant)
    assert err & mi.MI_DEVERR_BAD_QUERY
    assert np.all(got[:2] == 0)
    ref = oracle.paged_prefill_attention(q, kc, vc, bt, n_bad, qs, 0.125)
    assert_attention_close(got, ref, "m > n")
    # a bad block id: flagged, and the output stays finite
    bt_bad = bt.copy()
    bt_bad[1, 0] = kc.shape[0] + 3
    got, err = _attend(cuda_device, q, kc, vc, bt_bad, n, qs, 0.125, variant=variant)
    assert err & mi.MI_DEVERR_BAD_BLOCK
    assert np.all(np.isfinite(oracle.bf16_to_f64(got)))
    # a request longer than max_query_len is skipped (its rows untouched)
    got, err = _attend(cuda_device, q, kc, vc, bt, n, qs, 0.125, max_q=8, variant=variant)
    assert err & mi.MI_DEVERR_BAD_QUERY
    assert np.all(oracle.bf16_to_f64(got[6:]) == 7.0)
    ref = oracle.paged_prefill_attention(q, kc, vc, bt, n, qs, 0.125)
    assert_attention_close(got[:6], ref[:6], "request within max_query_len")
    # a context longer than a table row
    n_long = n.copy()
    n_long[1] = bt.shape[1] * BLOCK + 5
    _, err = _attend(cuda_device, q, kc, vc, bt, n_long, qs, 0.125, variant=variant)
    assert err & mi.MI_DEVERR_BAD_CONTEXT
    # query_start out of order
    qs_bad = np.array([0, 12, 6], np.int32)
    _, err = _attend(cuda_device, q[:6], kc, vc, bt, n, qs_bad, 0.125, max_q=12, variant=variant)
    assert err & mi.MI_DEVERR_BAD_QUERY
