"""CUDA-graph capture of the decode and prefill calls: a captured launch
keeps the kernel arguments of the capture, the split-KV merge's epoch
included, and is replayed many times over one workspace. Each replay must
give the bits of an eager call. Covered on the Qwen3-8B-shaped serving layer
(B = 64, contexts up to 8k, a fragmented pool, hundreds of units cut across
CTAs): the bf16, e4m3 and INT8 attention, the bf16 and e4m3 fused steps and
the INT8 append + attention, each replayed three times, and two launches
captured back to back on one workspace; and the causal prefill attention
with each of its kernels."""
import numpy as np
import pytest

from helpers import grow, pools_for, to_dev_i32, to_dev_u16
from workloads import BLOCK, WORKLOADS, device_fill_cache, new_token_values

pytestmark = pytest.mark.gpu

REPLAYS = 3


def _mi():
    import paged_kv_decode_25_gb300 as mi
    return mi


def _layer(device):
    import torch
    mi = _mi()
    w = WORKLOADS["qwen3_8b"]
    lib, _, ctx = pools_for(w)
    grow(lib, w.B, ctx + 1)
    bt, cl, _ = lib.batch_meta(range(w.B))
    shape = (w.num_blocks, w.Hkv, BLOCK, w.head_dim)
    kc = torch.empty(shape, dtype=torch.bfloat16, device=device)
    vc = torch.empty_like(kc)
    device_fill_cache(w, 0, kc, vc)
    q, k, v = new_token_values(w, 0)
    d = mi.dims(w.B, w.Hq, w.Hkv, w.head_dim, w.num_blocks, w.max_blocks_per_seq)
    lay = dict(w=w, d=d, bt=to_dev_i32(bt, device), cl=to_dev_i32(cl, device), kc=kc, vc=vc,
               q=to_dev_u16(q, device), k=to_dev_u16(k, device), v=to_dev_u16(v, device))
    return lay


def _workspace(mi, d, device):
    import torch
    # NaN bits everywhere: the call must not depend on the buffer's contents
    return torch.full((mi.mi_paged_decode_workspace_bytes(d) // 4 + 4,), float("nan"), dtype=torch.float32,
                      device=device)


def _bits(t):
    import torch
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.uint8)


def _replay_and_check(launch, outs, refs, err):
    """Capture launch() once, then replay it; before each replay the outputs
    are overwritten with NaN, after it they must equal refs bit for bit."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        launch()
    for _ in range(REPLAYS):
        for o in outs:
            o.fill_(float("nan"))
        err.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        for o, r in zip(outs, refs):
            assert torch.equal(_bits(o), _bits(r))


@pytest.mark.parametrize("kv", ["bf16", "e4m3", "int8"])
def test_graph_replay_attention(cuda_device, kv):
    import torch
    mi = _mi()
    lay = _layer(cuda_device)
    w, d = lay["w"], lay["d"]
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    if kv == "bf16":
        kc, vc = lay["kc"], lay["vc"]

        def call(out, ws):
            assert mi.mi_paged_decode_attention(d, lay["q"], kc, vc, lay["bt"], lay["cl"], w.scale, out, ws,
                                                dev_err=err) == 0
    else:
        ks = torch.full((w.Hkv,), 1.0 / 64, dtype=torch.float32, device=cuda_device)
        vs = torch.full((w.Hkv,), 1.0 / 32, dtype=torch.float32, device=cuda_device)
        kc = (lay["kc"].float() * 64).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
        vc = (lay["vc"].float() * 32).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)

        def call(out, ws):
            assert mi.mi_paged_decode_attention_fp8(d, lay["q"], kc, vc, ks, vs, lay["bt"], lay["cl"], w.scale, out,
                                                    ws, dev_err=err) == 0
    if kv == "int8":
        kc = (lay["kc"].float() * 32).round_().clamp_(-127, 127).to(torch.int8)
        vc = (lay["vc"].float() * 32).round_().clamp_(-127, 127).to(torch.int8)
        g = torch.Generator(device=cuda_device)
        g.manual_seed(3)
        ka = 3.5 + torch.rand(w.num_blocks * w.Hkv, generator=g, device=cuda_device)
        va = 3.5 + torch.rand(w.num_blocks * w.Hkv, generator=g, device=cuda_device)

        def call(out, ws):
            assert mi.mi_paged_decode_attention_int8(d, lay["q"], kc, vc, ka, va, lay["bt"], lay["cl"], w.scale, out,
                                                     ws, dev_err=err) == 0
    ref = torch.empty_like(lay["q"])
    call(ref, _workspace(mi, d, cuda_device))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ws = _workspace(mi, d, cuda_device)
    out = torch.empty_like(ref)
    _replay_and_check(lambda: call(out, ws), [out], [ref], err)
    # two launches captured back to back on one workspace (two layers of a step)
    out1, out2 = torch.empty_like(ref), torch.empty_like(ref)

    def two():
        call(out1, ws)
        call(out2, ws)
    _replay_and_check(two, [out1, out2], [ref, ref], err)


def test_graph_replay_step(cuda_device):
    """The fused step captured once and replayed: each replay writes the same
    new cache rows and q_out and gives the eager step's output."""
    import torch
    mi = _mi()
    lay = _layer(cuda_device)
    w, d = lay["w"], lay["d"]
    _, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos)
    tab = torch.from_numpy(table).to(cuda_device)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    kc_ref, vc_ref = lay["kc"].clone(), lay["vc"].clone()
    qo_ref, out_ref = torch.empty_like(lay["q"]), torch.empty_like(lay["q"])
    assert mi.mi_paged_decode_step(d, lay["q"], lay["k"], lay["v"], tab, w.max_pos, lay["bt"], lay["cl"], w.scale,
                                   qo_ref, kc_ref, vc_ref, out_ref, _workspace(mi, d, cuda_device), dev_err=err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ws = _workspace(mi, d, cuda_device)
    qo, out = torch.empty_like(qo_ref), torch.empty_like(out_ref)

    def step():
        assert mi.mi_paged_decode_step(d, lay["q"], lay["k"], lay["v"], tab, w.max_pos, lay["bt"], lay["cl"],
                                       w.scale, qo, lay["kc"], lay["vc"], out, ws, dev_err=err) == 0
    _replay_and_check(step, [qo, out], [qo_ref, out_ref], err)
    assert torch.equal(_bits(lay["kc"]), _bits(kc_ref))
    assert torch.equal(_bits(lay["vc"]), _bits(vc_ref))


def test_graph_replay_step_fp8(cuda_device):
    """The fused e4m3 step captured once and replayed: each replay writes the
    same quantised cache rows and q_out and gives the eager step's output."""
    import torch
    mi = _mi()
    lay = _layer(cuda_device)
    w, d = lay["w"], lay["d"]
    _, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos)
    tab = torch.from_numpy(table).to(cuda_device)
    ks = torch.full((w.Hkv,), 1.0 / 64, dtype=torch.float32, device=cuda_device)
    vs = torch.full((w.Hkv,), 1.0 / 32, dtype=torch.float32, device=cuda_device)
    kc = (lay["kc"].float() * 64).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    vc = (lay["vc"].float() * 32).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    kc_ref, vc_ref = kc.clone(), vc.clone()
    qo_ref, out_ref = torch.empty_like(lay["q"]), torch.empty_like(lay["q"])
    assert mi.mi_paged_decode_step_fp8(d, lay["q"], lay["k"], lay["v"], tab, w.max_pos, lay["bt"], lay["cl"], ks, vs,
                                       w.scale, qo_ref, kc_ref, vc_ref, out_ref, _workspace(mi, d, cuda_device),
                                       dev_err=err) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ws = _workspace(mi, d, cuda_device)
    qo, out = torch.empty_like(qo_ref), torch.empty_like(out_ref)

    def step():
        assert mi.mi_paged_decode_step_fp8(d, lay["q"], lay["k"], lay["v"], tab, w.max_pos, lay["bt"], lay["cl"], ks,
                                           vs, w.scale, qo, kc, vc, out, ws, dev_err=err) == 0
    _replay_and_check(step, [qo, out], [qo_ref, out_ref], err)
    assert torch.equal(kc, kc_ref)
    assert torch.equal(vc, vc_ref)


@pytest.mark.parametrize("variant", [0, 1, 2, 3])  # default (two-tile), mma.sync, single-tile tcgen05, two-tile
def test_graph_replay_prefill(cuda_device, variant):
    """Causal prefill attention captured once and replayed (requests with and
    without history, G = 4): each replay gives the eager call's bits."""
    import numpy as np
    import torch
    from test_prefill_gpu import _random_case
    mi = _mi()
    q, kc, vc, bt, n, qs = _random_case(31, 16, 4, 128, [0, 300, 1000, 5], [200, 64, 333, 1])
    T, Hq, dh = q.shape
    d = mi.dims(len(n), Hq, kc.shape[1], dh, kc.shape[0], bt.shape[1])
    q_d, kc_d, vc_d = (to_dev_u16(a, cuda_device) for a in (q, kc, vc))
    bt_d, n_d, qs_d = (to_dev_i32(a, cuda_device) for a in (bt, n, qs))
    max_q = int(np.diff(qs).max())
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    scale = 1.0 / np.sqrt(dh)

    def call(out):
        assert mi.mi_paged_prefill_attention_variant(d, T, max_q, q_d, kc_d, vc_d, bt_d, n_d, qs_d, scale, out,
                                                     variant=variant, dev_err=err) == 0
    ref = torch.empty_like(q_d)
    call(ref)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    out = torch.empty_like(ref)
    _replay_and_check(lambda: call(out), [out], [ref], err)


def test_graph_replay_int8_step(cuda_device):
    """The INT8 append (RoPE, the open group's bf16 rows, the group's codes
    and maxima) then the INT8 attention, captured once and replayed: the
    append of the same token is idempotent (the maximum it raised is the one
    it finds again), so every replay gives the same bits in q_out, codes,
    maxima, open rows and output."""
    import torch
    mi = _mi()
    lay = _layer(cuda_device)
    w, d = lay["w"], lay["d"]
    err = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    k8 = (lay["kc"].float() * 32).round_().clamp_(-127, 127).to(torch.int8)
    v8 = (lay["vc"].float() * 32).round_().clamp_(-127, 127).to(torch.int8)
    ka = torch.full((w.num_blocks * w.Hkv,), 4.0, dtype=torch.float32, device=cuda_device)
    va = torch.full_like(ka, 4.0)
    ko = torch.zeros((w.B, w.Hkv, 64, w.head_dim), dtype=torch.bfloat16, device=cuda_device)
    vo = torch.zeros_like(ko)
    slots = to_dev_i32(np.arange(w.B, dtype=np.int32), cuda_device)
    _, table = mi.mi_rope_table(w.theta, w.head_dim, w.max_pos)
    rope = torch.from_numpy(table).to(cuda_device)
    ws = _workspace(mi, d, cuda_device)
    qo, out = torch.empty_like(lay["q"]), torch.empty_like(lay["q"])

    def launch():
        assert mi.mi_paged_kv_append_int8(d, lay["q"], lay["k"], lay["v"], rope, w.max_pos, lay["bt"], lay["cl"],
                                          slots, qo, k8, v8, ka, va, ko, vo, err) == 0
        assert mi.mi_paged_decode_attention_int8(d, qo, k8, v8, ka, va, lay["bt"], lay["cl"], w.scale, out, ws,
                                                 dev_err=err) == 0
    launch()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    refs = [t.clone() for t in (qo, out, k8, v8, ka, va, ko, vo)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        launch()
    for _ in range(REPLAYS):
        qo.fill_(float("nan"))
        out.fill_(float("nan"))
        err.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        for t, r in zip((qo, out, k8, v8, ka, va, ko, vo), refs):
            assert torch.equal(_bits(t) if t.dtype != torch.float32 else t.view(torch.int32),
                               _bits(r) if r.dtype != torch.float32 else r.view(torch.int32))
