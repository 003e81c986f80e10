"""The five named workloads (and the ring, paged and attention-bias variants) at full size, in the launch configuration bench.py times,
checked against the fp64 oracle: every row for the tiny fp32 prompt, sampled rows (with the
band edges) for the large ones, and the appended present rows bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, out_rows, run_gpu
from helpers import storage
from sliding_window_gb300.inputs import WORKLOADS, make_case

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def sample_rows(w, n=192, seed=0):
    """Output rows compared at full size: n random rows, the band-edge rows, and one row of
    every CTA's output: a random row of each 128-row query tile for every q head (prefill),
    a random row of each (b, kv head) group (decode)."""
    rng = np.random.default_rng(seed)
    B, L, H = w.batch, w.q_len, w.q_heads
    rows = set(rng.integers(0, B * L * H, size=n).tolist())
    for b in (0, B - 1):
        for i in sorted({0, L - 1, L // 2, min(L - 1, 127), min(L - 1, 128), min(L - 1, 4095), min(L - 1, 4096)}):
            for h in (0, H - 1):
                rows.add((b * L + i) * H + h)
    G = H // w.kv_heads
    for b in range(B):
        if w.mode == "prefill":
            for t0 in range(0, L, 128):
                i = t0 + int(rng.integers(0, min(128, L - t0)))
                rows.update((b * L + i) * H + h for h in range(H))
        else:
            for hk in range(w.kv_heads):
                i, g = int(rng.integers(0, L)), int(rng.integers(0, G))
                rows.add((b * L + i) * H + hk * G + g)
    return np.array(sorted(rows), dtype=np.int64)


def check_workload(name, layer=0):
    w = WORKLOADS[name]
    dev = "cuda:0" if w.cap * w.batch * w.kv_heads * w.head_dim > (1 << 26) else "cpu"
    c = make_case(w, layer=layer, device=dev)
    # host copies of everything the oracle reads, taken before the in-place append
    host = make_host(c)
    r = run_gpu(c, w.mode)
    assert r["status"] == 0
    rows = None if w.batch * w.q_len * w.q_heads <= 4096 else sample_rows(w)
    p = c.params
    q_rot, pk, pv, st = oracle.rope_append(p, host["q"], host["k"], host["v"], host["past_k"], host["past_v"],
                                           host["seq"], host["cos"], host["sin"], present_k=host["past_k"],
                                           present_v=host["past_v"])
    assert st == 0
    gk, gv = r["present_k"], r["present_v"]
    for b, past in enumerate(host["seq"].tolist()):
        sl = slice(past, past + w.q_len)
        np.testing.assert_array_equal(storage(gk[b, :, sl]), pk[b, :, sl])
        np.testing.assert_array_equal(storage(gv[b, :, sl]), pv[b, :, sl])
    ref = oracle.attention(p, q_rot, pk, pv, host["seq"], host["sink"], rows=rows)
    got = out_rows(r["out"], c, rows)
    assert_close(got, ref, w.dtype, name)


def make_host(c):
    return dict(q=storage(c.q), k=storage(c.k), v=storage(c.v), past_k=storage(c.past_k).copy(),
                past_v=storage(c.past_v).copy(), seq=c.seqlens_k.cpu().numpy().copy(),
                cos=None if c.cos is None else storage(c.cos), sin=None if c.sin is None else storage(c.sin),
                sink=None if c.head_sink is None else c.head_sink.cpu().numpy())


def test_prefill_fp32_tiny():
    check_workload("prefill_fp32_tiny")


def test_decode_window_bf16():
    check_workload("decode_window_bf16")


def test_prefill_sink_softcap_bf16():
    check_workload("prefill_sink_softcap_bf16")


@pytest.mark.parametrize("layer", [0, 1])
def test_specdecode_rotary_f16(layer):
    check_workload("specdecode_rotary_f16", layer)


def test_decode_long_bf16():
    check_workload("decode_long_bf16")
    torch.cuda.empty_cache()


def test_decode_window_vdim_bf16():
    check_workload("decode_window_vdim_bf16")


def test_decode_window_ring_bf16():
    """The windowed decode over a ring of 1024 slots: sequences up to 4096 long, so most
    rings have wrapped; the appended slots bit for bit, sampled rows against the ring oracle."""
    w = WORKLOADS["decode_window_ring_bf16"]
    c = make_case(w, device="cpu")
    host = make_host(c)
    r = run_gpu(c, w.mode)
    assert r["status"] == 0
    p = c.params
    q_rot, pk, pv, st = oracle.rope_append_ring(p, host["q"], host["k"], host["v"], host["past_k"], host["past_v"],
                                                host["seq"], host["cos"], host["sin"])
    assert st == 0
    np.testing.assert_array_equal(storage(r["present_k"]), pk)
    np.testing.assert_array_equal(storage(r["present_v"]), pv)
    ref = oracle.attention_ring(p, q_rot, pk, pv, host["seq"], host["sink"])
    assert_close(out_rows(r["out"], c), ref, w.dtype, w.name)


def test_decode_window_paged_bf16():
    """The windowed decode through a shuffled pool of 64-position pages: the pages written bit
    for bit, sampled rows against the paged oracle."""
    from sliding_window_gb300 import gqa
    w = WORKLOADS["decode_window_paged_bf16"]
    c = make_case(w, device="cpu")
    B, Hkv, cap, D = c.past_k.shape
    mp = cap // gqa.PAGE
    table = np.random.default_rng(5).permutation(B * mp).reshape(B, mp).astype(np.int32)
    pools = []
    for lin in (storage(c.past_k), storage(c.past_v)):
        pool = np.empty((B * mp, Hkv, gqa.PAGE, D), dtype=lin.dtype)
        pool[table.ravel()] = lin.reshape(B, Hkv, mp, gqa.PAGE, D).transpose(0, 2, 1, 3, 4).reshape(-1, Hkv, gqa.PAGE, D)
        pools.append(pool)
    dev = [torch.from_numpy(x).view(torch.int16).view(torch.bfloat16).cuda() for x in pools]
    p = gqa.params_from_dict(c.params)
    out = torch.empty(c.q.shape, dtype=c.q.dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(max(16, gqa.gqa_workspace_bytes(p)), dtype=torch.uint8, device="cuda")
    gqa.check(gqa.gqa_attention_decode_paged(p, c.q.cuda(), c.k.cuda(), c.v.cuda(), c.seqlens_k.cuda(),
                                             torch.from_numpy(table).cuda(), B * mp, None, None, None, out, dev[0],
                                             dev[1], ws, st), "paged")
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    q_rot, pk, pv, s = oracle.rope_append_paged(c.params, storage(c.q), storage(c.k), storage(c.v), pools[0],
                                                pools[1], c.seqlens_k.numpy(), table, B * mp)
    assert s == 0
    np.testing.assert_array_equal(storage(dev[0]), pk)
    np.testing.assert_array_equal(storage(dev[1]), pv)
    ref = oracle.attention_paged(c.params, q_rot, pk, pv, c.seqlens_k.numpy(), table, B * mp)
    assert_close(out_rows(out, c), ref, w.dtype, w.name)


@pytest.mark.parametrize("name,kind", [("prefill_bias_bf16", "add"), ("prefill_blocksparse_bf16", "bool")])
def test_prefill_masked_workload(name, kind):
    """The long prompt with a mask [B, 1, S, S] through the masked prefill entry point
    (TMA-staged mask): a dense additive bias, or a block-sparse boolean mask whose removed
    128 x 128 blocks the kernel skips through its block map.  Sampled rows (band edges
    included) against the masked oracle, the appended rows bit for bit."""
    from sliding_window_gb300 import gqa
    w = WORKLOADS[name]
    c = make_case(w, device="cuda:0")
    host = make_host(c)
    mask_host = storage(c.extra["mask"]) if kind == "add" else c.extra["mask"].cpu().numpy()
    p = gqa.params_from_dict(c.params)
    out = torch.full_like(c.q, float("nan"))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(max(16, gqa.gqa_workspace_bytes(p)), dtype=torch.uint8, device="cuda")
    m = gqa.mask_from_tensor(c.extra["mask"], gqa.MASK_ADD if kind == "add" else gqa.MASK_KEEP)
    gqa.check(gqa.gqa_attention_prefill_masked(p, m, c.q, c.k, c.v, c.past_k, c.past_v, c.seqlens_k, c.cos, c.sin,
                                               c.head_sink, out, c.past_k, c.past_v, ws, st), name)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    q_rot, pk, pv, s = oracle.rope_append(c.params, host["q"], host["k"], host["v"], host["past_k"],
                                          host["past_v"], host["seq"], host["cos"], host["sin"],
                                          present_k=host["past_k"], present_v=host["past_v"])
    assert s == 0
    np.testing.assert_array_equal(storage(c.past_k[:, :, : w.q_len]), pk[:, :, : w.q_len])
    rows = sample_rows(w)
    ref = oracle.attention_masked(c.params, q_rot, pk, pv, host["seq"], mask_host, kind, host["sink"], rows=rows)
    assert_close(out_rows(out, c, rows), ref, w.dtype, w.name)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,fmt", [("decode_window_q8_bf16", "e4m3"), ("decode_window_i8_bf16", "int8")])
def test_decode_window_quantized_cache(name, fmt):
    """The windowed decode over a quantized cache (f8 or int8) at full size through its
    entry point: the appended codes bit for bit, sampled rows against the oracle."""
    from sliding_window_gb300 import gqa
    w = WORKLOADS[name]
    c = make_case(w, device="cpu")
    k8, v8 = c.extra["k8"].numpy().copy(), c.extra["v8"].numpy().copy()
    ks, vs = c.extra["k_scale"].numpy(), c.extra["v_scale"].numpy()
    p = gqa.params_from_dict(c.params)
    out = torch.full(c.q.shape, float("nan"), dtype=c.q.dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(max(16, gqa.gqa_workspace_bytes(p)), dtype=torch.uint8, device="cuda")
    gk, gv = torch.from_numpy(k8).cuda(), torch.from_numpy(v8).cuda()
    fn = gqa.gqa_attention_decode_q8 if fmt == "e4m3" else gqa.gqa_attention_decode_i8
    gqa.check(fn(p, c.q.cuda(), c.k.cuda(), c.v.cuda(), c.seqlens_k.cuda(), None, None, None,
                 c.extra["k_scale"].cuda(), c.extra["v_scale"].cuda(), out, gk, gv, ws, st), fmt)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rk, rv = k8.copy(), v8.copy()
    q_rot, s = oracle.rope_append_q8(c.params, storage(c.q), storage(c.k), storage(c.v), rk, rv,
                                     c.seqlens_k.numpy(), ks, vs, fmt=fmt)
    assert s == 0
    np.testing.assert_array_equal(gk.cpu().numpy(), rk)
    np.testing.assert_array_equal(gv.cpu().numpy(), rv)
    rows = sample_rows(w)
    ref = oracle.attention_q8(c.params, q_rot, rk, rv, c.seqlens_k.numpy(), ks, vs, None, rows=rows, fmt=fmt)
    assert_close(out_rows(out, c, rows), ref, w.dtype, w.name)
