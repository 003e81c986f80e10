"""Prefill, or a chunk of a prompt over a cache already filled, into the ring and paged
caches (OpenVINO PR #37423 "Sliding window": the rolling sliding_window_cache buffer;
ExecuTorch PR #21901 Summary: a cell cache whose slots belong to sequences).  The tensor-core
prefill reads the band as 128-position tiles (two pages, or a ring span that never
straddles the wrap) and the append kernel writes through the ring slots or the block table.
Parity with the fp64 ring / paged oracles on the same rounded inputs: the cache after the
step bit-exact, outputs within the bf16/f16 tolerance; chunks of 64 to 1024 tokens, rings
that have wrapped and rings that have not, windows across the past/current boundary, RoPE,
sinks, softcap, and a bad page that rejects only its sequence."""
import itertools
import zlib

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, oracle_ref, out_rows, run_gpu
from helpers import storage
from sliding_window_gb300.inputs import Workload, make_case
from test_gpu_paged import PAGE, oracle_paged, to_dev

pytestmark = pytest.mark.gpu


def ring_prefill_case(dtype, D, G, curr, cap, W, past_lo, past_hi, rotary=0, softcap=0.0, sink="head", B=2, Hkv=2,
                      seed=0):
    w = Workload("ringpf", 700 + seed, "prefill", dtype, B, G * Hkv, Hkv, D, curr, cap, past_lo, past_hi,
                 windows=(W,), softcap=softcap, head_sink=sink == "head", smooth_softmax=int(sink == "smooth"),
                 do_rotary=rotary, rope_len=past_hi + curr + 8 if rotary else 0, kv_ring=1)
    return make_case(w, seed_offset=seed)


RING = list(itertools.product(
    ["bf16", "f16"],
    [(128, 4), (64, 8)],                                  # (D, G)
    [(64, 4096, 4224), (300, 700, 1024), (1024, 1024, 2048), (200, 129, 384)],  # (chunk, window, ring slots)
    [(0, 40), (5000, 9000)],                              # past: ring not wrapped / wrapped
))


@pytest.mark.parametrize("dtype,dg,cwc,past", RING)
def test_ring_prefill_parity(dtype, dg, cwc, past):
    D, G = dg
    curr, W, cap = cwc
    lo, hi = past
    seed = zlib.crc32(repr((dtype, dg, cwc, past)).encode()) % 53
    c = ring_prefill_case(dtype, D, G, curr, cap, W, lo, hi, rotary=int(seed % 2 == 0),
                          softcap=30.0 if seed % 3 == 0 else 0.0, sink=("head", "smooth", "none")[seed % 3], seed=seed)
    r = run_gpu(c, "prefill")
    assert r["status"] == 0
    ref, pk, pv, st = oracle_ref(c)
    assert st == 0
    np.testing.assert_array_equal(storage(r["present_k"]), pk)
    np.testing.assert_array_equal(storage(r["present_v"]), pv)
    assert_close(out_rows(r["out"], c), ref, dtype, "ring prefill %s" % ((dtype, dg, cwc, past),))


def test_ring_chunked_prompt_matches_the_oracle_chunk_by_chunk():
    """A 1536-token prompt in six chunks of 256 through one ring of 1024 slots (window 700):
    after every chunk the GPU and oracle rings are bit-equal and the outputs agree."""
    from sliding_window_gb300 import gqa
    c = ring_prefill_case("bf16", 128, 4, 256, 1024, 700, 0, 0, rotary=1, seed=9)
    dev = torch.device("cuda:0")
    p = gqa.params_from_dict(dict(c.params, rope_len=2048))
    from sliding_window_gb300.inputs import rope_tables
    cos, sin = rope_tables(2048, 128, 10000.0, "bf16")
    ring_k, ring_v = c.past_k.to(dev), c.past_v.to(dev)
    hk, hv = storage(c.past_k), storage(c.past_v)
    ws = torch.zeros(max(16, gqa.gqa_workspace_bytes(p)), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    gen = torch.Generator().manual_seed(13)
    seq = torch.zeros(c.seqlens_k.shape, dtype=torch.int32)
    params = dict(c.params, rope_len=2048)
    for chunk in range(6):
        q = torch.randn(c.q.shape, generator=gen).to(c.q.dtype)
        k = torch.randn(c.k.shape, generator=gen).to(c.k.dtype)
        v = torch.randn(c.v.shape, generator=gen).to(c.v.dtype)
        out = torch.empty(q.shape, dtype=q.dtype, device=dev)
        gqa.check(gqa.gqa_attention_prefill(p, q.to(dev), k.to(dev), v.to(dev), ring_k, ring_v, seq.to(dev),
                                            cos.to(dev), sin.to(dev), c.head_sink.to(dev), out, ring_k, ring_v, ws,
                                            st), "ring prefill chunk")
        q_rot, hk, hv, s = oracle.rope_append_ring(params, storage(q), storage(k), storage(v), hk, hv, seq.numpy(),
                                                   storage(cos), storage(sin))
        ref = oracle.attention_ring(params, q_rot, hk, hv, seq.numpy(), c.head_sink.numpy())
        torch.cuda.synchronize()
        assert int(st.item()) == 0 and s == 0
        np.testing.assert_array_equal(storage(ring_k), hk)
        np.testing.assert_array_equal(storage(ring_v), hv)
        assert_close(out.cpu().to(torch.float64).numpy().reshape(ref.shape), ref, "bf16", "chunk %d" % chunk)
        seq = seq + 256


def paged_prefill_case(dtype, D, G, curr, cap, W, past_lo, past_hi, rotary=0, softcap=0.0, sink="head", B=2, Hkv=2,
                       seed=0, spare=7):
    w = Workload("pagedpf", 800 + seed, "prefill", dtype, B, G * Hkv, Hkv, D, curr, cap, past_lo, past_hi,
                 windows=(W,), softcap=softcap, head_sink=sink == "head", smooth_softmax=int(sink == "smooth"),
                 do_rotary=rotary, rope_len=cap + 8 if rotary else 0)
    c = make_case(w, seed_offset=seed)
    max_pages = cap // PAGE
    num_pages = B * max_pages + spare
    rng = np.random.default_rng(seed)
    table = rng.permutation(num_pages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)
    lk, lv = storage(c.past_k), storage(c.past_v)
    pool_k = np.zeros((num_pages, Hkv, PAGE, D), dtype=lk.dtype)
    pool_v = np.zeros_like(pool_k)
    for b in range(B):
        for n in range(max_pages):
            pool_k[table[b, n]] = lk[b, :, n * PAGE:(n + 1) * PAGE]
            pool_v[table[b, n]] = lv[b, :, n * PAGE:(n + 1) * PAGE]
    return c, table, num_pages, pool_k, pool_v


def run_prefill_paged(c, table, num_pages, pool_k, pool_v):
    from sliding_window_gb300 import gqa
    dt = c.params["dtype"]
    p = gqa.params_from_dict(c.params)
    dk, dv = to_dev(pool_k, dt), to_dev(pool_v, dt)
    tab = torch.from_numpy(table).cuda()
    out = torch.full(c.q.shape, float("nan"), dtype=c.q.dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(max(16, gqa.gqa_workspace_bytes(p)), dtype=torch.uint8, device="cuda")
    d = lambda x: None if x is None else x.cuda()  # noqa: E731
    gqa.check(gqa.gqa_attention_prefill_paged(p, d(c.q), d(c.k), d(c.v), d(c.seqlens_k), tab, num_pages, d(c.cos),
                                              d(c.sin), d(c.head_sink), out, dk, dv, ws, st), "prefill paged")
    torch.cuda.synchronize()
    return out, dk, dv, int(st.item())


PAGED = list(itertools.product(
    ["bf16", "f16"],
    [(128, 4), (64, 8)],                         # (D, G)
    [(64, -1), (200, 300), (700, 1000), (1024, -1)],  # (chunk, window)
    [(0, 0), (100, 1500)],                        # past: a first prompt / a chunk over a filled cache
))


@pytest.mark.parametrize("dtype,dg,cw,past", PAGED)
def test_paged_prefill_parity(dtype, dg, cw, past):
    D, G = dg
    curr, W = cw
    lo, hi = past
    cap = 2560
    seed = zlib.crc32(repr((dtype, dg, cw, past)).encode()) % 47
    c, table, npages, pk0, pv0 = paged_prefill_case(dtype, D, G, curr, cap, W, lo, hi, rotary=int(seed % 2 == 1),
                                                    softcap=30.0 if seed % 3 == 0 else 0.0,
                                                    sink=("head", "smooth", "none")[seed % 3], seed=seed)
    out, dk, dv, st = run_prefill_paged(c, table, npages, pk0, pv0)
    ref, pk, pv, s = oracle_paged(c, table, npages, pk0, pv0)
    assert st == 0 and s == 0
    np.testing.assert_array_equal(storage(dk), pk)
    np.testing.assert_array_equal(storage(dv), pv)
    B, L, Hq = c.q.shape[0], c.q.shape[1], c.params["q_heads"]
    assert_close(out.cpu().to(torch.float64).numpy().reshape(B, L, Hq, D), ref, dtype,
                 "paged prefill %s" % ((dtype, dg, cw, past),))


def test_paged_prefill_bad_page_rejects_only_its_sequence():
    c, table, npages, pk0, pv0 = paged_prefill_case("bf16", 128, 4, 300, 2048, -1, 500, 1500, seed=5)
    bad = table.copy()
    bad[1, 3] = npages + 11      # sequence 1 reads positions [192, 256) from a page that does not exist
    out, dk, dv, st = run_prefill_paged(c, bad, npages, pk0, pv0)
    ref, pk, pv, s = oracle_paged(c, bad, npages, pk0, pv0)
    assert st == 8 and s == 8
    np.testing.assert_array_equal(storage(dk), pk)  # nothing of sequence 1 appended
    o = out.cpu().to(torch.float64).numpy().reshape(ref.shape)
    assert np.all(o[1] == 0.0)
    assert_close(o[[0]], ref[[0]], "bf16")
