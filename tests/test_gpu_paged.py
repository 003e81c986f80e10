"""Paged KV cache on the GPU (ExecuTorch PR #21901 Summary: a cell cache whose slots belong
to sequences): a shared pool of 64-position pages, a shuffled block table per sequence, the
split-KV decode kernel reading and appending through the table.  Parity with the fp64
paged oracle on the same rounded inputs: the pool after the step bit-exact, outputs within
the bf16/f16 tolerance; bad page ids are reported and zero only their sequence."""
import itertools
import zlib

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close
from helpers import storage
from sliding_window_gb300.inputs import Workload, make_case

pytestmark = pytest.mark.gpu
PAGE = 64


def paged_case(dtype, D, G, curr, cap, W, sink="head", softcap=0.0, rotary=0, B=3, Hkv=2, seed=0, spare=5):
    w = Workload("pagedg", 600 + seed, "decode", dtype, B, G * Hkv, Hkv, D, curr, cap, 0, cap - curr, windows=(W,),
                 softcap=softcap, head_sink=sink == "head", smooth_softmax=int(sink == "smooth"), do_rotary=rotary,
                 rope_len=cap + 8 if rotary else 0)
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


def to_dev(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype != "f32":
        t = t.view(torch.int16).view(torch.float16 if dtype == "f16" else torch.bfloat16)
    return t.cuda()


def run_paged(c, table, num_pages, pool_k, pool_v, attend_only=False):
    from sliding_window_gb300 import gqa
    dt = c.params["dtype"]
    p = gqa.params_from_dict(c.params)
    dk, dv = to_dev(pool_k, dt), to_dev(pool_v, dt)
    tab = torch.from_numpy(table).cuda()
    out = torch.full(c.q.shape, float("nan"), dtype=c.q.dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(max(16, gqa.gqa_workspace_bytes(p)), dtype=torch.uint8, device="cuda")
    d = lambda x: None if x is None else x.cuda()  # noqa: E731
    q = d(c.q)
    if attend_only:
        q_rot, pk, pv, s = oracle.rope_append_paged(c.params, storage(c.q), storage(c.k), storage(c.v), pool_k, pool_v,
                                                    c.seqlens_k.numpy(), table, num_pages, PAGE,
                                                    None if c.cos is None else storage(c.cos),
                                                    None if c.sin is None else storage(c.sin))
        dk, dv = to_dev(pk, dt), to_dev(pv, dt)
        q = to_dev(q_rot.reshape(storage(c.q).shape), dt)
        p = gqa.params_from_dict(dict(c.params, do_rotary=0))
        gqa.check(gqa.gqa_attention_decode_paged(p, q, None, None, d(c.seqlens_k), tab, num_pages, None, None,
                                                 d(c.head_sink), out, dk, dv, ws, st), "paged attend-only")
    else:
        gqa.check(gqa.gqa_attention_decode_paged(p, q, d(c.k), d(c.v), d(c.seqlens_k), tab, num_pages, d(c.cos),
                                                 d(c.sin), d(c.head_sink), out, dk, dv, ws, st), "paged")
    torch.cuda.synchronize()
    return out, dk, dv, int(st.item())


def oracle_paged(c, table, num_pages, pool_k, pool_v):
    cs = None if c.cos is None else storage(c.cos)
    sn = None if c.sin is None else storage(c.sin)
    q_rot, pk, pv, st = oracle.rope_append_paged(c.params, storage(c.q), storage(c.k), storage(c.v), pool_k, pool_v,
                                                 c.seqlens_k.numpy(), table, num_pages, PAGE, cs, sn)
    sink = None if c.head_sink is None else c.head_sink.numpy()
    out = oracle.attention_paged(c.params, q_rot, pk, pv, c.seqlens_k.numpy(), table, num_pages, PAGE, sink)
    return out, pk, pv, st


SWEEP = list(itertools.product(
    ["bf16", "f16"],
    [(128, 8, 1), (128, 4, 4), (64, 8, 2), (128, 32, 1)],   # (D, G, curr)
    [(256, -1), (1024, 300), (1024, 1), (3072, -1)],         # (cap, window)
))


@pytest.mark.parametrize("dtype,dgc,capw", SWEEP)
def test_paged_decode_parity(dtype, dgc, capw):
    D, G, curr = dgc
    cap, W = capw
    seed = zlib.crc32(repr((dtype, dgc, capw)).encode()) % 61
    c, table, npages, pk0, pv0 = paged_case(dtype, D, G, curr, cap, W, rotary=int(seed % 2 == 0),
                                            softcap=30.0 if seed % 3 == 0 else 0.0, sink=("head", "smooth", "none")[seed % 3],
                                            seed=seed)
    out, dk, dv, st = run_paged(c, table, npages, pk0, pv0)
    ref, pk, pv, s = oracle_paged(c, table, npages, pk0, pv0)
    assert st == 0 and s == 0
    np.testing.assert_array_equal(storage(dk), pk)
    np.testing.assert_array_equal(storage(dv), pv)
    B, L, Hq = c.q.shape[0], c.q.shape[1], c.params["q_heads"]
    assert_close(out.cpu().to(torch.float64).numpy().reshape(B, L, Hq, D), ref, dtype, "paged %s" % ((dtype, dgc, capw),))


def test_paged_attend_only_matches_full_call():
    c, table, npages, pk0, pv0 = paged_case("bf16", 128, 4, 4, 1024, 500, rotary=1, seed=3)
    full, *_ = run_paged(c, table, npages, pk0, pv0)
    only, *_ = run_paged(c, table, npages, pk0, pv0, attend_only=True)
    assert torch.equal(full.view(torch.int16), only.view(torch.int16))


def test_bad_page_id_rejects_only_its_sequence():
    c, table, npages, pk0, pv0 = paged_case("bf16", 128, 8, 1, 1024, -1, seed=4)
    past = c.seqlens_k.numpy()
    bad = table.copy()
    bad[1, 0] = npages + 3        # sequence 1 reads position 0 from a page that does not exist
    out, dk, dv, st = run_paged(c, bad, npages, pk0, pv0)
    ref, pk, pv, s = oracle_paged(c, bad, npages, pk0, pv0)
    assert st == 8 and s == 8
    np.testing.assert_array_equal(storage(dk), pk)  # nothing of sequence 1 appended
    o = out.cpu().to(torch.float64).numpy().reshape(ref.shape)
    assert np.all(o[1] == 0.0)
    assert_close(o[[0, 2]], ref[[0, 2]], "bf16")
