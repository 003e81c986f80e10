"""Attention masks in the split-KV decode kernel (onnx-light-cpu "Attention Kernel Design",
"Layouts and semantics": boolean and FLOAT additive broadcast masks with the band; tract PR
#2645 "What changed": attention_bias summed with the band).  Parity with the fp64 masked
oracle on the same rounded inputs; masks that change nothing give the unmasked kernel's
bits; a mask too short for a sequence rejects it."""
import itertools
import zlib

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, out_rows
from helpers import storage
from sliding_window_gb300.inputs import Workload, make_case

pytestmark = pytest.mark.gpu


def case(dtype, D, G, curr, cap, W, sink="head", softcap=0.0, rotary=0, B=3, Hkv=2, seed=0, ring=0, lo=0, hi=None):
    w = Workload("mask", 700 + seed, "decode", dtype, B, G * Hkv, Hkv, D, curr, cap, lo,
                 hi if hi is not None else cap - curr, windows=(W,), softcap=softcap, head_sink=sink == "head",
                 smooth_softmax=int(sink == "smooth"), do_rotary=rotary, rope_len=(hi or cap) + curr + 8 if rotary else 0,
                 kv_ring=ring)
    return make_case(w, seed_offset=seed)


def draw_mask(kind, shape, dtype, rng):
    if kind == "bool":
        return (rng.random(shape) < 0.8).astype(np.uint8)
    vals = rng.standard_normal(shape) * 2.0
    return oracle.encode(vals, dtype)


def run(c, mask_np, kind, masked=True):
    from sliding_window_gb300 import gqa
    dt = c.params["dtype"]
    d = lambda x: None if x is None else x.cuda()  # noqa: E731
    p = gqa.params_from_dict(c.params)
    pk, pv = d(c.past_k), d(c.past_v)
    out = torch.full(c.q.shape, float("nan"), dtype=c.q.dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(max(16, gqa.gqa_workspace_bytes(p)), dtype=torch.uint8, device="cuda")
    if masked:
        mt = torch.from_numpy(np.ascontiguousarray(mask_np))
        if kind != "bool":
            mt = mt.view(torch.int16).view(torch.float16 if dt == "f16" else torch.bfloat16)
        mt = mt.cuda()
        m = gqa.mask_from_tensor(mt, gqa.MASK_KEEP if kind == "bool" else gqa.MASK_ADD)
        gqa.check(gqa.gqa_attention_decode_masked(p, m, d(c.q), d(c.k), d(c.v), pk, pv, d(c.seqlens_k), d(c.cos),
                                                  d(c.sin), d(c.head_sink), out, pk, pv, ws, st), "masked")
    else:
        gqa.check(gqa.gqa_attention_decode(p, d(c.q), d(c.k), d(c.v), pk, pv, d(c.seqlens_k), d(c.cos), d(c.sin),
                                           d(c.head_sink), out, pk, pv, ws, st), "decode")
    torch.cuda.synchronize()
    return out, pk, pv, int(st.item())


def oracle_masked(c, mask_np, kind):
    cs = None if c.cos is None else storage(c.cos)
    sn = None if c.sin is None else storage(c.sin)
    args = (storage(c.q), storage(c.k), storage(c.v), storage(c.past_k), storage(c.past_v), c.seqlens_k.numpy(), cs, sn)
    q_rot, pk, pv, st = oracle.rope_append(c.params, *args)
    sink = None if c.head_sink is None else c.head_sink.numpy()
    return oracle.attention_masked(c.params, q_rot, pk, pv, c.seqlens_k.numpy(), mask_np, kind, sink), pk, pv, st


SWEEP = list(itertools.product(
    ["bf16", "f16"],
    [(128, 8, 1), (128, 4, 4), (64, 16, 2)],                    # (D, G, curr)
    [(3000, -1), (3000, 200)],                                  # (cap, window)
    ["bool", "add"],
    ["full", "b1ik", "11ik"],                                   # mask shape: [B,Hq,L,K] / [B,1,L,K] / [1,1,L,K]
))


@pytest.mark.parametrize("dtype,dgc,capw,kind,shape", SWEEP)
def test_masked_decode_parity(dtype, dgc, capw, kind, shape):
    D, G, curr = dgc
    cap, W = capw
    seed = zlib.crc32(repr((dtype, dgc, capw, kind, shape)).encode()) % 53
    c = case(dtype, D, G, curr, cap, W, rotary=int(seed % 2 == 0), softcap=25.0 if seed % 3 == 0 else 0.0,
             sink=("head", "smooth", "none")[seed % 3], seed=seed)
    B, Hq = c.q.shape[0], c.params["q_heads"]
    full = {"full": (B, Hq, curr, cap), "b1ik": (B, 1, curr, cap), "11ik": (1, 1, curr, cap)}[shape]
    mask = draw_mask(kind, full, dtype, np.random.default_rng(seed))
    out, pk, pv, st = run(c, mask, kind)
    ref, rk, rv, s = oracle_masked(c, mask, kind)
    assert st == 0 and s == 0
    np.testing.assert_array_equal(storage(pk), rk)
    np.testing.assert_array_equal(storage(pv), rv)
    assert_close(out_rows(out, c), ref, dtype, "masked %s" % ((dtype, dgc, capw, kind, shape),))


@pytest.mark.parametrize("kind", ["bool", "add"])
def test_neutral_mask_gives_the_unmasked_bits(kind):
    c = case("bf16", 128, 8, 2, 3000, 500, rotary=1, seed=9)
    neutral = np.ones((1, 1, 2, 3000), np.uint8) if kind == "bool" else np.zeros((1, 1, 2, 3000), np.uint16)
    a, *_ = run(c, neutral, kind)
    b, *_ = run(c, None, kind, masked=False)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_mask_shorter_than_a_sequence_rejects_it():
    c = case("bf16", 128, 8, 1, 3000, -1, seed=10, lo=100, hi=2900)
    seq = c.seqlens_k.numpy()
    keys = int(np.sort(seq)[1]) + 1  # covers the shortest sequence only
    mask = np.ones((1, 1, 1, keys), np.uint8)
    out, pk, pv, st = run(c, mask, "bool")
    assert st & 1
    o = out_rows(out, c)
    for b in range(3):
        if seq[b] + 1 > keys:
            assert np.all(o[b] == 0.0)
