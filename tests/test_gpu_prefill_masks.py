"""Attention masks on prefill and on the CUDA-core path (onnx-light-cpu "Attention Kernel
Design", "Layouts and semantics": boolean and FLOAT additive broadcast masks with the
bottom-right band; tract PR #2645 "What changed": attention_bias summed with the band).
The tensor-core prefill stages 16-byte aligned masks by TMA; other masks, f32 and decode
shapes outside the split kernel run the CUDA-core kernel.  Parity with the fp64 masked
oracle on the same rounded inputs."""
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


def case(mode, dtype, D, G, S, past, W, sink="head", softcap=0.0, rotary=0, B=2, Hkv=2, seed=0, cap=None):
    cap = cap or past + S + 21
    w = Workload("pmask", 900 + seed, mode, dtype, B, G * Hkv, Hkv, D, S, cap, past, past, windows=(W,),
                 softcap=softcap, head_sink=sink == "head", smooth_softmax=int(sink == "smooth"), do_rotary=rotary,
                 rope_len=cap + 8 if rotary else 0)
    return make_case(w, seed_offset=seed)


def draw_mask(kind, shape, dtype, rng, keep=0.8):
    if kind == "bool":
        return (rng.random(shape) < keep).astype(np.uint8)
    vals = rng.standard_normal(shape) * 2.0
    return vals.astype(np.float32) if dtype == "f32" else oracle.encode(vals, dtype)


def to_device_mask(mask_np, kind, dtype):
    mt = torch.from_numpy(np.ascontiguousarray(mask_np))
    if kind != "bool" and dtype != "f32":
        mt = mt.view(torch.int16).view(torch.float16 if dtype == "f16" else torch.bfloat16)
    return mt.cuda()


def run(c, mask_np, kind, fn="gqa_attention_prefill_masked", padded_keys=None):
    """The masked entry point (fn) with mask_np, or the unmasked one for mask_np None.
    padded_keys: store the mask in rows of that many keys (a wider allocation, sliced)."""
    from sliding_window_gb300 import gqa
    dt = c.params["dtype"]
    d = lambda x: None if x is None else x.cuda()  # noqa: E731
    p = gqa.params_from_dict(c.params)
    pk, pv = d(c.past_k), d(c.past_v)
    out = torch.full(c.q.shape, float("nan"), dtype=c.q.dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(max(16, gqa.gqa_workspace_bytes(p)), dtype=torch.uint8, device="cuda")
    args = (d(c.q), d(c.k), d(c.v), pk, pv, d(c.seqlens_k), d(c.cos), d(c.sin), d(c.head_sink), out, pk, pv, ws, st)
    if mask_np is None:
        plain = fn.replace("_masked", "")
        gqa.check(getattr(gqa, plain)(p, *args), plain)
    else:
        mt = to_device_mask(mask_np, kind, dt)
        if padded_keys is not None:
            wide = torch.zeros(mt.shape[:3] + (padded_keys,), dtype=mt.dtype, device="cuda")
            wide[..., : mt.shape[3]] = mt
            mt = wide[..., : mt.shape[3]]
        m = gqa.mask_from_tensor(mt, gqa.MASK_KEEP if kind == "bool" else gqa.MASK_ADD)
        gqa.check(getattr(gqa, fn)(p, m, *args), fn)
    torch.cuda.synchronize()
    return out, pk, pv, int(st.item())


def oracle_masked(c, mask_np, kind):
    cs = None if c.cos is None else storage(c.cos)
    sn = None if c.sin is None else storage(c.sin)
    args = (storage(c.q), storage(c.k), storage(c.v), storage(c.past_k), storage(c.past_v), c.seqlens_k.numpy(), cs, sn)
    q_rot, pk, pv, st = oracle.rope_append(c.params, *args)
    sink = None if c.head_sink is None else c.head_sink.numpy()
    return oracle.attention_masked(c.params, q_rot, pk, pv, c.seqlens_k.numpy(), mask_np, kind, sink), pk, pv, st


def mask_shape(shape, B, Hq, S, keys):
    return {"full": (B, Hq, S, keys), "b1ik": (B, 1, S, keys), "11ik": (1, 1, S, keys),
            "b11k": (B, 1, 1, keys)}[shape]


SWEEP = list(itertools.product(
    ["bf16", "f16"],
    [(128, 2), (64, 4)],                                  # (D, G)
    [(300, 0, -1), (300, 0, 100), (200, 777, 256)],       # (prompt, past, window): several q tiles, ragged tail
    ["bool", "add"],
    ["full", "b1ik", "11ik", "b11k"],                     # [B,Hq,L,K] / [B,1,L,K] / [1,1,L,K] / [B,1,1,K]
))


@pytest.mark.parametrize("dtype,dg,spw,kind,shape", SWEEP)
def test_masked_prefill_parity(dtype, dg, spw, kind, shape):
    D, G = dg
    S, past, W = spw
    seed = zlib.crc32(repr((dtype, dg, spw, kind, shape)).encode()) % 61
    c = case("prefill", dtype, D, G, S, past, W, rotary=int(seed % 2 == 0), softcap=30.0 if seed % 3 == 0 else 0.0,
             sink=("head", "smooth", "none")[seed % 3], seed=seed)
    B, Hq = c.q.shape[0], c.params["q_heads"]
    keys = -(-(past + S) // 16) * 16  # rows of 16-byte multiples: the TMA path
    mask = draw_mask(kind, mask_shape(shape, B, Hq, S, keys), dtype, np.random.default_rng(seed))
    out, pk, pv, st = run(c, mask, kind)
    ref, rk, rv, s = oracle_masked(c, mask, kind)
    assert st == 0 and s == 0
    np.testing.assert_array_equal(storage(pk), rk)
    np.testing.assert_array_equal(storage(pv), rv)
    assert_close(out_rows(out, c), ref, dtype, "masked prefill %s" % ((dtype, dg, spw, kind, shape),))


@pytest.mark.parametrize("kind,softcap", [("bool", 0.0), ("bool", 20.0), ("add", 0.0), ("add", 20.0)])
def test_unaligned_mask_runs_the_cuda_core_kernel(kind, softcap):
    """Rows of past + S + 3 keys are not 16-byte multiples: same results within tolerance."""
    c = case("prefill", "bf16", 128, 4, 260, 40, 120, softcap=softcap, seed=11)
    B, Hq = c.q.shape[0], c.params["q_heads"]
    mask = draw_mask(kind, (B, 1, 260, 40 + 260 + 3), "bf16", np.random.default_rng(11))
    out, *_, st = run(c, mask, kind)
    ref, *_ = oracle_masked(c, mask, kind)
    assert st == 0
    assert_close(out_rows(out, c), ref, "bf16", "unaligned %s" % kind)


@pytest.mark.parametrize("kind", ["bool", "add"])
def test_padded_rows_take_the_tma_path(kind):
    """A mask allocated with wider rows (stride_i = 512 keys) and sliced to the keys in use."""
    c = case("prefill", "f16", 128, 2, 333, 0, -1, softcap=0.0, seed=12)
    B = c.q.shape[0]
    mask = draw_mask(kind, (B, 1, 333, 333), "f16", np.random.default_rng(12))
    out, *_, st = run(c, mask, kind, padded_keys=512)
    ref, *_ = oracle_masked(c, mask, kind)
    assert st == 0
    assert_close(out_rows(out, c), ref, "f16", "padded %s" % kind)


@pytest.mark.parametrize("mode,kind", list(itertools.product(["prefill", "decode"], ["bool", "add"])))
def test_f32_masks_on_the_cuda_core_kernel(mode, kind):
    S, past = (130, 50) if mode == "prefill" else (1, 900)
    c = case(mode, "f32", 64, 4, S, past, 300, sink="head", softcap=0.0 if kind == "bool" else 15.0, seed=13)
    B, Hq = c.q.shape[0], c.params["q_heads"]
    mask = draw_mask(kind, (B, Hq, S, past + S), "f32", np.random.default_rng(13))
    fn = "gqa_attention_prefill_masked" if mode == "prefill" else "gqa_attention_decode_masked"
    out, *_, st = run(c, mask, kind, fn=fn)
    ref, *_ = oracle_masked(c, mask, kind)
    assert st == 0
    assert_close(out_rows(out, c), ref, "f32", "f32 %s %s" % (mode, kind))


def test_decode_mask_outside_the_split_kernel():
    """64 query rows per kv head at D = 128 (G = 16, 4 new tokens): the CUDA-core kernel."""
    c = case("decode", "bf16", 128, 16, 4, 1500, 700, sink="smooth", seed=14)
    B, Hq = c.q.shape[0], c.params["q_heads"]
    mask = draw_mask("add", (B, Hq, 4, 1504), "bf16", np.random.default_rng(14))
    out, *_, st = run(c, mask, "add", fn="gqa_attention_decode_masked")
    ref, *_ = oracle_masked(c, mask, "add")
    assert st == 0
    assert_close(out_rows(out, c), ref, "bf16", "decode G=16 masked")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_additive_minus_inf_equals_key_removal(dtype):
    """Additive 0 / -inf (no softcap) removes the same keys as the boolean mask, bit for bit
    on the same kernel; a row with every key removed gives zeros."""
    c = case("prefill", dtype, 128 if dtype != "f32" else 64, 2, 200, 0, -1, sink="none", seed=15)
    B, Hq = c.q.shape[0], c.params["q_heads"]
    rng = np.random.default_rng(15)
    keep = (rng.random((B, Hq, 200, 208)) < 0.5).astype(np.uint8)
    keep[1, 1, 37, :] = 0
    keep[0, 2, 150:170, :] = 0
    vals = np.where(keep != 0, 0.0, -np.inf)
    add = vals.astype(np.float32) if dtype == "f32" else oracle.encode(vals, dtype)
    a, *_, sa = run(c, add, "add")
    b, *_, sb = run(c, keep, "bool")
    assert sa == 0 and sb == 0
    assert torch.equal(a.view(torch.int16) if dtype != "f32" else a, b.view(torch.int16) if dtype != "f32" else b)
    o = out_rows(a, c)
    assert np.all(o[1, 37, 1] == 0.0) and np.all(o[0, 150:170, 2] == 0.0)
    ref, *_ = oracle_masked(c, keep, "bool")
    assert_close(o, ref, dtype, "-inf mask")


@pytest.mark.parametrize("kind", ["bool", "add"])
def test_neutral_prefill_mask_gives_the_unmasked_bits(kind):
    """Without a window the masked kernel visits the same key tiles in the same order."""
    c = case("prefill", "bf16", 128, 4, 290, 0, -1, sink="head", seed=16)
    neutral = np.ones((1, 1, 290, 304), np.uint8) if kind == "bool" else np.zeros((1, 1, 290, 304), np.uint16)
    a, *_ = run(c, neutral, kind)
    b, *_ = run(c, None, kind)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_prefill_mask_shorter_than_a_sequence_rejects_it():
    c = case("prefill", "bf16", 128, 2, 100, 300, -1, seed=17)
    mask = np.ones((1, 1, 100, 304), np.uint8)  # 304 keys < past + S = 400
    out, *_, st = run(c, mask, "bool")
    assert st & 1
    assert np.all(out_rows(out, c) == 0.0)


@pytest.mark.parametrize("kind,shape,softcap", [("bool", "b1ik", 0.0), ("add", "b1ik", 25.0), ("add", "full", 0.0),
                                                ("add", "b11k", 25.0)])
def test_odd_group_size(kind, shape, softcap):
    """G = 3: the last CTA of each kv group holds one q head (a shared mask tile read by one
    softmax warpgroup)."""
    c = case("prefill", "bf16", 128, 3, 200, 64, 150, softcap=softcap, sink="smooth", seed=18)
    B, Hq = c.q.shape[0], c.params["q_heads"]
    mask = draw_mask(kind, mask_shape(shape, B, Hq, 200, 272), "bf16", np.random.default_rng(18))
    out, *_, st = run(c, mask, kind)
    ref, *_ = oracle_masked(c, mask, kind)
    assert st == 0
    assert_close(out_rows(out, c), ref, "bf16", "G=3 %s %s" % (kind, shape))
