"""Quantized KV caches with one scale per kv head for K and V, in both one-byte formats (f8
E4M3 and int8): the split-KV decode kernel (D = Dv = 128; code tiles by TMA, converted to
f16 MMA operands) and the RoPE/append + CUDA-core kernels (every other shape, prefill
included), against the fp64 oracle on the same codes: the appended codes bit for bit, the
outputs within the dtype's tolerance."""
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


FMTS = ["e4m3", "int8"]


def encode(x, fmt):
    return oracle.encode_e4m3(x) if fmt == "e4m3" else oracle.encode_i8(x).view(np.uint8)


def q8_case(mode, dtype, D, Dv, G, curr, cap, lo, hi, W, softcap=0.0, sink="head", rotary=0, B=3, Hkv=2, seed=0,
            seqlens=None, fmt="e4m3"):
    w = Workload("q8", 1300 + seed, mode, dtype, B, G * Hkv, Hkv, D, curr, cap, lo, hi, windows=(W,),
                 softcap=softcap, head_sink=sink == "head", smooth_softmax=int(sink == "smooth"), do_rotary=rotary,
                 rope_len=cap + 8 if rotary else 0, v_head_dim=Dv)
    c = make_case(w, seed_offset=seed, seqlens=seqlens)
    rng = np.random.default_rng(seed)
    # int8: scales near max|x| / 127 for N(0,1) rows, so that a few codes saturate
    lo_s, hi_s = (0.004, 0.03) if fmt == "e4m3" else (0.02, 0.04)
    ks = rng.uniform(lo_s, hi_s, size=Hkv).astype(np.float32)
    vs = rng.uniform(lo_s, hi_s, size=Hkv).astype(np.float32)
    # the past as codes of the drawn rows; stale slots hold random codes (E4M3 NaN codes among them)
    k8 = rng.integers(0, 256, size=(B, Hkv, cap, D), dtype=np.uint8)
    v8 = rng.integers(0, 256, size=(B, Hkv, cap, Dv), dtype=np.uint8)
    dec = (lambda a: a) if dtype == "f32" else (lambda a: oracle.decode(a, dtype))
    pk, pv = dec(storage(c.past_k)).astype(np.float32), dec(storage(c.past_v)).astype(np.float32)
    for b, past in enumerate(c.seqlens_k.tolist()):
        for h in range(Hkv):
            k8[b, h, :past] = encode(pk[b, h, :past] / ks[h], fmt)
            v8[b, h, :past] = encode(pv[b, h, :past] / vs[h], fmt)
    return c, k8, v8, ks, vs


def run_q8(c, k8, v8, ks, vs, attend_only=False, fmt="e4m3"):
    from sliding_window_gb300 import gqa
    d = lambda x: None if x is None else x.cuda()  # noqa: E731
    p = gqa.params_from_dict(c.params if not attend_only else dict(c.params, do_rotary=0))
    B, L, Hq = c.w.batch, c.w.q_len, c.w.q_heads
    Dv = c.w.v_head_dim or c.w.head_dim
    out = torch.full((B, L, Hq * Dv), float("nan"), dtype=c.q.dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(max(16, gqa.gqa_workspace_bytes(p)), dtype=torch.uint8, device="cuda")
    gk, gv = torch.from_numpy(k8.copy()).cuda(), torch.from_numpy(v8.copy()).cuda()
    sfx = "q8" if fmt == "e4m3" else "i8"
    fn = getattr(gqa, "gqa_attention_%s_%s" % ("decode" if c.w.mode == "decode" else "prefill", sfx))
    k, v = (None, None) if attend_only else (d(c.k), d(c.v))
    gqa.check(fn(p, d(c.q), k, v, d(c.seqlens_k), None if attend_only else d(c.cos),
                 None if attend_only else d(c.sin), d(c.head_sink), torch.from_numpy(ks).cuda(),
                 torch.from_numpy(vs).cuda(), out, gk, gv, ws, st), "q8")
    torch.cuda.synchronize()
    return out, gk.cpu().numpy(), gv.cpu().numpy(), int(st.item())


def oracle_q8(c, k8, v8, ks, vs, fmt="e4m3"):
    pk, pv = k8.copy(), v8.copy()
    cs = None if c.cos is None else storage(c.cos)
    sn = None if c.sin is None else storage(c.sin)
    q_rot, st = oracle.rope_append_q8(c.params, storage(c.q), storage(c.k), storage(c.v), pk, pv,
                                      c.seqlens_k.numpy(), ks, vs, cs, sn, fmt=fmt)
    sink = None if c.head_sink is None else c.head_sink.numpy()
    return oracle.attention_q8(c.params, q_rot, pk, pv, c.seqlens_k.numpy(), ks, vs, sink, fmt=fmt), pk, pv, st


def check(c, k8, v8, ks, vs, what, fmt="e4m3"):
    out, gk, gv, st = run_q8(c, k8, v8, ks, vs, fmt=fmt)
    ref, rk, rv, s = oracle_q8(c, k8, v8, ks, vs, fmt=fmt)
    assert st == 0 and s == 0
    np.testing.assert_array_equal(gk, rk)
    np.testing.assert_array_equal(gv, rv)
    assert_close(out_rows(out, c), ref, c.w.dtype, what)


SPLIT = list(itertools.product(FMTS, ["bf16", "f16"], [(4, 1), (2, 3), (4, 3), (8, 4)],
                               [(3000, 300), (20000, -1)]))


@pytest.mark.parametrize("fmt,dtype,gc,capw", SPLIT)
def test_split_decode_q8(fmt, dtype, gc, capw):
    G, curr = gc
    cap, W = capw
    seed = zlib.crc32(repr((dtype, gc, capw)).encode()) % 37
    c, k8, v8, ks, vs = q8_case("decode", dtype, 128, 128, G, curr, cap, 100, cap - curr, W,
                                softcap=30.0 if seed % 2 else 0.0, sink=("head", "smooth", "none")[seed % 3],
                                rotary=int(seed % 3 == 0), seed=seed, fmt=fmt)
    check(c, k8, v8, ks, vs, "split %s %s" % (fmt, (dtype, gc, capw)), fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_split_decode_q8_attention_only(fmt):
    c, k8, v8, ks, vs = q8_case("decode", "bf16", 128, 128, 4, 1, 2000, 50, 1990, 512, seed=3, fmt=fmt)
    # the step's rows appended first by the full call, then attention alone over them
    _, gk, gv, st = run_q8(c, k8, v8, ks, vs, fmt=fmt)
    assert st == 0
    out, _, _, st = run_q8(c, gk, gv, ks, vs, attend_only=True, fmt=fmt)
    ref, *_ = oracle_q8(c, k8, v8, ks, vs, fmt=fmt)
    assert st == 0
    assert_close(out_rows(out, c), ref, "bf16", "split %s attention only" % fmt)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("mode,dtype,D,Dv,G,curr", [
    ("decode", "f32", 64, 64, 4, 1), ("decode", "bf16", 128, 64, 4, 1), ("decode", "bf16", 128, 128, 16, 4),
    ("prefill", "bf16", 128, 128, 2, 150), ("prefill", "f32", 64, 64, 2, 70), ("prefill", "f16", 64, 128, 2, 90)])
def test_cuda_core_q8(fmt, mode, dtype, D, Dv, G, curr):
    past = 900 if mode == "decode" else 40
    c, k8, v8, ks, vs = q8_case(mode, dtype, D, Dv, G, curr, past + curr + 30, past, past, 200, softcap=20.0,
                                rotary=1, B=2, seed=5, fmt=fmt)
    check(c, k8, v8, ks, vs, "cuda-core %s %s" % (fmt, (mode, dtype, D, Dv, G, curr)), fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_q8_rejected_sequence(fmt):
    seq = np.array([100, 999], np.int32)  # 999 + 2 > 1000
    c, k8, v8, ks, vs = q8_case("decode", "bf16", 128, 128, 4, 2, 1000, 0, 998, -1, seed=6, B=2, seqlens=seq,
                                fmt=fmt)
    out, gk, gv, st = run_q8(c, k8, v8, ks, vs, fmt=fmt)
    assert st & 1
    o = out_rows(out, c)
    assert np.all(o[1] == 0.0) and np.all(np.isfinite(o[0]))
    np.testing.assert_array_equal(gk[1], k8[1])
    np.testing.assert_array_equal(gv[1], v8[1])


@pytest.mark.parametrize("mode,G,curr", [("decode", 4, 1), ("decode", 4, 3), ("prefill", 2, 40)])
def test_i8_append_saturates_and_maps_nan_to_zero(mode, G, curr):
    """New rows holding +-inf, NaN and values far past the scale: the split kernel's fused
    append (decode) and the RoPE/append kernel (prefill) write the oracle's codes bit for
    bit (127 / -128 for the infinities and the large values, 0 for NaN)."""
    past = 700
    c, k8, v8, ks, vs = q8_case(mode, "bf16", 128, 128, G, curr, past + curr + 20, past, past, 256, seed=7, B=2,
                                fmt="int8")
    specials = torch.tensor([float("inf"), float("-inf"), float("nan"), 1e6, -1e6, 3.0e3], dtype=torch.float32)
    for t in (c.k, c.v):
        flat = t.view(-1)
        idx = torch.arange(0, flat.numel(), 97)
        flat[idx] = specials[torch.arange(idx.numel()) % specials.numel()].to(t.dtype)
    out, gk, gv, st = run_q8(c, k8, v8, ks, vs, fmt="int8")
    ref, rk, rv, s = oracle_q8(c, k8, v8, ks, vs, fmt="int8")
    assert st == 0 and s == 0
    np.testing.assert_array_equal(gk, rk)
    np.testing.assert_array_equal(gv, rv)
    codes = np.concatenate([rk[b, :, past:past + curr].ravel() for b in range(2)]).view(np.int8)
    assert (codes == 127).any() and (codes == -128).any()
    assert_close(out_rows(out, c), ref, "bf16", "int8 specials %s" % mode)
