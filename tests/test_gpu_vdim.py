"""A V head dimension that differs from the Q/K one (onnx-light-cpu "Attention Kernel
Design", "Layouts and semantics"): the split-KV decode (cluster and ticket combines, with
and without a mask), the tensor-core prefill, and the CUDA-core kernel, against the fp64
oracle on the same rounded inputs; the appended K and V rows bit for bit."""
import itertools
import zlib

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, oracle_ref, out_rows, run_gpu
from helpers import storage
from sliding_window_gb300.inputs import Workload, make_case

pytestmark = pytest.mark.gpu

DIMS = [(128, 64), (64, 128)]


def case(mode, dtype, D, Dv, G, curr, cap, past_lo, past_hi, W, sink="head", softcap=0.0, rotary=0, B=3, Hkv=2,
         seed=0):
    w = Workload("vdim", 1100 + seed, mode, dtype, B, G * Hkv, Hkv, D, curr, cap, past_lo, past_hi, windows=(W,),
                 softcap=softcap, head_sink=sink == "head", smooth_softmax=int(sink == "smooth"), do_rotary=rotary,
                 rope_len=cap + 8 if rotary else 0, v_head_dim=Dv)
    return make_case(w, seed_offset=seed, garbage="nonfinite")


def check(c, mode, dtype, what, separate=False):
    r = run_gpu(c, mode, separate_present=separate)
    assert r["status"] == 0
    ref, pk, pv, st = oracle_ref(c)
    assert st == 0
    for b, past in enumerate(c.seqlens_k.tolist()):
        sl = slice(0, past + c.w.q_len)
        np.testing.assert_array_equal(storage(r["present_k"][b, :, sl]), pk[b, :, sl])
        np.testing.assert_array_equal(storage(r["present_v"][b, :, sl]), pv[b, :, sl])
    assert_close(out_rows(r["out"], c), ref, dtype, what)


DECODE = list(itertools.product(["bf16", "f16"], DIMS, [(4, 1), (2, 3), (4, 3), (8, 4)], [(3000, 300), (20000, -1)]))


@pytest.mark.parametrize("dtype,dims,gc,capw", DECODE)
def test_split_decode_vdim(dtype, dims, gc, capw):
    """(G, curr) = (4, 1) and (8, 4): 4 and 32 rows per group; a 3000-slot cache with a
    window (cluster combine) and a 20000-slot cache without (ticket combine)."""
    D, Dv = dims
    G, curr = gc
    cap, W = capw
    seed = zlib.crc32(repr((dtype, dims, gc, capw)).encode()) % 41
    c = case("decode", dtype, D, Dv, G, curr, cap, 100, cap - curr, W, sink=("head", "smooth", "none")[seed % 3],
             softcap=20.0 if seed % 2 else 0.0, rotary=int(seed % 3 == 0), seed=seed)
    check(c, "decode", dtype, "decode vdim %s" % ((dtype, dims, gc, capw),))


@pytest.mark.parametrize("dims,separate", list(itertools.product(DIMS, [False, True])))
def test_decode_vdim_separate_past(dims, separate):
    D, Dv = dims
    c = case("decode", "bf16", D, Dv, 4, 2, 1500, 10, 1400, 512, rotary=1, seed=5)
    check(c, "decode", "bf16", "decode vdim separate=%s" % separate, separate=separate)


@pytest.mark.parametrize("dims,kind", list(itertools.product(DIMS, ["bool", "add"])))
def test_masked_decode_vdim(dims, kind):
    from sliding_window_gb300 import gqa
    D, Dv = dims
    c = case("decode", "bf16", D, Dv, 4, 1, 2500, 100, 2400, -1, seed=6)
    B, Hq, cap = c.w.batch, c.w.q_heads, c.w.cap
    rng = np.random.default_rng(6)
    mask = (rng.random((B, 1, 1, cap)) < 0.8).astype(np.uint8) if kind == "bool" else \
        oracle.encode(rng.standard_normal((B, Hq, 1, cap)), "bf16")
    mt = torch.from_numpy(mask)
    if kind == "add":
        mt = mt.view(torch.int16).view(torch.bfloat16)
    mt = mt.cuda()
    m = gqa.mask_from_tensor(mt, gqa.MASK_KEEP if kind == "bool" else gqa.MASK_ADD)
    p = gqa.params_from_dict(c.params)
    d = lambda x: None if x is None else x.cuda()  # noqa: E731
    pk, pv = d(c.past_k), d(c.past_v)
    out = torch.full((B, 1, Hq * Dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(max(16, gqa.gqa_workspace_bytes(p)), dtype=torch.uint8, device="cuda")
    gqa.check(gqa.gqa_attention_decode_masked(p, m, d(c.q), d(c.k), d(c.v), pk, pv, d(c.seqlens_k), None, None,
                                              d(c.head_sink), out, pk, pv, ws, st), "masked vdim")
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    q_rot, rk, rv, _ = oracle.rope_append(c.params, storage(c.q), storage(c.k), storage(c.v), storage(c.past_k),
                                          storage(c.past_v), c.seqlens_k.numpy())
    ref = oracle.attention_masked(c.params, q_rot, rk, rv, c.seqlens_k.numpy(), mask, kind, c.head_sink.numpy())
    assert_close(out_rows(out, c), ref, "bf16", "masked decode vdim %s" % kind)


PREFILL = list(itertools.product(["bf16", "f16"], DIMS, [(300, 0, -1), (300, 0, 100), (200, 777, 256)],
                                 [0.0, 30.0]))


@pytest.mark.parametrize("dtype,dims,spw,softcap", PREFILL)
def test_prefill_vdim(dtype, dims, spw, softcap):
    D, Dv = dims
    S, past, W = spw
    seed = zlib.crc32(repr((dtype, dims, spw, softcap)).encode()) % 43
    c = case("prefill", dtype, D, Dv, 2, S, past + S + 29, past, past, W, sink=("head", "smooth", "none")[seed % 3],
             softcap=softcap, rotary=int(seed % 2 == 0), B=2, seed=seed)
    check(c, "prefill", dtype, "prefill vdim %s" % ((dtype, dims, spw, softcap),))


@pytest.mark.parametrize("mode,dims", list(itertools.product(["prefill", "decode"], DIMS)))
def test_cuda_core_kernel_vdim(mode, dims):
    """f32 (the CUDA-core kernel) in both modes, and a bf16 decode with 64 rows per group."""
    D, Dv = dims
    S, past = (130, 60) if mode == "prefill" else (1, 900)
    c = case(mode, "f32", D, Dv, 4, S, past + S + 9, past, past, 300, softcap=10.0, seed=7, B=2)
    check(c, mode, "f32", "f32 %s vdim" % mode)
    if mode == "decode":
        c = case("decode", "bf16", D, Dv, 16, 4, 2000, 500, 1990, 700, seed=8, B=2)
        check(c, "decode", "bf16", "decode vdim G=16")
