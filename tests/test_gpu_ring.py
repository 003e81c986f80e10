"""Ring cache on the GPU (OpenVINO PR #37423 "Sliding window": the rolling
sliding_window_cache buffer): position p in slot p mod cap, decode through the split-KV
kernel.  Parity with the fp64 ring oracle on the same rounded inputs: the ring after the
step bit-exact, outputs within the bf16/f16 tolerance; wrapped and unwrapped rings, bands
that start mid-tile, multi-token steps, RoPE, sinks and softcap."""
import itertools
import zlib

import numpy as np
import pytest
import torch

from gpu_util import assert_close, oracle_ref, out_rows, run_gpu
from helpers import storage
from sliding_window_gb300.inputs import Workload, make_case

pytestmark = pytest.mark.gpu


def ring_case(dtype, D, G, curr, cap, W, past_lo, past_hi, sink="head", softcap=0.0, rotary=0, B=3, Hkv=2,
              seed=0, garbage="normal"):
    w = Workload("ringg", 500 + seed, "decode", dtype, B, G * Hkv, Hkv, D, curr, cap, past_lo, past_hi,
                 windows=(W,), softcap=softcap, head_sink=sink == "head", smooth_softmax=int(sink == "smooth"),
                 do_rotary=rotary, rope_len=past_hi + curr + 8 if rotary else 0, kv_ring=1)
    return make_case(w, seed_offset=seed, garbage=garbage)


SWEEP = list(itertools.product(
    ["bf16", "f16"],
    [(128, 8, 1), (128, 4, 4), (64, 8, 2), (64, 16, 1)],       # (D, G, curr)
    [(64, None), (1024, None), (1024, 37), (1024, 300)],       # (cap, window: None = the largest valid)
    [(0, 50), (900, 5000)],                                    # past range: unwrapped / wrapped
))


@pytest.mark.parametrize("dtype,dgc,capw,past", SWEEP)
def test_ring_decode_parity(dtype, dgc, capw, past):
    D, G, curr = dgc
    cap, W = capw
    W = W or cap - curr + 1
    lo, hi = past
    seed = zlib.crc32(repr((dtype, dgc, capw, past)).encode()) % 71
    c = ring_case(dtype, D, G, curr, cap, W, lo, hi, rotary=int(seed % 2 == 0), softcap=30.0 if seed % 3 == 0 else 0.0,
                  seed=seed)
    r = run_gpu(c, "decode")
    assert r["status"] == 0
    ref, pk, pv, st = oracle_ref(c)
    assert st == 0
    np.testing.assert_array_equal(storage(r["present_k"]), pk)
    np.testing.assert_array_equal(storage(r["present_v"]), pv)
    assert_close(out_rows(r["out"], c), ref, dtype, "ring %s" % ((dtype, dgc, capw, past),))


def test_ring_consecutive_steps_match_the_oracle():
    """Eight decode steps of 3 tokens through one ring: GPU and oracle rings stay bit-equal."""
    import oracle
    c = ring_case("bf16", 128, 4, 3, 128, 100, 150, 190, rotary=1, seed=3)
    dev = torch.device("cuda:0")
    from sliding_window_gb300 import gqa
    p = gqa.params_from_dict(c.params)
    ring_k, ring_v = c.past_k.to(dev), c.past_v.to(dev)
    hk, hv = storage(c.past_k), storage(c.past_v)
    seq = c.seqlens_k.clone()
    ws = torch.zeros(max(16, gqa.gqa_workspace_bytes(p)), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    gen = torch.Generator().manual_seed(11)
    for step in range(8):
        q = torch.randn(c.q.shape, generator=gen).to(c.q.dtype)
        k = torch.randn(c.k.shape, generator=gen).to(c.k.dtype)
        v = torch.randn(c.v.shape, generator=gen).to(c.v.dtype)
        out = torch.empty(q.shape, dtype=q.dtype, device=dev)
        gqa.check(gqa.gqa_attention_decode(p, q.to(dev), k.to(dev), v.to(dev), ring_k, ring_v, seq.to(dev),
                                           c.cos.to(dev), c.sin.to(dev), c.head_sink.to(dev), out, ring_k, ring_v,
                                           ws, st), "decode")
        q_rot, hk, hv, s = oracle.rope_append_ring(c.params, storage(q), storage(k), storage(v), hk, hv, seq.numpy(),
                                                   storage(c.cos), storage(c.sin))
        ref = oracle.attention_ring(c.params, q_rot, hk, hv, seq.numpy(), c.head_sink.numpy())
        torch.cuda.synchronize()
        assert int(st.item()) == 0 and s == 0
        np.testing.assert_array_equal(storage(ring_k), hk)
        np.testing.assert_array_equal(storage(ring_v), hv)
        assert_close(out.cpu().to(torch.float64).numpy().reshape(ref.shape), ref, "bf16", "step %d" % step)
        seq = seq + 3


def test_ring_attend_only_and_rope_append_match_the_full_call():
    c = ring_case("f16", 128, 8, 2, 1024, 1000, 3000, 9000, sink="smooth", rotary=1, seed=4)
    full = run_gpu(c, "decode")
    split = run_gpu(c, "decode", attend_only=True)
    np.testing.assert_array_equal(storage(full["present_k"]), storage(split["present_k"]))
    assert torch.equal(full["out"].view(torch.int16), split["out"].view(torch.int16))


@pytest.mark.parametrize("garbage", ["huge", "nonfinite"])
def test_unwrapped_ring_never_reads_unwritten_slots(garbage):
    """Slots past the newest position of a ring that has not wrapped hold garbage."""
    a = ring_case("bf16", 128, 8, 1, 1024, 1024, 10, 900, seed=5)
    b = ring_case("bf16", 128, 8, 1, 1024, 1024, 10, 900, seed=5, garbage=garbage)
    ra, rb = run_gpu(a, "decode"), run_gpu(b, "decode")
    assert torch.equal(ra["out"].view(torch.int16), rb["out"].view(torch.int16))
