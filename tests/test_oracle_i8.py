"""Pins for the oracle's int8 KV cache (two's-complement codes in [-128, 127] with one scale
per kv head for K and for V; stored value = code * scale; code = round-half-even of the fp32
quotient x / scale, saturated, NaN to 0: the ONNX QuantizeLinear convention with a zero point
of 0, the reading taken for a format the pages leave open).  The codes are pinned against
numpy's rint and clip (library routines), the append against the pinned unquantized append
followed by numpy's fp32 division, rint and clip, and the attention against the unquantized
oracle run on the cache dequantized by numpy."""
import numpy as np
import pytest

import oracle
from helpers import storage
from sliding_window_gb300.inputs import Workload, make_case


def np_quantize(x):
    """numpy's statement of the code: rint (half to even), clip, NaN to 0."""
    x = np.asarray(x, dtype=np.float32)
    r = np.clip(np.rint(x.astype(np.float64)), -128, 127)
    r[np.isnan(x)] = 0
    return r.astype(np.int8)


def test_decode_is_the_twos_complement_value_of_every_code():
    codes = np.arange(256, dtype=np.uint8).view(np.int8)
    np.testing.assert_array_equal(oracle.decode_i8(codes), codes.astype(np.float64))
    assert oracle.decode_i8(np.array([0x80], np.uint8).view(np.int8))[0] == -128.0


def test_encode_matches_rint_and_clip():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(4000) * 40.0,
        rng.uniform(-300, 300, 3000),
        np.arange(-130, 131) + 0.5,                  # every tie in range and just beyond it
        np.arange(-130, 131).astype(np.float64),     # every integer
        np.nextafter(np.arange(-129, 129) + 0.5, 0),  # just below each tie (towards zero)
        [0.0, -0.0, 0.49999997, -0.49999997, 126.5, 127.5, -127.5, -128.5, 1e30, -1e30]])
    x = vals.astype(np.float32)
    np.testing.assert_array_equal(oracle.encode_i8(x), np_quantize(x))


def test_ties_go_to_even_and_saturation_and_nan():
    x = np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 127.5, 128.0, np.inf, -128.5, -129.0, -np.inf, np.nan],
                 dtype=np.float32)
    np.testing.assert_array_equal(oracle.encode_i8(x), [0, 2, 2, 0, -2, -2, 127, 127, 127, -128, -128, -128, 0])


def i8_case(dtype="bf16", D=64, Dv=64, curr=3, cap=40, rotary=1, B=2, Hq=4, Hkv=2, W=-1, seed=0):
    w = Workload("i8", 500 + seed, "decode", dtype, B, Hq, Hkv, D, curr, cap, 0, cap - curr, windows=(W,),
                 head_sink=True, do_rotary=rotary, rope_len=cap + 4 if rotary else 0, v_head_dim=Dv)
    return make_case(w, seed_offset=seed)


@pytest.mark.parametrize("dtype,rotary,Dv", [("bf16", 1, 64), ("f16", 0, 64), ("bf16", 0, 128), ("f32", 1, 64)])
def test_append_is_the_unquantized_append_then_the_code(dtype, rotary, Dv):
    c = i8_case(dtype=dtype, rotary=rotary, Dv=Dv, seed=1)
    p = c.params
    B, Hkv, cap, D = p["batch"], p["kv_heads"], p["cap_present"], p["head_dim"]
    seq = c.seqlens_k.numpy()
    cs = None if c.cos is None else storage(c.cos)
    sn = None if c.sin is None else storage(c.sin)
    q_rot_ref, pk, pv, st = oracle.rope_append(p, storage(c.q), storage(c.k), storage(c.v), storage(c.past_k),
                                               storage(c.past_v), seq, cs, sn)
    assert st == 0
    ks = np.array([0.021, 0.033], dtype=np.float32)  # |x| / scale reaches past 127 for N(0,1) rows
    vs = np.array([0.017, 0.011], dtype=np.float32)
    k8 = np.zeros((B, Hkv, cap, D), np.uint8)
    v8 = np.zeros((B, Hkv, cap, Dv), np.uint8)
    q_rot, st8 = oracle.rope_append_q8(p, storage(c.q), storage(c.k), storage(c.v), k8, v8, seq, ks, vs, cs, sn,
                                       fmt="int8")
    assert st8 == 0
    np.testing.assert_array_equal(q_rot, q_rot_ref)
    dec = (lambda a: a) if dtype == "f32" else (lambda a: oracle.decode(a, dtype))
    saturated = 0
    for b in range(B):
        rows = slice(int(seq[b]), int(seq[b]) + p["q_len"])
        for h in range(Hkv):
            kf = dec(pk[b, h, rows]).astype(np.float32)
            vf = dec(pv[b, h, rows]).astype(np.float32)
            kq = kf / np.float32(ks[h])  # fp32 division
            vq = vf / np.float32(vs[h])
            saturated += int((np.abs(kq) > 127.5).sum() + (np.abs(vq) > 127.5).sum())
            np.testing.assert_array_equal(k8[b, h, rows].view(np.int8), np_quantize(kq))
            np.testing.assert_array_equal(v8[b, h, rows].view(np.int8), np_quantize(vq))
        untouched = np.ones(cap, bool)
        untouched[rows] = False
        assert not k8[b, :, untouched].any() and not v8[b, :, untouched].any()
    assert saturated > 0  # the clip is exercised


@pytest.mark.parametrize("W,Dv,pow2", [(-1, 64, True), (5, 64, True), (-1, 128, True), (7, 64, False)])
def test_attention_is_the_oracle_on_the_dequantized_cache(W, Dv, pow2):
    c = i8_case(W=W, Dv=Dv, curr=2, cap=30, seed=2)
    p = c.params
    B, Hkv, cap, D = p["batch"], p["kv_heads"], p["cap_present"], p["head_dim"]
    rng = np.random.default_rng(3)
    k8 = rng.integers(0, 256, size=(B, Hkv, cap, D), dtype=np.uint8)
    v8 = rng.integers(0, 256, size=(B, Hkv, cap, Dv), dtype=np.uint8)
    if pow2:  # code * scale is then exact in fp32 too, and the two oracles agree to the bit
        ks, vs = np.array([2.0 ** -6, 2.0 ** -8], np.float32), np.array([2.0 ** -7, 2.0 ** -5], np.float32)
    else:
        ks, vs = np.array([0.0137, 0.0091], np.float32), np.array([0.0073, 0.0119], np.float32)
    seq = c.seqlens_k.numpy()
    q = storage(c.q)
    sink = c.head_sink.numpy()
    got = oracle.attention_q8(p, q, k8, v8, seq, ks, vs, sink, fmt="int8")
    kd = k8.view(np.int8).astype(np.float32) * ks[None, :, None, None]
    vd = v8.view(np.int8).astype(np.float32) * vs[None, :, None, None]
    qf = oracle.decode(q, "bf16").astype(np.float32)  # exact
    want = oracle.attention(dict(p, dtype="f32"), qf, kd, vd, seq, sink)
    if pow2:
        np.testing.assert_array_equal(got, want)
    else:
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-6)


def test_rejected_sequence_gives_zeros_and_appends_nothing():
    c = i8_case(curr=3, cap=20, rotary=0, seed=4)
    p = c.params
    seq = np.array([17, 18], np.int32)  # 18 + 3 > 20: the second sequence is rejected
    k8 = np.zeros((2, 2, 20, 64), np.uint8)
    v8 = np.zeros((2, 2, 20, 64), np.uint8)
    ks = vs = np.full(2, 0.01, np.float32)
    _, st = oracle.rope_append_q8(p, storage(c.q), storage(c.k), storage(c.v), k8, v8, seq, ks, vs, fmt="int8")
    assert st == 1 and not k8[1].any() and not v8[1].any() and k8[0].any()
    out = oracle.attention_q8(p, storage(c.q), k8, v8, seq, ks, vs, c.head_sink.numpy(), fmt="int8")
    assert np.all(out[1] == 0.0) and np.any(out[0] != 0.0)
