"""Pins for the oracle's quantized KV cache (an f8 E4M3 cache with one scale per kv head
for K and for V; the pages leave a quantized cache out of their own designs, so the format
is this oracle's reading).  The E4M3 codes are pinned against torch's float8_e4m3fn (a
library routine), the append against the pinned unquantized append followed by torch's
division and cast, and the attention against the unquantized oracle run on the
dequantized cache."""
import numpy as np
import pytest
import torch

import oracle
from helpers import storage
from sliding_window_gb300.inputs import Workload, make_case


def test_decode_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    got = oracle.decode_e4m3(codes)
    nan = np.isnan(want)
    assert np.array_equal(nan, np.isnan(got)) and nan.sum() == 2  # S.1111.111
    np.testing.assert_array_equal(got[~nan], want[~nan])


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(4000) * 10.0,
        rng.uniform(-460, 460, 2000),
        rng.standard_normal(2000) * 1e-2,                               # subnormals
        oracle.decode_e4m3(np.arange(0, 126, dtype=np.uint8)),          # every finite code
        (oracle.decode_e4m3(np.arange(0, 125, dtype=np.uint8)) +
         oracle.decode_e4m3(np.arange(1, 126, dtype=np.uint8))) / 2,    # ties between neighbours
        [0.0, -0.0, 2.0 ** -10, -2.0 ** -10, 463.9]])
    x = vals.astype(np.float32)
    x = np.concatenate([x, -x])
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.encode_e4m3(x), want)


def test_saturation_and_nan():
    x = np.array([464.0, 480.0, 1e6, np.inf, -464.0, -1e30, -np.inf, np.nan], dtype=np.float32)
    np.testing.assert_array_equal(oracle.encode_e4m3(x), [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0xFE, 0x7F])


def q8_case(dtype="bf16", D=64, Dv=64, curr=3, cap=40, rotary=1, B=2, Hq=4, Hkv=2, W=-1, seed=0):
    w = Workload("q8", 300 + seed, "decode", dtype, B, Hq, Hkv, D, curr, cap, 0, cap - curr, windows=(W,),
                 head_sink=True, do_rotary=rotary, rope_len=cap + 4 if rotary else 0, v_head_dim=Dv)
    return make_case(w, seed_offset=seed)


def quantize_torch(rows_f32, scale):
    """Independent statement of the append's quantization: fp32 division, torch's cast."""
    return (torch.from_numpy(rows_f32) / torch.tensor(scale, dtype=torch.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("dtype,rotary,Dv", [("bf16", 1, 64), ("f16", 0, 64), ("bf16", 0, 128), ("f32", 1, 64)])
def test_append_is_the_unquantized_append_then_the_cast(dtype, rotary, Dv):
    c = q8_case(dtype=dtype, rotary=rotary, Dv=Dv, seed=1)
    p = c.params
    B, Hkv, cap = p["batch"], p["kv_heads"], p["cap_present"]
    D = p["head_dim"]
    seq = c.seqlens_k.numpy()
    q_rot_ref, pk, pv, st = oracle.rope_append(p, storage(c.q), storage(c.k), storage(c.v), storage(c.past_k),
                                               storage(c.past_v), seq,
                                               None if c.cos is None else storage(c.cos),
                                               None if c.sin is None else storage(c.sin))
    assert st == 0
    ks = np.array([0.013, 0.021], dtype=np.float32)  # |x| / scale stays below 448 for N(0,1) rows
    vs = np.array([0.017, 0.011], dtype=np.float32)
    k8 = np.zeros((B, Hkv, cap, D), np.uint8)
    v8 = np.zeros((B, Hkv, cap, Dv), np.uint8)
    q_rot, st8 = oracle.rope_append_q8(p, storage(c.q), storage(c.k), storage(c.v), k8, v8, seq, ks, vs,
                                       None if c.cos is None else storage(c.cos),
                                       None if c.sin is None else storage(c.sin))
    assert st8 == 0
    np.testing.assert_array_equal(q_rot, q_rot_ref)
    dec = (lambda a: a) if dtype == "f32" else (lambda a: oracle.decode(a, dtype))
    for b in range(B):
        rows = slice(int(seq[b]), int(seq[b]) + p["q_len"])
        for h in range(Hkv):
            kf = dec(pk[b, h, rows]).astype(np.float32)
            vf = dec(pv[b, h, rows]).astype(np.float32)
            assert np.abs(kf / ks[h]).max() < 448 and np.abs(vf / vs[h]).max() < 448
            np.testing.assert_array_equal(k8[b, h, rows], quantize_torch(kf, ks[h]))
            np.testing.assert_array_equal(v8[b, h, rows], quantize_torch(vf, vs[h]))
        untouched = np.ones(cap, bool)
        untouched[rows] = False
        assert not k8[b, :, untouched].any() and not v8[b, :, untouched].any()


@pytest.mark.parametrize("W,Dv,pow2", [(-1, 64, True), (5, 64, True), (-1, 128, True), (7, 64, False)])
def test_attention_is_the_oracle_on_the_dequantized_cache(W, Dv, pow2):
    c = q8_case(W=W, Dv=Dv, curr=2, cap=30, seed=2)
    p = c.params
    B, Hq, Hkv, cap, D = p["batch"], p["q_heads"], p["kv_heads"], p["cap_present"], p["head_dim"]
    rng = np.random.default_rng(3)
    k8 = rng.integers(0, 256, size=(B, Hkv, cap, D), dtype=np.uint8)
    v8 = rng.integers(0, 256, size=(B, Hkv, cap, Dv), dtype=np.uint8)
    k8[(k8 & 0x7F) == 0x7F] = 0x10  # no NaN codes in the resident rows
    v8[(v8 & 0x7F) == 0x7F] = 0x11
    if pow2:  # code * scale is then exact in fp32 too, and the two oracles agree to the bit
        ks, vs = np.array([0.25, 2.0 ** -5], np.float32), np.array([0.5, 2.0 ** -7], np.float32)
    else:
        ks, vs = np.array([0.0137, 0.0291], np.float32), np.array([0.0173, 0.0119], np.float32)
    seq = c.seqlens_k.numpy()
    q = storage(c.q)
    sink = c.head_sink.numpy()
    got = oracle.attention_q8(p, q, k8, v8, seq, ks, vs, sink)
    kd = (torch.from_numpy(k8).view(torch.float8_e4m3fn).to(torch.float32) *
          torch.from_numpy(ks)[None, :, None, None]).numpy()
    vd = (torch.from_numpy(v8).view(torch.float8_e4m3fn).to(torch.float32) *
          torch.from_numpy(vs)[None, :, None, None]).numpy()
    qf = oracle.decode(q, "bf16").astype(np.float32)  # exact
    want = oracle.attention(dict(p, dtype="f32"), qf, kd, vd, seq, sink)
    if pow2:
        np.testing.assert_array_equal(got, want)
    else:
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-6)


def test_rejected_sequence_gives_zeros_and_appends_nothing():
    c = q8_case(curr=3, cap=20, rotary=0, seed=4)
    p = c.params
    seq = np.array([17, 18], np.int32)  # 18 + 3 > 20: the second sequence is rejected
    k8 = np.zeros((2, 2, 20, 64), np.uint8)
    v8 = np.zeros((2, 2, 20, 64), np.uint8)
    ks = vs = np.ones(2, np.float32)
    _, st = oracle.rope_append_q8(p, storage(c.q), storage(c.k), storage(c.v), k8, v8, seq, ks, vs)
    assert st == 1 and not k8[1].any() and not v8[1].any() and k8[0].any()
    out = oracle.attention_q8(p, storage(c.q), k8, v8, seq, ks, vs, c.head_sink.numpy())
    assert np.all(out[1] == 0.0) and np.any(out[0] != 0.0)
