"""Pins for the oracle's RoPE + append emulation (tract PR #2645, "What changed": do_rotary
with the cos/sin halves widened to the head size, K rotated before it enters the cache,
past concatenated into present)."""
import numpy as np
import pytest
import torch

import oracle
from helpers import storage
from sliding_window_gb300.inputs import Workload, make_case


def case(dtype, curr=3, cap=24, seed=0, rope_len=64, D=16):
    w = Workload("rope", 60 + seed, "decode", dtype, 2, 4, 2, D, curr, cap, 0, min(cap - curr, rope_len - curr),
                 do_rotary=1, rope_len=rope_len)
    return make_case(w, seed_offset=seed)


def numpy_rotate(x, cos, sin, pos, dtype):
    """Second implementation: numpy float32 arithmetic (one rounding per op), then the
    storage rounding done by numpy (f16) or torch (bf16)."""
    half = x.shape[-1] // 2
    x1 = x[..., :half].astype(np.float32)
    x2 = x[..., half:].astype(np.float32)
    c = cos[pos].astype(np.float32)
    s = sin[pos].astype(np.float32)
    y1 = np.subtract(np.multiply(x1, c, dtype=np.float32), np.multiply(x2, s, dtype=np.float32), dtype=np.float32)
    y2 = np.add(np.multiply(x2, c, dtype=np.float32), np.multiply(x1, s, dtype=np.float32), dtype=np.float32)
    y = np.concatenate([y1, y2], axis=-1)
    if dtype == "f32":
        return y
    if dtype == "f16":
        return y.astype(np.float16).view(np.uint16)
    return torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f32_of(t):
    return t.detach().cpu().to(torch.float32).numpy()


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_rope_append_bitwise_against_numpy(dtype):
    c = case(dtype, seed=1)
    p = c.params
    q_rot, pk, pv, st = oracle.rope_append(p, storage(c.q), storage(c.k), storage(c.v), storage(c.past_k),
                                           storage(c.past_v), c.seqlens_k.numpy(), storage(c.cos), storage(c.sin))
    assert st == 0
    B, Hq, Hkv, D, L, cap = 2, 4, 2, 16, 3, 24
    cos, sin = f32_of(c.cos), f32_of(c.sin)
    qf = f32_of(c.q).reshape(B, L, Hq, D)
    kf = f32_of(c.k).reshape(B, L, Hkv, D)
    pkv = pk.reshape(B, Hkv, cap, D)
    pvv = pv.reshape(B, Hkv, cap, D)
    vst = storage(c.v).reshape(B, L, Hkv, D)
    qr = q_rot.reshape(B, L, Hq, D)
    for b in range(B):
        past = int(c.seqlens_k[b])
        for i in range(L):
            pos = past + i
            np.testing.assert_array_equal(qr[b, i], numpy_rotate(qf[b, i], cos, sin, pos, dtype))
            np.testing.assert_array_equal(pkv[b, :, pos], numpy_rotate(kf[b, i], cos, sin, pos, dtype))
            np.testing.assert_array_equal(pvv[b, :, pos], vst[b, i])
    # rows outside [past, past+curr) untouched (compared as raw bits, NaN-safe)
    orig = storage(c.past_k).reshape(B, Hkv, cap, D).view(np.uint32 if dtype == "f32" else np.uint16)
    now = pkv.view(np.uint32 if dtype == "f32" else np.uint16)
    for b in range(B):
        past = int(c.seqlens_k[b])
        np.testing.assert_array_equal(now[b, :, :past], orig[b, :, :past])
        np.testing.assert_array_equal(now[b, :, past + L:], orig[b, :, past + L:])


def test_position_zero_is_identity():
    c = case("bf16", seed=2)
    p = dict(c.params)
    seq = np.zeros(2, np.int32)
    q_rot, pk, _, _ = oracle.rope_append(dict(p, q_len=1), storage(c.q)[:, :1].copy(), storage(c.k)[:, :1].copy(),
                                         storage(c.v)[:, :1].copy(), storage(c.past_k), storage(c.past_v), seq,
                                         storage(c.cos), storage(c.sin))
    np.testing.assert_array_equal(q_rot, storage(c.q)[:, :1])
    np.testing.assert_array_equal(pk.reshape(2, 2, 24, 16)[:, :, 0], storage(c.k)[:, 0].reshape(2, 2, 16))


def test_rotation_preserves_norm_and_relative_position():
    """fp32 tables: ||rope(x)|| = ||x|| and <rope(q,m), rope(k,n)> depends on m - n only."""
    D, rope_len = 32, 200
    w = Workload("rope_f32", 70, "decode", "f32", 1, 1, 1, D, 1, 256, 0, 0, do_rotary=1, rope_len=rope_len)
    c = make_case(w)
    p = c.params
    q = storage(c.q)
    k = storage(c.k).reshape(1, 1, D)

    def rot(x, pos):
        qr, pk, _, st = oracle.rope_append(p, x.reshape(1, 1, D), x.reshape(1, 1, D), x.reshape(1, 1, D),
                                           storage(c.past_k), storage(c.past_v), np.array([pos], np.int32),
                                           storage(c.cos), storage(c.sin))
        assert st == 0
        return qr.reshape(D).astype(np.float64)

    for pos in (0, 1, 17, 150):
        r = rot(q, pos)
        assert abs(np.linalg.norm(r) - np.linalg.norm(q.astype(np.float64))) < 1e-5 * np.linalg.norm(q)
    base = rot(q, 40) @ rot(k, 30)
    for shift in (1, 25, 100):
        np.testing.assert_allclose(rot(q, 40 + shift) @ rot(k, 30 + shift), base, rtol=1e-4, atol=1e-4)


def test_separate_past_is_copied_and_rest_untouched():
    c = case("bf16", seed=3)
    p = c.params
    B, Hkv, cap, D, L = 2, 2, 24, 16, 3
    present_k = np.full((B, Hkv, cap, D), 0x7FC0, np.uint16)  # bf16 NaN everywhere first
    present_v = present_k.copy()
    _, pk, pv, st = oracle.rope_append(p, storage(c.q), storage(c.k), storage(c.v), storage(c.past_k),
                                       storage(c.past_v), c.seqlens_k.numpy(), storage(c.cos), storage(c.sin),
                                       present_k=present_k, present_v=present_v)
    assert st == 0
    past_k = storage(c.past_k).reshape(B, Hkv, cap, D)
    for b in range(B):
        s = int(c.seqlens_k[b])
        np.testing.assert_array_equal(pk[b, :, :s], past_k[b, :, :s])
        assert np.all(pk[b, :, s + L:] == 0x7FC0)
        assert not np.any(pk[b, :, s:s + L] == 0x7FC0)
