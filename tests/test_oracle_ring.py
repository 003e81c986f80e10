"""Pins for the oracle's ring layout of the cache (OpenVINO PR #37423 "Sliding window": the
rolling sliding_window_cache buffer, whose memory is bounded by the window; ExecuTorch PR
#21901 Summary: the window is a per-layer setting).  Position p lives in slot p mod cap.
Each pin ties the ring functions to the linear-layout oracle, which is pinned on its own,
through an independent re-layout done here with numpy indexing."""
import itertools

import numpy as np
import pytest

import oracle
from helpers import storage
from sliding_window_gb300.inputs import Workload, make_case


def test_validity_rule_is_exactly_residency_by_brute_force():
    """W + curr - 1 <= cap (W >= 1) holds iff, for every past length, every key that some
    query of the step sees is still resident once the step's rows are in the ring."""
    for cap, curr, W in itertools.product(range(1, 9), range(1, 5), list(range(1, 11)) + [-1]):
        all_resident = True
        for past in range(0, 3 * cap + 2):
            total = past + curr
            resident = set(range(max(0, total - cap), total))
            for i in range(curr):
                q_abs = past + i
                seen = {j for j in range(total) if j <= q_abs and (W < 0 or q_abs - j < W)}
                if not seen <= resident:
                    all_resident = False
        assert oracle.ring_valid(curr, cap, W) == all_resident, (cap, curr, W)


def ring_case(dtype="bf16", curr=2, cap=16, W=9, past_lo=0, past_hi=60, rotary=1, seed=0, B=3, D=16, rope_len=None):
    w = Workload("ring", 80 + seed, "decode", dtype, B, 4, 2, D, curr, cap, past_lo, past_hi, windows=(W,),
                 head_sink=True, do_rotary=rotary, rope_len=rope_len or past_hi + curr + 8, kv_ring=1)
    return make_case(w, seed_offset=seed)


def unroll(ring: np.ndarray, past: int, curr: int, cap: int, fill) -> np.ndarray:
    """[Hkv, cap, D] ring of one sequence -> [Hkv, total, D] in position order; positions
    no longer resident are set to `fill` (they must never be read)."""
    total = past + curr
    lin = np.full((ring.shape[0], total, ring.shape[2]), fill, dtype=ring.dtype)
    for pos in range(max(0, total - cap), total):
        lin[:, pos] = ring[:, pos % cap]
    return lin


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_ring_append_keeps_the_last_cap_positions_of_the_linear_history(dtype):
    """Several decode steps through a ring and through a linear cache from the same start:
    afterwards ring[p % cap] == linear[p] bit for bit for every resident position p."""
    cap, curr, W, steps = 16, 3, 10, 9
    c = ring_case(dtype, curr=curr, cap=cap, W=W, past_lo=0, past_hi=0, seed=1, rope_len=64)
    p_ring = dict(c.params)
    p_lin = dict(c.params, kv_ring=0, cap_past=256, cap_present=256)
    B, Hkv, D = 3, 2, 16
    ring_k, ring_v = storage(c.past_k), storage(c.past_v)
    lin_k = np.zeros((B, Hkv, 256, D), dtype=ring_k.dtype)
    lin_v = np.zeros_like(lin_k)
    rng = np.random.default_rng(7)
    past = np.zeros(B, dtype=np.int32)
    for s in range(steps):
        k = oracle.encode(rng.standard_normal((B, curr, Hkv * D)), dtype) if dtype != "f32" else \
            rng.standard_normal((B, curr, Hkv * D)).astype(np.float32)
        v = oracle.encode(rng.standard_normal((B, curr, Hkv * D)), dtype) if dtype != "f32" else \
            rng.standard_normal((B, curr, Hkv * D)).astype(np.float32)
        q = storage(c.q)
        _, ring_k, ring_v, st = oracle.rope_append_ring(p_ring, q, k, v, ring_k, ring_v, past, storage(c.cos),
                                                        storage(c.sin))
        assert st == 0
        _, lin_k, lin_v, st = oracle.rope_append(p_lin, q, k, v, lin_k, lin_v, past, storage(c.cos), storage(c.sin),
                                                 present_k=lin_k, present_v=lin_v)
        assert st == 0
        past = past + curr
    rk, rv = ring_k.reshape(B, Hkv, cap, D), ring_v.reshape(B, Hkv, cap, D)
    for b in range(B):
        total = int(past[b])
        for pos in range(total - cap, total):
            np.testing.assert_array_equal(rk[b, :, pos % cap], lin_k[b, :, pos])
            np.testing.assert_array_equal(rv[b, :, pos % cap], lin_v[b, :, pos])


@pytest.mark.parametrize("dtype,curr,cap,W", [("bf16", 1, 16, 16), ("f16", 3, 16, 9), ("f32", 2, 24, 7),
                                              ("bf16", 4, 32, 29)])
def test_ring_attention_equals_linear_attention_on_the_unrolled_cache(dtype, curr, cap, W):
    """The ring oracle on a wrapped ring equals the linear oracle on the same positions laid
    out in order, with every evicted position filled with NaN (never visible): bitwise."""
    c = ring_case(dtype, curr=curr, cap=cap, W=W, past_lo=0, past_hi=70, seed=2)
    p = dict(c.params)
    out_r, rk, rv, q_rot, st = oracle.gqa(p, storage(c.q), storage(c.k), storage(c.v), storage(c.past_k),
                                          storage(c.past_v), c.seqlens_k.numpy(), storage(c.cos), storage(c.sin),
                                          c.head_sink.numpy())
    assert st == 0
    B, Hkv, D = 3, 2, 16
    nan = np.float32("nan") if dtype == "f32" else np.uint16(0x7FC0 if dtype == "bf16" else 0x7E00)
    rk, rv = rk.reshape(B, Hkv, cap, D), rv.reshape(B, Hkv, cap, D)
    seq = c.seqlens_k.numpy()
    for b in range(B):
        past = int(seq[b])
        total = past + curr
        pl = dict(p, kv_ring=0, batch=1, cap_past=total, cap_present=total)
        lk = unroll(rk[b], past, curr, cap, nan)[None]
        lv = unroll(rv[b], past, curr, cap, nan)[None]
        ref = oracle.attention(pl, q_rot.reshape(B, curr, -1)[b:b + 1], lk, lv, np.array([past], np.int32),
                               c.head_sink.numpy())
        np.testing.assert_array_equal(out_r[b], ref[0])
        assert np.all(np.isfinite(out_r[b]))


def test_unwrapped_ring_is_the_linear_layout():
    """While past + curr <= cap nothing wraps: the ring oracle equals the linear oracle on the
    very same buffers (slot = position), bitwise, including the stale slots being ignored."""
    c = ring_case("bf16", curr=2, cap=64, W=40, past_lo=3, past_hi=62, seed=3)
    args = (storage(c.q), storage(c.k), storage(c.v), storage(c.past_k), storage(c.past_v), c.seqlens_k.numpy(),
            storage(c.cos), storage(c.sin), c.head_sink.numpy())
    out_r, rk, rv, _, st_r = oracle.gqa(dict(c.params), *args)
    out_l, lk, lv, _, st_l = oracle.gqa(dict(c.params, kv_ring=0), *args)
    assert st_r == st_l == 0
    np.testing.assert_array_equal(out_r, out_l)
    np.testing.assert_array_equal(rk, lk)
    np.testing.assert_array_equal(rv, lv)


def test_ring_that_cannot_hold_the_band_gives_zeros():
    c = ring_case("bf16", curr=3, cap=16, W=15, past_lo=20, past_hi=40, seed=4)  # 15 + 3 - 1 > 16
    assert not oracle.ring_valid(3, 16, 15)
    out, *_ = oracle.gqa(dict(c.params), storage(c.q), storage(c.k), storage(c.v), storage(c.past_k),
                         storage(c.past_v), c.seqlens_k.numpy(), storage(c.cos), storage(c.sin), c.head_sink.numpy())
    assert np.all(out == 0.0)
