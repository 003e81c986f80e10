"""Pins for the oracle's attention (fp64), each against something other than the oracle:
the pure-Python brute force, torch's scaled_dot_product_attention in fp64 (a library
routine) in the special cases that reduce to it, closed forms, and invariants.

Pages: OpenVINO PR #37423 ("Sliding window", "smooth_softmax / head_sink", "Testing"),
tract PR #2645 ("What changed"), ExecuTorch PR #21901 (Summary: mask, don't evict),
onnx-light-cpu "Attention Kernel Design" ("Layouts and semantics", "Compute paths",
"Scheduling, precision, and invariants").
"""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import brute_force
import oracle
from helpers import as_f64, nested, storage
from sliding_window_gb300.inputs import Workload, make_case


def tiny(B=2, Hq=4, Hkv=2, D=8, curr=1, cap=12, dtype="f32", seqlens=None, window=-1, causal=1,
         softcap=0.0, head_sink=False, smooth=0, rotary=0, rope_len=0, scale=0.0, seed=0, garbage="normal",
         Dv=0):
    w = Workload("tiny", 50 + seed, "decode", dtype, B, Hq, Hkv, D, curr, cap, 0, cap - curr,
                 windows=(window,), causal=causal, scale=scale, softcap=softcap, head_sink=head_sink,
                 smooth_softmax=smooth, do_rotary=rotary, rope_len=rope_len, v_head_dim=Dv)
    return make_case(w, seed_offset=seed, seqlens=seqlens, garbage=garbage)


def run_oracle(c, rows=None):
    p = c.params
    q_rot, pk, pv, st = oracle.rope_append(
        p, storage(c.q), storage(c.k), storage(c.v), storage(c.past_k), storage(c.past_v),
        c.seqlens_k.numpy(), None if c.cos is None else storage(c.cos), None if c.sin is None else storage(c.sin))
    sink = None if c.head_sink is None else c.head_sink.numpy()
    out = oracle.attention(p, q_rot, pk, pv, c.seqlens_k.numpy(), sink, rows=rows)
    return out, pk, pv, q_rot, st


def concat_present(c):
    """Independent statement of past->present concat (no rotary): fp64 copies."""
    B, Hq, Hkv, D, L = c.w.batch, c.w.q_heads, c.w.kv_heads, c.w.head_dim, c.w.q_len
    Dv = c.w.v_head_dim or D
    pk = as_f64(c.past_k).copy()
    pv = as_f64(c.past_v).copy()
    k = as_f64(c.k).reshape(B, L, Hkv, D)
    v = as_f64(c.v).reshape(B, L, Hkv, Dv)
    for b in range(B):
        s = int(c.seqlens_k[b])
        pk[b, :, s:s + L] = k[b].transpose(1, 0, 2)
        pv[b, :, s:s + L] = v[b].transpose(1, 0, 2)
    return pk, pv


COMBOS = list(itertools.product([1, 2, 3], [-1, 1, 2, 3, 50], [0, 1], ["none", "smooth", "head"],
                                [0.0, 2.0], ["f32", "bf16"]))


@pytest.mark.parametrize("curr,window,causal,sink,softcap,dtype", COMBOS)
def test_oracle_matches_brute_force(curr, window, causal, sink, softcap, dtype):
    B, Hq, Hkv, D, cap = 2, 4, 2, 8, 12
    rng = np.random.default_rng(curr * 1000 + window * 10 + causal)
    seq = rng.integers(0, cap - curr, endpoint=True, size=B).astype(np.int32)
    c = tiny(B, Hq, Hkv, D, curr, cap, dtype, seq, window, causal, softcap, sink == "head",
             int(sink == "smooth"), seed=len(COMBOS) % 7)
    out, *_ = run_oracle(c)
    pk, pv = concat_present(c)
    q = as_f64(c.q).reshape(B, curr, Hq, D)
    sinks = None
    if sink == "head":
        sinks = c.head_sink.double().tolist()
    elif sink == "smooth":
        sinks = [0.0] * Hq
    want = brute_force.attention(nested(q), nested(pk), nested(pv), seq.tolist(), B, Hq, Hkv, D, curr,
                                 window, causal, 1.0 / math.sqrt(D), softcap, sinks)
    np.testing.assert_allclose(out, np.array(want), rtol=0, atol=1e-12)


def test_window_one_returns_own_value_exactly():
    c = tiny(B=2, Hq=4, Hkv=2, D=16, curr=3, cap=20, window=1, seed=3)
    out, pk, pv, _, _ = run_oracle(c)
    pvd = pv.reshape(2, 2, 20, 16)
    for b in range(2):
        for i in range(3):
            for hq in range(4):
                qa = int(c.seqlens_k[b]) + i
                np.testing.assert_array_equal(out[b, i, hq], pvd[b, hq // 2, qa].astype(np.float64))


def test_window_at_least_history_is_plain_causal_bitwise():
    for window in (12, 13, 40):
        a = tiny(curr=3, cap=12, window=window, seed=4, head_sink=True, softcap=3.0)
        b = tiny(curr=3, cap=12, window=-1, seed=4, head_sink=True, softcap=3.0)
        oa, *_ = run_oracle(a)
        ob, *_ = run_oracle(b)
        np.testing.assert_array_equal(oa, ob)


def test_fp32_prefill_matches_torch_sdpa():
    """First prompt, causal, no window, no sink: the textbook causal SDPA after repeating the
    K/V heads (the tiny fp32 workload's shape)."""
    c = tiny(B=1, Hq=4, Hkv=2, D=64, curr=128, cap=128, seqlens=np.zeros(1, np.int32), scale=1.0 / 8, seed=5)
    out, *_ = run_oracle(c)
    q = torch.from_numpy(as_f64(c.q).reshape(1, 128, 4, 64)).transpose(1, 2)
    k = torch.from_numpy(as_f64(c.k).reshape(1, 128, 2, 64)).transpose(1, 2).repeat_interleave(2, dim=1)
    v = torch.from_numpy(as_f64(c.v).reshape(1, 128, 2, 64)).transpose(1, 2).repeat_interleave(2, dim=1)
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=True, scale=1.0 / 8).transpose(1, 2).numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def _sdpa_decode(c, extra_logit=None):
    """Single-token decode with no window: every slot below total is visible, so plain
    unmasked SDPA over present[:total] applies.  extra_logit (per q head) appends one zero
    key/value whose score is forced to that value through an additive mask."""
    B, Hq, Hkv, D = c.w.batch, c.w.q_heads, c.w.kv_heads, c.w.head_dim
    G = Hq // Hkv
    pk, pv = concat_present(c)
    q = as_f64(c.q).reshape(B, 1, Hq, D)
    outs = []
    for b in range(B):
        tot = int(c.seqlens_k[b]) + 1
        qb = torch.from_numpy(q[b]).transpose(0, 1)[None]                 # [1, Hq, 1, D]
        kb = torch.from_numpy(pk[b, :, :tot]).repeat_interleave(G, 0)[None]  # [1, Hq, tot, D]
        vb = torch.from_numpy(pv[b, :, :tot]).repeat_interleave(G, 0)[None]
        mask = None
        if extra_logit is not None:
            kb = torch.cat([kb, torch.zeros(1, Hq, 1, D, dtype=torch.float64)], 2)
            vb = torch.cat([vb, torch.zeros(1, Hq, 1, D, dtype=torch.float64)], 2)
            mask = torch.zeros(1, Hq, 1, tot + 1, dtype=torch.float64)
            mask[0, :, 0, tot] = torch.as_tensor(extra_logit, dtype=torch.float64)
        o = F.scaled_dot_product_attention(qb, kb, vb, attn_mask=mask, scale=1.0 / math.sqrt(D))
        outs.append(o[0].transpose(0, 1).numpy())
    return np.stack(outs)


def test_decode_no_window_matches_torch_sdpa():
    c = tiny(B=3, Hq=8, Hkv=2, D=32, curr=1, cap=40, seed=6)
    out, *_ = run_oracle(c)
    np.testing.assert_allclose(out, _sdpa_decode(c), rtol=0, atol=1e-12)


def test_zero_sink_equals_softmax_with_extra_zero_logit():
    """smooth_softmax: a zero sink = one more key whose score is 0 and whose value is 0."""
    c = tiny(B=3, Hq=8, Hkv=2, D=32, curr=1, cap=40, smooth=1, seed=7)
    out, *_ = run_oracle(c)
    np.testing.assert_allclose(out, _sdpa_decode(c, extra_logit=np.zeros(8)), rtol=0, atol=1e-12)


def test_head_sink_equals_softmax_with_extra_logit_per_head():
    c = tiny(B=3, Hq=8, Hkv=2, D=32, curr=1, cap=40, head_sink=True, seed=8)
    out, *_ = run_oracle(c)
    z = c.head_sink.double().numpy()
    np.testing.assert_allclose(out, _sdpa_decode(c, extra_logit=z), rtol=0, atol=1e-12)


def test_very_negative_sink_is_plain_softmax():
    c = tiny(B=2, Hq=4, Hkv=2, D=16, curr=2, cap=16, head_sink=True, window=3, seed=9)
    c.head_sink.fill_(-1e30)
    with_sink, *_ = run_oracle(c)
    c.head_sink = None
    plain, *_ = run_oracle(c)
    np.testing.assert_allclose(with_sink, plain, rtol=0, atol=1e-15)


def test_head_sink_is_per_head():
    c = tiny(B=2, Hq=4, Hkv=2, D=16, curr=2, cap=16, head_sink=True, seed=10)
    base, *_ = run_oracle(c)
    c.head_sink[2] += 3.0
    moved, *_ = run_oracle(c)
    for h in range(4):
        if h == 2:
            assert np.abs(moved[:, :, h] - base[:, :, h]).max() > 1e-3
        else:
            np.testing.assert_array_equal(moved[:, :, h], base[:, :, h])


def test_gqa_equals_mha_with_repeated_kv():
    """group_size = Hq/Hkv maps q head hq to kv head hq // G ("Layouts and semantics")."""
    c = tiny(B=2, Hq=8, Hkv=2, D=16, curr=2, cap=20, window=5, head_sink=True, softcap=4.0, seed=11)
    out, pk, pv, q_rot, _ = run_oracle(c)
    p = dict(c.params, kv_heads=8)
    pk4 = pk.reshape(2, 2, 20, 16).repeat(4, axis=1)
    pv4 = pv.reshape(2, 2, 20, 16).repeat(4, axis=1)
    mha = oracle.attention(p, q_rot, pk4, pv4, c.seqlens_k.numpy(), c.head_sink.numpy())
    np.testing.assert_array_equal(out, mha)


@pytest.mark.parametrize("garbage", ["huge", "nonfinite"])
def test_stale_slots_never_change_output(garbage):
    """[P1] "Testing": stale buffer slots are fully masked."""
    a = tiny(B=2, Hq=4, Hkv=2, D=16, curr=2, cap=24, window=4, head_sink=True, dtype="bf16", seed=12)
    b = tiny(B=2, Hq=4, Hkv=2, D=16, curr=2, cap=24, window=4, head_sink=True, dtype="bf16", seed=12,
             garbage=garbage)
    oa, *_ = run_oracle(a)
    ob, *_ = run_oracle(b)
    np.testing.assert_array_equal(oa, ob)


def test_softcap_two_key_logistic_identity():
    """With two visible keys, a zero second key and one-hot values, out[0] = sigmoid(s1')
    where s1' = c * tanh(scale * <q, k1> / c): the cap acts on the scaled score."""
    D, c_cap = 4, 3.0
    for trial in range(5):
        rng = np.random.default_rng(trial)
        q = rng.standard_normal(D).astype(np.float32)
        k1 = rng.standard_normal(D).astype(np.float32) * np.float32(2.0)
        keys = np.stack([k1, np.zeros(D, np.float32)])
        vals = np.zeros((2, D), np.float32)
        vals[0, 0] = 1.0
        scale = 0.7
        out = oracle.attend_row(q.astype(np.float64), keys, vals, np.array([1, 1], np.uint8), "f32",
                                scale, softcap=c_cap)
        s1 = scale * math.fsum(float(a) * float(b) for a, b in zip(q, k1))
        want = c_cap * math.tanh(s1 / c_cap)
        got = math.log(out[0] / (1.0 - out[0]))
        assert abs(got - want) < 1e-9
        assert out[1:].tolist() == [0.0] * (D - 1)


def test_huge_softcap_is_no_softcap():
    a = tiny(B=2, Hq=4, Hkv=2, D=16, curr=2, cap=16, softcap=1e30, seed=13)
    b = tiny(B=2, Hq=4, Hkv=2, D=16, curr=2, cap=16, softcap=0.0, seed=13)
    oa, *_ = run_oracle(a)
    ob, *_ = run_oracle(b)
    np.testing.assert_allclose(oa, ob, rtol=0, atol=1e-12)


@pytest.mark.parametrize("sink", [None, 0.0, 1.5])
def test_fully_masked_row_gives_zeros(sink):
    """[P4] "Scheduling, precision, and invariants": a fully masked row produces zeros."""
    D = 8
    keys = np.full((5, D), np.nan, np.float32)
    vals = np.full((5, D), np.inf, np.float32)
    out = oracle.attend_row(np.ones(D), keys, vals, np.zeros(5, np.uint8), "f32", 0.3, 2.0, sink)
    assert out.tolist() == [0.0] * D


@pytest.mark.parametrize("window,sink", [(-1, None), (3, None), (-1, "smooth"), (4, "head"), (1, "head")])
def test_uniform_values_closed_form(window, sink):
    """Zero keys and identical value rows u: every visible score is 0, so
    out = u * n / (n + e^z) with n the number of visible slots (n / n = 1 without a sink)."""
    B, Hq, Hkv, D, curr, cap = 2, 4, 2, 8, 3, 16
    c = tiny(B, Hq, Hkv, D, curr, cap, window=window, head_sink=sink == "head", smooth=int(sink == "smooth"),
             seed=14)
    c.k.zero_()
    c.past_k.zero_()
    u = torch.linspace(-1.0, 1.0, D)
    c.v[:] = u.repeat(Hkv)
    c.past_v[:] = u
    out, *_ = run_oracle(c)
    for b in range(B):
        past = int(c.seqlens_k[b])
        for i in range(curr):
            n = past + i + 1 if window < 0 else min(past + i + 1, window)
            for hq in range(Hq):
                z = None if sink is None else (0.0 if sink == "smooth" else float(c.head_sink[hq]))
                frac = 1.0 if z is None else n / (n + math.exp(z))
                np.testing.assert_allclose(out[b, i, hq], u.double().numpy() * frac, rtol=0, atol=1e-14)


@pytest.mark.parametrize("window,rotary", [(-1, 0), (3, 0), (5, 1)])
def test_prefill_equals_sequential_decodes(window, rotary):
    """A first prompt of S tokens equals S single-token decode steps (bottom-right band,
    RoPE positions 0..S-1 for the prompt and seqlens_k for each generated token)."""
    B, Hq, Hkv, D, S, cap = 2, 4, 2, 16, 7, 10
    pre = tiny(B, Hq, Hkv, D, S, cap, dtype="bf16", seqlens=np.zeros(B, np.int32), window=window,
               head_sink=True, softcap=5.0, rotary=rotary, rope_len=16, seed=15)
    out_pre, pk_pre, pv_pre, _, _ = run_oracle(pre)
    p1 = dict(pre.params, q_len=1)
    present_k = storage(pre.past_k).copy()
    present_v = storage(pre.past_v).copy()
    q = storage(pre.q).reshape(B, S, Hq * D)
    k = storage(pre.k).reshape(B, S, Hkv * D)
    v = storage(pre.v).reshape(B, S, Hkv * D)
    cs = None if pre.cos is None else storage(pre.cos)
    sn = None if pre.sin is None else storage(pre.sin)
    for t in range(S):
        seq = np.full(B, t, np.int32)
        q_rot, present_k, present_v, st = oracle.rope_append(
            p1, q[:, t:t + 1].copy(), k[:, t:t + 1].copy(), v[:, t:t + 1].copy(), present_k, present_v, seq,
            cs, sn, present_k=present_k, present_v=present_v)
        assert st == 0
        o = oracle.attention(p1, q_rot, present_k, present_v, seq, pre.head_sink.numpy())
        np.testing.assert_allclose(o[:, 0], out_pre[:, t], rtol=0, atol=1e-12)
    rows = np.arange(S)
    np.testing.assert_array_equal(present_k.reshape(B, Hkv, cap, D)[:, :, rows],
                                  pk_pre.reshape(B, Hkv, cap, D)[:, :, rows])


def test_rejected_sequences_give_zeros_and_status():
    c = tiny(B=3, Hq=4, Hkv=2, D=8, curr=2, cap=10, seqlens=np.array([3, 9, -1], np.int32), seed=16)
    out, pk, pv, _, st = run_oracle(c)
    assert st == 1
    assert np.all(out[1] == 0) and np.all(out[2] == 0)
    assert np.abs(out[0]).max() > 0
    # nothing of a rejected sequence is appended
    np.testing.assert_array_equal(pk.reshape(3, 2, 10, 8)[1:], storage(c.past_k)[1:])
