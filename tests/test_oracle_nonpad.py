"""Pins for the oracle's attention over a padded K/V cache (onnx-light-cpu "Attention Kernel
Design", "Layouts and semantics": the opset-24 nonpad_kv_seqlen input; "Compute paths":
padding frontiers).  Reading: sequence b has n_b valid keys, rows [0, n_b); rows at or past
n_b are padding; the q_len queries are the last q_len valid tokens (bottom-right, query i at
position n_b - q_len + i); n_b < q_len or n_b > cap rejects the sequence (zeros).

Each pin is independent of the oracle's code: a set-based brute force that builds the
visible keys from the definition, torch SDPA in fp64 for the special cases that reduce to
it, and invariance to whatever the padding rows hold."""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from helpers import storage
from sliding_window_gb300.inputs import Workload, make_case


def padded_case(B=2, Hq=4, Hkv=2, D=8, curr=2, cap=12, dtype="f32", window=-1, causal=1, softcap=0.0,
                head_sink=False, smooth=0, seed=0, garbage="normal"):
    """q [B, curr, Hq*D] and a cache [B, Hkv, cap, D] from the seeded generator; the rows
    beyond each sequence's valid keys are drawn as garbage of the given kind."""
    w = Workload("pad", 70 + seed, "decode", dtype, B, Hq, Hkv, D, curr, cap, 0, cap - curr, windows=(window,),
                 causal=causal, softcap=softcap, head_sink=head_sink, smooth_softmax=smooth)
    return w, make_case(w, seed_offset=seed, garbage=garbage)


def brute(q, kc, vc, nonpad, B, Hq, Hkv, D, curr, window, causal, scale, softcap=0.0, sinks=None):
    """The definition, written out: keys {j < n} (the padding frontier), intersected with the
    causal band {j <= n - curr + i} and the window {j > n - curr + i - W}; math.fsum sums."""
    G = Hq // Hkv
    out = np.zeros((B, curr, Hq, D))
    for b, i, hq in itertools.product(range(B), range(curr), range(Hq)):
        n = int(nonpad[b])
        if n < curr or n > kc.shape[2]:
            continue
        q_abs = n - curr + i
        keys = set(range(n))
        if causal:
            keys &= set(range(q_abs + 1))
        if window > 0:
            keys &= set(range(q_abs - window + 1, n))
        logits, vals = [], []
        for j in sorted(keys):
            s = scale * math.fsum(float(a) * float(c) for a, c in zip(q[b, i, hq], kc[b, hq // G, j]))
            if softcap > 0:
                s = softcap * math.tanh(s / softcap)
            logits.append(s)
            vals.append(vc[b, hq // G, j])
        if not vals:
            continue
        if sinks is not None:
            logits.append(float(sinks[hq]))
        m = max(logits)
        e = [math.exp(x - m) for x in logits]
        den = math.fsum(e)
        out[b, i, hq] = [math.fsum(e[t] / den * float(vals[t][d]) for t in range(len(vals))) for d in range(D)]
    return out


@pytest.mark.parametrize("curr,window,causal,softcap,sink", [
    (1, -1, 1, 0.0, False), (2, -1, 1, 0.0, True), (3, 2, 1, 0.0, False), (2, 1, 1, 0.0, True),
    (3, 4, 0, 0.0, False), (1, 3, 1, 2.0, True), (4, -1, 0, 0.0, True)])
def test_nonpad_matches_set_brute_force(curr, window, causal, softcap, sink):
    B, Hq, Hkv, D, cap = 3, 4, 2, 8, 12
    w, c = padded_case(B, Hq, Hkv, D, curr, cap, window=window, causal=causal, softcap=softcap, head_sink=sink,
                       seed=curr + 10 * max(window, 0))
    nonpad = np.array([curr, 7, cap], dtype=np.int64)  # shortest, middle, no padding
    q = c.q.double().numpy().reshape(B, curr, Hq, D)
    kc, vc = c.past_k.double().numpy(), c.past_v.double().numpy()
    scale = 1.0 / math.sqrt(D)
    sinks = None if c.head_sink is None else c.head_sink.numpy()
    got = oracle.attention_nonpad(c.params, storage(c.q), storage(c.past_k), storage(c.past_v), nonpad, sinks)
    want = brute(q, kc, vc, nonpad, B, Hq, Hkv, D, curr, window, causal, scale, softcap, sinks)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("garbage", ["huge", "nonfinite"])
def test_padding_rows_are_never_read(garbage):
    """Whatever the padding rows hold (+-1e4, NaN, +-Inf) the outputs are bit-identical."""
    B, Hq, Hkv, D, curr, cap = 2, 4, 2, 8, 2, 16
    nonpad = np.array([5, 11], dtype=np.int64)
    _, c0 = padded_case(B, Hq, Hkv, D, curr, cap, seed=3)
    kc, vc = storage(c0.past_k).copy(), storage(c0.past_v).copy()
    _, cg = padded_case(B, Hq, Hkv, D, curr, cap, seed=3, garbage=garbage)
    gk, gv = storage(cg.past_k), storage(cg.past_v)
    for b, n in enumerate(nonpad):  # valid rows from the clean draw, padding from the garbage one
        kc[b, :, n:], vc[b, :, n:] = gk[b, :, n:], gv[b, :, n:]
    a = oracle.attention_nonpad(c0.params, storage(c0.q), storage(c0.past_k), storage(c0.past_v), nonpad)
    bb = oracle.attention_nonpad(c0.params, storage(c0.q), kc, vc, nonpad)
    assert np.isfinite(bb).all()
    np.testing.assert_array_equal(a, bb)


def test_no_padding_no_mask_is_sdpa():
    """n = cap, causal = 0, no window: plain softmax attention over every key (torch SDPA)."""
    B, Hq, Hkv, D, curr, cap = 2, 4, 2, 8, 3, 10
    w, c = padded_case(B, Hq, Hkv, D, curr, cap, causal=0, seed=5)
    nonpad = np.full(B, cap, dtype=np.int64)
    got = oracle.attention_nonpad(c.params, storage(c.q), storage(c.past_k), storage(c.past_v), nonpad)
    q = c.q.double().view(B, curr, Hq, D).transpose(1, 2)
    k = c.past_k.double().repeat_interleave(Hq // Hkv, dim=1)
    v = c.past_v.double().repeat_interleave(Hq // Hkv, dim=1)
    want = F.scaled_dot_product_attention(q, k, v).transpose(1, 2).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_full_prompt_is_causal_sdpa():
    """curr = n (the queries are every valid token): the bottom-right band is the ordinary
    lower-triangular causal mask over the first n keys (torch SDPA, is_causal)."""
    B, Hq, Hkv, D, cap, n = 1, 4, 2, 8, 12, 9
    w, c = padded_case(B, Hq, Hkv, D, n, cap, causal=1, seed=6)
    got = oracle.attention_nonpad(c.params, storage(c.q), storage(c.past_k), storage(c.past_v),
                                  np.array([n], dtype=np.int64))
    q = c.q.double().view(B, n, Hq, D).transpose(1, 2)
    k = c.past_k.double()[:, :, :n].repeat_interleave(Hq // Hkv, dim=1)
    v = c.past_v.double()[:, :, :n].repeat_interleave(Hq // Hkv, dim=1)
    want = F.scaled_dot_product_attention(q, k, v, is_causal=True).transpose(1, 2).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("n", [0, 1, 13, -4])
def test_out_of_range_lengths_give_zeros(n):
    """n < q_len (the queries would not be valid tokens) or n > cap: zeros for that sequence,
    the other sequence unaffected."""
    B, Hq, Hkv, D, curr, cap = 2, 4, 2, 8, 2, 12
    w, c = padded_case(B, Hq, Hkv, D, curr, cap, seed=7)
    nonpad = np.array([n, 8], dtype=np.int64)
    got = oracle.attention_nonpad(c.params, storage(c.q), storage(c.past_k), storage(c.past_v), nonpad)
    assert (got[0] == 0).all()
    ok = oracle.attention_nonpad(c.params, storage(c.q), storage(c.past_k), storage(c.past_v),
                                 np.array([8, 8], dtype=np.int64))
    np.testing.assert_array_equal(got[1], ok[1])
