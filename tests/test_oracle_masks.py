"""Pins for the oracle's attention masks (onnx-light-cpu "Attention Kernel Design", "Layouts
and semantics": boolean and FLOAT additive broadcast masks with the bottom-right causal band;
tract PR #2645 "What changed": attention_bias summed with the causal band): the pure-Python
brute force with the mask as key removal / added logit, the unmasked oracle for masks that
change nothing, the window attribute for a boolean mask that encodes the same band, and
broadcasting against the explicit full mask."""
import itertools
import math

import numpy as np
import pytest

import brute_force
import oracle
from helpers import as_f64, nested, storage
from test_oracle_attention import concat_present, run_oracle, tiny


def run_masked(c, mask, kind):
    p = c.params
    q_rot, pk, pv, st = oracle.rope_append(p, storage(c.q), storage(c.k), storage(c.v), storage(c.past_k),
                                           storage(c.past_v), c.seqlens_k.numpy())
    sink = None if c.head_sink is None else c.head_sink.numpy()
    return oracle.attention_masked(p, q_rot, pk, pv, c.seqlens_k.numpy(), mask, kind, sink)


COMBOS = list(itertools.product([1, 3], [-1, 2], ["none", "head"], [0.0, 2.0], ["bool", "add"], ["f32", "bf16"]))


@pytest.mark.parametrize("curr,window,sink,softcap,kind,dtype", COMBOS)
def test_masked_oracle_matches_brute_force(curr, window, sink, softcap, kind, dtype):
    B, Hq, Hkv, D, cap = 2, 4, 2, 8, 12
    rng = np.random.default_rng(curr * 100 + window + 7)
    seq = rng.integers(0, cap - curr, endpoint=True, size=B).astype(np.int32)
    c = tiny(B, Hq, Hkv, D, curr, cap, dtype, seq, window, 1, softcap, sink == "head", seed=3)
    if kind == "bool":
        mask = (rng.random((B, Hq, curr, cap)) < 0.7).astype(np.uint8)
        keep = lambda b, h, i, j: bool(mask[b, h, i, j])  # noqa: E731
        bias = None
    else:
        vals = rng.standard_normal((B, 1, curr, cap)) * 3.0
        mask = oracle.encode(vals, dtype) if dtype != "f32" else vals.astype(np.float32)
        dec = oracle.decode(mask, dtype) if dtype != "f32" else mask.astype(np.float64)
        keep = None
        bias = lambda b, h, i, j: float(dec[b, 0, i, j])  # noqa: E731
    out = run_masked(c, mask, kind)
    pk, pv = concat_present(c)
    q = as_f64(c.q).reshape(B, curr, Hq, D)
    sinks = c.head_sink.double().tolist() if sink == "head" else None
    want = brute_force.attention(nested(q), nested(pk), nested(pv), seq.tolist(), B, Hq, Hkv, D, curr, window, 1,
                                 1.0 / math.sqrt(D), softcap, sinks, keep=keep, bias=bias)
    np.testing.assert_allclose(out, np.array(want), rtol=0, atol=1e-12)


def test_masks_that_change_nothing_equal_the_unmasked_oracle():
    c = tiny(B=2, Hq=4, Hkv=2, D=16, curr=2, cap=20, dtype="bf16", window=5, head_sink=True, seed=4)
    ref, *_ = run_oracle(c)
    ones = np.ones((1, 1, 2, 20), np.uint8)
    zeros = np.zeros((2, 4, 2, 20), np.uint16)  # bf16 +0.0
    np.testing.assert_array_equal(run_masked(c, ones, "bool"), ref)
    np.testing.assert_array_equal(run_masked(c, zeros, "add"), ref)


def test_boolean_mask_of_a_band_equals_the_window_attribute():
    W, curr, cap = 4, 3, 24
    c_w = tiny(B=2, Hq=4, Hkv=2, D=16, curr=curr, cap=cap, dtype="f16", window=W, head_sink=True, seed=5)
    c_m = tiny(B=2, Hq=4, Hkv=2, D=16, curr=curr, cap=cap, dtype="f16", window=-1, head_sink=True, seed=5)
    seq = c_m.seqlens_k.numpy()
    mask = np.zeros((2, 1, curr, cap), np.uint8)
    for b in range(2):
        for i in range(curr):
            q_abs = int(seq[b]) + i
            mask[b, 0, i, max(0, q_abs - W + 1):] = 1
    ref, *_ = run_oracle(c_w)
    np.testing.assert_array_equal(run_masked(c_m, mask, "bool"), ref)


def test_broadcast_mask_equals_the_explicit_mask():
    c = tiny(B=2, Hq=4, Hkv=2, D=8, curr=2, cap=16, dtype="bf16", seed=6)
    rng = np.random.default_rng(6)
    small = oracle.encode(rng.standard_normal((1, 4, 1, 16)), "bf16")
    full = np.broadcast_to(small, (2, 4, 2, 16)).copy()
    np.testing.assert_array_equal(run_masked(c, small, "add"), run_masked(c, full, "add"))


def test_additive_constant_per_row_cancels_without_softcap():
    c = tiny(B=2, Hq=4, Hkv=2, D=8, curr=2, cap=16, dtype="f32", seed=7)
    ref, *_ = run_oracle(c)
    const = np.full((2, 4, 2, 16), 3.25, np.float32)
    np.testing.assert_allclose(run_masked(c, const, "add"), ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_additive_minus_inf_equals_key_removal_without_softcap(dtype):
    """0 / -inf additive values remove exactly the -inf keys, like a boolean mask; a row whose
    keys all carry -inf is fully masked and gives zeros (with or without a sink)."""
    for sink in (False, True):
        c = tiny(B=2, Hq=4, Hkv=2, D=8, curr=3, cap=16, dtype=dtype, window=6, head_sink=sink, seed=8)
        rng = np.random.default_rng(8)
        keep = (rng.random((2, 4, 3, 16)) < 0.6).astype(np.uint8)
        keep[1, 2, 1, :] = 0  # one row with every key removed
        vals = np.where(keep != 0, 0.0, -np.inf)
        add = oracle.encode(vals, dtype) if dtype != "f32" else vals.astype(np.float32)
        out_add = run_masked(c, add, "add")
        np.testing.assert_array_equal(out_add, run_masked(c, keep, "bool"))
        assert np.all(out_add[1, 1, 2] == 0.0)
        assert np.isfinite(out_add).all()


def test_additive_minus_inf_under_softcap_is_the_capped_floor():
    """With a softcap the bias joins before the cap, so -inf becomes the finite score -softcap
    (tanh(-inf) = -1): the key keeps a small weight.  Brute force agrees."""
    B, Hq, Hkv, D, curr, cap, softcap = 1, 2, 1, 8, 2, 10, 1.5
    c = tiny(B, Hq, Hkv, D, curr, cap, "f32", np.array([6], np.int32), -1, 1, softcap, False, seed=9)
    vals = np.zeros((1, 1, curr, cap))
    vals[0, 0, :, ::2] = -np.inf
    out = run_masked(c, vals.astype(np.float32), "add")
    pk, pv = concat_present(c)
    q = as_f64(c.q).reshape(B, curr, Hq, D)
    want = brute_force.attention(nested(q), nested(pk), nested(pv), [6], B, Hq, Hkv, D, curr, -1, 1,
                                 1.0 / math.sqrt(D), softcap, None, bias=lambda b, h, i, j: float(vals[0, 0, i, j]))
    np.testing.assert_allclose(out, np.array(want), rtol=0, atol=1e-12)
    assert np.isfinite(out).all()
