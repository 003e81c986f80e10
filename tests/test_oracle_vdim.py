"""Pins for a V head dimension that differs from the Q/K one (onnx-light-cpu "Attention
Kernel Design", "Layouts and semantics": the V head dimension may differ from the Q/K head
dimension): the pure-Python brute force, the column split of V (each output column depends
only on the same V column, so V = [V1 | V2] gives [out(V1) | out(V2)] through the oracle's
equal-dimension path), and the append copying V rows of their own width."""
import itertools
import math

import numpy as np
import pytest

import brute_force
import oracle
from helpers import as_f64, nested, storage
from test_oracle_attention import concat_present, run_oracle, tiny


@pytest.mark.parametrize("D,Dv,curr,window,softcap,dtype", list(itertools.product(
    [8, 16], [4, 8, 24], [1, 3], [-1, 2], [0.0, 2.0], ["f32", "bf16"])))
def test_vdim_matches_brute_force(D, Dv, curr, window, softcap, dtype):
    B, Hq, Hkv, cap = 2, 4, 2, 12
    rng = np.random.default_rng(D * 100 + Dv + curr)
    seq = rng.integers(0, cap - curr, endpoint=True, size=B).astype(np.int32)
    c = tiny(B, Hq, Hkv, D, curr, cap, dtype, seq, window, 1, softcap, True, seed=11, Dv=Dv)
    out, *_ = run_oracle(c)
    assert out.shape == (B, curr, Hq, Dv)
    pk, pv = concat_present(c)
    q = as_f64(c.q).reshape(B, curr, Hq, D)
    want = brute_force.attention(nested(q), nested(pk), nested(pv), seq.tolist(), B, Hq, Hkv, D, curr, window, 1,
                                 1.0 / math.sqrt(D), softcap, c.head_sink.double().tolist(), Dv=Dv)
    np.testing.assert_allclose(out, np.array(want), rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_v_column_split(dtype):
    """out with V = [V1 | V2] is [out(V1) | out(V2)], the halves through Dv = D."""
    D, Dh = 16, 16
    c = tiny(B=2, Hq=4, Hkv=2, D=D, curr=2, cap=20, dtype=dtype, window=7, head_sink=True, seed=12, Dv=2 * Dh)
    q_rot, pk, pv, st = oracle.rope_append(c.params, storage(c.q), storage(c.k), storage(c.v), storage(c.past_k),
                                           storage(c.past_v), c.seqlens_k.numpy())
    assert st == 0
    sink = c.head_sink.numpy()
    full = oracle.attention(c.params, q_rot, pk, pv, c.seqlens_k.numpy(), sink)
    p_half = dict(c.params, v_head_dim=0)
    for h in range(2):
        half = np.ascontiguousarray(pv[..., h * Dh:(h + 1) * Dh])
        part = oracle.attention(p_half, q_rot, pk, half, c.seqlens_k.numpy(), sink)
        np.testing.assert_array_equal(full[..., h * Dh:(h + 1) * Dh], part)


def test_append_copies_v_rows_of_their_own_width():
    B, Hkv, L, D, Dv = 2, 2, 3, 8, 24
    c = tiny(B=B, Hq=4, Hkv=Hkv, D=D, curr=L, cap=16, dtype="bf16", seed=13, Dv=Dv)
    _, pk, pv, st = oracle.rope_append(c.params, storage(c.q), storage(c.k), storage(c.v), storage(c.past_k),
                                       storage(c.past_v), c.seqlens_k.numpy())
    assert st == 0 and pv.shape == (B, Hkv, 16, Dv)
    v = storage(c.v).reshape(B, L, Hkv, Dv)
    old = storage(c.past_v)
    for b in range(B):
        s = int(c.seqlens_k[b])
        np.testing.assert_array_equal(pv[b, :, s:s + L], v[b].transpose(1, 0, 2))
        np.testing.assert_array_equal(pv[b, :, :s], old[b, :, :s])


def test_masked_oracle_with_vdim():
    c = tiny(B=2, Hq=4, Hkv=2, D=8, curr=2, cap=14, dtype="f32", window=5, head_sink=True, seed=14, Dv=16)
    q_rot, pk, pv, _ = oracle.rope_append(c.params, storage(c.q), storage(c.k), storage(c.v), storage(c.past_k),
                                          storage(c.past_v), c.seqlens_k.numpy())
    ones = np.ones((1, 1, 2, 14), np.uint8)
    ref = oracle.attention(c.params, q_rot, pk, pv, c.seqlens_k.numpy(), c.head_sink.numpy())
    np.testing.assert_array_equal(oracle.attention_masked(c.params, q_rot, pk, pv, c.seqlens_k.numpy(), ones, "bool",
                                                          c.head_sink.numpy()), ref)
