"""K1 parity: RoPE + append into present and the rotated queries, bit-exact against the
oracle's emulation (tract PR #2645, "What changed")."""
import numpy as np
import pytest
import torch

import oracle
from helpers import storage
from sliding_window_gb300.inputs import Workload, make_case

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("rotary", [0, 1])
@pytest.mark.parametrize("separate", [False, True])
@pytest.mark.parametrize("D,curr", [(128, 1), (64, 3), (128, 5)])
def test_rope_append_bit_exact(dtype, rotary, separate, D, curr):
    from sliding_window_gb300 import gqa
    w = Workload("k1", 200 + D + curr, "decode", dtype, 3, 8, 2, D, curr, 300, 0, 290, do_rotary=rotary,
                 rope_len=400 if rotary else 0)
    c = make_case(w, seed_offset=rotary + 2 * separate, garbage="nonfinite")
    dev = torch.device("cuda:0")
    p = gqa.params_from_dict(c.params)
    q, k, v = c.q.to(dev), c.k.to(dev), c.v.to(dev)
    past_k, past_v = c.past_k.to(dev), c.past_v.to(dev)
    if separate:
        present_k = torch.zeros_like(past_k)
        present_v = torch.zeros_like(past_v)
    else:
        present_k, present_v = past_k, past_v
    cos = None if c.cos is None else c.cos.to(dev)
    sin = None if c.sin is None else c.sin.to(dev)
    q_rot = torch.empty_like(q)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    gqa.check(gqa.gqa_rope_append_kv(p, q, k, v, past_k, past_v, c.seqlens_k.to(dev), cos, sin, q_rot, present_k,
                                     present_v, st))
    torch.cuda.synchronize()
    assert st.item() == 0
    pk0 = storage(c.past_k)
    pv0 = storage(c.past_v)
    init_k = np.zeros_like(pk0) if separate else pk0.copy()
    init_v = np.zeros_like(pv0) if separate else pv0.copy()
    qr, pk, pv, s = oracle.rope_append(c.params, storage(c.q), storage(c.k), storage(c.v), pk0, pv0,
                                       c.seqlens_k.numpy(), None if cos is None else storage(c.cos),
                                       None if sin is None else storage(c.sin), present_k=init_k, present_v=init_v)
    assert s == 0
    u = np.uint32 if dtype == "f32" else np.uint16
    np.testing.assert_array_equal(storage(present_k).view(u), pk.view(u))
    np.testing.assert_array_equal(storage(present_v).view(u), pv.view(u))
    np.testing.assert_array_equal(storage(q_rot).view(u), qr.view(u))


def test_rope_append_rejects_bad_sequences():
    from sliding_window_gb300 import gqa
    w = Workload("k1bad", 230, "decode", "bf16", 4, 4, 2, 128, 2, 64, 0, 60, do_rotary=1, rope_len=50)
    seq = np.array([10, -1, 63, 49], np.int32)  # ok, negative, overflow, rope position out of range
    c = make_case(w, seqlens=seq)
    dev = torch.device("cuda:0")
    p = gqa.params_from_dict(c.params)
    pk, pv = c.past_k.to(dev), c.past_v.to(dev)
    before = storage(pk).copy()
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    gqa.check(gqa.gqa_rope_append_kv(p, c.q.to(dev), c.k.to(dev), c.v.to(dev), pk, pv, c.seqlens_k.to(dev),
                                     c.cos.to(dev), c.sin.to(dev), None, pk, pv, st))
    torch.cuda.synchronize()
    assert st.item() == 3
    after = storage(pk)
    np.testing.assert_array_equal(after[1:], before[1:])
    assert not np.array_equal(after[0], before[0])
