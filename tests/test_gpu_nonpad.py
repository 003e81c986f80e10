"""gqa_attention_nonpad against the fp64 oracle (onnx-light-cpu "Attention Kernel Design",
"Layouts and semantics": opset-24 nonpad_kv_seqlen; "Compute paths": padding frontiers).
Sequence b has n_b valid keys in rows [0, n_b) of its cache, the rows past n_b hold NaN/Inf
padding that must never be read, and the q_len queries are the last q_len valid tokens.
One case per kernel the entry point routes to: the split-KV decode (one and four query
tokens), the tensor-core prefill and the fp32 kernel; plus lengths the call must reject."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close
from helpers import storage
from sliding_window_gb300.inputs import Workload, make_case

pytestmark = pytest.mark.gpu

CASES = {
    "decode": (Workload("np_dec", 601, "decode", "bf16", 4, 32, 8, 128, 1, 2048, 0, 0, windows=(700,),
                        head_sink=True), [1, 333, 1500, 2048]),
    "decode_multi": (Workload("np_spec", 602, "decode", "f16", 3, 32, 4, 128, 4, 4096, 0, 0, windows=(-1,),
                              smooth_softmax=1), [4, 2049, 4096]),
    "prefill": (Workload("np_pre", 603, "prefill", "bf16", 2, 8, 2, 128, 300, 512, 0, 0, windows=(200,),
                         softcap=30.0, head_sink=True), [300, 477]),
    "fp32": (Workload("np_f32", 604, "prefill", "f32", 2, 4, 2, 64, 20, 128, 0, 0, windows=(-1,)), [20, 97]),
}


def run(w, lengths, seed=0):
    from sliding_window_gb300 import gqa
    c = make_case(w, seqlens=np.array(lengths, dtype=np.int32), garbage="nonfinite", seed_offset=seed)
    dev = torch.device("cuda:0")
    q, kc, vc = c.q.to(dev), c.past_k.to(dev), c.past_v.to(dev)
    sink = None if c.head_sink is None else c.head_sink.to(dev)
    nonpad = torch.tensor(lengths, dtype=torch.int64, device=dev)
    p = gqa.params_from_dict(c.params)
    ws = torch.zeros(max(16, gqa.gqa_workspace_bytes(p)), dtype=torch.uint8, device=dev)
    out = torch.full_like(q, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    gqa.check(gqa.gqa_attention_nonpad(p, nonpad, q, kc, vc, sink, out, ws, status), "nonpad")
    torch.cuda.synchronize()
    ref = oracle.attention_nonpad(c.params, storage(c.q), storage(c.past_k), storage(c.past_v),
                                  np.array(lengths, dtype=np.int64), None if sink is None else c.head_sink.numpy())
    return out.double().cpu().numpy().reshape(ref.shape), ref, int(status.item())


@pytest.mark.parametrize("name", list(CASES))
def test_nonpad_matches_oracle(name):
    w, lengths = CASES[name]
    got, ref, st = run(w, lengths)
    assert st == 0
    assert_close(got, ref, w.dtype, name)


def test_nonpad_rejects_lengths_that_cannot_hold_the_queries():
    from sliding_window_gb300 import gqa
    w = Workload("np_bad", 605, "decode", "bf16", 3, 16, 4, 128, 2, 256, 0, 0, windows=(-1,), head_sink=True)
    got, ref, st = run(w, [1, 100, 256])
    assert st & gqa.GQA_DEV_BAD_SEQLEN
    assert (got[0] == 0).all()                     # one valid key for two queries: rejected
    assert_close(got[1:], ref[1:], w.dtype, "valid sequences")
