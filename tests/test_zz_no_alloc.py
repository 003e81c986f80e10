"""The workspace-free decode entry point, gqa_attention_decode_noalloc.

It exists for callers that cannot allocate device memory where they run attention (a
plugin inside an engine that owns all device memory, a latency-critical loop where a
cudaMalloc is not acceptable); it keeps its scratch in a static device array of the
library.  These tests call it through the C ABI twice in a row and compare each output
with gqa_attention_decode's on the same inputs, within the decode parity tolerance, and
with the fp64 oracle on sampled rows.
Collected last on purpose, so that a failure here never hides another test's result."""
import numpy as np
import pytest
import torch

from gpu_util import assert_close, oracle_ref, out_rows
from sliding_window_gb300.inputs import Workload, make_case

pytestmark = pytest.mark.gpu


def _tensors(case, dev):
    return {n: (None if getattr(case, n) is None else getattr(case, n).to(dev))
            for n in ("q", "k", "v", "past_k", "past_v", "seqlens_k", "cos", "sin", "head_sink")}


@pytest.mark.parametrize("case_id", ["window_decode", "rotary_multi_token"])
def test_noalloc_matches_workspace_decode_twice(case_id):
    from sliding_window_gb300 import gqa
    if case_id == "window_decode":
        # a band long enough to be split across CTAs, so the call needs its chunk partials
        w = Workload("noalloc_win", 76, "decode", "bf16", 8, 32, 8, 128, 1, 16384, 9000, 16383, windows=(12000,),
                     head_sink=True)
        case = make_case(w)
    else:
        w = Workload("noalloc_rot", 77, "decode", "f16", 4, 32, 4, 128, 4, 6000, 1000, 5990, windows=(-1,),
                     smooth_softmax=1, do_rotary=1, rope_len=6000)
        case = make_case(w)
    dev = torch.device("cuda:0")
    t = _tensors(case, dev)
    p = gqa.params_from_dict(case.params)
    need = gqa.gqa_workspace_bytes(p)
    assert 0 < need <= gqa.NOALLOC_SCRATCH_BYTES  # the case really uses scratch
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    # the existing entry point with a caller-allocated workspace
    pk, pv = t["past_k"].clone(), t["past_v"].clone()
    ref = torch.empty_like(t["q"])
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    gqa.check(gqa.gqa_attention_decode(p, t["q"], t["k"], t["v"], pk, pv, t["seqlens_k"], t["cos"], t["sin"],
                                       t["head_sink"], ref, pk, pv, ws, status))
    torch.cuda.synchronize()
    ref64 = ref.double().cpu().numpy()
    # the oracle on the same rounded inputs, on a sample of rows (every sequence, first and
    # last q head of each kv group)
    G = w.q_heads // w.kv_heads
    rows = np.array([(b * w.q_len + i) * w.q_heads + h for b in range(w.batch) for i in range(w.q_len)
                     for h in range(w.q_heads) if h % G in (0, G - 1)], dtype=np.int64)
    want, _, _, st = oracle_ref(case, rows=rows)
    assert st == 0
    for _ in range(2):  # two calls in a row share (and must clean up) the static scratch
        qk, qv = t["past_k"].clone(), t["past_v"].clone()
        out = torch.full_like(t["q"], float("nan"))
        gqa.check(gqa.gqa_attention_decode_noalloc(p, t["q"], t["k"], t["v"], qk, qv, t["seqlens_k"], t["cos"],
                                                   t["sin"], t["head_sink"], out, qk, qv, status))
        torch.cuda.synchronize()
        assert status.item() == 0
        assert_close(out.double().cpu().numpy(), ref64, case.w.dtype, "noalloc vs workspace decode")
        assert_close(out_rows(out, case, rows), want, case.w.dtype, "noalloc vs oracle")
        assert torch.equal(qk.view(torch.int16), pk.view(torch.int16))


def test_noalloc_rejects_params_beyond_its_scratch():
    from sliding_window_gb300 import gqa
    p = gqa.params(batch=256, q_heads=64, kv_heads=8, head_dim=128, q_len=4, cap_present=65536, dtype="bf16")
    assert gqa.gqa_workspace_bytes(p) > gqa.NOALLOC_SCRATCH_BYTES
    dev = torch.device("cuda:0")
    dummy = torch.zeros(16, dtype=torch.uint8, device=dev)
    rc = gqa.gqa_attention_decode_noalloc(p, dummy, dummy, dummy, None, None, dummy, None, None, None, dummy,
                                          dummy, dummy, None)
    assert rc == gqa.GQA_ERR_WORKSPACE
