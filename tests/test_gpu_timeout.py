"""The failure path of the bounded pipeline waits (onnx-light-cpu "Attention Kernel Design",
"Scheduling, precision, and invariants": invalid situations fail explicitly).

With the test hook gqa_test_stall_waits(cycles) every launch of the split-KV decode and the
tensor-core prefill kernels first waits on an mbarrier that nothing completes, bounded by
`cycles` SM cycles.  The wait gives up, the CTA lets the copies and MMAs it already issued
land, frees its tensor memory and returns: the call returns, the device status carries
GQA_DEV_TIMEOUT, and the GPU stays usable.  The next normal call on the same workspace (its
tickets back at zero) matches the fp64 oracle."""
import numpy as np
import pytest
import torch

from gpu_util import assert_close, oracle_ref, out_rows, run_gpu
from sliding_window_gb300.inputs import Workload, make_case

pytestmark = pytest.mark.gpu

CASES = {
    # one wave of 2..8 chunks per group: combined in distributed shared memory
    "decode_cluster": Workload("to_dc", 501, "decode", "bf16", 4, 32, 8, 128, 1, 2048, 900, 2000,
                               windows=(-1,), head_sink=True),
    # 64 chunks per group: partials in the workspace, combined by the last CTA (tickets)
    "decode_ticket": Workload("to_dt", 502, "decode", "bf16", 1, 8, 2, 128, 1, 16384, 16000, 16383,
                              windows=(-1,), head_sink=True),
    "prefill": Workload("to_pf", 503, "prefill", "bf16", 1, 8, 2, 128, 300, 384, 0, 0, windows=(200,),
                        softcap=30.0, head_sink=True),
}


@pytest.fixture
def gqa():
    from sliding_window_gb300 import gqa as g
    yield g
    g.gqa_test_stall_waits(0)


@pytest.mark.parametrize("name", list(CASES))
def test_wait_gives_up_then_next_call_is_correct(gqa, name):
    w = CASES[name]
    case = make_case(w)
    p = gqa.params_from_dict(case.params)
    ws = torch.zeros(max(16, gqa.gqa_workspace_bytes(p)), dtype=torch.uint8, device="cuda:0")
    if name == "decode_ticket":
        assert gqa.gqa_workspace_bytes(p) > 0  # the ticket path really uses the workspace
    # a wait that nothing completes, given 200k SM cycles (about 0.1 ms)
    assert gqa.gqa_test_stall_waits(200_000) == gqa.GQA_OK
    r = run_gpu(case, w.mode, workspace=ws)
    assert r["status"] & gqa.GQA_DEV_TIMEOUT
    # normal operation on the same workspace
    assert gqa.gqa_test_stall_waits(0) == gqa.GQA_OK
    r = run_gpu(make_case(w), w.mode, workspace=ws)
    assert r["status"] == 0
    ref, pk, pv, st = oracle_ref(case)
    assert st == 0
    assert_close(out_rows(r["out"], case), ref, w.dtype, name)
