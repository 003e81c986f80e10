"""Prefill parity: the tcgen05/TMEM tensor-core kernel (f16/bf16) and the fp32 SIMT kernel
against the fp64 oracle on the same rounded inputs (onnx-light-cpu "Attention Kernel
Design" "Compute paths"; OpenVINO PR #37423 "Sliding window", "smooth_softmax /
head_sink"; tract PR #2645 "What changed")."""
import itertools
import zlib

import numpy as np
import pytest

from gpu_util import assert_close, oracle_ref, out_rows, run_gpu
from helpers import storage
from sliding_window_gb300.inputs import Workload, make_case

pytestmark = pytest.mark.gpu


def prefill_case(dtype, D, G, S, window, sink, softcap, causal=1, past=0, cap=None, B=2, Hkv=2, seed=0,
                 garbage="normal", rotary=0):
    cap = cap or (past + S + 37)
    w = Workload("pre", 400 + seed, "prefill", dtype, B, G * Hkv, Hkv, D, S, cap, past, past, windows=(window,),
                 causal=causal, softcap=softcap, head_sink=sink == "head", smooth_softmax=int(sink == "smooth"),
                 do_rotary=rotary, rope_len=cap + 8 if rotary else 0)
    return make_case(w, seed_offset=seed, garbage=garbage)


TC_SWEEP = list(itertools.product(
    ["bf16", "f16"], [128, 64], [1, 100, 128, 300, 700], [-1, 1, 64, 200], ["none", "head"], [0.0, 30.0]))


@pytest.mark.parametrize("dtype,D,S,window,sink,softcap", TC_SWEEP)
def test_prefill_tc_parity(dtype, D, S, window, sink, softcap):
    c = prefill_case(dtype, D, 2, S, window, sink, softcap, seed=zlib.crc32(repr((dtype, D, S, window, sink, softcap)).encode()) % 89)
    r = run_gpu(c, "prefill")
    assert r["status"] == 0
    ref, pk, pv, _ = oracle_ref(c)
    np.testing.assert_array_equal(storage(r["present_k"]), pk)
    assert_close(out_rows(r["out"], c), ref, dtype, "prefill %s" % ((dtype, D, S, window, sink, softcap),))


@pytest.mark.parametrize("causal,window", [(0, -1), (0, 50), (1, 129)])
def test_prefill_tc_noncausal_and_window_edges(causal, window):
    c = prefill_case("bf16", 128, 4, 390, window, "smooth", 0.0, causal=causal, seed=3)
    r = run_gpu(c, "prefill")
    ref, *_ = oracle_ref(c)
    assert_close(out_rows(r["out"], c), ref, "bf16")


@pytest.mark.parametrize("past,S,window", [(1000, 300, -1), (1000, 300, 256), (77, 129, 100), (5000, 64, 4096)])
def test_prefill_over_nonempty_past(past, S, window):
    """A prompt continued over a cached past: bottom-right band, appended at seqlens_k."""
    c = prefill_case("bf16", 128, 8, S, window, "head", 50.0, past=past, seed=4, garbage="nonfinite")
    r = run_gpu(c, "prefill")
    ref, *_ = oracle_ref(c)
    assert_close(out_rows(r["out"], c), ref, "bf16")


def test_prefill_rotary():
    c = prefill_case("f16", 128, 4, 200, 64, "none", 0.0, past=33, rotary=1, seed=5)
    r = run_gpu(c, "prefill")
    ref, pk, *_ = oracle_ref(c)
    np.testing.assert_array_equal(storage(r["present_k"]), pk)
    assert_close(out_rows(r["out"], c), ref, "f16")


@pytest.mark.parametrize("S,window,sink", [(128, -1, "none"), (77, 5, "head"), (260, 64, "smooth")])
def test_prefill_fp32_parity(S, window, sink):
    c = prefill_case("f32", 64, 2, S, window, sink, 0.0, seed=6)
    r = run_gpu(c, "prefill")
    ref, *_ = oracle_ref(c)
    assert_close(out_rows(r["out"], c), ref, "f32")


def test_prefill_stale_garbage_is_masked():
    c = prefill_case("bf16", 128, 2, 200, -1, "head", 0.0, cap=512, seed=7, garbage="nonfinite")
    r = run_gpu(c, "prefill")
    ref, *_ = oracle_ref(c)
    assert_close(out_rows(r["out"], c), ref, "bf16")


@pytest.mark.parametrize("dtype,softcap", [("bf16", 0.0), ("f16", 0.0), ("bf16", 50.0)])
def test_prefill_tc_sharp_scores(dtype, softcap):
    """Scale 1 (scores of standard deviation ~11): exp2 arguments far below -125 in tiles
    with no masked key, whose weights must flush to zero without NaN."""
    w = Workload("presharp", 420, "prefill", dtype, 2, 8, 2, 128, 700, 740, 0, 0, windows=(-1,), scale=1.0,
                 softcap=softcap, head_sink=True)
    c = make_case(w, seed_offset=1)
    r = run_gpu(c, "prefill")
    assert r["status"] == 0
    ref, *_ = oracle_ref(c)
    assert_close(out_rows(r["out"], c), ref, dtype, "sharp %s" % ((dtype, softcap),))


@pytest.mark.parametrize("softcap", [0.5, 2.0])
def test_prefill_tc_small_softcap_masks_exactly(softcap):
    """With a small softcap every capped score is within [-softcap, softcap], so a key removed
    by the band must get exactly zero weight, not the weight of a score of -softcap."""
    c = prefill_case("bf16", 128, 2, 300, 70, "head", softcap, seed=11)
    r = run_gpu(c, "prefill")
    ref, *_ = oracle_ref(c)
    assert_close(out_rows(r["out"], c), ref, "bf16", "softcap %g" % softcap)
