"""Decode parity: the split-KV kernel (and the SIMT kernel outside its envelope) against the
fp64 oracle on the same rounded inputs, plus the device-status paths and robustness to
stale-slot garbage (OpenVINO PR #37423 "Sliding window" / "smooth_softmax / head_sink" /
"Testing"; tract PR #2645 "What changed"; onnx-light-cpu "Attention Kernel Design")."""
import itertools
import zlib

import numpy as np
import pytest
import torch

from gpu_util import assert_close, oracle_ref, out_rows, run_gpu
from helpers import storage
from sliding_window_gb300.inputs import Workload, make_case

pytestmark = pytest.mark.gpu

SWEEP = list(itertools.product(
    ["bf16", "f16"],
    [(128, 8, 1), (128, 4, 4), (128, 1, 3), (64, 8, 8), (64, 16, 1), (128, 32, 1), (128, 16, 4)],  # (D, G, curr)
    [-1, 1, 7, 300],
    ["none", "smooth", "head"],
    [0.0, 20.0],
))


def small_case(dtype, D, G, curr, window, sink, softcap, seed=0, cap=3000, B=3, Hkv=2, lo=0, garbage="normal",
               rotary=0):
    w = Workload("dec", 300 + seed, "decode", dtype, B, G * Hkv, Hkv, D, curr, cap, lo, cap - curr,
                 windows=(window,), softcap=softcap, head_sink=sink == "head", smooth_softmax=int(sink == "smooth"),
                 do_rotary=rotary, rope_len=cap + 16 if rotary else 0)
    return make_case(w, seed_offset=seed, garbage=garbage)


@pytest.mark.parametrize("dtype,dgc,window,sink,softcap", SWEEP)
def test_decode_parity_sweep(dtype, dgc, window, sink, softcap):
    D, G, curr = dgc
    c = small_case(dtype, D, G, curr, window, sink, softcap, seed=zlib.crc32(repr((dtype, dgc, window, sink, softcap)).encode()) % 97)
    r = run_gpu(c, "decode")
    assert r["status"] == 0
    ref, pk, pv, st = oracle_ref(c)
    assert st == 0
    np.testing.assert_array_equal(storage(r["present_k"]), pk)
    np.testing.assert_array_equal(storage(r["present_v"]), pv)
    assert_close(out_rows(r["out"], c), ref, dtype, "decode %s" % ((dtype, dgc, window, sink, softcap),))


@pytest.mark.parametrize("seqlens", [[0, 1, 2], [255, 256, 257], [2999, 2998, 1000], [4096 - 1, 511, 512]])
def test_decode_chunk_boundaries(seqlens):
    """Past lengths on and around chunk (256) and tile (64) boundaries, one to many chunks."""
    cap = 4096
    w = Workload("decb", 320, "decode", "bf16", 3, 16, 2, 128, 1, cap, 0, cap - 1, head_sink=True)
    c = make_case(w, seqlens=np.array(seqlens, np.int32))
    r = run_gpu(c, "decode")
    ref, *_ = oracle_ref(c)
    assert_close(out_rows(r["out"], c), ref, "bf16")


def plan_splits(B, Hkv, cap, window, curr):
    """Chunks per group as the library plans them (mirrors the host planner's rule)."""
    lmax = cap if window < 0 else min(cap, window + curr - 1)
    s = max(-(-608 // (B * Hkv)), -(-lmax // 4096))
    return min(64, max(1, min(s, max(1, -(-lmax // 256)))))


@pytest.mark.parametrize("dgc", [(128, 8, 1), (128, 4, 4), (128, 8, 4), (64, 16, 4), (64, 8, 1)])
@pytest.mark.parametrize("cap,S", [(520, 3), (1100, 5), (2000, 8)])
@pytest.mark.parametrize("sink,softcap", [("head", 0.0), ("smooth", 30.0), ("none", 0.0)])
def test_decode_cluster_combine(dgc, cap, S, sink, softcap):
    """Groups of 2..8 chunks combined through distributed shared memory: sequences of one
    chunk (finished in place), of fewer chunks than the cluster (idle CTAs still take part)
    and of every chunk; output slices that do not divide evenly among the CTAs."""
    D, G, curr = dgc
    B, Hkv = 4, 2
    assert plan_splits(B, Hkv, cap, -1, curr) == S and B * Hkv * S <= 304
    w = Workload("decc", 340, "decode", "f16" if softcap else "bf16", B, G * Hkv, Hkv, D, curr, cap, 0, cap - curr,
                 softcap=softcap, head_sink=sink == "head", smooth_softmax=int(sink == "smooth"))
    seqlens = np.array([0, 70, cap // 2 + 3, cap - curr], np.int32)
    c = make_case(w, seed_offset=S, seqlens=seqlens)
    r = run_gpu(c, "decode")
    assert r["status"] == 0
    ref, pk, pv, st = oracle_ref(c)
    assert st == 0
    np.testing.assert_array_equal(storage(r["present_k"]), pk)
    np.testing.assert_array_equal(storage(r["present_v"]), pv)
    assert_close(out_rows(r["out"], c), ref, w.dtype, "cluster %s" % ((dgc, cap, S, sink, softcap),))


@pytest.mark.parametrize("garbage", ["huge", "nonfinite"])
def test_stale_slots_do_not_change_output(garbage):
    base = small_case("bf16", 128, 8, 2, 50, "head", 0.0, seed=5)
    other = small_case("bf16", 128, 8, 2, 50, "head", 0.0, seed=5, garbage=garbage)
    a = run_gpu(base, "decode")["out"]
    b = run_gpu(other, "decode")["out"]
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_rotary_multi_token_decode():
    c = small_case("f16", 128, 8, 4, 4096, "smooth", 0.0, seed=6, cap=6000, rotary=1)
    r = run_gpu(c, "decode")
    ref, pk, pv, _ = oracle_ref(c)
    np.testing.assert_array_equal(storage(r["present_k"]), pk)
    assert_close(out_rows(r["out"], c), ref, "f16")


def test_attention_only_matches_full_call():
    c = small_case("f16", 128, 8, 4, 1000, "smooth", 0.0, seed=7, cap=3000, rotary=1)
    full = run_gpu(c, "decode")["out"]
    split = run_gpu(c, "decode", attend_only=True)["out"]
    assert torch.equal(full.view(torch.int16), split.view(torch.int16))


def test_separate_present_buffer():
    c = small_case("bf16", 128, 4, 2, -1, "head", 0.0, seed=8)
    r = run_gpu(c, "decode", separate_present=True)
    ref, pk, pv, _ = oracle_ref(c)
    B, Hkv = 3, 2
    got_k = storage(r["present_k"])
    for b in range(B):
        tot = int(c.seqlens_k[b]) + 2
        np.testing.assert_array_equal(got_k[b, :, :tot], pk[b, :, :tot])
    assert_close(out_rows(r["out"], c), ref, "bf16")


def test_workspace_reused_across_calls():
    """Every call leaves its tickets at zero: repeated calls on one workspace agree."""
    c = small_case("bf16", 128, 8, 1, -1, "head", 0.0, seed=9, cap=4000, lo=3000)
    r1 = run_gpu(c, "decode")
    r2 = run_gpu(c, "decode", workspace=r1["workspace"])
    r3 = run_gpu(c, "decode", workspace=r1["workspace"])
    assert torch.equal(r1["out"].view(torch.int16), r2["out"].view(torch.int16))
    assert torch.equal(r1["out"].view(torch.int16), r3["out"].view(torch.int16))


def test_bad_sequences_give_zeros_and_status():
    w = Workload("decbad", 330, "decode", "bf16", 4, 8, 2, 128, 2, 512, 0, 500, windows=(64,), head_sink=True)
    c = make_case(w, seqlens=np.array([100, -5, 511, 300], np.int32))
    r = run_gpu(c, "decode")
    assert r["status"] == 1
    out = out_rows(r["out"], c)
    assert np.all(out[1] == 0) and np.all(out[2] == 0)
    ref, *_ = oracle_ref(c)
    assert_close(out[[0, 3]], ref[[0, 3]], "bf16")


def test_status_is_ored_not_overwritten():
    w = Workload("decor", 331, "decode", "bf16", 2, 8, 2, 128, 1, 512, 0, 500)
    c = make_case(w, seqlens=np.array([100, 600], np.int32))
    r = run_gpu(c, "decode", status_init=4)
    assert r["status"] == 5
