"""The bench's algorithmic accounting, checked against counts written out by hand from the
definitions: decode reads every visible K row (D elements) and V row (Dv elements) of each
(b, kv head) once, plus q read, out written and the new K/V read and appended; prefill does
2·D (scores) + 2·Dv (weighted sum) flops per visible (query, key) pair.  Also the launch
count the bench claims per layer."""
import dataclasses

import numpy as np
import pytest

import bench
from sliding_window_gb300.inputs import WORKLOADS, make_case


def test_decode_bytes_by_hand():
    w = WORKLOADS["decode_window_bf16"].scaled(batch=2)
    seqs = [np.array([100, 3000], dtype=np.int32)]
    # band lengths: window 1024 -> seq 100: [0, 101) = 101 keys; seq 3000: [1977, 3001) = 1024 keys
    keys = 101 + 1024
    kv = keys * w.kv_heads * (128 + 128) * 2
    io = 2 * 1 * 2 * (w.q_heads + 2 * w.kv_heads) * (128 + 128)
    units, kunits, unit = bench.step_work(w, seqs)
    assert unit == "GB/s"
    assert units == pytest.approx((kv + io) / 1e9, rel=0, abs=1e-15)
    append = 2 * 2 * 1 * w.kv_heads * 256 * 2
    assert kunits == pytest.approx((kv + io - append) / 1e9, rel=0, abs=1e-15)


def test_decode_bytes_with_a_narrower_v():
    w = WORKLOADS["decode_window_vdim_bf16"].scaled(batch=1)
    seqs = [np.array([5000 - 1], dtype=np.int32)]
    units, _, _ = bench.step_work(w, seqs)
    kv = 1024 * w.kv_heads * (128 + 64) * 2
    io = 1 * 1 * 2 * (w.q_heads + 2 * w.kv_heads) * (128 + 64)
    assert units == pytest.approx((kv + io) / 1e9, rel=0, abs=1e-15)


@pytest.mark.parametrize("dv", [0, 64])
def test_prefill_flops_by_hand(dv):
    w = WORKLOADS["prefill_sink_softcap_bf16"].scaled(batch=1, q_len=10, cap=10, windows=(4,), v_head_dim=dv)
    seqs = [np.array([0], dtype=np.int32)]
    # causal with window 4 over a 10-token prompt: row i sees min(i + 1, 4) keys
    pairs = sum(min(i + 1, 4) for i in range(10)) * w.q_heads
    d = 128 + (dv or 128)
    flops, kflops, unit = bench.step_work(w, seqs)
    assert unit == "TFLOP/s" and flops == kflops == pytest.approx(2 * d * pairs / 1e12, rel=1e-12)


@pytest.mark.parametrize("name,launches", [
    ("prefill_fp32_tiny", 2), ("decode_window_bf16", 1), ("prefill_sink_softcap_bf16", 2),
    ("specdecode_rotary_f16", 1), ("decode_long_bf16", 1), ("decode_window_ring_bf16", 1),
    ("decode_window_paged_bf16", 1), ("decode_window_vdim_bf16", 1), ("prefill_bias_bf16", 2),
    ("decode_window_q8_bf16", 1), ("decode_window_i8_bf16", 1), ("prefill_blocksparse_bf16", 3)])
def test_kernels_per_layer(name, launches):
    """One fused launch for the split-KV decode (it appends and rotates itself), else the
    RoPE/append kernel and the attention kernel, with the block-map kernel between them for a
    boolean mask.  The speculative decode's 8 q heads x 4 tokens = 32 rows per group at
    D = 128 fit the split kernel."""
    w = WORKLOADS[name]
    assert bench.kernels_per_layer(w) == launches


def test_f8_cache_bytes_by_hand():
    """An f8 cache: one byte per cached element read and appended; q, out and the new rows
    read in the dtype."""
    w = WORKLOADS["decode_window_q8_bf16"].scaled(batch=1)
    seqs = [np.array([2000], dtype=np.int32)]
    units, kunits, _ = bench.step_work(w, seqs)
    kv = 1024 * w.kv_heads * 256 * 1
    io = 1 * 1 * (w.q_heads * 2 + w.kv_heads * (2 + 1)) * 256
    assert units == pytest.approx((kv + io) / 1e9, rel=0, abs=1e-15)
    assert kunits == pytest.approx((kv + io - w.kv_heads * 256 * 3) / 1e9, rel=0, abs=1e-15)


@pytest.mark.parametrize("name,kernel,bound", [
    ("decode_long_bf16", "decode_split", "hbm"), ("decode_window_bf16", "decode_split", "hbm"),
    ("specdecode_rotary_f16", "decode_split", "hbm"), ("prefill_sink_softcap_bf16", "prefill_tc", "tensor"),
    ("prefill_fp32_tiny", "attn_simt", "alu")])
def test_dominant_kernel_and_bound(name, kernel, bound):
    w = WORKLOADS[name]
    assert bench.kernel_name(w) == kernel
    b, peak, unit, _ = bench.roofline_peak(w, {"hbm_gbs": 6777.6, "bf16_tflops": 1929.0}, "measured")
    assert b == bound
    assert unit == ("GB/s" if bound == "hbm" else "TFLOP/s")
    if bound == "alu":  # 152 SMs x 128 FP32 lanes x 2 flop x 2.07 GHz
        assert peak == pytest.approx(80.55, abs=0.01)


def test_headline_is_the_largest_single_gpu_workload_and_subrecords_cover_the_rest():
    named = ["prefill_fp32_tiny", "decode_window_bf16", "prefill_sink_softcap_bf16", "specdecode_rotary_f16",
             "decode_long_bf16"]
    assert bench.HEADLINE == "decode_long_bf16"
    assert set(bench.SUB_WORKLOADS) | {bench.HEADLINE} == set(named)


@pytest.mark.parametrize("q_len,cap,window", [(300, 300, -1), (700, 700, 200), (1000, 1000, 4096)])
def test_block_sparse_pairs_by_brute_force(q_len, cap, window):
    """The FLOP count of the block-sparse boolean workload counts the keys its mask keeps
    inside the band: brute force over the mask the input generator builds."""
    w = WORKLOADS["prefill_blocksparse_bf16"].scaled(batch=1)
    w = dataclasses.replace(w, q_len=q_len, cap=cap, windows=(window,), q_heads=1, kv_heads=1)
    c = make_case(w, device="cpu")
    m = c.extra["mask"][0, 0].numpy().astype(bool)
    seqs = [np.array([0], dtype=np.int32)]
    qa = np.arange(q_len)[:, None]
    k = np.arange(cap)[None, :]
    band = (k <= qa) & ((window < 0) | (qa - k < window))
    want = int((band & m).sum()) * 2 * (w.head_dim + w.head_dim)
    units, kunits, _ = bench.step_work(w, seqs)
    assert units == pytest.approx(want / 1e12, rel=0, abs=1e-18)
    assert 0 < (band & m).sum() < band.sum()
