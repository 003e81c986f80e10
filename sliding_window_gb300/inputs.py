"""Seeded synthetic workloads for sliding-window GQA over a KV cache.

This module only draws and lays out inputs (Gaussian Q/K/V, uniform past lengths, stale
garbage beyond each past, RoPE cos/sin tables and per-head sinks).  It holds none of the
attention arithmetic, so the CUDA path and the CPU oracle can both be fed from it without
sharing any of the method.

The five named workloads follow the shapes of the pages' cases: a tiny fp32 first prompt,
a windowed single-token decode, a long windowed prefill with per-head sink and softcap,
a multi-token speculative decode with rotary over two layers with alternating windows,
and a large-batch long-context decode.  Layouts:
    q [B, curr, Hq*D], k/v [B, curr, Hkv*D], past/present [B, Hkv, cap, D],
    cos/sin [rope_len, D/2], seqlens_k int32 [B], head_sink fp32 [Hq].
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np
import torch

TORCH_DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    index: int              # seed offset: torch seed 1000+index, numpy seed 2000+index
    mode: str               # "prefill" or "decode"
    dtype: str              # "f32" | "f16" | "bf16"
    batch: int
    q_heads: int
    kv_heads: int
    head_dim: int
    q_len: int              # new tokens per sequence (S for a prompt, curr for decode)
    cap: int                # present (and past) capacity in tokens
    past_lo: int            # seqlens_k drawn uniformly from [past_lo, past_hi]
    past_hi: int
    windows: tuple = (-1,)  # one entry per layer; -1 = no window
    causal: int = 1
    scale: float = 0.0      # 0 -> 1/sqrt(D)
    softcap: float = 0.0
    head_sink: bool = False  # per-head sink drawn N(0,1)
    smooth_softmax: int = 0  # zero sink when head_sink is absent
    do_rotary: int = 0
    rope_len: int = 0
    rope_theta: float = 10000.0
    garbage_std: float = 10.0
    kv_ring: int = 0        # 1: the cache is a ring of `cap` slots, position p in slot p % cap
    kv_paged: int = 0       # 1: the cache is a shared pool of 64-position pages behind a block table
    mask: str = ""          # "add": an additive attention bias [B, 1, S, cap] of the dtype, N(0,1);
                            # "blocks": a block-sparse boolean mask [B, 1, S, cap] (block_live)
    v_head_dim: int = 0     # Dv; 0: the same as head_dim
    kv_q8: int = 0          # the cache holds one-byte codes with one scale per kv head for K and V: 1 f8 E4M3, 2 int8

    @property
    def layers(self) -> int:
        return len(self.windows)

    def params(self, layer: int = 0) -> dict:
        """The op attributes of one layer as a plain dict (keys shared by the oracle
        wrapper and the C-ABI binding)."""
        return dict(batch=self.batch, q_heads=self.q_heads, kv_heads=self.kv_heads,
                    head_dim=self.head_dim, q_len=self.q_len, cap_past=self.cap,
                    cap_present=self.cap, rope_len=self.rope_len, dtype=self.dtype,
                    scale=self.scale, softcap=self.softcap, window=self.windows[layer],
                    causal=self.causal, do_rotary=self.do_rotary, rotary_interleaved=0,
                    smooth_softmax=self.smooth_softmax, kv_ring=self.kv_ring, v_head_dim=self.v_head_dim)

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("prefill_fp32_tiny", 0, "prefill", "f32", 1, 4, 2, 64, 128, 128, 0, 0,
                 windows=(-1,), scale=1.0 / 8.0),
        Workload("decode_window_bf16", 1, "decode", "bf16", 8, 32, 8, 128, 1, 4096, 512, 4095,
                 windows=(1024,)),
        Workload("prefill_sink_softcap_bf16", 2, "prefill", "bf16", 2, 64, 8, 128, 8192, 8192, 0, 0,
                 windows=(4096,), softcap=50.0, head_sink=True),
        Workload("specdecode_rotary_f16", 3, "decode", "f16", 16, 32, 4, 128, 4, 16384, 1024, 16380,
                 windows=(-1, 4096), smooth_softmax=1, do_rotary=1, rope_len=32768),
        Workload("decode_long_bf16", 4, "decode", "bf16", 64, 64, 8, 128, 1, 32768, 8192, 32767,
                 windows=(-1,), head_sink=True),
        # the windowed decode over a ring of 1024 slots (W + curr - 1 = 1024): the same band,
        # a quarter of the cache memory
        Workload("decode_window_ring_bf16", 5, "decode", "bf16", 8, 32, 8, 128, 1, 1024, 512, 4095,
                 windows=(1024,), kv_ring=1),
        # the windowed decode over a paged cache: the same rows in a shuffled pool of pages
        Workload("decode_window_paged_bf16", 6, "decode", "bf16", 8, 32, 8, 128, 1, 4096, 512, 4095,
                 windows=(1024,), kv_paged=1),
        # the windowed decode with a V head dim of 64 under a Q/K head dim of 128
        Workload("decode_window_vdim_bf16", 8, "decode", "bf16", 8, 32, 8, 128, 1, 4096, 512, 4095,
                 windows=(1024,), v_head_dim=64),
        # the windowed decode over an f8 cache (one byte per cached element)
        Workload("decode_window_q8_bf16", 9, "decode", "bf16", 8, 32, 8, 128, 1, 4096, 512, 4095,
                 windows=(1024,), kv_q8=1),
        # the same with an int8 cache
        Workload("decode_window_i8_bf16", 10, "decode", "bf16", 8, 32, 8, 128, 1, 4096, 512, 4095,
                 windows=(1024,), kv_q8=2),
        # the long prompt with a dense additive attention bias, broadcast over the heads
        Workload("prefill_bias_bf16", 7, "prefill", "bf16", 2, 64, 8, 128, 8192, 8192, 0, 0,
                 windows=(4096,), softcap=50.0, head_sink=True, mask="add"),
        # the long prompt with a block-sparse boolean mask: half of the 128 x 128 blocks removed
        Workload("prefill_blocksparse_bf16", 11, "prefill", "bf16", 2, 64, 8, 128, 8192, 8192, 0, 0,
                 windows=(4096,), softcap=50.0, head_sink=True, mask="blocks"),
    ]
}

WORKLOAD_ORDER = ["prefill_fp32_tiny", "decode_window_bf16", "prefill_sink_softcap_bf16",
                  "specdecode_rotary_f16", "decode_long_bf16"]


MASK_BLOCK = 128  # rows and keys of one block of the "blocks" mask


def block_live(qb, kb):
    """Whether block (query block qb, key block kb) of the "blocks" mask keeps its keys."""
    return (qb + kb) % 2 == 0


def rope_tables(rope_len: int, head_dim: int, theta: float, dtype: str, device="cpu"):
    """cos/sin tables [rope_len, D/2]: angle(pos, k) = pos * theta^(-2k/D), in fp64, then
    rounded to the storage dtype."""
    half = head_dim // 2
    pos = torch.arange(rope_len, dtype=torch.float64)
    inv = theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / head_dim)
    ang = pos[:, None] * inv[None, :]
    t = TORCH_DTYPES[dtype]
    return torch.cos(ang).to(t).to(device), torch.sin(ang).to(t).to(device)


def draw_seqlens(w: Workload, seed_offset: int = 0) -> np.ndarray:
    rng = np.random.default_rng(2000 + w.index + 7919 * seed_offset)
    hi = w.past_hi if w.kv_ring else min(w.past_hi, w.cap - w.q_len)
    return rng.integers(w.past_lo, hi, endpoint=True, size=w.batch).astype(np.int32)


def _fill_garbage(t: torch.Tensor, mode: str, std: float, gen: torch.Generator):
    if mode == "normal":
        t.normal_(0.0, std, generator=gen)
    elif mode == "huge":
        t.copy_(torch.where(torch.rand(t.shape, generator=gen, device=t.device) < 0.5,
                            torch.tensor(1e4, device=t.device), torch.tensor(-1e4, device=t.device)))
    elif mode == "nonfinite":
        r = torch.rand(t.shape, generator=gen, device=t.device)
        vals = torch.where(r < 0.34, torch.tensor(float("nan"), device=t.device),
                           torch.where(r < 0.67, torch.tensor(float("inf"), device=t.device),
                                       torch.tensor(float("-inf"), device=t.device)))
        t.copy_(vals)
    else:
        raise ValueError(mode)


@dataclass
class Case:
    """One layer's worth of inputs, as torch tensors on `device`."""
    w: Workload
    layer: int
    params: dict
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    past_k: torch.Tensor
    past_v: torch.Tensor
    seqlens_k: torch.Tensor
    cos: torch.Tensor | None
    sin: torch.Tensor | None
    head_sink: torch.Tensor | None
    extra: dict = field(default_factory=dict)


def make_case(w: Workload, layer: int = 0, device="cpu", seed_offset: int = 0, garbage: str = "normal",
              seqlens: np.ndarray | None = None) -> Case:
    """Draw one layer of a workload.  Past rows [0, seqlens_k[b]) are N(0,1); rows beyond
    are stale garbage (N(0, garbage_std^2), +-1e4, or NaN/+-Inf) that must never be read.
    For a ring cache the resident slots (every slot once the past fills the ring) are
    N(0,1) and only slots of a ring that has not wrapped yet hold garbage."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 + w.index + 104729 * layer + 7919 * seed_offset)
    # stale slots draw from their own stream, so the garbage mode never shifts the real data
    junk = torch.Generator(device=dev)
    junk.manual_seed(5000 + w.index + 104729 * layer + 7919 * seed_offset)
    t = TORCH_DTYPES[w.dtype]
    B, Hq, Hkv, D, L, cap = w.batch, w.q_heads, w.kv_heads, w.head_dim, w.q_len, w.cap
    Dv = w.v_head_dim or D

    def randn(*shape):
        return torch.randn(*shape, generator=gen, device=dev, dtype=torch.float32).to(t)

    q = randn(B, L, Hq * D)
    k = randn(B, L, Hkv * D)
    v = randn(B, L, Hkv * Dv)
    seq = draw_seqlens(w, seed_offset) if seqlens is None else np.asarray(seqlens, dtype=np.int32)
    past_k = torch.empty(B, Hkv, cap, D, dtype=t, device=dev)
    past_v = torch.empty(B, Hkv, cap, Dv, dtype=t, device=dev)
    # rows are drawn per sequence so that the large caches never need an fp32 copy in full
    for b in range(B):
        n = min(int(seq[b]), cap) if w.kv_ring else int(seq[b])
        for buf in (past_k, past_v):
            tmp = torch.empty(Hkv, cap, buf.shape[-1], dtype=torch.float32, device=dev)
            tmp[:, :n].normal_(0.0, 1.0, generator=gen)
            _fill_garbage(tmp[:, n:], garbage, w.garbage_std, junk)
            buf[b].copy_(tmp)
            del tmp
    cos = sin = None
    if w.do_rotary:
        cos, sin = rope_tables(w.rope_len, D, w.rope_theta, w.dtype, device=dev)
    sink = None
    if w.head_sink:
        sink = torch.randn(Hq, generator=gen, device=dev, dtype=torch.float32)
    extra = {}
    if w.mask == "add":  # its own stream: the other inputs match the unmasked workload's draw
        mg = torch.Generator(device=dev)
        mg.manual_seed(6000 + w.index + 104729 * layer + 7919 * seed_offset)
        m = torch.empty(B, 1, L, cap, dtype=t, device=dev)
        for b in range(B):
            m[b].copy_(torch.randn(1, L, cap, generator=mg, device=dev, dtype=torch.float32))
        extra["mask"] = m
    elif w.mask == "blocks":  # a fixed checkerboard of 128 x 128 blocks, every key of a live block kept
        qb = torch.arange(L, device=dev) // MASK_BLOCK
        kb = torch.arange(cap, device=dev) // MASK_BLOCK
        live = block_live(qb[:, None], kb[None, :]).to(torch.uint8)
        extra["mask"] = live[None, None].expand(B, 1, L, cap).contiguous()
    elif w.mask:
        raise ValueError(w.mask)
    if w.kv_q8:
        # quantized cache: the past as random codes drawn directly as bytes (f8: finite E4M3
        # codes, sign, exponent field 1..11, fraction; int8: uniform over [-127, 127]), scales
        # U[0.01, 0.02] per kv head; q/k/v stay in the dtype
        qg = torch.Generator(device=dev)
        qg.manual_seed(7000 + w.index + 104729 * layer + 7919 * seed_offset)
        Dv = w.v_head_dim or D

        def codes(*shape):
            if w.kv_q8 == 2:
                return torch.randint(-127, 128, shape, generator=qg, device=dev, dtype=torch.int32).to(
                    torch.int8).view(torch.uint8)
            sign = torch.randint(0, 2, shape, generator=qg, device=dev, dtype=torch.int32) << 7
            expo = torch.randint(1, 12, shape, generator=qg, device=dev, dtype=torch.int32) << 3
            frac = torch.randint(0, 8, shape, generator=qg, device=dev, dtype=torch.int32)
            return (sign | expo | frac).to(torch.uint8)

        extra["k8"] = codes(B, Hkv, cap, D)
        extra["v8"] = codes(B, Hkv, cap, Dv)
        extra["k_scale"] = torch.rand(Hkv, generator=qg, device=dev, dtype=torch.float32) * 0.01 + 0.01
        extra["v_scale"] = torch.rand(Hkv, generator=qg, device=dev, dtype=torch.float32) * 0.01 + 0.01
    return Case(w, layer, w.params(layer), q, k, v, past_k, past_v,
                torch.from_numpy(seq).to(dev), cos, sin, sink, extra)


def small_variant(w: Workload, **kw) -> Workload:
    """A reduced copy of a workload for oracle-speed parity checks (same features)."""
    return replace(w, **kw)
