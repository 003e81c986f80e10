"""Python binding of libgqa.so (ctypes): the same entry points as include/gqa.h, with
argument marshalling only.  Tensors are passed as device pointers; every step of the
computation runs in the library's CUDA kernels.  Importing this module loads the library
and raises if it has not been built (there is no fallback of any kind).

    from sliding_window_gb300 import gqa
    p = gqa.params(batch=..., q_heads=..., ...)          # a gqa_params struct
    ws = torch.zeros(gqa.gqa_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    gqa.check(gqa.gqa_attention_decode(p, q, k, v, past_k, past_v, seqlens_k, cos, sin,
                                       head_sink, out, present_k, present_v, ws, status))
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# GQA_CHECKED_BUILD=1: the bounds-checked debug library (build(checked=True))
LIB_PATH = os.path.join(_HERE, "_build_checked" if os.environ.get("GQA_CHECKED_BUILD") == "1" else "_build",
                        "libgqa.so")

GQA_OK = 0
GQA_ERR_INVALID_ARG = 1
GQA_ERR_UNSUPPORTED = 2
GQA_ERR_CAPACITY = 3
GQA_ERR_CUDA = 4
GQA_ERR_WORKSPACE = 5
GQA_DEV_BAD_SEQLEN = 1
GQA_DEV_BAD_ROPE_POS = 2
GQA_DEV_TIMEOUT = 4
GQA_DEV_BAD_PAGE = 8
GQA_DEV_BOUNDS = 16  # bounds-checked debug build only
DTYPES = {"f32": 0, "f16": 1, "bf16": 2}
TORCH_DTYPE_CODES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}

EXPORTED = ["gqa_workspace_bytes", "gqa_attention_prefill", "gqa_attention_decode", "gqa_rope_append_kv",
            "gqa_status_string", "gqa_abi_version", "gqa_attention_decode_noalloc", "gqa_attention_decode_paged",
            "gqa_attention_decode_masked", "gqa_attention_prefill_masked", "gqa_attention_decode_q8",
            "gqa_attention_prefill_q8", "gqa_test_stall_waits", "gqa_attention_nonpad",
            "gqa_attention_prefill_paged", "gqa_attention_decode_i8", "gqa_attention_prefill_i8"]
MASK_KEEP, MASK_ADD = 1, 2
PAGE = 64  # positions per page of a paged cache
NOALLOC_SCRATCH_BYTES = 32 << 20  # GQA_NOALLOC_SCRATCH_BYTES


class GqaParams(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("q_heads", ctypes.c_int32), ("kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("q_len", ctypes.c_int32), ("cap_past", ctypes.c_int32),
                ("cap_present", ctypes.c_int32), ("rope_len", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("scale", ctypes.c_float), ("softcap", ctypes.c_float), ("window", ctypes.c_int32),
                ("causal", ctypes.c_int32), ("do_rotary", ctypes.c_int32), ("rotary_interleaved", ctypes.c_int32),
                ("smooth_softmax", ctypes.c_int32), ("kv_ring", ctypes.c_int32), ("v_head_dim", ctypes.c_int32)]


class GqaMask(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("kind", ctypes.c_int32), ("keys", ctypes.c_int32),
                ("stride_b", ctypes.c_int64), ("stride_h", ctypes.c_int64), ("stride_i", ctypes.c_int64)]


def mask_from_tensor(m, kind: int) -> GqaMask:
    """A gqa_mask for a CUDA tensor of 4 dims [B or 1, Hq or 1, q_len or 1, keys] (size-1
    dims broadcast; the key dim contiguous).  kind MASK_KEEP: uint8/bool; MASK_ADD: the dtype."""
    if m.dim() != 4 or m.stride(3) != 1:
        raise ValueError("a mask is a 4-dim tensor with contiguous keys")
    if not m.is_cuda:
        raise ValueError("libgqa takes device tensors; got a mask on %s" % m.device)
    st = [0 if m.shape[d] == 1 else m.stride(d) for d in range(3)]  # any other strides are explicit
    g = GqaMask(m.data_ptr(), kind, m.shape[3], st[0], st[1], st[2])
    g.tensor = m  # the struct holds a raw pointer: keep the memory alive as long as the struct
    return g


class GqaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        super().__init__("%s: gqa status %d (%s)" % (what or "gqa call", status, gqa_status_string(status)))
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libgqa.so is not built (%s); run `python -c \"import __graft_entry__ as g; "
                          "g.build()\"` on a machine with the CUDA toolkit" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
    pp = ctypes.POINTER(GqaParams)
    lib.gqa_workspace_bytes.argtypes = [pp]
    lib.gqa_workspace_bytes.restype = sz
    for name in ("gqa_attention_prefill", "gqa_attention_decode"):
        fn = getattr(lib, name)
        fn.argtypes = [pp] + [vp] * 13 + [sz, vp, vp]
        fn.restype = i32
    lib.gqa_rope_append_kv.argtypes = [pp] + [vp] * 13
    lib.gqa_rope_append_kv.restype = i32
    lib.gqa_attention_decode_noalloc.argtypes = [pp] + [vp] * 12 + [vp, vp]
    lib.gqa_attention_decode_noalloc.restype = i32
    for name in ("gqa_attention_decode_paged", "gqa_attention_prefill_paged"):
        getattr(lib, name).argtypes = [pp] + [vp] * 5 + [i32, i32] + [vp] * 7 + [sz, vp, vp]
        getattr(lib, name).restype = i32
    lib.gqa_attention_decode_masked.argtypes = [pp, ctypes.POINTER(GqaMask)] + [vp] * 13 + [sz, vp, vp]
    lib.gqa_attention_decode_masked.restype = i32
    lib.gqa_attention_prefill_masked.argtypes = [pp, ctypes.POINTER(GqaMask)] + [vp] * 13 + [sz, vp, vp]
    lib.gqa_attention_prefill_masked.restype = i32
    for name in ("gqa_attention_decode_q8", "gqa_attention_prefill_q8", "gqa_attention_decode_i8",
                 "gqa_attention_prefill_i8"):
        getattr(lib, name).argtypes = [pp] + [vp] * 13 + [sz, vp, vp]
        getattr(lib, name).restype = i32
    lib.gqa_status_string.argtypes = [i32]
    lib.gqa_status_string.restype = ctypes.c_char_p
    lib.gqa_abi_version.argtypes = []
    lib.gqa_abi_version.restype = i32
    lib.gqa_attention_nonpad.argtypes = [pp] + [vp] * 7 + [sz, vp, vp]
    lib.gqa_attention_nonpad.restype = i32
    lib.gqa_test_stall_waits.argtypes = [ctypes.c_int64]
    lib.gqa_test_stall_waits.restype = i32
    return lib


lib = _load()


def params(batch, q_heads, kv_heads, head_dim, q_len, cap_present, dtype, cap_past=None, rope_len=0, scale=0.0,
           softcap=0.0, window=-1, causal=1, do_rotary=0, rotary_interleaved=0, smooth_softmax=0,
           kv_ring=0, v_head_dim=0) -> GqaParams:
    """Build a gqa_params struct (dtype: "f32" | "f16" | "bf16" or its integer code)."""
    dt = DTYPES[dtype] if isinstance(dtype, str) else int(dtype)
    return GqaParams(batch, q_heads, kv_heads, head_dim, q_len, cap_present if cap_past is None else cap_past,
                     cap_present, rope_len, dt, scale, softcap, window, causal, do_rotary, rotary_interleaved,
                     smooth_softmax, kv_ring, v_head_dim)


def params_from_dict(d: dict) -> GqaParams:
    return params(d["batch"], d["q_heads"], d["kv_heads"], d["head_dim"], d["q_len"], d["cap_present"], d["dtype"],
                  cap_past=d.get("cap_past"), rope_len=d.get("rope_len", 0), scale=d.get("scale", 0.0),
                  softcap=d.get("softcap", 0.0), window=d.get("window", -1), causal=d.get("causal", 1),
                  do_rotary=d.get("do_rotary", 0), rotary_interleaved=d.get("rotary_interleaved", 0),
                  smooth_softmax=d.get("smooth_softmax", 0), kv_ring=d.get("kv_ring", 0),
                  v_head_dim=d.get("v_head_dim", 0))


def _ptr(t):
    """Device pointer of a CUDA tensor (or an int address, or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if not t.is_cuda:
        raise ValueError("libgqa takes device tensors; got a tensor on %s" % t.device)
    if not t.is_contiguous():
        raise ValueError("libgqa takes dense row-major tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def gqa_workspace_bytes(p: GqaParams) -> int:
    return int(lib.gqa_workspace_bytes(ctypes.byref(p)))


def gqa_attention_prefill(p, q, k, v, past_k, past_v, seqlens_k, cos_cache, sin_cache, head_sink, out, present_k,
                          present_v, workspace, dev_status, stream=None) -> int:
    return int(lib.gqa_attention_prefill(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(past_k), _ptr(past_v),
                                         _ptr(seqlens_k), _ptr(cos_cache), _ptr(sin_cache), _ptr(head_sink),
                                         _ptr(out), _ptr(present_k), _ptr(present_v), _ptr(workspace),
                                         _nbytes(workspace), _ptr(dev_status), _stream(stream)))


def gqa_attention_decode(p, q, k, v, past_k, past_v, seqlens_k, cos_cache, sin_cache, head_sink, out, present_k,
                         present_v, workspace, dev_status, stream=None) -> int:
    return int(lib.gqa_attention_decode(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(past_k), _ptr(past_v),
                                        _ptr(seqlens_k), _ptr(cos_cache), _ptr(sin_cache), _ptr(head_sink),
                                        _ptr(out), _ptr(present_k), _ptr(present_v), _ptr(workspace),
                                        _nbytes(workspace), _ptr(dev_status), _stream(stream)))


def gqa_attention_decode_noalloc(p, q, k, v, past_k, past_v, seqlens_k, cos_cache, sin_cache, head_sink, out,
                                 present_k, present_v, dev_status, stream=None) -> int:
    """Decode with the library's static scratch instead of a workspace (for callers that
    cannot allocate device memory; see include/gqa.h)."""
    return int(lib.gqa_attention_decode_noalloc(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(past_k),
                                                _ptr(past_v), _ptr(seqlens_k), _ptr(cos_cache), _ptr(sin_cache),
                                                _ptr(head_sink), _ptr(out), _ptr(present_k), _ptr(present_v),
                                                _ptr(dev_status), _stream(stream)))


def gqa_attention_decode_masked(p, mask: "GqaMask", q, k, v, past_k, past_v, seqlens_k, cos_cache, sin_cache,
                                head_sink, out, present_k, present_v, workspace, dev_status, stream=None) -> int:
    """Decode with a boolean or additive attention mask (see include/gqa.h)."""
    return int(lib.gqa_attention_decode_masked(ctypes.byref(p), ctypes.byref(mask), _ptr(q), _ptr(k), _ptr(v),
                                               _ptr(past_k), _ptr(past_v), _ptr(seqlens_k), _ptr(cos_cache),
                                               _ptr(sin_cache), _ptr(head_sink), _ptr(out), _ptr(present_k),
                                               _ptr(present_v), _ptr(workspace), _nbytes(workspace),
                                               _ptr(dev_status), _stream(stream)))


def gqa_attention_prefill_masked(p, mask: "GqaMask", q, k, v, past_k, past_v, seqlens_k, cos_cache, sin_cache,
                                 head_sink, out, present_k, present_v, workspace, dev_status, stream=None) -> int:
    """Prefill (or any step) with a boolean or additive attention mask (see include/gqa.h)."""
    return int(lib.gqa_attention_prefill_masked(ctypes.byref(p), ctypes.byref(mask), _ptr(q), _ptr(k), _ptr(v),
                                                _ptr(past_k), _ptr(past_v), _ptr(seqlens_k), _ptr(cos_cache),
                                                _ptr(sin_cache), _ptr(head_sink), _ptr(out), _ptr(present_k),
                                                _ptr(present_v), _ptr(workspace), _nbytes(workspace),
                                                _ptr(dev_status), _stream(stream)))


def _q8(name, p, q, k, v, seqlens_k, cos_cache, sin_cache, head_sink, k_scale, v_scale, out, present_k8, present_v8,
        workspace, dev_status, stream):
    return int(getattr(lib, name)(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(seqlens_k), _ptr(cos_cache),
                                  _ptr(sin_cache), _ptr(head_sink), _ptr(k_scale), _ptr(v_scale), _ptr(out),
                                  _ptr(present_k8), _ptr(present_v8), _ptr(workspace), _nbytes(workspace),
                                  _ptr(dev_status), _stream(stream)))


def gqa_attention_decode_q8(p, q, k, v, seqlens_k, cos_cache, sin_cache, head_sink, k_scale, v_scale, out,
                            present_k8, present_v8, workspace, dev_status, stream=None) -> int:
    """Decode over an f8 (E4M3) cache with per-kv-head scales (see include/gqa.h)."""
    return _q8("gqa_attention_decode_q8", p, q, k, v, seqlens_k, cos_cache, sin_cache, head_sink, k_scale, v_scale,
               out, present_k8, present_v8, workspace, dev_status, stream)


def gqa_attention_prefill_q8(p, q, k, v, seqlens_k, cos_cache, sin_cache, head_sink, k_scale, v_scale, out,
                             present_k8, present_v8, workspace, dev_status, stream=None) -> int:
    """Prefill over an f8 (E4M3) cache with per-kv-head scales (see include/gqa.h)."""
    return _q8("gqa_attention_prefill_q8", p, q, k, v, seqlens_k, cos_cache, sin_cache, head_sink, k_scale, v_scale,
               out, present_k8, present_v8, workspace, dev_status, stream)


def gqa_attention_decode_i8(p, q, k, v, seqlens_k, cos_cache, sin_cache, head_sink, k_scale, v_scale, out,
                            present_k8, present_v8, workspace, dev_status, stream=None) -> int:
    """Decode over an int8 cache with per-kv-head scales (see include/gqa.h)."""
    return _q8("gqa_attention_decode_i8", p, q, k, v, seqlens_k, cos_cache, sin_cache, head_sink, k_scale, v_scale,
               out, present_k8, present_v8, workspace, dev_status, stream)


def gqa_attention_prefill_i8(p, q, k, v, seqlens_k, cos_cache, sin_cache, head_sink, k_scale, v_scale, out,
                             present_k8, present_v8, workspace, dev_status, stream=None) -> int:
    """Prefill over an int8 cache with per-kv-head scales (see include/gqa.h)."""
    return _q8("gqa_attention_prefill_i8", p, q, k, v, seqlens_k, cos_cache, sin_cache, head_sink, k_scale, v_scale,
               out, present_k8, present_v8, workspace, dev_status, stream)


def _paged(name, p, q, k, v, seqlens_k, block_table, num_pages, cos_cache, sin_cache, head_sink, out, k_pool, v_pool,
           workspace, dev_status, stream):
    return int(getattr(lib, name)(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(seqlens_k), _ptr(block_table),
                                  int(block_table.shape[1]), int(num_pages), _ptr(cos_cache), _ptr(sin_cache),
                                  _ptr(head_sink), _ptr(out), _ptr(k_pool), _ptr(v_pool), _ptr(workspace),
                                  _nbytes(workspace), _ptr(dev_status), _stream(stream)))


def gqa_attention_decode_paged(p, q, k, v, seqlens_k, block_table, num_pages, cos_cache, sin_cache, head_sink, out,
                               k_pool, v_pool, workspace, dev_status, stream=None) -> int:
    """Decode over a paged cache: pools [num_pages, Hkv, 64, D], block_table int32
    [B, max_pages] on the device (see include/gqa.h)."""
    return _paged("gqa_attention_decode_paged", p, q, k, v, seqlens_k, block_table, num_pages, cos_cache, sin_cache,
                  head_sink, out, k_pool, v_pool, workspace, dev_status, stream)


def gqa_attention_prefill_paged(p, q, k, v, seqlens_k, block_table, num_pages, cos_cache, sin_cache, head_sink, out,
                                k_pool, v_pool, workspace, dev_status, stream=None) -> int:
    """Prefill (or a chunk of one) into a paged cache (see include/gqa.h)."""
    return _paged("gqa_attention_prefill_paged", p, q, k, v, seqlens_k, block_table, num_pages, cos_cache, sin_cache,
                  head_sink, out, k_pool, v_pool, workspace, dev_status, stream)


def gqa_rope_append_kv(p, q, k, v, past_k, past_v, seqlens_k, cos_cache, sin_cache, q_rot, present_k, present_v,
                       dev_status, stream=None) -> int:
    return int(lib.gqa_rope_append_kv(ctypes.byref(p), _ptr(q), _ptr(k), _ptr(v), _ptr(past_k), _ptr(past_v),
                                      _ptr(seqlens_k), _ptr(cos_cache), _ptr(sin_cache), _ptr(q_rot),
                                      _ptr(present_k), _ptr(present_v), _ptr(dev_status), _stream(stream)))


def gqa_status_string(status: int) -> str:
    return lib.gqa_status_string(int(status)).decode()


def gqa_abi_version() -> int:
    return int(lib.gqa_abi_version())


def gqa_attention_nonpad(p, nonpad_kv_seqlen, q, k_cache, v_cache, head_sink, out, workspace, dev_status,
                         stream=None) -> int:
    """Attention over a padded K/V cache: nonpad_kv_seqlen int64 [B] valid keys per sequence,
    the queries the last q_len of them (see include/gqa.h)."""
    return int(lib.gqa_attention_nonpad(ctypes.byref(p), _ptr(nonpad_kv_seqlen), _ptr(q), _ptr(k_cache),
                                        _ptr(v_cache), _ptr(head_sink), _ptr(out), _ptr(workspace),
                                        _nbytes(workspace), _ptr(dev_status), _stream(stream)))


def gqa_test_stall_waits(cycles: int) -> int:
    """Failure-path test hook (see include/gqa.h): > 0 makes the kernels' first wait run out
    after that many SM cycles; 0 restores normal operation."""
    return int(lib.gqa_test_stall_waits(int(cycles)))


def check(status: int, what: str = "") -> None:
    if status != GQA_OK:
        raise GqaError(status, what)
