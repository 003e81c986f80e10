"""fp64 CPU oracle for sliding-window grouped-query attention over a KV cache.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline
leg may import this package; the product path (``sliding_window_gb300``) never does, and
this package imports nothing from it.  The arithmetic lives in ``gqa_oracle.c`` (plain C,
fp64, one materialized row at a time); this module only builds it with gcc, marshals numpy
arrays and returns numpy results.

Pages followed (each function cites its section):
  [P1] OpenVINO PR #37423 "[NPUW] Support GQA sliding-window and smooth-softmax in
       DecomposeGQA" -- "Sliding window", "smooth_softmax / head_sink".
  [P2] tract PR #2645 "onnx: import GroupQueryAttention decode steps and its internal
       rotary" -- "What changed".
  [P3] ExecuTorch PR #21901 "Add sliding windows to the off-graph KV-cache reference".
  [P4] onnx-light-cpu "Attention Kernel Design" -- "Layouts and semantics", "Compute
       paths", "Scheduling, precision, and invariants".

Every function is pinned by a ``-m "not gpu"`` test in tests/test_oracle_*.py against
something other than itself (library routines, closed forms, brute force, hand-derived
fixtures under tests/golden/).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}


def v_dim(p: dict) -> int:
    """The V head dimension: v_head_dim when given and nonzero, else head_dim ([P4] "Layouts
    and semantics": it may differ from the Q/K head dimension)."""
    return int(p.get("v_head_dim", 0) or p["head_dim"])
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gqa_oracle.c into oracle/_build/liboracle.so (gcc, fp64, OpenMP if present)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    try:
        subprocess.run(base + ["-fopenmp", _SRC, "-o", tmp, "-lm"], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + [_SRC, "-o", tmp, "-lm"], check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i32, i64, f64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.oracle_encode_f16.argtypes = [ctypes.c_float]
        lib.oracle_encode_f16.restype = ctypes.c_uint16
        lib.oracle_encode_bf16.argtypes = [ctypes.c_float]
        lib.oracle_encode_bf16.restype = ctypes.c_uint16
        lib.oracle_decode_f16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_f16.restype = f64
        lib.oracle_decode_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_decode_bf16.restype = f64
        lib.oracle_sequence_status.argtypes = [i32] * 7
        lib.oracle_sequence_status.restype = i32
        lib.oracle_visible.argtypes = [i64, i64, i64, i32, i32]
        lib.oracle_visible.restype = i32
        lib.oracle_rope_append.argtypes = [i32] * 11 + [vp] * 11 + [ctypes.POINTER(i32)]
        lib.oracle_rope_append.restype = None
        lib.oracle_attend_row.argtypes = [vp, vp, vp, i64, i64, vp, i32, i32, i32, f64, f64, i32, f64, vp]
        lib.oracle_attend_row.restype = None
        lib.oracle_attention.argtypes = [i32] * 10 + [f64, f64] + [i32] * 5 + [vp] * 6 + [i64, vp]
        # B, Hq, Hkv, D, Dv, curr, cap, dtype; scale, softcap; window, causal, smooth; q, k, v,
        # nonpad, sink, rows; nrows; out
        lib.oracle_attention_nonpad.argtypes = [i32] * 8 + [f64, f64] + [i32] * 3 + [vp] * 6 + [i64, vp]
        lib.oracle_ring_valid.argtypes = [i32] * 3
        lib.oracle_ring_valid.restype = i32
        lib.oracle_ring_status.argtypes = [i32] * 4
        lib.oracle_ring_status.restype = i32
        lib.oracle_rope_append_ring.argtypes = [i32] * 9 + [vp] * 9 + [ctypes.POINTER(i32)]
        lib.oracle_attention_ring.argtypes = [i32] * 8 + [f64, f64] + [i32] * 4 + [vp] * 6 + [i64, vp]
        lib.oracle_attention_masked.argtypes = [i32] * 9 + [f64, f64] + [i32] * 5 + [vp, i64, i64, i64, i32] + \
            [vp] * 6 + [i64, vp]
        lib.oracle_paged_status.argtypes = [i32] * 6 + [vp, i32, i32]
        lib.oracle_paged_status.restype = i32
        lib.oracle_rope_append_paged.argtypes = [i32] * 12 + [vp] * 10 + [ctypes.POINTER(i32)]
        lib.oracle_attention_paged.argtypes = [i32] * 10 + [f64, f64] + [i32] * 4 + [vp] * 7 + [i64, vp]
        lib.oracle_attention.restype = None
        lib.oracle_encode_e4m3.argtypes = [ctypes.c_float]
        lib.oracle_encode_e4m3.restype = ctypes.c_uint8
        lib.oracle_decode_e4m3.argtypes = [ctypes.c_uint8]
        lib.oracle_decode_e4m3.restype = f64
        lib.oracle_encode_i8.argtypes = [ctypes.c_float]
        lib.oracle_encode_i8.restype = ctypes.c_int8
        lib.oracle_decode_i8.argtypes = [ctypes.c_int8]
        lib.oracle_decode_i8.restype = f64
        lib.oracle_rope_append_q8.argtypes = [i32] * 10 + [vp] * 11 + [ctypes.POINTER(i32), i32]
        lib.oracle_attention_q8.argtypes = [i32] * 9 + [f64, f64] + [i32] * 4 + [vp] * 8 + [i64, vp, i32]
        lib.oracle_has_openmp.restype = i32
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits(a: np.ndarray, dtype: str) -> np.ndarray:
    """Storage view of an array in the given dtype: float32 for f32, uint16 bits otherwise."""
    if dtype == "f32":
        return np.ascontiguousarray(a, dtype=np.float32)
    a = np.ascontiguousarray(a)
    if a.dtype not in (np.uint16, np.int16, np.float16):
        raise TypeError("f16/bf16 oracle inputs are passed as their 16-bit storage (uint16 view)")
    return a.view(np.uint16)


def has_openmp() -> bool:
    return bool(_load().oracle_has_openmp())


# --------------------------------------------------------------------------------------
# Number formats (IEEE-754 binary16 / bfloat16 definitions, round to nearest even)
# --------------------------------------------------------------------------------------
def encode(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 values -> uint16 storage bits of f16 or bf16, ties to even."""
    lib = _load()
    fn = lib.oracle_encode_f16 if dtype == "f16" else lib.oracle_encode_bf16
    flat = np.ascontiguousarray(x, dtype=np.float32).ravel()
    return np.fromiter((fn(float(v)) for v in flat), dtype=np.uint16, count=flat.size).reshape(np.shape(x))


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """uint16 storage bits of f16 or bf16 -> float64 (exact)."""
    lib = _load()
    fn = lib.oracle_decode_f16 if dtype == "f16" else lib.oracle_decode_bf16
    flat = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    return np.fromiter((fn(int(v)) for v in flat), dtype=np.float64, count=flat.size).reshape(np.shape(bits))


# --------------------------------------------------------------------------------------
# Band predicate and per-sequence validity
# --------------------------------------------------------------------------------------
def visible(q_abs: int, j: int, total: int, causal: bool, window: int) -> bool:
    """[P1] "Sliding window" / [P2] "What changed": slot j visible to query q_abs."""
    return bool(_load().oracle_visible(q_abs, j, total, int(causal), window))


def sequence_status(past, curr, cap_past, cap_present, past_is_separate, do_rotary, rope_len) -> int:
    """0 for a valid sequence, else 1 (bad seqlens_k) or 2 (RoPE position past the cache)."""
    return int(_load().oracle_sequence_status(past, curr, cap_past, cap_present,
                                              int(past_is_separate), int(do_rotary), rope_len))


# --------------------------------------------------------------------------------------
# RoPE + append ([P2] "What changed")
# --------------------------------------------------------------------------------------
def rope_append(p: dict, q, k, v, past_k, past_v, seqlens_k, cos_cache=None, sin_cache=None,
                present_k=None, present_v=None):
    """Emulate the append step bit for bit.

    Arrays are numpy storage arrays (float32 for f32, uint16 bits for f16/bf16).
    present_k/present_v, when given, are updated in place (aliasing past is allowed: pass
    the same array as past_k and present_k); otherwise fresh copies of past are used.
    Returns (q_rot, present_k, present_v, status_bits).
    """
    lib = _load()
    dt = p["dtype"]
    q, k, v = _bits(q, dt), _bits(k, dt), _bits(v, dt)
    if present_k is None:
        present_k = _bits(past_k, dt).copy()
        present_v = _bits(past_v, dt).copy()
        pk, pv = None, None  # treat as aliased: present already holds past
    else:
        pk = None if past_k is None or past_k is present_k else _bits(past_k, dt)
        pv = None if past_v is None or past_v is present_v else _bits(past_v, dt)
    q_rot = np.empty_like(q)
    st = ctypes.c_int32(0)
    cs = _bits(cos_cache, dt) if cos_cache is not None else None
    sn = _bits(sin_cache, dt) if sin_cache is not None else None
    seq = np.ascontiguousarray(seqlens_k, dtype=np.int32)
    lib.oracle_rope_append(p["batch"], p["q_heads"], p["kv_heads"], p["head_dim"], v_dim(p), p["q_len"],
                           p.get("cap_past", p["cap_present"]), p["cap_present"], p.get("rope_len", 0),
                           DTYPE_CODES[dt], int(p.get("do_rotary", 0)),
                           _ptr(q), _ptr(k), _ptr(v), _ptr(pk), _ptr(pv), _ptr(seq), _ptr(cs), _ptr(sn),
                           _ptr(q_rot), _ptr(present_k), _ptr(present_v), ctypes.byref(st))
    return q_rot, present_k, present_v, int(st.value)


# --------------------------------------------------------------------------------------
# Attention ([P1], [P2], [P4]) in fp64
# --------------------------------------------------------------------------------------
def attend_row(q: np.ndarray, k: np.ndarray, v: np.ndarray, visible_mask: np.ndarray, dtype: str,
               scale: float, softcap: float = 0.0, sink=None) -> np.ndarray:
    """One query row (q: D floats) over n cache rows (k: [n, D], v: [n, Dv]) with an
    explicit visibility mask; returns Dv floats."""
    lib = _load()
    qd = np.ascontiguousarray(q, dtype=np.float64)
    kb, vb = _bits(k, dtype), _bits(v, dtype)
    vis = np.ascontiguousarray(visible_mask, dtype=np.uint8)
    dv = vb.size // max(1, vis.shape[0])
    out = np.zeros(dv, dtype=np.float64)
    lib.oracle_attend_row(_ptr(qd), _ptr(kb), _ptr(vb), 0, vis.shape[0], _ptr(vis), qd.shape[0], dv,
                          DTYPE_CODES[dtype], float(scale), float(softcap), int(sink is not None),
                          float(sink if sink is not None else 0.0), _ptr(out))
    return out


def attention(p: dict, q_rot, present_k, present_v, seqlens_k, head_sink=None, rows=None,
              past_is_separate: bool = False) -> np.ndarray:
    """Attention output in fp64.

    q_rot: the query as it enters the scores, [B, curr, Hq*D] storage array.
    rows: None for every row (result [B, curr, Hq, D]) or an int array of flat row indices
    r = ((b*curr)+i)*Hq + hq (result [len(rows), D]).
    """
    lib = _load()
    dt = p["dtype"]
    qb = _bits(q_rot, dt)
    kb, vb = _bits(present_k, dt), _bits(present_v, dt)
    seq = np.ascontiguousarray(seqlens_k, dtype=np.int32)
    sink = None if head_sink is None else np.ascontiguousarray(head_sink, dtype=np.float32)
    B, Hq, D, curr, Dv = p["batch"], p["q_heads"], p["head_dim"], p["q_len"], v_dim(p)
    if rows is None:
        ridx, n = None, B * curr * Hq
    else:
        ridx = np.ascontiguousarray(rows, dtype=np.int64)
        n = ridx.shape[0]
    out = np.zeros((n, Dv), dtype=np.float64)
    lib.oracle_attention(B, Hq, p["kv_heads"], D, Dv, curr, p.get("cap_past", p["cap_present"]),
                         p["cap_present"], p.get("rope_len", 0), DTYPE_CODES[dt],
                         float(p.get("scale", 0.0)), float(p.get("softcap", 0.0)), int(p.get("window", -1)),
                         int(p.get("causal", 1)), int(p.get("do_rotary", 0)), int(p.get("smooth_softmax", 0)),
                         int(past_is_separate), _ptr(qb), _ptr(kb), _ptr(vb), _ptr(seq), _ptr(sink),
                         _ptr(ridx), n, _ptr(out))
    if rows is None:
        return out.reshape(B, curr, Hq, Dv)
    return out


def attention_nonpad(p: dict, q, k_cache, v_cache, nonpad_kv_seqlen, head_sink=None, rows=None) -> np.ndarray:
    """Attention in fp64 over a padded K/V cache ([P4] "Layouts and semantics": opset-24
    nonpad_kv_seqlen).  Sequence b has n_b = nonpad_kv_seqlen[b] valid keys (rows [0, n_b) of
    its cache, p["cap_present"] rows); its q_len queries are the last q_len valid tokens
    (query i at position n_b - q_len + i); n_b < q_len or n_b > cap gives zeros.  Same
    conventions as attention() otherwise (q as it enters the scores; rows selection)."""
    lib = _load()
    dt = p["dtype"]
    qb = _bits(q, dt)
    kb, vb = _bits(k_cache, dt), _bits(v_cache, dt)
    npd = np.ascontiguousarray(nonpad_kv_seqlen, dtype=np.int64)
    sink = None if head_sink is None else np.ascontiguousarray(head_sink, dtype=np.float32)
    B, Hq, D, curr, Dv = p["batch"], p["q_heads"], p["head_dim"], p["q_len"], v_dim(p)
    if rows is None:
        ridx, n = None, B * curr * Hq
    else:
        ridx = np.ascontiguousarray(rows, dtype=np.int64)
        n = ridx.shape[0]
    out = np.zeros((n, Dv), dtype=np.float64)
    lib.oracle_attention_nonpad(B, Hq, p["kv_heads"], D, Dv, curr, p["cap_present"], DTYPE_CODES[dt],
                                float(p.get("scale", 0.0)), float(p.get("softcap", 0.0)), int(p.get("window", -1)),
                                int(p.get("causal", 1)), int(p.get("smooth_softmax", 0)), _ptr(qb), _ptr(kb),
                                _ptr(vb), _ptr(npd), _ptr(sink), _ptr(ridx), n, _ptr(out))
    if rows is None:
        return out.reshape(B, curr, Hq, Dv)
    return out


def gqa(p: dict, q, k, v, past_k, past_v, seqlens_k, cos_cache=None, sin_cache=None, head_sink=None,
        rows=None):
    """Whole step: append (+RoPE) into present, then attention.  Returns
    (out_fp64, present_k, present_v, q_rot, status_bits).  p["kv_ring"] = 1 selects the
    ring layout (present updated in place from past_k/past_v, which hold the ring)."""
    if p.get("kv_ring", 0):
        q_rot, pk, pv, st = rope_append_ring(p, q, k, v, past_k, past_v, seqlens_k, cos_cache, sin_cache)
        out = attention_ring(p, q_rot, pk, pv, seqlens_k, head_sink, rows)
        return out, pk, pv, q_rot, st
    q_rot, pk, pv, st = rope_append(p, q, k, v, past_k, past_v, seqlens_k, cos_cache, sin_cache)
    out = attention(p, q_rot, pk, pv, seqlens_k, head_sink, rows)
    return out, pk, pv, q_rot, st


# --------------------------------------------------------------------------------------
# Ring layout ([P1] "Sliding window": the rolling sliding_window_cache buffer)
# --------------------------------------------------------------------------------------
def ring_valid(curr: int, cap: int, window: int) -> bool:
    """A ring of cap slots can serve a step of curr tokens with window W iff
    W >= 1 and W + curr - 1 <= cap."""
    return bool(_load().oracle_ring_valid(curr, cap, window))


def rope_append_ring(p: dict, q, k, v, ring_k, ring_v, seqlens_k, cos_cache=None, sin_cache=None):
    """Append (+RoPE) into a ring of p["cap_present"] slots: position p goes to slot
    p mod cap.  Works on copies of ring_k/ring_v; returns (q_rot, ring_k, ring_v, status)."""
    lib = _load()
    dt = p["dtype"]
    q, k, v = _bits(q, dt), _bits(k, dt), _bits(v, dt)
    rk, rv = _bits(ring_k, dt).copy(), _bits(ring_v, dt).copy()
    q_rot = np.empty_like(q)
    st = ctypes.c_int32(0)
    cs = _bits(cos_cache, dt) if cos_cache is not None else None
    sn = _bits(sin_cache, dt) if sin_cache is not None else None
    seq = np.ascontiguousarray(seqlens_k, dtype=np.int32)
    lib.oracle_rope_append_ring(p["batch"], p["q_heads"], p["kv_heads"], p["head_dim"], p["q_len"],
                                p["cap_present"], p.get("rope_len", 0), DTYPE_CODES[dt], int(p.get("do_rotary", 0)),
                                _ptr(q), _ptr(k), _ptr(v), _ptr(seq), _ptr(cs), _ptr(sn), _ptr(q_rot),
                                _ptr(rk), _ptr(rv), ctypes.byref(st))
    return q_rot, rk, rv, int(st.value)


def attention_ring(p: dict, q_rot, ring_k, ring_v, seqlens_k, head_sink=None, rows=None) -> np.ndarray:
    """Attention in fp64 over a ring cache (same conventions as attention())."""
    lib = _load()
    dt = p["dtype"]
    qb = _bits(q_rot, dt)
    kb, vb = _bits(ring_k, dt), _bits(ring_v, dt)
    seq = np.ascontiguousarray(seqlens_k, dtype=np.int32)
    sink = None if head_sink is None else np.ascontiguousarray(head_sink, dtype=np.float32)
    B, Hq, D, curr = p["batch"], p["q_heads"], p["head_dim"], p["q_len"]
    if rows is None:
        ridx, n = None, B * curr * Hq
    else:
        ridx = np.ascontiguousarray(rows, dtype=np.int64)
        n = ridx.shape[0]
    out = np.zeros((n, D), dtype=np.float64)
    lib.oracle_attention_ring(B, Hq, p["kv_heads"], D, curr, p["cap_present"], p.get("rope_len", 0),
                              DTYPE_CODES[dt], float(p.get("scale", 0.0)), float(p.get("softcap", 0.0)),
                              int(p.get("window", -1)), int(p.get("causal", 1)), int(p.get("do_rotary", 0)),
                              int(p.get("smooth_softmax", 0)), _ptr(qb), _ptr(kb), _ptr(vb), _ptr(seq),
                              _ptr(sink), _ptr(ridx), n, _ptr(out))
    if rows is None:
        return out.reshape(B, curr, Hq, D)
    return out


# --------------------------------------------------------------------------------------
# Paged layout ([P3] Summary: a cell cache with per-sequence membership)
# --------------------------------------------------------------------------------------
def rope_append_paged(p: dict, q, k, v, pool_k, pool_v, seqlens_k, table, num_pages, page=64, cos_cache=None,
                      sin_cache=None):
    """Append (+RoPE) into a paged pool [num_pages, Hkv, page, D] through a block table
    [B, max_pages]; works on copies of the pools.  Returns (q_rot, pool_k, pool_v, status)."""
    lib = _load()
    dt = p["dtype"]
    q, k, v = _bits(q, dt), _bits(k, dt), _bits(v, dt)
    pk, pv = _bits(pool_k, dt).copy(), _bits(pool_v, dt).copy()
    tab = np.ascontiguousarray(table, dtype=np.int32)
    q_rot = np.empty_like(q)
    st = ctypes.c_int32(0)
    cs = _bits(cos_cache, dt) if cos_cache is not None else None
    sn = _bits(sin_cache, dt) if sin_cache is not None else None
    seq = np.ascontiguousarray(seqlens_k, dtype=np.int32)
    lib.oracle_rope_append_paged(p["batch"], p["q_heads"], p["kv_heads"], p["head_dim"], p["q_len"], page,
                                 tab.shape[1], num_pages, p.get("rope_len", 0), DTYPE_CODES[dt],
                                 int(p.get("do_rotary", 0)), int(p.get("window", -1)), _ptr(tab), _ptr(q), _ptr(k),
                                 _ptr(v), _ptr(seq), _ptr(cs), _ptr(sn), _ptr(q_rot), _ptr(pk), _ptr(pv),
                                 ctypes.byref(st))
    return q_rot, pk, pv, int(st.value)


def attention_paged(p: dict, q_rot, pool_k, pool_v, seqlens_k, table, num_pages, page=64, head_sink=None,
                    rows=None) -> np.ndarray:
    """Attention in fp64 over a paged cache (same conventions as attention())."""
    lib = _load()
    dt = p["dtype"]
    qb = _bits(q_rot, dt)
    kb, vb = _bits(pool_k, dt), _bits(pool_v, dt)
    tab = np.ascontiguousarray(table, dtype=np.int32)
    seq = np.ascontiguousarray(seqlens_k, dtype=np.int32)
    sink = None if head_sink is None else np.ascontiguousarray(head_sink, dtype=np.float32)
    B, Hq, D, curr = p["batch"], p["q_heads"], p["head_dim"], p["q_len"]
    if rows is None:
        ridx, n = None, B * curr * Hq
    else:
        ridx = np.ascontiguousarray(rows, dtype=np.int64)
        n = ridx.shape[0]
    out = np.zeros((n, D), dtype=np.float64)
    lib.oracle_attention_paged(B, Hq, p["kv_heads"], D, curr, page, tab.shape[1], num_pages, p.get("rope_len", 0),
                               DTYPE_CODES[dt], float(p.get("scale", 0.0)), float(p.get("softcap", 0.0)),
                               int(p.get("window", -1)), int(p.get("causal", 1)), int(p.get("do_rotary", 0)),
                               int(p.get("smooth_softmax", 0)), _ptr(tab), _ptr(qb), _ptr(kb), _ptr(vb), _ptr(seq),
                               _ptr(sink), _ptr(ridx), n, _ptr(out))
    if rows is None:
        return out.reshape(B, curr, Hq, D)
    return out


# --------------------------------------------------------------------------------------
# Attention masks ([P4] "Layouts and semantics"; [P2] "What changed": attention_bias)
# --------------------------------------------------------------------------------------
def attention_masked(p: dict, q_rot, present_k, present_v, seqlens_k, mask, kind: str, head_sink=None,
                     rows=None) -> np.ndarray:
    """Attention in fp64 with a mask broadcastable to [B, Hq, curr, keys] (numpy array with
    4 dims, size-1 dims broadcast): kind "bool" (nonzero keeps) or "add" (values of the
    dtype, storage bits for f16/bf16, added to the scaled score before the softcap)."""
    lib = _load()
    dt = p["dtype"]
    qb = _bits(q_rot, dt)
    kb, vb = _bits(present_k, dt), _bits(present_v, dt)
    seq = np.ascontiguousarray(seqlens_k, dtype=np.int32)
    sink = None if head_sink is None else np.ascontiguousarray(head_sink, dtype=np.float32)
    m = np.ascontiguousarray(mask, dtype=np.uint8) if kind == "bool" else _bits(mask, dt)
    assert m.ndim == 4
    st = [0 if m.shape[d] == 1 else int(np.prod(m.shape[d + 1:])) for d in range(3)]
    B, Hq, D, curr, Dv = p["batch"], p["q_heads"], p["head_dim"], p["q_len"], v_dim(p)
    if rows is None:
        ridx, n = None, B * curr * Hq
    else:
        ridx = np.ascontiguousarray(rows, dtype=np.int64)
        n = ridx.shape[0]
    out = np.zeros((n, Dv), dtype=np.float64)
    lib.oracle_attention_masked(B, Hq, p["kv_heads"], D, Dv, curr, p["cap_present"], p.get("rope_len", 0),
                                DTYPE_CODES[dt], float(p.get("scale", 0.0)), float(p.get("softcap", 0.0)),
                                int(p.get("window", -1)), int(p.get("causal", 1)), int(p.get("do_rotary", 0)),
                                int(p.get("smooth_softmax", 0)), 1 if kind == "bool" else 2, _ptr(m), st[0], st[1],
                                st[2], m.shape[3], _ptr(qb), _ptr(kb), _ptr(vb), _ptr(seq), _ptr(sink), _ptr(ridx), n,
                                _ptr(out))
    if rows is None:
        return out.reshape(B, curr, Hq, Dv)
    return out


# --------------------------------------------------------------------------------------
# Quantized (f8 E4M3) KV cache: codes with one scale per kv head for K and for V
# --------------------------------------------------------------------------------------
def encode_e4m3(x) -> np.ndarray:
    """E4M3 codes (uint8) of float32 values: nearest, ties to even, saturating at +-448
    (infinity included), NaN to NaN."""
    lib = _load()
    a = np.ascontiguousarray(x, dtype=np.float32)
    return np.array([lib.oracle_encode_e4m3(float(v)) for v in a.ravel()], dtype=np.uint8).reshape(a.shape)


def decode_e4m3(codes) -> np.ndarray:
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    return np.array([lib.oracle_decode_e4m3(int(v)) for v in c.ravel()], dtype=np.float64).reshape(c.shape)


def encode_i8(x) -> np.ndarray:
    """int8 codes of float32 values: nearest, ties to even, saturating at -128 and 127
    (infinities included), NaN to 0."""
    lib = _load()
    a = np.ascontiguousarray(x, dtype=np.float32)
    return np.array([lib.oracle_encode_i8(float(v)) for v in a.ravel()], dtype=np.int8).reshape(a.shape)


def decode_i8(codes) -> np.ndarray:
    lib = _load()
    c = np.ascontiguousarray(codes, dtype=np.int8)
    return np.array([lib.oracle_decode_i8(int(v)) for v in c.ravel()], dtype=np.float64).reshape(c.shape)


KV_FORMATS = {"e4m3": 0, "int8": 1}


def rope_append_q8(p: dict, q, k, v, present_k8, present_v8, seqlens_k, k_scale, v_scale, cos_cache=None,
                   sin_cache=None, fmt="e4m3"):
    """Append into a quantized cache in place: K (rotated, rounded to the dtype) and V divided
    by their kv head's scale in fp32 and encoded as `fmt` codes ("e4m3" or "int8", one byte
    each).  present_k8 [B, Hkv, cap, D] and present_v8 [B, Hkv, cap, Dv] are uint8 arrays (the
    codes' bytes) updated in place.  Returns (q_rot, status_bits)."""
    lib = _load()
    dt = p["dtype"]
    q, k, v = _bits(q, dt), _bits(k, dt), _bits(v, dt)
    assert present_k8.dtype == np.uint8 and present_k8.flags.c_contiguous
    assert present_v8.dtype == np.uint8 and present_v8.flags.c_contiguous
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    cs = _bits(cos_cache, dt) if cos_cache is not None else None
    sn = _bits(sin_cache, dt) if sin_cache is not None else None
    seq = np.ascontiguousarray(seqlens_k, dtype=np.int32)
    q_rot = np.empty_like(q)
    st = ctypes.c_int32(0)
    lib.oracle_rope_append_q8(p["batch"], p["q_heads"], p["kv_heads"], p["head_dim"], v_dim(p), p["q_len"],
                              p["cap_present"], p.get("rope_len", 0), DTYPE_CODES[dt], int(p.get("do_rotary", 0)),
                              _ptr(q), _ptr(k), _ptr(v), _ptr(seq), _ptr(cs), _ptr(sn), _ptr(ks), _ptr(vs),
                              _ptr(q_rot), _ptr(present_k8), _ptr(present_v8), ctypes.byref(st), KV_FORMATS[fmt])
    return q_rot, int(st.value)


def attention_q8(p: dict, q_rot, present_k8, present_v8, seqlens_k, k_scale, v_scale, head_sink=None,
                 rows=None, fmt="e4m3") -> np.ndarray:
    """Attention in fp64 over the dequantized cache (code * scale of its kv head; `fmt` codes)."""
    lib = _load()
    dt = p["dtype"]
    qb = _bits(q_rot, dt)
    kb = np.ascontiguousarray(present_k8, dtype=np.uint8)
    vb = np.ascontiguousarray(present_v8, dtype=np.uint8)
    ks = np.ascontiguousarray(k_scale, dtype=np.float32)
    vs = np.ascontiguousarray(v_scale, dtype=np.float32)
    seq = np.ascontiguousarray(seqlens_k, dtype=np.int32)
    sink = None if head_sink is None else np.ascontiguousarray(head_sink, dtype=np.float32)
    B, Hq, D, curr, Dv = p["batch"], p["q_heads"], p["head_dim"], p["q_len"], v_dim(p)
    if rows is None:
        ridx, n = None, B * curr * Hq
    else:
        ridx = np.ascontiguousarray(rows, dtype=np.int64)
        n = ridx.shape[0]
    out = np.zeros((n, Dv), dtype=np.float64)
    lib.oracle_attention_q8(B, Hq, p["kv_heads"], D, Dv, curr, p["cap_present"], p.get("rope_len", 0),
                            DTYPE_CODES[dt], float(p.get("scale", 0.0)), float(p.get("softcap", 0.0)),
                            int(p.get("window", -1)), int(p.get("causal", 1)), int(p.get("do_rotary", 0)),
                            int(p.get("smooth_softmax", 0)), _ptr(qb), _ptr(kb), _ptr(vb), _ptr(ks), _ptr(vs),
                            _ptr(seq), _ptr(sink), _ptr(ridx), n, _ptr(out), KV_FORMATS[fmt])
    if rows is None:
        return out.reshape(B, curr, Hq, Dv)
    return out
