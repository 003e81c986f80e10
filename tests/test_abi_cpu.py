"""Host-side checks of the C ABI that need no GPU: the library loads, exports every function
that include/gqa.h declares, the Python struct matches the C struct byte for byte, and
invalid calls return their error codes before anything is launched (onnx-light-cpu
"Attention Kernel Design", "Scheduling, precision, and invariants": invalid pairings fail
explicitly)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gqa.h")


@pytest.fixture(scope="module")
def g():
    import __graft_entry__
    __graft_entry__.build()
    from sliding_window_gb300 import gqa
    return gqa


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(gqa_\w+)\s*\(", text, re.M)))


def test_exports_every_declared_symbol(g):
    names = declared_functions()
    assert set(names) == set(g.EXPORTED)
    out = subprocess.run(["nm", "-D", "--defined-only", g.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (gqa_\w+)", out))
    for n in names:
        assert n in exported, n
        assert hasattr(g.lib, n)


def test_struct_layout_matches_header(g, tmp_path):
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "gqa.h"\nint main(void){\n'
                   'printf("%zu", sizeof(gqa_params));\n'
                   + "".join('printf(" %%zu", offsetof(gqa_params, %s));\n' % f for f, _ in g.GqaParams._fields_)
                   + "return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    vals = list(map(int, subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()))
    assert vals[0] == ctypes.sizeof(g.GqaParams)
    assert vals[1:] == [getattr(g.GqaParams, f).offset for f, _ in g.GqaParams._fields_]


def test_mask_struct_layout_matches_header(g, tmp_path):
    src = tmp_path / "mask.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "gqa.h"\nint main(void){\n'
                   'printf("%zu", sizeof(gqa_mask));\n'
                   + "".join('printf(" %%zu", offsetof(gqa_mask, %s));\n' % f for f, _ in g.GqaMask._fields_)
                   + "return 0;}\n")
    exe = tmp_path / "mask"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    vals = list(map(int, subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()))
    assert vals[0] == ctypes.sizeof(g.GqaMask)
    assert vals[1:] == [getattr(g.GqaMask, f).offset for f, _ in g.GqaMask._fields_]


def test_version_and_status_strings(g):
    assert g.gqa_abi_version() == 8
    for s in range(6):
        assert g.gqa_status_string(s) and g.gqa_status_string(s) != "unknown status"
    assert g.gqa_status_string(99) == "unknown status"


def good_params(g, **kw):
    d = dict(batch=2, q_heads=8, kv_heads=2, head_dim=128, q_len=1, cap_present=1024, dtype="bf16", window=256)
    d.update(kw)
    return g.params(**d)


FAKE = 1 << 20  # a 16-byte aligned address that is never dereferenced: every case fails first


def call(g, p, fn="gqa_attention_decode", ws_bytes=0, **ptrs):
    names = ["q", "k", "v", "past_k", "past_v", "seqlens_k", "cos", "sin", "head_sink", "out", "present_k",
             "present_v", "workspace"]
    vals = {n: FAKE for n in names}
    vals.update(ptrs)
    args = [ctypes.c_void_p(vals[n]) if vals[n] is not None else None for n in names]
    return getattr(g.lib, fn)(ctypes.byref(p), *args, ws_bytes, None, None)


@pytest.mark.parametrize("fn", ["gqa_attention_decode", "gqa_attention_prefill"])
@pytest.mark.parametrize("kw,code", [
    (dict(q_heads=6, kv_heads=4), 1),          # heads not divisible
    (dict(kv_heads=0), 1),
    (dict(batch=0), 1),
    (dict(q_len=0), 1),
    (dict(head_dim=96), 2),                    # valid op, not implemented
    (dict(dtype=7), 1),
    (dict(window=0), 1),                       # window must be -1 or >= 1
    (dict(window=-2), 1),
    (dict(scale=-1.0), 1),
    (dict(softcap=-2.0), 1),
    (dict(causal=2), 1),
    (dict(rotary_interleaved=1), 2),
    (dict(cap_present=0), 3),
    (dict(q_len=8, cap_present=4), 3),
    (dict(do_rotary=1, rope_len=0), 1),
    (dict(kv_ring=2), 1),
    (dict(kv_ring=1, window=-1), 1),            # a ring needs a window
    (dict(kv_ring=1, window=1024, q_len=2), 3),  # W + curr - 1 > cap: a visible key would be overwritten
    (dict(kv_ring=1, window=100, cap_present=1000), 2),  # ring capacity not a multiple of 64
    (dict(v_head_dim=-1), 1),
    (dict(v_head_dim=96), 2),                                  # V head dim 64 or 128 only
    (dict(kv_ring=1, window=1000, v_head_dim=64), 2),          # a ring holds K and V rows of one width
])
def test_invalid_params_rejected(g, fn, kw, code):
    assert call(g, good_params(g, **kw), fn) == code
    assert g.lib.gqa_workspace_bytes(ctypes.byref(good_params(g, **kw))) == 0


@pytest.mark.parametrize("ptrs,code", [
    (dict(q=None), 1), (dict(seqlens_k=None), 1), (dict(present_k=None), 1), (dict(out=None), 1),
    (dict(k=None), 1),                              # k without v
    (dict(q=FAKE + 8), 1), (dict(present_v=FAKE + 4), 1), (dict(out=FAKE + 2), 1),
    (dict(seqlens_k=FAKE + 2), 1), (dict(past_k=None), 1),  # past_k without past_v
])
def test_invalid_pointers_rejected(g, ptrs, code):
    assert call(g, good_params(g), **ptrs) == code


def test_ring_rules(g):
    ring = good_params(g, kv_ring=1, window=1000, cap_present=1024, q_len=4)
    assert call(g, ring, past_k=FAKE + 4096, past_v=FAKE + 4096) == 1  # a ring is updated in place
    # prefill reads a ring in 128-position tiles: a capacity that is not a multiple of 128,
    # fp32 and masks are not supported
    assert call(g, good_params(g, kv_ring=1, window=1000, cap_present=1088, q_len=4), fn="gqa_attention_prefill") == 2
    assert call(g, good_params(g, kv_ring=1, window=1000, cap_present=1024, q_len=4, dtype="f32"),
                fn="gqa_attention_prefill") == 2
    assert call(g, good_params(g, kv_ring=1, window=1000, cap_present=1024, q_len=4, dtype="f32")) == 2


def call_paged(g, p, table=FAKE, max_pages=16, num_pages=40, ws_bytes=0, fn="gqa_attention_decode_paged", **ptrs):
    names = ["q", "k", "v", "seqlens_k", "cos", "sin", "head_sink", "out", "k_pool", "v_pool", "workspace"]
    vals = {n: FAKE for n in names}
    vals.update(ptrs)
    a = [ctypes.c_void_p(vals[n]) if vals[n] is not None else None for n in names]
    tab = ctypes.c_void_p(table) if table is not None else None
    return getattr(g.lib, fn)(ctypes.byref(p), a[0], a[1], a[2], a[3], tab, max_pages, num_pages,
                              a[4], a[5], a[6], a[7], a[8], a[9], a[10], ws_bytes, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(table=None), 1), (dict(table=FAKE + 2), 1),      # missing or misaligned block table
    (dict(max_pages=0), 1), (dict(num_pages=0), 1),
    (dict(max_pages=15), 3),                              # cap_present must be 64 * max_pages
    (dict(out=None), 1), (dict(k_pool=FAKE + 8), 1),
])
@pytest.mark.parametrize("fn", ["gqa_attention_decode_paged", "gqa_attention_prefill_paged"])
def test_paged_invalid_arguments(g, kw, code, fn):
    assert call_paged(g, good_params(g), fn=fn, **kw) == code


def test_paged_rejects_ring_and_unsupported_shapes(g):
    pf = "gqa_attention_prefill_paged"
    assert call_paged(g, good_params(g, kv_ring=1, window=1000), fn=pf) == 1
    assert call_paged(g, good_params(g, v_head_dim=64), fn=pf) == 2
    assert call_paged(g, good_params(g, dtype="f32"), fn=pf) == 2           # the tensor-core prefill reads pages
    assert call_paged(g, good_params(g, kv_ring=1, window=1000)) == 1
    assert call_paged(g, good_params(g, v_head_dim=64)) == 2       # pages hold K and V rows of one width
    assert call_paged(g, good_params(g, dtype="f32")) == 2          # only the split decode kernel reads pages
    assert call_paged(g, good_params(g, q_heads=64, q_len=2)) == 2  # 64 rows per group at D=128


def call_masked(g, p, mask, fn="gqa_attention_decode_masked", **ptrs):
    names = ["q", "k", "v", "past_k", "past_v", "seqlens_k", "cos", "sin", "head_sink", "out", "present_k",
             "present_v", "workspace"]
    vals = {n: FAKE for n in names}
    vals.update(ptrs)
    a = [ctypes.c_void_p(vals[n]) if vals[n] is not None else None for n in names]
    m = ctypes.byref(mask) if mask is not None else None
    return getattr(g.lib, fn)(ctypes.byref(p), m, *a, 0, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(data=None), 1), (dict(kind=3), 1), (dict(keys=0), 1), (dict(stride_h=-1), 1),
    (dict(data=FAKE + 1, kind=2), 1),                       # additive values must be 2-byte aligned
])
@pytest.mark.parametrize("fn", ["gqa_attention_decode_masked", "gqa_attention_prefill_masked"])
def test_masked_invalid_arguments(g, kw, code, fn):
    d = dict(data=FAKE, kind=1, keys=1024, stride_b=0, stride_h=0, stride_i=0)
    d.update(kw)
    m = g.GqaMask(d["data"], d["kind"], d["keys"], d["stride_b"], d["stride_h"], d["stride_i"])
    assert call_masked(g, good_params(g), m, fn) == code


@pytest.mark.parametrize("fn", ["gqa_attention_decode_masked", "gqa_attention_prefill_masked"])
def test_masked_argument_rules(g, fn):
    m = g.GqaMask(FAKE, 1, 1024, 0, 0, 0)
    assert call_masked(g, good_params(g), None, fn) == 1
    # f32 additive values are aligned to 4 bytes
    assert call_masked(g, good_params(g, dtype="f32"), g.GqaMask(FAKE + 2, 2, 1024, 0, 0, 0), fn) == 1
    # a ring is read by the split decode kernel only: f32, large groups and prefill reject it
    ring = dict(kv_ring=1, window=1000, cap_present=1024)
    assert call_masked(g, good_params(g, dtype="f32", **ring), m, fn) == 2
    assert call_masked(g, good_params(g, q_heads=64, q_len=2, **ring), m, fn) == 2


def test_attention_only_rejects_rotary(g):
    p = good_params(g, do_rotary=1, rope_len=4096)
    assert call(g, p, k=None, v=None) == 1


def test_rotary_needs_tables(g):
    p = good_params(g, do_rotary=1, rope_len=4096)
    assert call(g, p, cos=None) == 1


def test_workspace_checked_before_launch(g):
    p = good_params(g, batch=4, cap_present=16384, window=-1)  # band too long for one chunk
    need = g.lib.gqa_workspace_bytes(ctypes.byref(p))
    assert need > 0
    assert call(g, p, ws_bytes=need - 1) == 5
    assert call(g, p, ws_bytes=need, workspace=None) == 5
    assert call(g, p, ws_bytes=need, workspace=FAKE + 8) == 5


def bound_splits(B, Hkv, cap, window, curr=1):
    """Chunks per group of the largest plan any GPU of up to 512 SMs would choose (it sizes
    the workspace): one wave of two CTAs per SM (1024 slots), chunks of at most 4096 keys
    and at least 256 keys, at most 64 chunks."""
    lmax = cap if window < 0 else min(cap, window + curr - 1)
    units = B * Hkv
    s = max(1024 // units, -(-lmax // 4096))
    return min(64, max(1, min(s, max(1, -(-lmax // 256)))))


def decode_ws(B, Hkv, R, D, S):
    """Split decode workspace: fp32 acc [R][D] and (m, l) per (group, chunk) slot, one ticket
    per group; 256-byte aligned.  Nothing when a group is one chunk."""
    if S == 1:
        return 0
    al = lambda x: (x + 255) // 256 * 256
    slots = B * Hkv * S
    return al(slots * R * D * 4) + al(slots * R * 2 * 4) + al(B * Hkv * 4)


def test_workspace_sizes(g):
    ws = lambda **kw: g.lib.gqa_workspace_bytes(ctypes.byref(good_params(g, **kw)))
    # decode: B=2, Hq=8, Hkv=2 -> G=4, R=4 rows per group
    S = bound_splits(2, 2, 1024, 200)
    assert S == 1 and ws(window=200) == 0  # the band fits one chunk
    S = bound_splits(2, 2, 16384, -1)
    assert S == 64 and ws(window=-1, cap_present=16384) == decode_ws(2, 2, 4, 128, S)
    # partial accumulators are rows of the V head dim
    assert ws(window=-1, cap_present=16384, v_head_dim=64) == decode_ws(2, 2, 4, 64, S)
    assert ws(window=-1, cap_present=16384, head_dim=64, v_head_dim=128) == decode_ws(2, 2, 4, 128, S)
    # rotary adds room for the rotated queries (prefill path): B*curr*Hq*D*2 bytes
    assert ws(do_rotary=1, rope_len=64, window=-1, cap_present=16384) == \
        2 * 1 * 8 * 128 * 2 + decode_ws(2, 2, 4, 128, S)
    # long decode: G=8, R=8, 8 chunks of up to 4096 keys
    S = bound_splits(64, 8, 32768, -1)
    assert S == 8
    assert ws(batch=64, q_heads=64, kv_heads=8, cap_present=32768, window=-1) == decode_ws(64, 8, 8, 128, S) > 0
    # the sliding-window decode: 64 groups, bands of at most 1024 keys -> 4 chunks
    S = bound_splits(8, 8, 4096, 1024)
    assert S == 4
    assert ws(batch=8, q_heads=32, kv_heads=8, cap_present=4096, window=1024) == decode_ws(8, 8, 4, 128, S)
    # more than 32 query rows per group at D=128: the SIMT kernel, no split workspace; with more
    # than one query token the boolean-mask block map: one bit per (b, q head, 128-row query
    # tile, 16-key chunk of the cache), 32 chunks a word
    blockmap = lambda B, Hq, L, cap: B * Hq * -(-L // 128) * -(-cap // 512) * 4
    assert ws(q_heads=64, kv_heads=2, q_len=2, window=-1) == blockmap(2, 64, 2, 1024)
    # prefill-sized q_len never needs decode partials, only the block map
    assert ws(batch=2, q_heads=64, kv_heads=8, q_len=8192, cap_present=8192, window=4096) == blockmap(2, 64, 8192, 8192)
    assert ws(batch=2, q_heads=64, kv_heads=8, q_len=8192, cap_present=8192, window=4096, dtype="f32") == 0
    assert ws(batch=2, q_heads=8, kv_heads=2, q_len=300, cap_present=1024, head_dim=128, v_head_dim=64) == 0


def test_binding_refuses_host_tensors(g):
    import torch
    with pytest.raises(ValueError):
        g._ptr(torch.zeros(4))


def call_q8(g, p, fn="gqa_attention_decode_q8", **ptrs):
    names = ["q", "k", "v", "seqlens_k", "cos", "sin", "head_sink", "k_scale", "v_scale", "out", "present_k",
             "present_v", "workspace"]
    vals = {n: FAKE for n in names}
    vals.update(ptrs)
    a = [ctypes.c_void_p(vals[n]) if vals[n] is not None else None for n in names]
    return getattr(g.lib, fn)(ctypes.byref(p), *a, 0, None, None)


@pytest.mark.parametrize("fn", ["gqa_attention_decode_q8", "gqa_attention_prefill_q8", "gqa_attention_decode_i8",
                                "gqa_attention_prefill_i8"])
@pytest.mark.parametrize("ptrs,code", [
    (dict(k_scale=None), 1), (dict(v_scale=None), 1), (dict(k_scale=FAKE + 2), 1),  # scales: fp32, aligned
    (dict(present_k=FAKE + 8), 1), (dict(out=None), 1), (dict(q=None), 1),
])
def test_q8_invalid_arguments(g, fn, ptrs, code):
    assert call_q8(g, good_params(g), fn, **ptrs) == code


@pytest.mark.parametrize("fn", ["gqa_attention_decode_q8", "gqa_attention_prefill_q8", "gqa_attention_decode_i8",
                                "gqa_attention_prefill_i8"])
def test_q8_rejects_a_ring(g, fn):
    assert call_q8(g, good_params(g, kv_ring=1, window=1000), fn) == 2


def call_noalloc(g, p, **ptrs):
    names = ["q", "k", "v", "past_k", "past_v", "seqlens_k", "cos", "sin", "head_sink", "out", "present_k",
             "present_v"]
    vals = {n: FAKE for n in names}
    vals.update(ptrs)
    a = [ctypes.c_void_p(vals[n]) if vals[n] is not None else None for n in names]
    return g.lib.gqa_attention_decode_noalloc(ctypes.byref(p), *a, None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(kv_heads=0), 1),                                   # would divide by zero in the scratch plan
    (dict(batch=1 << 20, dtype=7), 1),                       # invalid dtype with a huge batch
    (dict(batch=1 << 20, head_dim=96), 2),                   # unsupported head dim with a huge batch
    (dict(batch=1 << 20, window=-1, cap_present=1 << 16, kv_ring=2), 1),
])
def test_noalloc_validates_before_touching_its_scratch(g, kw, code):
    """Invalid params are rejected by the same checks as gqa_attention_decode, before the
    entry point plans or clears anything in its static scratch (no GPU is needed: nothing
    is launched, and no CUDA call is made)."""
    assert call_noalloc(g, good_params(g, **kw)) == code


def test_noalloc_rejects_pointers_like_decode(g):
    assert call_noalloc(g, good_params(g), q=None) == 1
    assert call_noalloc(g, good_params(g), out=FAKE + 2) == 1


def test_stall_hook_arguments(g):
    """The failure-path test hook takes a non-negative cycle count (0 = normal operation)
    and launches nothing by itself."""
    assert g.gqa_test_stall_waits(-1) == g.GQA_ERR_INVALID_ARG
    assert g.gqa_test_stall_waits(0) == g.GQA_OK


def call_nonpad(g, p, nonpad=FAKE, **ptrs):
    names = ["q", "k_cache", "v_cache", "head_sink", "out", "workspace"]
    vals = {n: FAKE for n in names}
    vals.update(ptrs)
    a = [ctypes.c_void_p(vals[n]) if vals[n] is not None else None for n in names]
    npd = ctypes.c_void_p(nonpad) if nonpad is not None else None
    return g.lib.gqa_attention_nonpad(ctypes.byref(p), npd, a[0], a[1], a[2], a[3], a[4], a[5], 0, None, None)


@pytest.mark.parametrize("kw,ptrs,code", [
    (dict(), dict(nonpad=None), 1), (dict(), dict(nonpad=FAKE + 4), 1),  # int64 lengths, 8-byte aligned
    (dict(do_rotary=1, rope_len=64), dict(), 1),                        # q is used as given
    (dict(kv_ring=1, window=1000), dict(), 1),                          # a plain cache only
    (dict(), dict(q=None), 1), (dict(), dict(out=FAKE + 2), 1), (dict(kv_heads=3), dict(), 1),
])
def test_nonpad_invalid_arguments(g, kw, ptrs, code):
    assert call_nonpad(g, good_params(g, **kw), **ptrs) == code
