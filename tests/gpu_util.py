"""Helpers for the GPU parity tests: run one seeded case through the C ABI and through the
fp64 oracle on the same rounded inputs, and compare.

Tolerances: present_k/present_v and q_rot bit-exact; fp32 outputs max abs error <= 2e-5;
f16/bf16 outputs |gpu - oracle| <= 1e-2 + 1e-2*|oracle| element-wise."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from helpers import storage
from sliding_window_gb300.inputs import Case

TOL_F32 = 2e-5
TOL_ABS, TOL_REL = 1e-2, 1e-2


GUARD_BYTES = 4096  # margin on each side of a guarded buffer (a multiple of 16: the interior stays aligned)


class Guarded:
    """A device tensor placed inside a larger buffer whose margins hold a seeded random bit
    pattern; check() asserts the margins are bit for bit what they were, so a kernel that
    writes past either end of the tensor fails the test (the stand-in for a bounds checker)."""
    _seed = 0

    def __init__(self, shape, dtype, device, fill=None):
        esize = torch.empty((), dtype=dtype).element_size()
        self.g = GUARD_BYTES // esize
        n = int(np.prod(shape))
        self.whole = torch.empty(n + 2 * self.g, dtype=dtype, device=device)
        Guarded._seed += 1
        gen = torch.Generator(device="cpu").manual_seed(9000 + Guarded._seed)
        pattern = torch.randint(0, 256, (2 * GUARD_BYTES,), dtype=torch.uint8, generator=gen).to(device)
        raw = self.whole.view(torch.uint8)
        raw[:GUARD_BYTES].copy_(pattern[:GUARD_BYTES])
        raw[raw.numel() - GUARD_BYTES:].copy_(pattern[GUARD_BYTES:])
        self.pattern = pattern
        self.t = self.whole[self.g:self.g + n].view(shape)
        if fill is not None:
            self.t.copy_(fill) if torch.is_tensor(fill) else self.t.fill_(fill)

    def check(self, what: str):
        raw = self.whole.view(torch.uint8)
        assert torch.equal(raw[:GUARD_BYTES], self.pattern[:GUARD_BYTES]), "%s: write before the buffer" % what
        assert torch.equal(raw[raw.numel() - GUARD_BYTES:], self.pattern[GUARD_BYTES:]), \
            "%s: write past the buffer" % what


def run_gpu(case: Case, mode: str, separate_present: bool = False, attend_only: bool = False,
            status_init: int = 0, workspace=None):
    """Run one call on cuda:0.  Returns dict(out, present_k, present_v, status) on the device.
    out and present sit inside guarded buffers whose margins are checked after the call."""
    from sliding_window_gb300 import gqa
    dev = torch.device("cuda:0")

    def d(x):
        return None if x is None else x.to(dev)

    q, k, v = d(case.q), d(case.k), d(case.v)
    seq = d(case.seqlens_k)
    cos, sin, sink = d(case.cos), d(case.sin), d(case.head_sink)
    p = gqa.params_from_dict(case.params)
    gk = Guarded(case.past_k.shape, case.past_k.dtype, dev, fill=case.past_k.to(dev))
    gv = Guarded(case.past_v.shape, case.past_v.dtype, dev, fill=case.past_v.to(dev))
    guards = [(gk, "present_k"), (gv, "present_v")]
    past_k, past_v = gk.t, gv.t
    if separate_present:
        pk_g = Guarded(case.past_k.shape, case.past_k.dtype, dev, fill=float("nan"))
        pv_g = Guarded(case.past_v.shape, case.past_v.dtype, dev, fill=float("nan"))
        guards = [(gk, "past_k"), (gv, "past_v"), (pk_g, "present_k"), (pv_g, "present_v")]
        present_k, present_v = pk_g.t, pv_g.t
    else:
        present_k, present_v = past_k, past_v
    dv = case.w.v_head_dim or case.w.head_dim
    go = Guarded((q.shape[0], q.shape[1], case.w.q_heads * dv), q.dtype, dev, fill=float("nan"))
    guards.append((go, "out"))
    out = go.t
    status = torch.full((1,), status_init, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.zeros(max(16, gqa.gqa_workspace_bytes(p)), dtype=torch.uint8, device=dev)
    fn = gqa.gqa_attention_decode if mode == "decode" else gqa.gqa_attention_prefill
    if attend_only:
        q_rot = torch.empty_like(q)
        gqa.check(gqa.gqa_rope_append_kv(p, q, k, v, past_k, past_v, seq, cos, sin, q_rot, present_k, present_v,
                                         status), "rope_append")
        p2 = gqa.params_from_dict(dict(case.params, do_rotary=0))
        gqa.check(fn(p2, q_rot, None, None, None, None, seq, None, None, sink, out, present_k, present_v, workspace,
                     status), mode)
    else:
        gqa.check(fn(p, q, k, v, past_k, past_v, seq, cos, sin, sink, out, present_k, present_v, workspace, status),
                  mode)
    torch.cuda.synchronize()
    for g, what in guards:
        g.check(what)
    return dict(out=out, present_k=present_k, present_v=present_v, status=int(status.item()), workspace=workspace)


def oracle_ref(case: Case, rows=None, host_present=None):
    """Oracle on the case's rounded inputs.  Returns (out_fp64, present_k, present_v, status).
    host_present=(pk, pv): numpy storage arrays updated in place (saves a copy at full size)."""
    p = case.params
    cs = None if case.cos is None else storage(case.cos)
    sn = None if case.sin is None else storage(case.sin)
    if p.get("kv_ring", 0):
        q_rot, pk, pv, st = oracle.rope_append_ring(p, storage(case.q), storage(case.k), storage(case.v),
                                                    storage(case.past_k), storage(case.past_v),
                                                    case.seqlens_k.cpu().numpy(), cs, sn)
        sink = None if case.head_sink is None else case.head_sink.cpu().numpy()
        return oracle.attention_ring(p, q_rot, pk, pv, case.seqlens_k.cpu().numpy(), sink, rows=rows), pk, pv, st
    if host_present is None:
        q_rot, pk, pv, st = oracle.rope_append(p, storage(case.q), storage(case.k), storage(case.v),
                                               storage(case.past_k), storage(case.past_v),
                                               case.seqlens_k.cpu().numpy(), cs, sn)
    else:
        pk, pv = host_present
        q_rot, pk, pv, st = oracle.rope_append(p, storage(case.q), storage(case.k), storage(case.v), pk, pv,
                                               case.seqlens_k.cpu().numpy(), cs, sn, present_k=pk, present_v=pv)
    sink = None if case.head_sink is None else case.head_sink.cpu().numpy()
    out = oracle.attention(p, q_rot, pk, pv, case.seqlens_k.cpu().numpy(), sink, rows=rows)
    return out, pk, pv, st


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    got = np.asarray(got, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite output" % what
    if dtype == "f32":
        err = np.abs(got - ref).max()
        assert err <= TOL_F32, "%s: max abs error %.3g > %.1g" % (what, err, TOL_F32)
    else:
        excess = np.abs(got - ref) - (TOL_ABS + TOL_REL * np.abs(ref))
        i = np.unravel_index(np.argmax(excess), excess.shape)
        assert excess.max() <= 0, "%s: error %.3g at %s (ref %.4g, got %.4g)" % (
            what, abs(got[i] - ref[i]), i, ref[i], got[i])


def out_rows(out: torch.Tensor, case: Case, rows=None) -> np.ndarray:
    """GPU output as fp64 [B, curr, Hq, Dv] (or [len(rows), Dv])."""
    w = case.w
    dv = w.v_head_dim or w.head_dim
    o = out.detach().to(torch.float64).cpu().numpy().reshape(w.batch * w.q_len * w.q_heads, dv)
    if rows is None:
        return o.reshape(w.batch, w.q_len, w.q_heads, dv)
    return o[np.asarray(rows)]
