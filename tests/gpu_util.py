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


def run_gpu(case: Case, mode: str, separate_present: bool = False, attend_only: bool = False,
            status_init: int = 0, workspace=None):
    """Run one call on cuda:0.  Returns dict(out, present_k, present_v, status) on the device."""
    from sliding_window_gb300 import gqa
    dev = torch.device("cuda:0")

    def d(x):
        return None if x is None else x.to(dev)

    q, k, v = d(case.q), d(case.k), d(case.v)
    past_k, past_v, seq = d(case.past_k), d(case.past_v), d(case.seqlens_k)
    cos, sin, sink = d(case.cos), d(case.sin), d(case.head_sink)
    p = gqa.params_from_dict(case.params)
    if separate_present:
        present_k = torch.full_like(past_k, float("nan"))
        present_v = torch.full_like(past_v, float("nan"))
    else:
        present_k, present_v = past_k, past_v
    dv = case.w.v_head_dim or case.w.head_dim
    out = torch.full((q.shape[0], q.shape[1], case.w.q_heads * dv), float("nan"), dtype=q.dtype, device=dev)
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
