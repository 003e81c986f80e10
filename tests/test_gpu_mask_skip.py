"""Skipping the key tiles a boolean mask removes entirely (onnx-light-cpu "Attention Kernel
Design", "Compute paths": an all-false boolean-mask block is skipped).  The tensor-core
prefill reads a block map of the mask (one bit per 128-row query tile and 16-key chunk,
built in the workspace) and streams only the 128-key tiles in which the mask keeps a key of
its query tile.  Parity with the fp64 masked oracle for block-sparse masks of every broadcast
shape, with and without a window, with query tiles whose mask keeps nothing, and with a
workspace too small for the map (every tile streamed).  The evidence that dead tiles are
never read: their K/V rows hold NaN, which a streamed tile would carry into the output
(0 * NaN in the PV product), yet the output is finite and matches the oracle."""
import itertools
import zlib

import numpy as np
import pytest
import torch

from gpu_util import assert_close, out_rows
from helpers import storage
from test_gpu_prefill_masks import case, mask_shape, oracle_masked, to_device_mask

pytestmark = pytest.mark.gpu


def block_sparse(shape, S, keys, rng, dead_tiles=(), dead_frac=0.4, keep=0.7, origin=0):
    """A boolean mask whose 128-row x 128-key blocks (key blocks counted from `origin`) are
    all-false with probability dead_frac, and all-false in the key tiles `dead_tiles` for
    every row; other blocks keep each key with probability `keep`."""
    m = (rng.random(shape) < keep).astype(np.uint8)
    nq = shape[2]
    for qb in range(0, nq, 128):
        for kb in range(origin, keys, 128):
            if rng.random() < dead_frac:
                m[..., qb:qb + 128, max(0, kb):kb + 128] = 0
    for t in dead_tiles:
        m[..., origin + 128 * t:origin + 128 * (t + 1)] = 0
    return m


def run_ws(c, mask_np, ws_bytes=None):
    """The masked prefill with the workspace gqa_workspace_bytes gives (the map fits), or with
    ws_bytes (too small for the map: every tile is streamed)."""
    from sliding_window_gb300 import gqa
    d = lambda x: None if x is None else x.cuda()  # noqa: E731
    p = gqa.params_from_dict(c.params)
    pk, pv = d(c.past_k), d(c.past_v)
    out = torch.full(c.q.shape, float("nan"), dtype=c.q.dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    n = gqa.gqa_workspace_bytes(p) if ws_bytes is None else ws_bytes
    ws = torch.zeros(max(16, n), dtype=torch.uint8, device="cuda")
    m = gqa.mask_from_tensor(to_device_mask(mask_np, "bool", c.params["dtype"]), gqa.MASK_KEEP)
    gqa.check(gqa.gqa_attention_prefill_masked(p, m, d(c.q), d(c.k), d(c.v), pk, pv, d(c.seqlens_k), d(c.cos),
                                               d(c.sin), d(c.head_sink), out, pk, pv, ws, st), "masked prefill")
    torch.cuda.synchronize()
    return out, pk, pv, int(st.item())


SHAPES = ["full", "b1ik", "11ik", "b11k"]


@pytest.mark.parametrize("dtype,shape,spw,softcap", list(itertools.product(
    ["bf16", "f16"], SHAPES, [(384, 512, -1), (300, 700, 300), (200, 0, -1)], [0.0, 25.0])))
def test_block_sparse_mask_parity(dtype, shape, spw, softcap):
    S, past, W = spw
    seed = zlib.crc32(repr((dtype, shape, spw, softcap)).encode()) % 1000
    c = case("prefill", dtype, 128, 2, S, past, W, softcap=softcap, seed=seed % 53)
    B, Hq = c.q.shape[0], c.params["q_heads"]
    keys = -(-(past + S) // 16) * 16
    mask = block_sparse(mask_shape(shape, B, Hq, S, keys), S, keys, np.random.default_rng(seed))
    ref, rk, rv, s = oracle_masked(c, mask, "bool")
    for ws_bytes in (None, 16):  # with the block map; without it (every tile streamed)
        out, pk, pv, st = run_ws(c, mask, ws_bytes)
        assert st == 0 and s == 0
        np.testing.assert_array_equal(storage(pk), rk)
        np.testing.assert_array_equal(storage(pv), rv)
        assert_close(out_rows(out, c), ref, dtype, "block-sparse %s ws %s" % ((dtype, shape, spw), ws_bytes))


@pytest.mark.parametrize("shape", SHAPES)
def test_dead_tiles_are_never_read(shape):
    """Key tiles 1 and 3 (keys [128, 256) and [384, 512) of the past) are all-false for every
    row: their K and V rows are NaN.  Streamed, they would make the output NaN."""
    S, past = 384, 512
    c = case("prefill", "bf16", 128, 2, S, past, -1, seed=5)
    B, Hq = c.q.shape[0], c.params["q_heads"]
    keys = past + S
    mask = block_sparse(mask_shape(shape, B, Hq, S, keys), S, keys, np.random.default_rng(5), dead_tiles=(1, 3),
                        dead_frac=0.2)
    for t in (c.past_k, c.past_v):
        t[:, :, 128:256] = float("nan")
        t[:, :, 384:512] = float("nan")
    ref, *_ = oracle_masked(c, mask, "bool")
    out, _, _, st = run_ws(c, mask)
    assert st == 0
    assert_close(out_rows(out, c), ref, "bf16", "dead tiles %s" % shape)


def test_query_tile_with_nothing_kept_gives_zeros():
    """A query tile whose mask keeps no key streams no tile: its rows are zeros (with a sink
    too: a fully masked row gives zeros), other tiles are unaffected."""
    S, past = 384, 100
    c = case("prefill", "bf16", 128, 2, S, past, -1, sink="head", seed=9)
    B, Hq = c.q.shape[0], c.params["q_heads"]
    keys = -(-(past + S) // 16) * 16
    mask = block_sparse((B, Hq, S, keys), S, keys, np.random.default_rng(9), dead_frac=0.0)
    mask[1, :, 128:256, :] = 0  # batch 1, query tile 1: nothing kept
    mask[0, 2:4, 0:128, :] = 0  # batch 0, heads 2 and 3 (one CTA), query tile 0
    ref, *_ = oracle_masked(c, mask, "bool")
    out, _, _, st = run_ws(c, mask)
    assert st == 0
    o = out_rows(out, c)
    assert np.all(o[1, 128:256] == 0.0) and np.all(o[0, 0:128, 2:4] == 0.0)
    assert_close(o, ref, "bf16", "empty query tiles")
