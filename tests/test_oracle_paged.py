"""Pins for the oracle's paged layout of the cache (ExecuTorch PR #21901 Summary: a cell
cache whose slots belong to sequences, masked rather than evicted).  A pool of 64-position
pages [num_pages, Hkv, 64, D] and a block table [B, max_pages].  Each pin ties the paged
functions to the contiguous-layout oracle (pinned on its own) through a re-layout done here
with numpy indexing."""
import numpy as np
import pytest

import oracle
from helpers import storage
from sliding_window_gb300.inputs import Workload, make_case

PAGE = 64


def linear_case(dtype, curr, cap, W, rotary, seed, B=3, D=16, past_lo=0, past_hi=None):
    w = Workload("paged", 90 + seed, "decode", dtype, B, 4, 2, D, curr, cap, past_lo,
                 past_hi if past_hi is not None else cap - curr, windows=(W,), head_sink=True, do_rotary=rotary,
                 rope_len=cap + 8)
    return make_case(w, seed_offset=seed)


def to_paged(lin: np.ndarray, table: np.ndarray, num_pages: int, fill):
    """[B, Hkv, cap, D] contiguous cache -> pool [num_pages, Hkv, 64, D] via the table;
    pages no sequence owns keep `fill`."""
    B, Hkv, cap, D = lin.shape
    pool = np.full((num_pages, Hkv, PAGE, D), fill, dtype=lin.dtype)
    for b in range(B):
        for n in range(cap // PAGE):
            pool[table[b, n]] = lin[b, :, n * PAGE:(n + 1) * PAGE]
    return pool


def shuffled_table(B, max_pages, num_pages, seed):
    rng = np.random.default_rng(seed)
    return rng.permutation(num_pages)[:B * max_pages].reshape(B, max_pages).astype(np.int32)


@pytest.mark.parametrize("dtype,curr,W,rotary", [("bf16", 1, -1, 0), ("f16", 3, 100, 1), ("f32", 2, 64, 1),
                                                 ("bf16", 4, 1, 0)])
def test_paged_step_equals_contiguous_step(dtype, curr, W, rotary):
    """The same step through a shuffled, shared pool and through the contiguous cache: the
    pages written hold exactly the contiguous rows, and the outputs are bitwise equal."""
    cap, B, num_pages = 256, 3, 20
    c = linear_case(dtype, curr, cap, W, rotary, seed=curr)
    p = dict(c.params)
    table = shuffled_table(B, cap // PAGE, num_pages, seed=curr)
    nan = np.float32("nan") if dtype == "f32" else np.uint16(0x7FC0)
    pool_k = to_paged(storage(c.past_k), table, num_pages, nan)
    pool_v = to_paged(storage(c.past_v), table, num_pages, nan)
    seq = c.seqlens_k.numpy()
    cs, sn = (storage(c.cos), storage(c.sin)) if rotary else (None, None)
    out_l, lk, lv, qr_l, st_l = oracle.gqa(p, storage(c.q), storage(c.k), storage(c.v), storage(c.past_k),
                                           storage(c.past_v), seq, cs, sn, c.head_sink.numpy())
    qr_p, pk, pv, st_p = oracle.rope_append_paged(p, storage(c.q), storage(c.k), storage(c.v), pool_k, pool_v, seq,
                                                  table, num_pages, PAGE, cs, sn)
    assert st_l == st_p == 0
    np.testing.assert_array_equal(qr_p, qr_l)
    np.testing.assert_array_equal(pk.view(np.uint8), to_paged(lk, table, num_pages, nan).view(np.uint8))
    np.testing.assert_array_equal(pv.view(np.uint8), to_paged(lv, table, num_pages, nan).view(np.uint8))
    out_p = oracle.attention_paged(p, qr_p, pk, pv, seq, table, num_pages, PAGE, c.head_sink.numpy())
    np.testing.assert_array_equal(out_p, out_l)


def test_unused_pages_and_table_entries_are_never_read():
    """Pages before the window's first page, pages past the last position and table entries
    no position uses may hold anything (NaN, or an out-of-range page index)."""
    cap, B, num_pages, W, curr = 512, 2, 24, 70, 1
    c = linear_case("bf16", curr, cap, W, 0, seed=7, B=B, past_lo=300, past_hi=400)
    p = dict(c.params)
    table = shuffled_table(B, cap // PAGE, num_pages, seed=7)
    seq = c.seqlens_k.numpy()
    pool_k = to_paged(storage(c.past_k), table, num_pages, np.uint16(0x7FC0))
    pool_v = to_paged(storage(c.past_v), table, num_pages, np.uint16(0x7FC0))
    ref, *_ = oracle.gqa(p, storage(c.q), storage(c.k), storage(c.v), storage(c.past_k), storage(c.past_v), seq,
                         None, None, c.head_sink.numpy())
    bad = table.copy()
    for b in range(B):
        lo_page = max(0, int(seq[b]) - W + 1) // PAGE
        hi_page = (int(seq[b]) + curr - 1) // PAGE
        bad[b, :lo_page] = -5
        bad[b, hi_page + 1:] = 10 ** 6
        for n in list(range(lo_page)) + list(range(hi_page + 1, cap // PAGE)):
            pool_k[table[b, n]] = np.uint16(0x7FC0)
            pool_v[table[b, n]] = np.uint16(0x7FC0)
    qr, pk, pv, st = oracle.rope_append_paged(p, storage(c.q), storage(c.k), storage(c.v), pool_k, pool_v, seq, bad,
                                              num_pages, PAGE)
    assert st == 0
    out = oracle.attention_paged(p, qr, pk, pv, seq, bad, num_pages, PAGE, c.head_sink.numpy())
    np.testing.assert_array_equal(out, ref)


def test_out_of_range_page_in_use_rejects_the_sequence():
    cap, B, num_pages = 256, 2, 10
    c = linear_case("bf16", 1, cap, -1, 0, seed=8, B=B, past_lo=100, past_hi=200)
    p = dict(c.params)
    table = shuffled_table(B, cap // PAGE, num_pages, seed=8)
    table[1, 0] = num_pages  # sequence 1 reads position 0 from a page that does not exist
    pool_k = np.zeros((num_pages, 2, PAGE, 16), np.uint16)
    qr, pk, pv, st = oracle.rope_append_paged(p, storage(c.q), storage(c.k), storage(c.v), pool_k, pool_k.copy(),
                                              c.seqlens_k.numpy(), table, num_pages, PAGE)
    assert st == 8
    out = oracle.attention_paged(p, qr, pk, pv, c.seqlens_k.numpy(), table, num_pages, PAGE, c.head_sink.numpy())
    assert np.all(out[1] == 0.0) and np.any(out[0] != 0.0)
