"""The indexer + top-k entry point that allocates nothing (v4a_index_topk_noalloc).

It serves callers that can neither allocate device memory nor lend the library a
workspace (a runtime that owns all device memory, or a path where an allocation would
synchronise or break a fixed memory budget). Its scores live in a fixed scratch array in
the library's device image. These tests call it through the C ABI and check that it
returns the same lists as v4a_index_topk on the same inputs, twice in a row (the second
call runs over a smaller region than the first, so stale scratch contents would show),
and that requests larger than the scratch are refused. This file is collected last.
"""
import numpy as np
import pytest
import torch

import compressed_sparse_long_gb300 as v4a
import workloads as wl
from helpers import DevInputs, check_topk, device_layer, oracle_pools
from oracle import v4a_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    yield
    torch.cuda.synchronize()


def _both(w, k=512):
    h = w.layers[0]
    lay, x = device_layer(h), DevInputs(w)
    ref = lay.index_topk(x.q_seq, x.q_pos, x.max_pos, x.q_idx, x.w, k=k)
    got = torch.full_like(ref, -7)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    v4a.v4a_index_topk_noalloc(lay.cfg, len(w.queries.pos), x.q_seq, x.q_pos, x.max_pos,
                               x.q_idx, x.w, lay.idx.c, k, got, err)
    assert v4a.v4a_get_error(err) == 0
    return got.cpu().numpy(), ref.cpu().numpy()


def test_noalloc_matches_workspace_call_twice():
    # first call: 32 queries over 8191 entries each (1 MiB of scores)
    w1 = wl.c4a_decode(seed=31, B=32, L=32768)
    got, ref = _both(w1)
    assert np.array_equal(got, ref)
    # second call: fewer queries, shorter rows, different data; the scratch still holds the
    # first call's scores beyond this call's region
    w2 = wl.c4a_decode(seed=32, B=5, L=4096)
    got2, ref2 = _both(w2)
    assert np.array_equal(got2, ref2)
    # and both agree with the oracle within the top-k tie band
    h = w2.layers[0]
    q = w2.queries
    o_top, scores = O.index_topk(h.spec, oracle_pools(h), q.seq, q.pos, q.q_idx, q.w, 512)
    check_topk(got2, o_top, scores, 512)


def test_noalloc_with_the_fp4_cache():
    w = wl.c4a_decode(seed=34, B=8, L=8192, idx_fp4=True)
    got, ref = _both(w)
    assert np.array_equal(got, ref)


def test_noalloc_rows_longer_than_32768_entries():
    """Two queries that each see 39,999 entries: the selection stages each row in shared
    memory (the path for rows of 32,768 to 49,152 entries). Same lists as the workspace
    call, and the oracle's within the tie band."""
    w = wl.c4a_decode(seed=35, B=2, L=160000)
    got, ref = _both(w)
    assert np.array_equal(got, ref)
    h = w.layers[0]
    q = w.queries
    o_top, scores = O.index_topk(h.spec, oracle_pools(h), q.seq, q.pos, q.q_idx, q.w, 512)
    assert len(scores[0]) == 39999
    check_topk(got, o_top, scores, 512)


def test_noalloc_request_exactly_at_capacity():
    """64 queries whose score rows fill the scratch exactly: max_pos = 131,067 gives 32,765
    visible entries, rows of 32,768 floats, 64 x 32,768 = the capacity. The chunk's own
    entries are inserted first, so every visible entry holds a key."""
    cap = v4a.v4a_index_topk_noalloc_capacity()
    w = wl.c4a_prefill(seed=36, cached=131004, chunk=64)
    h = w.layers[0]
    lay, x = device_layer(h), DevInputs(w)
    assert x.max_pos == 131067
    assert 64 * v4a.v4a_index_scores_row_stride(lay.cfg, x.max_pos) == cap
    lay.compress_insert(x.cu, x.start, x.kv, x.s, x.ik, x.is_)
    ref = lay.index_topk(x.q_seq, x.q_pos, x.max_pos, x.q_idx, x.w)
    got = torch.full_like(ref, -7)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    v4a.v4a_index_topk_noalloc(lay.cfg, 64, x.q_seq, x.q_pos, x.max_pos, x.q_idx, x.w,
                               lay.idx.c, 512, got, err)
    assert v4a.v4a_get_error(err) == 0
    assert torch.equal(got, ref)
    # the next larger row (max_pos 131,080: 32,769 visible entries, rows of 32,772 floats)
    # no longer fits and is refused
    assert 64 * v4a.v4a_index_scores_row_stride(lay.cfg, 131080) > cap
    with pytest.raises(v4a.V4AError) as e:
        v4a.v4a_index_topk_noalloc(lay.cfg, 64, x.q_seq, x.q_pos, 131080, x.q_idx,
                                   x.w, lay.idx.c, 512, got)
    assert e.value.code == -5


def test_noalloc_refuses_requests_beyond_the_scratch():
    cap = v4a.v4a_index_topk_noalloc_capacity()
    assert cap == (8 << 20) // 4
    w = wl.c4a_decode(seed=33, B=2, L=1024)
    h = w.layers[0]
    lay, x = device_layer(h), DevInputs(w)
    out = torch.empty((2, 512), dtype=torch.int32, device="cuda")
    max_pos = 4 * (cap // 2) + 8 + 4 * 16        # 2 rows of more than cap/2 entries each
    with pytest.raises(v4a.V4AError) as e:
        v4a.v4a_index_topk_noalloc(lay.cfg, 2, x.q_seq, x.q_pos, max_pos, x.q_idx, x.w,
                                   lay.idx.c, 512, out)
    assert e.value.code == -5
