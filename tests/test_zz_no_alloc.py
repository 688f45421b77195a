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
