"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the same seeded
inputs. Marked gpu; the acceptance rules are in helpers.py."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import compressed_sparse_long_gb300 as v4a
import workloads as wl
from helpers import (DevInputs, T, check_fp4_rows, check_fp8_rows, check_out, check_topk,
                     device_layer, device_pools, oracle_insert, oracle_pools)
from oracle import v4a_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    torch.cuda.synchronize()
    yield
    torch.cuda.synchronize()


def _err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _gpu_rows(pool):
    d = pool.data.cpu()
    if d.dtype == torch.bfloat16:
        d = d.float()
    return d.numpy(), None if pool.scale is None else pool.scale.cpu().numpy()


def _compare_written(dev_layer, pools, writes, fp8):
    """Rows the oracle wrote must match the GPU's rows at the same pool slots."""
    n_close = 0
    for kind in ("attn", "idx", "swa", "state"):
        slots = sorted({s for (k, _, _, s) in writes if k == kind and s >= 0})
        if not slots:
            continue
        g_data, g_scale = _gpu_rows(getattr(dev_layer, kind))
        ref = getattr(pools, kind)
        if kind == "state":
            assert np.array_equal(g_data[slots], ref.data[slots]), "residual rows differ"
        elif fp8:
            n_close += check_fp8_rows(g_data, g_scale, ref, slots)
        else:
            d = np.abs(g_data[slots] - ref.data[slots])
            assert d.max() <= 1e-5, (kind, d.max())
    return n_close


# ------------------------------------------------------------------------- fp32 layer
@pytest.mark.parametrize("win_off", [0, -4])
def test_tiny_fp32_layer_every_position(win_off):
    """Tiny fp32 c4a layer, one sequence of 1024 tokens, all 1024 positions queried:
    insert (every written row), index + top-64 (tie band, every row) and attention on the
    GPU's own lists over the GPU-written rows (every row, max-abs 1e-4)."""
    w = wl.tiny_prefill(seed=0, L=1024, win_off=win_off)
    h = w.layers[0]
    lay, x, err = device_layer(h), DevInputs(w), _err()
    out, topk = lay.step(x.cu, x.start, x.kv, x.s, x.ik, x.is_, x.q_seq, x.q_pos, x.max_pos,
                         x.q, x.q_idx, x.w, prefill=True, dev_err=err)
    assert v4a.v4a_get_error(err) == 0
    pools = oracle_pools(h)
    writes = oracle_insert(w, h, pools)
    _compare_written(lay, pools, writes, fp8=False)
    _check_rows(w, h, lay, out.cpu().numpy(), topk.cpu().numpy(), np.arange(len(w.queries.pos)))


def test_tiny_fp32_decode_splits_and_merge():
    """fp32 layer, a few late queries through the decode call (keys split over CTAs and
    merged), against the oracle on the same stored rows."""
    w = wl.tiny_prefill(seed=9, L=1024)
    h = w.layers[0]
    lay, x = device_layer(h), DevInputs(w)
    lay.compress_insert(x.cu, x.start, x.kv, x.s, x.ik, x.is_)
    sel = np.array([300, 511, 777, 1000, 1023])
    topk = lay.index_topk(x.q_seq[sel], x.q_pos[sel], 1023, x.q_idx[sel].contiguous(),
                          x.w[sel].contiguous())
    out = lay.attention(x.q_seq[sel], x.q_pos[sel], 1023, x.q[sel].contiguous(), topk)
    assert lay.cfg.n_heads == 8
    sub = wl.Workload(w.name, w.layers, w.batch, wl.Queries(
        w.queries.seq[sel], w.queries.pos[sel], w.queries.q[sel], w.queries.q_idx[sel],
        w.queries.w[sel]))
    _check_rows(sub, h, lay, out.cpu().numpy(), topk.cpu().numpy(), np.arange(len(sel)))


def test_slot_mapping_bit_exact():
    rng = np.random.default_rng(0)
    for R in (256, 64, 2):
        need = [set(rng.choice(40, 25, replace=False).tolist()) for _ in range(3)]
        bt, n_pages = wl.block_table(rng, need, 40)
        n = 5000
        seq = rng.integers(0, 3, n).astype(np.int32)
        row = rng.integers(-3, 40 * R + 10, n).astype(np.int64)
        data = torch.zeros((n_pages * R, 16), dtype=torch.uint8, device="cuda")
        bt_dev = T(bt, torch.int32)                 # must outlive the launch
        c = v4a.cache(data, None, bt_dev, R)
        slots = torch.empty(n, dtype=torch.int32, device="cuda")
        v4a.v4a_slot_mapping(c, n, T(seq, torch.int32), T(row, torch.int64), slots)
        want = np.array([O.slot(bt, R, int(s), int(r)) for s, r in zip(seq, row)])
        assert np.array_equal(slots.cpu().numpy(), want)


# ------------------------------------------------------------------------ compressor
@pytest.mark.parametrize("kind", ["c4a", "c128a"])
def test_compress_insert_fp8_ragged_chunks(kind):
    """Several sequences with ragged contexts and chunks (windows spanning the residual
    pool, partial windows left behind); every written row is compared."""
    spec = wl.LayerSpec(kind, True)
    rng = np.random.default_rng(21)
    ctx = [1000, 37, 127, 4096] if kind == "c4a" else [1000, 130, 127, 4096]
    new = [300, 1, 129, 257]
    h = wl.make_layer(rng, spec, ctx, new, prefill_cache=True)
    h.bias, h.gamma, h.ibias = wl.layer_params(rng, spec)
    b = wl.make_batch(rng, spec, ctx, new)
    w = wl.Workload("ragged", [h], b, wl.make_queries(rng, spec, np.arange(4), np.array(ctx),
                                                      False))
    lay, x, err = device_layer(h), DevInputs(w), _err()
    lay.compress_insert(x.cu, x.start, x.kv, x.s, x.ik, x.is_, dev_err=err)
    assert v4a.v4a_get_error(err) == 0
    pools = oracle_pools(h)
    writes = oracle_insert(w, h, pools)
    assert any(k == "attn" for (k, _, _, _) in writes)
    _compare_written(lay, pools, writes, fp8=True)


def test_compress_chunking_invariance_gpu():
    """One call or several ragged calls write identical bytes on the GPU."""
    w = wl.c4a_prefill(seed=3, cached=4096, chunk=1000)
    h = w.layers[0]
    one, many = device_layer(h), device_layer(h)
    x = DevInputs(w)
    one.compress_insert(x.cu, x.start, x.kv, x.s, x.ik, x.is_)
    cuts = [0, 3, 4, 77, 500, 999, 1000]
    for a, b in zip(cuts[:-1], cuts[1:]):
        cu = torch.tensor([0, b - a], dtype=torch.int32, device="cuda")
        st = torch.tensor([4096 + a], dtype=torch.int64, device="cuda")
        many.compress_insert(cu, st, x.kv[a:b].contiguous(), x.s[a:b].contiguous(),
                             x.ik[a:b].contiguous(), x.is_[a:b].contiguous())
    for name in ("attn", "idx", "swa"):
        p1, p2 = getattr(one, name), getattr(many, name)
        assert torch.equal(p1.data, p2.data) and torch.equal(p1.scale, p2.scale), name


# -------------------------------------------------------------------- indexer / top-k
def _pools_equal(a, b):
    for kind in ("attn", "idx", "swa", "state"):
        pa, pb = getattr(a, kind), getattr(b, kind)
        if pa is None:
            continue
        assert torch.equal(pa.data, pb.data), kind
        if pa.scale is not None:
            assert torch.equal(pa.scale, pb.scale), kind


@pytest.mark.parametrize("fp8", [True, False])
def test_compress_insert_qnorm(fp8):
    """Fusion 3 (static warp dispatch): the insert warps of v4a_compress_insert_qnorm write
    the same bytes as v4a_compress_insert; every (query, head) row of q_out is the oracle's
    per-head RMSNorm to within one rounding to the output type (bf16: 2^-8 relative; fp32:
    1e-5 relative), and within the layer tolerances; q_out == q gives the same rows in
    place; n_tokens = 0 runs the norm alone and leaves the pools untouched."""
    w = wl.c4a_decode(seed=31, B=8, L=4096) if fp8 else wl.tiny_prefill(seed=32, L=300)
    h = w.layers[0]
    rng = np.random.default_rng(33)
    dt = torch.bfloat16 if fp8 else torch.float32
    q_gamma = rng.normal(1.0, 0.1, h.spec.D)
    # heads at very different scales, as a joint or wrong-axis norm would not survive
    q_host = np.asarray(w.queries.q, dtype=np.float64) * \
        (2.0 ** ((np.arange(h.spec.H) % 9) - 4.0))[None, :, None]
    q_host = T(q_host, dt).float().cpu().numpy().astype(np.float64)   # what the kernel reads
    lay, x, err = device_layer(h), DevInputs(w), _err()
    ref_lay = lay.clone_pools()
    qd, gd = T(q_host, dt), T(q_gamma, torch.float32)
    q_out = lay.compress_insert_qnorm(x.cu, x.start, x.kv, x.s, x.ik, x.is_, qd, gd,
                                      dev_err=err)
    ref_lay.compress_insert(x.cu, x.start, x.kv, x.s, x.ik, x.is_, dev_err=err)
    torch.cuda.synchronize()
    assert v4a.v4a_get_error(err) == 0
    _pools_equal(lay, ref_lay)

    o = O.q_norm(q_host, q_gamma, h.spec.eps)
    g = q_out.float().cpu().numpy()
    d = np.abs(g - o)
    rel = 2.0 ** -8 * 1.001 if fp8 else 1e-5
    assert np.all(d <= rel * np.abs(o) + 1e-6), d.max()
    if fp8:
        assert d.max() <= 3e-2 and d.mean() <= 3e-3
    else:
        assert d.max() <= 1e-4

    # in place, and the norm alone
    q_in = qd.clone()
    before = lay.clone_pools()
    lay.compress_insert_qnorm(x.cu[:1], x.start[:0], x.kv[:0], x.s[:0],
                              None if x.ik is None else x.ik[:0],
                              None if x.is_ is None else x.is_[:0], q_in, gd, q_out=q_in,
                              dev_err=err)
    torch.cuda.synchronize()
    assert torch.equal(q_in, q_out)
    _pools_equal(lay, before)


def _inject_subnormal_keys(h, rng, n=200):
    """Give some indexer rows only subnormal e4m3 codes and a large scale, so a wrong
    decoding of subnormal codes changes the scores."""
    used = np.nonzero(h.idx.data.any(axis=1))[0]
    rows = rng.choice(used, size=min(n, len(used)), replace=False)
    codes = rng.integers(0, 8, size=(len(rows), h.idx.data.shape[1]))
    codes |= rng.integers(0, 2, size=codes.shape) << 7
    h.idx.data[rows] = codes.astype(np.uint8)
    h.idx.scale[rows] = 2000.0


def test_index_topk_fp8_decode():
    w = wl.c4a_decode(seed=1, B=8, L=8192)
    h = w.layers[0]
    _inject_subnormal_keys(h, np.random.default_rng(5))
    lay, x, err = device_layer(h), DevInputs(w), _err()
    topk = lay.index_topk(x.q_seq, x.q_pos, x.max_pos, x.q_idx, x.w, dev_err=err)
    assert v4a.v4a_get_error(err) == 0
    pools = oracle_pools(h)
    q = w.queries
    ref, scores = O.index_topk(h.spec, pools, q.seq, q.pos, q.q_idx, q.w, 512)
    same = check_topk(topk.cpu().numpy(), ref, scores, 512)
    assert len(same) >= 6


def test_compress_insert_fp4_indexer_rows():
    """fp4 indexer cache: the insert writes each completed indexer entry as packed e2m1
    codes + amax/6 row scale equal to the oracle's (codes may differ by one grid step only
    at a rounding tie); attention and window rows are the fp8 rows of the default layer."""
    spec = wl.LayerSpec("c4a", True, idx_fp4=True)
    rng = np.random.default_rng(41)
    ctx, new = [1000, 37, 127, 4096], [300, 1, 129, 257]
    h = wl.make_layer(rng, spec, ctx, new, prefill_cache=True)
    h.bias, h.gamma, h.ibias = wl.layer_params(rng, spec)
    b = wl.make_batch(rng, spec, ctx, new)
    w = wl.Workload("ragged fp4", [h], b, wl.make_queries(rng, spec, np.arange(4), np.array(ctx),
                                                         False))
    lay, x, err = device_layer(h), DevInputs(w), _err()
    assert lay.idx.data.shape[1] == 64 and lay.idx.c.row_width == 128
    lay.compress_insert(x.cu, x.start, x.kv, x.s, x.ik, x.is_, dev_err=err)
    assert v4a.v4a_get_error(err) == 0
    pools = oracle_pools(h)
    writes = oracle_insert(w, h, pools)
    slots = sorted({sl for (k, _, _, sl) in writes if k == "idx" and sl >= 0})
    assert len(slots) > 100
    g_data, g_scale = _gpu_rows(lay.idx)
    check_fp4_rows(g_data.astype(np.uint8), g_scale, pools.idx, slots)
    _compare_written(lay, pools, [wr for wr in writes if wr[0] != "idx"], fp8=True)


@pytest.mark.parametrize("B,L", [(8, 8192), (32, 32768)])
def test_index_topk_fp4_decode(B, L):
    """Indexer over an fp4 cache (packed pages expanded on chip to exact e4m3 operands):
    the top-k lists equal the oracle's over the same dequantised keys except near-ties."""
    w = wl.c4a_decode(seed=43, B=B, L=L, idx_fp4=True)
    h = w.layers[0]
    lay, x, err = device_layer(h), DevInputs(w), _err()
    topk = lay.index_topk(x.q_seq, x.q_pos, x.max_pos, x.q_idx, x.w, dev_err=err)
    assert v4a.v4a_get_error(err) == 0
    q = w.queries
    sample = np.arange(B) if B <= 8 else np.array([0, 5, 17, 31])
    pools = oracle_pools(h)
    ref, scores = O.index_topk(h.spec, pools, q.seq[sample], q.pos[sample], q.q_idx[sample],
                               q.w[sample], 512)
    same = check_topk(topk.cpu().numpy()[sample], ref, scores, 512)
    assert len(same) >= len(sample) - 1


def test_index_topk_fp4_prefill_two_queries_per_group():
    """A prefill chunk of 1024 queries over an fp4 indexer cache runs the fp4 kernel with two
    queries per group (N = 256 operand rows); sampled rows match the oracle's top-k."""
    w = wl.c4a_prefill(seed=44, cached=8192, chunk=1024, idx_fp4=True)
    h = w.layers[0]
    lay, x, err = device_layer(h), DevInputs(w), _err()
    lay.compress_insert(x.cu, x.start, x.kv, x.s, x.ik, x.is_, dev_err=err)
    topk = lay.index_topk(x.q_seq, x.q_pos, x.max_pos, x.q_idx, x.w, dev_err=err)
    assert v4a.v4a_get_error(err) == 0
    pools = oracle_pools(h)
    oracle_insert(w, h, pools)
    q = w.queries
    sample = np.array([0, 1, 511, 512, 1022, 1023])
    ref, scores = O.index_topk(h.spec, pools, q.seq[sample], q.pos[sample], q.q_idx[sample],
                               q.w[sample], 512)
    same = check_topk(topk.cpu().numpy()[sample], ref, scores, 512)
    assert len(same) >= len(sample) - 1


@pytest.mark.parametrize("n_q,k", [(16, 512), (5, 64), (3, 2048)])
def test_index_topk_prefill_positions(n_q, k):
    """Queries at many positions of one sequence (ragged visibility, rows shorter and
    longer than k)."""
    w = wl.c4a_prefill(seed=3, cached=16384, chunk=n_q)
    h = w.layers[0]
    q = w.queries
    q.pos = np.sort(np.random.default_rng(1).integers(0, 16384, n_q)).astype(np.int64)
    q.pos[0] = 9                                   # two visible entries
    lay, x = device_layer(h), DevInputs(w)
    topk = lay.index_topk(x.q_seq, x.q_pos, int(q.pos.max()), x.q_idx, x.w, k=k)
    pools = oracle_pools(h)
    ref, scores = O.index_topk(h.spec, pools, q.seq, q.pos, q.q_idx, q.w, k)
    check_topk(topk.cpu().numpy(), ref, scores, k)


@pytest.mark.parametrize("k", [64, 512, 1024, 1025, 2048])
def test_index_topk_streaming_rows(k):
    """Rows longer than the register-resident selection holds (up to 16,383 entries), five
    rows (1024 threads a row): the streaming selection with its candidate floor (each warp's
    ceil(k / 32)-th largest candidate; k <= 2048) against the oracle's lists; one row is
    shorter than k."""
    w = wl.c4a_prefill(seed=61, cached=65536, chunk=5)
    h = w.layers[0]
    q = w.queries
    q.pos = np.array([65536 + 4, 60001, 40000, 33000, 900], np.int64)
    lay, x = device_layer(h), DevInputs(w)
    assert O.visible_entries(h.spec.S, h.spec.W, h.spec.win_off, 65540) > 8192
    topk = lay.index_topk(x.q_seq, x.q_pos, int(q.pos.max()), x.q_idx, x.w, k=k)
    pools = oracle_pools(h)
    ref, scores = O.index_topk(h.spec, pools, q.seq, q.pos, q.q_idx, q.w, k)
    same = check_topk(topk.cpu().numpy(), ref, scores, k)
    assert len(same) >= len(q.pos) - 1


def test_index_topk_streaming_many_rows():
    """A call with more rows (320) than two per SM, each longer than the register-resident
    selection holds: the streaming selection with 256 threads a row (calls with fewer rows
    use 1024); sampled rows against the oracle's lists."""
    w = wl.c4a_prefill(seed=62, cached=40000, chunk=320)
    h = w.layers[0]
    q = w.queries
    q.pos = np.linspace(33000, 40000, 320).astype(np.int64)
    lay, x = device_layer(h), DevInputs(w)
    assert O.visible_entries(h.spec.S, h.spec.W, h.spec.win_off, 33000) > 8192
    topk = lay.index_topk(x.q_seq, x.q_pos, int(q.pos.max()), x.q_idx, x.w).cpu().numpy()
    sample = np.array([0, 1, 77, 150, 151, 200, 318, 319])
    ref, scores = O.index_topk(h.spec, oracle_pools(h), q.seq[sample], q.pos[sample],
                               q.q_idx[sample], q.w[sample], 512)
    same = check_topk(topk[sample], ref, scores, 512)
    assert len(same) >= len(sample) - 1


@pytest.mark.parametrize("L", [4096, 65536])
def test_topk_ties_take_smaller_index(L):
    """Equal scores: identical keys tie exactly; the smaller entry indices win (rows held in
    registers at L=4096; at L=65536 the streaming selection, whose constant rows take the
    radix passes)."""
    w = wl.c4a_decode(seed=7, B=2, L=L)
    h = w.layers[0]
    h.idx.data[:] = h.idx.data[0]
    h.idx.scale[:] = h.idx.scale[0]
    lay, x = device_layer(h), DevInputs(w)
    topk = lay.index_topk(x.q_seq, x.q_pos, x.max_pos, x.q_idx, x.w).cpu().numpy()
    for i in range(2):
        assert np.array_equal(topk[i], np.arange(512))


@pytest.mark.parametrize("n_tied,rank,L", [(300, 0, 16384), (300, 412, 16384), (1200, 0, 16384),
                                           (300, 0, 65536), (300, 412, 65536), (1200, 0, 65536),
                                           (3000, 0, 65536)])
def test_topk_tied_block(n_tied, rank, L):
    """A block of identical indexer keys (so identical scores) placed wholly above the k-th
    score, across it, or larger than k at the top of the row: the output holds every entry
    scoring above the block and exactly the smallest-index members of the block (rows of
    4095 entries held in registers, rows of 16383 in the streaming selection; a block of
    3000 puts more entries at the streaming selection's floor than its 2048-entry buffer
    holds, so that row takes the whole-row radix passes)."""
    w = wl.c4a_decode(seed=11, B=2, L=L)
    h = w.layers[0]
    q = w.queries
    rng = np.random.default_rng(17)
    _, scores = O.index_topk(h.spec, oracle_pools(h), q.seq, q.pos, q.q_idx, q.w, 512)
    tied = []
    for i in range(len(q.pos)):
        b, sc = int(q.seq[i]), np.asarray(scores[i])
        src = int(np.argsort(-sc, kind="stable")[rank])
        others = rng.choice(np.setdiff1d(np.arange(len(sc)), [src]), n_tied - 1, replace=False)
        r0 = O.slot(h.idx.bt, 64, b, src)
        for j in others:
            r = O.slot(h.idx.bt, 64, b, int(j))
            h.idx.data[r], h.idx.scale[r] = h.idx.data[r0], h.idx.scale[r0]
        tied.append(np.sort(np.append(others, src)))
    lay, x = device_layer(h), DevInputs(w)
    got = lay.index_topk(x.q_seq, x.q_pos, x.max_pos, x.q_idx, x.w).cpu().numpy()
    ref, scores = O.index_topk(h.spec, oracle_pools(h), q.seq, q.pos, q.q_idx, q.w, 512)
    check_topk(got, ref, scores, 512)
    for i in range(len(q.pos)):
        sel = np.intersect1d(got[i], tied[i])
        assert np.array_equal(sel, tied[i][:len(sel)]), "tied block must be taken by index"
        if rank == 0:
            assert len(sel) == min(n_tied, 512)


# ------------------------------------------------------------------------- attention
def _random_lists(rng, pos, spec, k, n_pad=3):
    out = np.full((len(pos), k), -1, np.int32)
    for i, p in enumerate(pos):
        n = O.visible_entries(spec.S, spec.W, spec.win_off, int(p))
        m = max(0, min(k - n_pad, n))
        out[i, :m] = np.sort(rng.choice(n, m, replace=False))
    return out


def _fill_query_window_row(h, w):
    """Random stored window row at each query position (normally written by the insert)."""
    rng = np.random.default_rng(99)
    for b, p in zip(w.queries.seq, w.queries.pos):
        s = O.slot(h.swa.bt, 256, int(b), int(p))
        c, sc = wl.random_fp8_rows(rng, 1, h.spec.D)
        h.swa.data[s], h.swa.scale[s] = c[0], sc[0]


@pytest.mark.parametrize("prefill", [False, True])
def test_attention_fp8_c4a_lists(prefill):
    w = wl.c4a_decode(seed=11, B=8, L=8192)
    h = w.layers[0]
    _fill_query_window_row(h, w)
    q = w.queries
    lists = _random_lists(np.random.default_rng(3), q.pos, h.spec, 512)
    lay, x, err = device_layer(h), DevInputs(w), _err()
    out = lay.attention(x.q_seq, x.q_pos, x.max_pos, x.q, T(lists, torch.int32),
                        prefill=prefill, dev_err=err)
    assert v4a.v4a_get_error(err) == 0
    ref = O.attention(h.spec, oracle_pools(h), q.seq, q.pos, q.q, lists)
    check_out(out.float().cpu().numpy(), ref, fp8=True)


@pytest.mark.parametrize("B,L,width,plan", [
    (32, 4096, 512, (3, 2)), (40, 4096, 128, (2, 2)), (24, 8192, 896, (4, 2)),
    (32, 600, 512, (3, 2)), (16, 4096, 512, (5, 2)), (160, 4096, 512, (1, 1)),
    (16, 8192, 1024, (9, 2)), (8, 600, 1024, (9, 2))])
def test_attention_split_merge_modes(B, L, width, plan):
    """Decode attention with 2, 3, 4, 5 or 9 key ranges per query (partials combined by the
    merge kernel) and without a split. At L=600 a query sees 149 entries: its middle range
    of three (512-wide lists), or most of its nine (1024-wide lists), hold only masked
    entries."""
    w = wl.c4a_decode(seed=17, B=B, L=L)
    h = w.layers[0]
    _fill_query_window_row(h, w)
    q = w.queries
    lists = _random_lists(np.random.default_rng(5), q.pos, h.spec, width)
    lay, x, err = device_layer(h), DevInputs(w), _err()
    assert v4a.v4a_attn_plan(lay.cfg, B, x.max_pos, width) == plan
    tk = T(lists, torch.int32)
    out = lay.attention(x.q_seq, x.q_pos, x.max_pos, x.q, tk, dev_err=err)
    assert v4a.v4a_get_error(err) == 0
    again = lay.attention(x.q_seq, x.q_pos, x.max_pos, x.q, tk, dev_err=err)
    assert torch.equal(again, out)                  # the same bytes on a second call
    ref = O.attention(h.spec, oracle_pools(h), q.seq, q.pos, q.q, lists)
    check_out(out.float().cpu().numpy(), ref, fp8=True)


def _lists_with_masked_blocks(rng, pos, spec, width=512, masked=(0, 2)):
    """Top-`width` lists whose 128-entry blocks named in `masked` are all -1 and whose other
    blocks hold distinct visible entries, each block sorted: with 128-key tiles, a key range
    may then begin with a tile that has no key."""
    out = np.full((len(pos), width), -1, np.int32)
    keep = [t for t in range(width // 128) if t not in masked]
    for i, p in enumerate(pos):
        n = O.visible_entries(spec.S, spec.W, spec.win_off, int(p))
        e = rng.choice(n, 128 * len(keep), replace=False)
        for j, t in enumerate(keep):
            out[i, 128 * t:128 * (t + 1)] = np.sort(e[128 * j:128 * (j + 1)])
    return out


@pytest.mark.parametrize("mode", ["split", "split_wide", "prefill"])
def test_attention_key_range_starting_with_a_masked_tile(mode):
    """Attention where key ranges begin with tiles that hold only masked list entries:
    decode with 3 ranges of 2/2/1 tiles (tiles 0 and 2 masked), decode with 3 ranges of 3
    tiles over 1024-wide lists (tiles 0, 3 and 6 masked: every range) and prefill (one range
    of 5 tiles, tiles 0 and 2 masked). The scaling of P' must be set by the first tile that
    has a key, not by the range's first tile."""
    L, width, masked = (8192, 1024, (0, 3, 6)) if mode == "split_wide" else (4096, 512, (0, 2))
    w = wl.c4a_decode(seed=23, B=32, L=L)
    h = w.layers[0]
    _fill_query_window_row(h, w)
    q = w.queries
    lists = _lists_with_masked_blocks(np.random.default_rng(8), q.pos, h.spec, width, masked)
    lay, x, err = device_layer(h), DevInputs(w), _err()
    if mode != "prefill":
        assert v4a.v4a_attn_plan(lay.cfg, 32, x.max_pos, width) == (3, 2)
    out = lay.attention(x.q_seq, x.q_pos, x.max_pos, x.q, T(lists, torch.int32),
                        prefill=mode == "prefill", dev_err=err)
    assert v4a.v4a_get_error(err) == 0
    ref = O.attention(h.spec, oracle_pools(h), q.seq, q.pos, q.q, lists)
    check_out(out.float().cpu().numpy(), ref, fp8=True)


def _e4m3_step(v):
    """Grid step of the e4m3 value nearest |v| (the spacing a rounding error is bounded by)."""
    g = O.e4m3_values()
    a = np.minimum(np.abs(v), 448.0)
    hi = np.clip(np.searchsorted(g, a, side="left"), 1, len(g) - 1)
    return g[hi] - g[hi - 1]


@pytest.mark.parametrize("B,L", [(8, 8192), (4, 48)])
def test_attention_q8_output(B, L):
    """fp8 output epilogue ([notes] 融合 2：Inverse RoPE + FP8 Quant): per (query, head) row the
    scale is amax/448 and the codes are e4m3 RNE of out/scale. The rule is checked against the
    same attention's bf16 output, the values against the oracle. The lists are 1024 wide (9 key
    tiles), so the bf16 call and the fp8 one split the keys into the same 9 ranges and share
    their arithmetic up to the merge; the short context leaves most ranges empty (the merge
    must skip them)."""
    w = wl.c4a_decode(seed=21, B=B, L=L)
    h = w.layers[0]
    q = w.queries
    width = 1024
    lists = _random_lists(np.random.default_rng(5), q.pos, h.spec, width)
    _fill_query_window_row(h, w)
    lay, x = device_layer(h), DevInputs(w)
    assert v4a.v4a_attn_plan(lay.cfg, B, x.max_pos, width) == (9, 2)
    assert (v4a.v4a_attn_q8_workspace_size(lay.cfg, B, x.max_pos, width)
            == v4a.v4a_attn_workspace_size(lay.cfg, B, x.max_pos, width, False))
    tk = torch.from_numpy(lists).cuda()
    err = _err()
    out = lay.attention(x.q_seq, x.q_pos, x.max_pos, x.q, tk, dev_err=err)
    codes, scale = lay.attention_q8(x.q_seq, x.q_pos, x.max_pos, x.q, tk, dev_err=err)
    assert v4a.v4a_get_error(err) == 0
    out = out.float().cpu().numpy()
    codes, scale = codes.cpu().numpy(), scale.cpu().numpy().astype(np.float64)
    assert np.isfinite(scale).all() and (scale > 0).all()
    # the rule, against the same call's output (bf16 rounds the fp32 values by <= 2^-9)
    amax = np.abs(out).max(axis=-1)
    assert np.allclose(scale, np.where(amax > 0, amax / 448.0, 1.0), rtol=2.0 ** -8)
    deq = O.e4m3_decode(codes) * scale[..., None]
    half = 0.5 * _e4m3_step(out / scale[..., None]) * scale[..., None]
    assert (np.abs(deq - out) <= half * 1.05 + np.abs(out) * 2.0 ** -8 + 1e-12).all()
    # against the oracle: its quantised rows, within the attention tolerance plus one step
    ref = O.attention(h.spec, oracle_pools(h), q.seq, q.pos, q.q, lists)
    codes_o, scale_o = O.quantize(ref)
    assert np.allclose(scale, scale_o, rtol=3e-2, atol=1e-6)
    deq_o = O.e4m3_decode(codes_o) * scale_o[..., None]
    step_o = _e4m3_step(ref / scale_o[..., None]) * scale_o[..., None]
    assert (np.abs(deq - deq_o) <= step_o * 1.05 + 3e-2).all()
    # fp8 rounding itself (half a step, ~3% of a value) is in both: compare the quantised
    # outputs with the bf16 output's mean tolerance
    assert np.abs(deq - deq_o).mean() <= 3e-3


def test_attention_q8_c128a_dense():
    """The fp8 output epilogue on a dense c128a layer (every visible entry + window): the
    quantised rows match the oracle's within one e4m3 step plus the attention tolerance."""
    w = wl.c128a_decode(seed=24, B=2, L=32768)
    h = w.layers[0]
    _fill_query_window_row(h, w)
    q = w.queries
    lay, x, err = device_layer(h), DevInputs(w), _err()
    codes, scale = lay.attention_q8(x.q_seq, x.q_pos, x.max_pos, x.q, None, dev_err=err)
    assert v4a.v4a_get_error(err) == 0
    codes, scale = codes.cpu().numpy(), scale.cpu().numpy().astype(np.float64)
    ref = O.attention(h.spec, oracle_pools(h), q.seq, q.pos, q.q, None)
    codes_o, scale_o = O.quantize(ref)
    assert np.allclose(scale, scale_o, rtol=3e-2, atol=1e-6)
    deq = O.e4m3_decode(codes) * scale[..., None]
    deq_o = O.e4m3_decode(codes_o) * scale_o[..., None]
    step_o = _e4m3_step(ref / scale_o[..., None]) * scale_o[..., None]
    assert (np.abs(deq - deq_o) <= step_o * 1.05 + 3e-2).all()
    assert np.abs(deq - deq_o).mean() <= 3e-3


def test_attention_fp8_c128a_dense():
    w = wl.c128a_decode(seed=2, B=4, L=65536)
    h = w.layers[0]
    _fill_query_window_row(h, w)
    q = w.queries
    lay, x = device_layer(h), DevInputs(w)
    out = lay.attention(x.q_seq, x.q_pos, x.max_pos, x.q, None)
    ref = O.attention(h.spec, oracle_pools(h), q.seq, q.pos, q.q, None)
    check_out(out.float().cpu().numpy(), ref, fp8=True)


def test_attention_split_with_empty_ranges():
    """Dense c128a decode of sequences of 32768, 256, 100 and 20000 tokens: 3 key tiles at
    the longest, so 3 ranges per query. The 256-token query has one entry and 128 window
    rows (its third range is empty), the 100-token query only its 101 window rows (two
    empty ranges): an empty range writes no partial and must not enter the merge."""
    spec = wl.LayerSpec("c128a", True)
    rng = np.random.default_rng(31)
    ctx = [32768, 256, 100, 20000]
    h = wl.make_layer(rng, spec, ctx, [1] * 4, prefill_cache=True)
    h.bias, h.gamma, _ = wl.layer_params(rng, spec)
    b = wl.make_batch(rng, spec, ctx, [1] * 4)
    w = wl.Workload("c128a mixed", [h], b, wl.make_queries(rng, spec, np.arange(4),
                                                           np.array(ctx), False))
    _fill_query_window_row(h, w)
    q = w.queries
    lay, x, err = device_layer(h), DevInputs(w), _err()
    assert v4a.v4a_attn_plan(lay.cfg, 4, x.max_pos, 0) == (3, 2)
    out = lay.attention(x.q_seq, x.q_pos, x.max_pos, x.q, None, dev_err=err)
    assert v4a.v4a_get_error(err) == 0
    ref = O.attention(h.spec, oracle_pools(h), q.seq, q.pos, q.q, None)
    check_out(out.float().cpu().numpy(), ref, fp8=True)


def test_attention_k_covers_all_equals_dense():
    """A top-k list holding every visible entry gives the dense result."""
    w = wl.c4a_decode(seed=12, B=4, L=1024)
    h = w.layers[0]
    _fill_query_window_row(h, w)
    lay, x = device_layer(h), DevInputs(w)
    n = O.visible_entries(4, 8, 0, 1024)
    lists = np.tile(np.concatenate([np.arange(n), -np.ones(512 - n)]).astype(np.int32), (4, 1))
    a = lay.attention(x.q_seq, x.q_pos, x.max_pos, x.q, T(lists, torch.int32))
    d = lay.attention(x.q_seq, x.q_pos, x.max_pos, x.q, None)
    diff = (a.float() - d.float()).abs().max().item()
    assert diff <= 1e-2, diff


def test_attention_no_visible_entries_window_only():
    """Queries before position 8 see no c4a entry: the layer is window attention."""
    w = wl.tiny_prefill(seed=4, L=8)
    h = w.layers[0]
    lay, x = device_layer(h), DevInputs(w)
    out, topk = lay.step(x.cu, x.start, x.kv, x.s, x.ik, x.is_, x.q_seq, x.q_pos, x.max_pos, x.q,
                         x.q_idx, x.w, prefill=True)
    assert (topk.cpu().numpy() == -1).all()
    pools = oracle_pools(h)
    oracle_insert(w, h, pools)
    q = w.queries
    ref = O.attention(h.spec, pools, q.seq, q.pos, q.q, np.full((8, 64), -1))
    check_out(out.cpu().numpy(), ref, fp8=False)


# ---------------------------------------------------------------------- device errors
def test_missing_page_and_bad_index_raise_device_error():
    w = wl.c4a_decode(seed=13, B=2, L=2048)
    h = w.layers[0]
    _fill_query_window_row(h, w)
    h.attn.bt[1, 3] = -1                                   # hole in sequence 1's entries
    lay, x, err = device_layer(h), DevInputs(w), _err()
    lists = np.tile(np.arange(512, dtype=np.int32), (2, 1))
    lay.attention(x.q_seq, x.q_pos, x.max_pos, x.q, T(lists, torch.int32), dev_err=err)
    assert v4a.v4a_get_error(err) & v4a.DEV_MISSING_PAGE
    assert v4a.v4a_get_error(err) == 0                     # read clears the word
    lists[0, -1] = 600                                     # not visible at p = 2048
    lists[1] = np.arange(512)
    lay.attention(x.q_seq, x.q_pos, x.max_pos, x.q, T(lists, torch.int32), dev_err=err)
    assert v4a.v4a_get_error(err) & v4a.DEV_BAD_INDEX


def test_empty_calls_are_noops():
    w = wl.c4a_decode(seed=14, B=2, L=1024)
    lay = device_layer(w.layers[0])
    z32 = torch.zeros(1, dtype=torch.int32, device="cuda")
    z64 = torch.zeros(0, dtype=torch.int64, device="cuda")
    lay.compress_insert(torch.zeros(2, dtype=torch.int32, device="cuda"),
                        torch.zeros(1, dtype=torch.int64, device="cuda"),
                        torch.empty((0, 512), dtype=torch.bfloat16, device="cuda"),
                        torch.empty((0, 512), dtype=torch.bfloat16, device="cuda"),
                        torch.empty((0, 128), dtype=torch.bfloat16, device="cuda"),
                        torch.empty((0, 128), dtype=torch.bfloat16, device="cuda"))
    out = lay.attention(z32[:0], z64, 0, torch.empty((0, 64, 512), dtype=torch.bfloat16,
                                                     device="cuda"), None)
    assert out.shape[0] == 0


# ------------------------------------------------------------- full-size workloads
def _full_step(w, li=0, prefill=False, side=False):
    h = w.layers[li]
    lay, x, err = device_layer(h), DevInputs(w), _err()
    out, topk = lay.step(x.cu, x.start, x.kv, x.s, x.ik, x.is_, x.q_seq, x.q_pos, x.max_pos,
                         x.q, x.q_idx, x.w, prefill=prefill, dev_err=err,
                         side_stream=torch.cuda.Stream() if side else None)
    torch.cuda.synchronize()
    assert v4a.v4a_get_error(err) == 0
    return h, out.float().cpu().numpy(), None if topk is None else topk.cpu().numpy()


def _check_rows(w, h, lay, out, topk, rows):
    """Oracle parity of a layer step for the query rows `rows`, over the pools as the GPU
    left them (the same dequantised values on both sides): top-k lists within the tie band
    (c4a), and attention on the GPU's own lists for every row (no row is skipped)."""
    dp = device_pools(lay, h.spec)
    q = w.queries
    rows = np.asarray(rows)
    lists = None
    if h.spec.has_indexer:
        ref_top, scores = O.index_topk(h.spec, dp, q.seq[rows], q.pos[rows], q.q_idx[rows],
                                       q.w[rows], h.spec.top_k)
        check_topk(topk[rows], ref_top, scores, h.spec.top_k)
        lists = topk[rows]
    ref = O.attention(h.spec, dp, q.seq[rows], q.pos[rows], q.q[rows], lists)
    return check_out(out[rows], ref, fp8=h.spec.fp8)


def _check_insert(w, h, lay):
    """Every row the step's insert wrote, against the oracle's own insert."""
    pools = oracle_pools(h)
    writes = oracle_insert(w, h, pools)
    _compare_written(lay, pools, writes, fp8=h.spec.fp8)


def _full_step(w, li=0, prefill=False, side=False):
    h = w.layers[li]
    lay, x, err = device_layer(h), DevInputs(w), _err()
    out, topk = lay.step(x.cu, x.start, x.kv, x.s, x.ik, x.is_, x.q_seq, x.q_pos, x.max_pos,
                         x.q, x.q_idx, x.w, prefill=prefill, dev_err=err,
                         side_stream=torch.cuda.Stream() if side else None)
    torch.cuda.synchronize()
    assert v4a.v4a_get_error(err) == 0
    return h, lay, out.float().cpu().numpy(), None if topk is None else topk.cpu().numpy()


def test_c4a_decode_full_size_every_query():
    """B=32 sequences of 32768 tokens, one new token and query each: the full layer step as
    the benchmark runs it (the insert on a side stream beside the indexer; on a 152-SM GB300
    the attention call splits each query's keys into 3 ranges). All 32 queries."""
    w = wl.c4a_decode()
    cfg = device_layer(w.layers[0]).cfg
    assert v4a.v4a_attn_plan(cfg, 32, 32768, 512) == (3, 2)
    h, lay, out, topk = _full_step(w, side=True)
    _check_insert(w, h, lay)
    _check_rows(w, h, lay, out, topk, np.arange(32))


def test_side_stream_step_equals_serial_step():
    """The decode step with the insert on a side stream, run eagerly and replayed from a
    CUDA graph, writes the same bytes (pools, top-k lists, outputs) as the serial step."""
    w = wl.c4a_decode(seed=41, B=8, L=8192)
    h = w.layers[0]
    x, err = DevInputs(w), _err()
    ser, side_e, side_g = device_layer(h), device_layer(h), device_layer(h)
    args = (x.cu, x.start, x.kv, x.s, x.ik, x.is_, x.q_seq, x.q_pos, x.max_pos, x.q, x.q_idx,
            x.w)
    o_ser, t_ser = ser.step(*args, dev_err=err)
    side = torch.cuda.Stream()
    o_e, t_e = side_e.step(*args, dev_err=err, side_stream=side)
    torch.cuda.synchronize()
    # graph: warm the workspaces on a scratch copy, capture on the third layer, replay once
    side_g.clone_pools().step(*args, dev_err=err, side_stream=side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        o_g, t_g = side_g.step(*args, dev_err=err, side_stream=side)
    g.replay()
    torch.cuda.synchronize()
    assert v4a.v4a_get_error(err) == 0
    for o, t, lay in ((o_e, t_e, side_e), (o_g, t_g, side_g)):
        assert torch.equal(t, t_ser)
        assert torch.equal(o, o_ser)
        _pools_equal(lay, ser)


def test_c128a_decode_full_size_every_query():
    """B=8 sequences of 2^20 tokens, dense over 8192 entries + window; all 8 queries."""
    w = wl.c128a_decode()
    h, lay, out, _ = _full_step(w)
    _check_insert(w, h, lay)
    _check_rows(w, h, lay, out, None, np.arange(8))


def prefill_rows(cached, chunk, n=256, seed=0):
    """Stratified chunk queries of the prefill workload (offsets into the chunk): the first
    and last four; pairs just before and after an entry becomes visible (p = 4j+7, the
    entry's last token, and p = 4j+8); positions at the edges of a 256-token window block
    and where the window's first token crosses one (p-127 at a block edge); positions where
    the visible count crosses a 128-entry indexer tile; the rest drawn uniformly."""
    rng = np.random.default_rng(seed)
    p0 = cached
    offs = set(range(4)) | set(range(chunk - 4, chunk))
    ps = np.arange(p0, p0 + chunk)
    before = ps[(ps % 4) == 3]                                # p = 4j + 7: entry j not yet seen
    pick = rng.choice(before, 24, replace=False)
    offs |= set((pick - p0).tolist()) | set((pick + 1 - p0).tolist())
    edges = ps[np.isin(ps % 256, (0, 255)) | np.isin((ps - 127) % 256, (0, 255))]
    offs |= set((rng.choice(edges, 48, replace=False) - p0).tolist())
    vis = (ps - 8) // 4 + 1
    tiles = ps[np.isin(vis % 128, (0, 1))]
    offs |= set((rng.choice(tiles, 48, replace=False) - p0).tolist())
    offs = {o for o in offs if 0 <= o < chunk}
    rest = np.setdiff1d(np.arange(chunk), sorted(offs))
    offs |= set(rng.choice(rest, n - len(offs), replace=False).tolist())
    return np.array(sorted(offs))


def test_c4a_prefill_full_size_stratified():
    """122880 cached tokens plus a chunk of 8192: every row the insert wrote, and 256
    stratified chunk queries (top-k and attention)."""
    w = wl.c4a_prefill()
    h, lay, out, topk = _full_step(w, prefill=True)
    _check_insert(w, h, lay)
    rows = prefill_rows(122880, 8192)
    assert len(rows) == 256
    _check_rows(w, h, lay, out, topk, rows)


def test_mixed_decode_full_size_every_query():
    """64 sequences, log-uniform lengths in [4096, 2^20), a c4a and a c128a layer; all 64
    queries of each layer."""
    w = wl.mixed_decode()
    for li in (0, 1):
        h, lay, out, topk = _full_step(w, li)
        _check_insert(w, h, lay)
        _check_rows(w, h, lay, out, topk, np.arange(64))


# ---------------------------------------------------------------- indexer scores alone
def _score_bound(spec, dp, seq, pos, q_idx, w):
    """A-priori bound on the rounding of one score row: scale_j * sum_h |w_h| max|q_h| *
    sum_d |code_jd| (it covers the fp32 accumulation and the e4m3 split of the query)."""
    n = O.visible_entries(spec.S, spec.W, spec.win_off, int(pos))
    keys = dp.idx.read_many(int(seq), np.arange(n), spec.fp8)
    qa = np.abs(np.asarray(q_idx, np.float64)).max(axis=1)
    return np.abs(keys).sum(axis=1) * float((np.abs(np.asarray(w, np.float64)) * qa).sum())


@pytest.mark.parametrize("case", ["fp8_decode", "fp4_decode", "fp8_prefill", "fp8_prefill_pairs",
                                  "fp8_prefill_quads", "fp4_prefill_pairs", "fp32_tiny"])
def test_index_scores_elementwise(case):
    """v4a_index_scores against the oracle's scores, element by element, for every visible
    entry of every query: |gpu - oracle| <= 3e-5 x the row's a-priori rounding bound (fp32
    accumulation of exact products, 2^-17 relative loss of the split query below the e4m3
    subnormal step). The pair cases run the kernel that takes two queries per key tile and
    accumulates the query's two e4m3 terms in one product; the quads case (>= 4096 queries over
    four sequences with ragged chunks, so groups of four straddle sequence boundaries) runs the
    kernel that takes four queries per key tile and accumulates each query's two terms in the
    same accumulator columns."""
    if case == "fp8_decode":
        w = wl.c4a_decode(seed=51, B=8, L=8192)
        _inject_subnormal_keys(w.layers[0], np.random.default_rng(52))
    elif case == "fp4_decode":
        w = wl.c4a_decode(seed=53, B=8, L=8192, idx_fp4=True)
    elif case == "fp8_prefill":
        w = wl.c4a_prefill(seed=54, cached=8192, chunk=300)
    elif case == "fp8_prefill_pairs":        # >= 1024 queries: two queries per key tile
        w = wl.c4a_prefill(seed=56, cached=8192, chunk=1024)
    elif case == "fp8_prefill_quads":        # >= 4096 queries: four queries per key tile
        spec = wl.LayerSpec("c4a", True)
        rng = np.random.default_rng(58)
        ctx, new = [1000, 37, 127, 2048], [1501, 1, 1298, 1303]
        h = wl.make_layer(rng, spec, ctx, new, prefill_cache=True)
        h.bias, h.gamma, h.ibias = wl.layer_params(rng, spec)
        seq = np.repeat(np.arange(4), new)
        pos = np.concatenate([c + np.arange(n) for c, n in zip(ctx, new)])
        w = wl.Workload("ragged quads", [h], wl.make_batch(rng, spec, ctx, new),
                        wl.make_queries(rng, spec, seq, pos, False))
        assert len(seq) >= 4096 and len(seq) % 4 != 0
    elif case == "fp4_prefill_pairs":
        w = wl.c4a_prefill(seed=57, cached=8192, chunk=1024, idx_fp4=True)
    else:
        w = wl.tiny_prefill(seed=55, L=700)
    h = w.layers[0]
    lay, x, err = device_layer(h), DevInputs(w), _err()
    lay.compress_insert(x.cu, x.start, x.kv, x.s, x.ik, x.is_, dev_err=err)
    got = lay.index_scores(x.q_seq, x.q_pos, x.max_pos, x.q_idx, x.w, dev_err=err)
    assert v4a.v4a_get_error(err) == 0
    got = got.cpu().numpy()               # columns past a row's visible count are not written
    dp = device_pools(lay, h.spec)
    q = w.queries
    _, scores = O.index_topk(h.spec, dp, q.seq, q.pos, q.q_idx, q.w, h.spec.top_k)
    worst = 0.0
    for i in range(len(q.pos)):
        n = len(scores[i])
        bound = _score_bound(h.spec, dp, q.seq[i], q.pos[i], q.q_idx[i], q.w[i])
        d = np.abs(got[i, :n].astype(np.float64) - scores[i])
        assert (d <= 3e-5 * bound + 1e-30).all(), (i, d.max(), bound[np.argmax(d)])
        if n:
            worst = max(worst, float((d / np.maximum(bound, 1e-300)).max()))
    assert worst < 3e-5
