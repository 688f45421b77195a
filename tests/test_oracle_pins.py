"""Pins of the fp64 oracle against things other than itself: figures the pages print,
closed forms, brute force on tiny inputs, library routines in special cases, and
invariants the pages state. CPU only."""
import json
import math
import os
from dataclasses import replace

import numpy as np
import pytest
import torch

import workloads as wl
from oracle import v4a_oracle as O

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")))


# ------------------------------------------------------------------------------ RoPE
def test_rope_closed_form_pairs():
    # D=4, d_r=4, base=100: theta_0 = 1, theta_1 = 100^(-1/2) = 0.1, adjacent pairs.
    x = np.array([1.0, 0.0, 0.0, 2.0])
    y = O.rope(x, 3, 4, 100.0)
    want = [math.cos(3.0), math.sin(3.0), -2.0 * math.sin(0.3), 2.0 * math.cos(0.3)]
    assert np.allclose(y, want, atol=1e-15)
    # only the tail rotates
    x = np.arange(8.0)
    y = O.rope(x, 5, 2, 10000.0)
    assert np.array_equal(y[:6], x[:6])
    assert np.allclose(y[6:], [6 * math.cos(5) - 7 * math.sin(5), 6 * math.sin(5) + 7 * math.cos(5)])


def test_rope_inverse_isometry_relative():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 64))
    p = np.array([0, 7, 1000, 123456, 1 << 20])
    y = O.rope(x, p, 32, 10000.0)
    assert np.allclose(O.rope(y, p, 32, 10000.0, inverse=True), x, atol=1e-12)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), atol=1e-12)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    d0 = O.rope(q, 900, 32, 1e4) @ O.rope(k, 37, 32, 1e4)
    d1 = O.rope(q, 900 + 4096, 32, 1e4) @ O.rope(k, 37 + 4096, 32, 1e4)
    assert abs(d0 - d1) < 1e-10


# ------------------------------------------------------------------------------ fp8
def test_e4m3_decode_matches_torch_all_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(O.e4m3_decode(codes), want)


def test_e4m3_encode_matches_torch_on_all_bf16_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    ok = np.isfinite(v) & (np.abs(v) <= 448.0)
    v = v[ok]
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_encode(v)
    zero = v == 0
    assert np.array_equal(got[~zero], want[~zero])
    assert np.all(O.e4m3_decode(got[zero]) == 0)
    # saturation (satfinite): beyond the largest finite value the code is +-448
    assert list(O.e4m3_encode([449.0, 1e6, -1e6])) == [0x7E, 0x7E, 0xFE]


def test_e2m1_table_matches_the_published_format():
    fmt = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "e2m1_format.json")))
    vals = O.e2m1_values()
    assert np.array_equal(vals, fmt["magnitudes"])
    assert vals.max() == fmt["max_normal"] and vals[2] == fmt["min_normal"]
    assert vals[1] == fmt["max_subnormal"]
    # every e2m1 value is an e4m3 value (so an exact e4m3 operand can carry it)
    assert set(vals.tolist()) <= set(O.e4m3_values().tolist())
    assert np.array_equal(O.e2m1_decode(np.arange(16)), np.concatenate([vals, -vals]))


def test_e2m1_encode_is_nearest_even_by_brute_force():
    """Against a brute-force search over the 16 codes: nearest value, ties to the code with
    a zero mantissa bit, saturation at +-6, the sign kept for zero."""
    vals = O.e2m1_decode(np.arange(16))
    grid = np.unique(np.abs(vals))
    mids = 0.5 * (grid[1:] + grid[:-1])
    v = np.concatenate([grid, mids, mids + 1e-9, mids - 1e-9, np.linspace(-9, 9, 4001),
                        np.random.default_rng(7).standard_normal(2000) * 3, [-0.0, 0.0, 1e-30]])
    got = O.e2m1_encode(v)
    for x, c in zip(v, got):
        a = min(abs(x), 6.0)
        d = np.abs(np.abs(vals[:8]) - a)
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else best[best % 2 == 0][0]
        want |= 8 if np.signbit(x) else 0
        assert c == want, (x, c, want)


def test_e2m1_packing_and_row_quantisation():
    codes = np.array([[1, 2, 3, 15, 8, 0]], dtype=np.uint8)
    packed = O.pack_e2m1(codes)
    assert packed.tolist() == [[0x21, 0xF3, 0x08]]          # element 2i in the low nibble
    assert np.array_equal(O.unpack_e2m1(packed), codes)
    rng = np.random.default_rng(11)
    y = rng.standard_normal((64, 128)) * rng.uniform(0.1, 10, (64, 1))
    p, sc = O.quantize_fp4(y)
    assert p.shape == (64, 64) and p.dtype == np.uint8
    assert np.allclose(sc, np.abs(y).max(axis=1) / 6.0)
    deq = O.e2m1_decode(O.unpack_e2m1(p)) * sc[:, None]
    # the largest element of each row is stored exactly; every other within half a step
    i = np.abs(y).argmax(axis=1)
    assert np.allclose(deq[np.arange(64), i], y[np.arange(64), i])
    step = np.diff(np.concatenate([O.e2m1_values(), [8.0]]))
    a = np.abs(y) / sc[:, None]
    k = np.minimum(np.searchsorted(O.e2m1_values(), a, side="right") - 1, 7)
    assert np.all(np.abs(deq - y) <= 0.5 * step[k] * sc[:, None] + 1e-12)
    z, zs = O.quantize_fp4(np.zeros((1, 128)))
    assert zs[0] == 1.0 and not z.any()


def test_fp4_indexer_rows_written_by_the_compressor():
    """With the fp4 indexer cache, the insert stores each indexer entry as packed e2m1
    codes + row scale whose dequantised values are within half an e2m1 step (times the
    row scale) of the exact compressed vector; the attention entries stay fp8."""
    w = wl.c4a_prefill(seed=5, cached=64, chunk=96, idx_fp4=True)
    pools = _fresh_pools(w)
    assert pools.idx.fp4 and pools.idx.data.shape[1] == 64
    writes = _run_compress(w, pools)
    idx_slots = [sl for (k, _, _, sl) in writes if k == "idx" and sl >= 0]
    assert len(idx_slots) >= 20
    step = np.diff(np.concatenate([O.e2m1_values(), [8.0]]))
    for sl in idx_slots:
        y = pools.idx.raw[sl]
        sc = pools.idx.scale[sl]
        assert np.isclose(sc, np.abs(y).max() / 6.0)
        deq = O.e2m1_decode(O.unpack_e2m1(pools.idx.data[sl])) * sc
        k = np.minimum(np.searchsorted(O.e2m1_values(), np.abs(y) / sc, side="right") - 1, 7)
        assert np.all(np.abs(deq - y) <= 0.5 * step[k] * sc + 1e-12)
    a_sl = [sl for (k, _, _, sl) in writes if k == "attn" and sl >= 0]
    assert pools.attn.data.shape[1] == 512 and len(a_sl) == len(idx_slots)


def test_quantize_rows():
    y = np.array([[0.5, -3.0, 1.0], [0.0, 0.0, 0.0]])
    codes, scale = O.quantize(y)
    assert scale[0] == 3.0 / 448.0 and scale[1] == 1.0
    assert codes[0, 1] == 0xFE and np.all(codes[1] == 0)
    assert np.allclose(O.e4m3_decode(codes[0]) * scale[0], y[0], rtol=2 ** -4)


# ------------------------------------------------------------------------ paged layout
def test_block_geometry_matches_pages():
    assert GOLD["block_native_positions"]["value"] == O.BLOCK
    for kind, key in (("c4a", "c4a_entries_per_block"), ("c128a", "c128a_entries_per_block")):
        assert wl.LayerSpec(kind, True).rows_per_block == GOLD[key]["value"]
    assert [wl.LayerSpec("c4a", True).W, wl.LayerSpec("c4a", True).S] == GOLD["c4a_window_stride"]["value"]
    assert [wl.LayerSpec("c128a", True).W, wl.LayerSpec("c128a", True).S] == \
        GOLD["c128a_window_stride"]["value"]


@pytest.mark.parametrize("R", [256, 64, 2])
def test_slot_mapping_is_a_bijection_onto_pages(R):
    rng = np.random.default_rng(1)
    bt, n_pages = wl.block_table(rng, [set(range(5)), {0, 2, 3}, set()], 6)
    seen = {}
    for seq in range(3):
        for r in range(6 * R):
            s = O.slot(bt, R, seq, r)
            blk = r * (256 // R) // 256            # block of native position r*256/R
            if bt[seq, blk] < 0:
                assert s == -1
                continue
            assert s not in seen
            seen[s] = (seq, r)
            # rows of one page are consecutive logical rows of one block, in order
            assert s // R == bt[seq, blk] and s % R == r - blk * R
    assert sorted(seen) == list(range(n_pages * R))
    assert O.slot(bt, R, 0, 6 * R) == -1


# -------------------------------------------------------------------------- compressor
def test_compress_window_closed_forms():
    rng = np.random.default_rng(2)
    kv = rng.standard_normal((8, 16))
    # constant gates, no bias -> plain mean over the window
    assert np.allclose(O.compress_window(kv, np.full((8, 16), 0.3), np.zeros((8, 16))),
                       kv.mean(axis=0), atol=1e-14)
    # per-channel one-hot gate: channel d takes token o_d (softmax is per channel)
    o = rng.integers(0, 8, 16)
    s = np.zeros((8, 16))
    s[o, np.arange(16)] = 60.0
    assert np.allclose(O.compress_window(kv, s, np.zeros((8, 16))), kv[o, np.arange(16)],
                       atol=1e-20 + 1e-20)
    # the bias enters the gate: a one-hot bias selects like a one-hot score
    b = np.zeros((8, 16))
    b[o, np.arange(16)] = 60.0
    assert np.allclose(O.compress_window(kv, np.zeros((8, 16)), b), kv[o, np.arange(16)])
    # weights sum to one
    assert np.allclose(O.compress_window(np.ones((8, 16)), rng.standard_normal((8, 16)),
                                         rng.standard_normal((8, 16))), 1.0)


def test_rmsnorm_closed_form():
    c = np.array([3.0, 4.0])
    g = np.array([2.0, -1.0])
    y = O.rmsnorm(c, g, 0.0)
    r = math.sqrt((9 + 16) / 2)
    assert np.allclose(y, [6 / r, -4 / r])
    rng = np.random.default_rng(3)
    c = rng.standard_normal(512) * 7
    y = O.rmsnorm(c, np.ones(512), 1e-6)
    assert abs(math.sqrt(np.mean(y * y)) - 1.0) < 1e-6


def test_q_norm_by_hand_per_head():
    """Two heads of D=2 worked out by hand: each head is divided by its own RMS and
    multiplied by the per-dim gamma (R13)."""
    q = np.array([[[3.0, 4.0], [1.0, 0.0]]])
    g = np.array([2.0, -1.0])
    y = O.q_norm(q, g, 0.0)
    r0, r1 = math.sqrt(12.5), math.sqrt(0.5)
    assert np.allclose(y, [[[6 / r0, -4 / r0], [2 / r1, 0.0]]])


def test_q_norm_heads_are_independent_and_unit_rms():
    """Heads at scales 1e-2 .. 1e3 each come out with RMS 1 (gamma = 1), and scaling one
    head leaves every row unchanged (eps = 0): a norm taken over all heads jointly, or over
    the wrong axis, fails here."""
    rng = np.random.default_rng(5)
    q = rng.standard_normal((3, 6, 64)) * (10.0 ** np.arange(-2, 4))[None, :, None]
    y = O.q_norm(q, np.ones(64), 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, atol=1e-12)
    q2 = q.copy()
    q2[1, 4] *= 37.0
    assert np.allclose(O.q_norm(q2, np.ones(64), 0.0), y, atol=1e-12)
    # eps enters inside the root: a zero row stays zero, a row of RMS sqrt(eps) shrinks by 1/sqrt(2)
    z = np.zeros((1, 2, 4))
    z[0, 1] = math.sqrt(1e-6)
    yz = O.q_norm(z, np.ones(4), 1e-6)
    assert np.all(yz[0, 0] == 0.0) and np.allclose(yz[0, 1], 1 / math.sqrt(2))


def _fresh_pools(w):
    L = w.layers[0]
    return O.Pools(L.spec, L.attn, L.idx, L.swa, L.state)


def _run_compress(w, pools, cu=None, start=None, rows=None):
    L, B = w.layers[0], w.batch
    sl = slice(None) if rows is None else rows
    return O.compress_insert(L.spec, L.bias, L.gamma, L.ibias, pools,
                             B.cu if cu is None else cu, B.start if start is None else start,
                             B.kv[sl], B.s[sl], None if B.ik is None else B.ik[sl],
                             None if B.is_ is None else B.is_[sl])


@pytest.mark.parametrize("kind", ["c4a", "c128a"])
def test_compressor_picks_the_window_tokens(kind):
    """Gate +80 on the tokens with t % S == o and -80 elsewhere, bias 0: entry j is then
    the mean of the covered tokens with that residue (two for c4a, whose 8-token windows
    hold two such tokens; one for c128a), RMS-normalised and rotated at position S*j.
    kv carries the token index in channel 0, so a wrong window shows up directly."""
    w = wl.tiny_prefill(seed=5, L=512, kind=kind)
    L, spec = w.layers[0], w.layers[0].spec
    o = 3
    L.bias = np.zeros_like(L.bias)
    pos = np.arange(512)
    kv = np.zeros_like(w.batch.kv)
    kv[:, 0] = pos
    kv[:, 1] = 1.0
    kv[:, spec.D - spec.d_r] = 1.0
    s = np.where((pos % spec.S == o)[:, None], 80.0, -80.0) * np.ones_like(w.batch.s)
    w.batch.kv, w.batch.s = kv, s
    pools = _fresh_pools(w)
    _run_compress(w, pools)
    n_e = O.visible_entries(spec.S, spec.W, spec.win_off, 512)
    assert n_e == (512 - spec.W) // spec.S + 1
    for j in range(n_e):
        toks = [t for t in range(spec.S * j, spec.S * j + spec.W) if t % spec.S == o]
        c = np.zeros(spec.D)
        c[0], c[1], c[spec.D - spec.d_r] = np.mean(toks), 1.0, 1.0
        want = O.rope(O.rmsnorm(c, L.gamma.astype(np.float64), spec.eps), spec.S * j,
                      spec.d_r, spec.rope_base)
        assert np.allclose(pools.attn.read(0, j, False), want, atol=1e-9), j


def test_compressor_uniform_gate_is_plain_mean_c128a():
    """c128a with constant gates and zero bias: the entry is the 128-token mean."""
    w = wl.tiny_prefill(seed=6, L=300, kind="c128a")
    L, spec = w.layers[0], w.layers[0].spec
    L.bias = np.zeros_like(L.bias)
    w.batch.s = np.full_like(w.batch.s, 0.7)
    pools = _fresh_pools(w)
    _run_compress(w, pools)
    for j in range(2):
        c = w.batch.kv[128 * j:128 * j + 128].astype(np.float64).mean(axis=0)
        want = O.rope(O.rmsnorm(c, L.gamma.astype(np.float64), spec.eps), 128 * j, spec.d_r,
                      spec.rope_base)
        assert np.allclose(pools.attn.read(0, j, False), want, atol=1e-12)


@pytest.mark.parametrize("fp8,kind", [(False, "c4a"), (True, "c4a"), (False, "c128a")])
def test_chunking_invariance(fp8, kind):
    """Inserting a sequence in one call or in ragged chunks (the residual pool carrying
    the partial windows between calls) writes identical caches."""
    over = dict(kind=kind, fp8=fp8)
    w = wl.tiny_prefill(seed=7, L=700, **over)
    one = _fresh_pools(w)
    _run_compress(w, one)
    many = _fresh_pools(w)
    cuts = [0, 1, 5, 130, 131, 400, 699, 700]
    for a, b in zip(cuts[:-1], cuts[1:]):
        _run_compress(w, many, cu=np.array([0, b - a]), start=np.array([a]), rows=slice(a, b))
    for name in ("attn", "idx", "swa"):
        x, y = getattr(one, name), getattr(many, name)
        if x is None:
            continue
        assert np.array_equal(x.data, y.data), name
        if x.scale is not None:
            assert np.array_equal(x.scale, y.scale), name


# ------------------------------------------------------------------------ visibility
@pytest.mark.parametrize("S,W,off", [(4, 8, 0), (128, 128, 0), (4, 8, -4)])
def test_visibility_brute_force(S, W, off):
    for p in range(0, 700):
        want = sum(1 for j in range(p + 10)
                   if all(t < p for t in range(S * j + off, S * j + off + W)))
        assert O.visible_entries(S, W, off, p) == want


def test_decode_insert_is_invisible_to_its_own_queries():
    """R15 (the side stream's condition), by brute force with the oracle: in a decode step
    the only new token sits at the query's own position, so the entry it completes covers
    that position and no query of the step can see it; the indexer's scores and top-k are
    the same computed before or after the insert. In a prefill chunk later queries do see
    entries completed by earlier tokens of the same call, so there they differ."""
    for L in (1027, 1031):                        # the token completes an entry at 1031 (4j+7)
        w = wl.c4a_decode(seed=61, B=3, L=L, top_k=64)
        h, q = w.layers[0], w.queries
        before = _fresh_pools(w)
        t0, s0 = O.index_topk(h.spec, before, q.seq, q.pos, q.q_idx, q.w, 64)
        after = _fresh_pools(w)
        writes = _run_compress(w, after)
        if L == 1031:
            assert any(k == "idx" for (k, _, _, _) in writes)   # an entry was completed
        t1, s1 = O.index_topk(h.spec, after, q.seq, q.pos, q.q_idx, q.w, 64)
        assert np.array_equal(t0, t1)
        assert all(np.array_equal(a, b) for a, b in zip(s0, s1))
    w = wl.c4a_prefill(seed=62, cached=256, chunk=64, top_k=64)
    h, q = w.layers[0], w.queries
    before = _fresh_pools(w)
    _, s0 = O.index_topk(h.spec, before, q.seq[-4:], q.pos[-4:], q.q_idx[-4:], q.w[-4:], 64)
    after = _fresh_pools(w)
    _run_compress(w, after)
    _, s1 = O.index_topk(h.spec, after, q.seq[-4:], q.pos[-4:], q.q_idx[-4:], q.w[-4:], 64)
    assert any(not np.array_equal(a, b) for a, b in zip(s0, s1))


def test_entry_counts_at_one_million():
    n4 = O.visible_entries(4, 8, 0, 1 << 20)
    n128 = O.visible_entries(128, 128, 0, 1 << 20)
    assert n4 == 262143 and n128 == 8191 + 1 - 0 or n128 == 8192
    # the pages round these to ~250k and ~8k
    assert abs(n4 - GOLD["c4a_entries_at_1m"]["value"]) / n4 < 0.05
    assert abs(n128 - GOLD["c128a_entries_at_1m"]["value"]) / n128 < 0.05
    # no c128a entry is usable before position 128 (C128A 的因果性约束)
    assert O.visible_entries(128, 128, 0, 128) == 1 and O.visible_entries(128, 128, 0, 127) == 0


# -------------------------------------------------------------------- indexer + top-k
def test_index_scores_by_hand():
    q = np.array([[1.0, 0.0], [0.0, 1.0]])
    w = np.array([2.0, 3.0])
    keys = np.array([[1.0, -1.0], [-2.0, 5.0], [-1.0, -1.0]])
    assert np.allclose(O.index_scores(q, w, keys), [2.0, 15.0, 0.0])


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(8)
    for trial in range(200):
        n = int(rng.integers(0, 40))
        k = int(rng.integers(1, 12))
        sc = rng.integers(-3, 4, n).astype(np.float64)        # many ties
        want = sorted(sorted(range(n), key=lambda j: (-sc[j], j))[:k])
        got = O.select_topk(sc, k)
        assert list(got[:len(want)]) == want and np.all(got[len(want):] == -1)


# ------------------------------------------------------------------------ attention
def _attend_loops(q, p, keys, scale, d_r, base):
    """Attention written with explicit loops and math.exp (no numpy matmul)."""
    qr = O.rope(q, p, d_r, base)
    H, D = q.shape
    out = np.zeros((H, D))
    for h in range(H):
        lg = [scale * sum(qr[h, d] * keys[x, d] for d in range(D)) for x in range(len(keys))]
        m = max(lg)
        e = [math.exp(v - m) for v in lg]
        z = sum(e)
        for x in range(len(keys)):
            out[h] += (e[x] / z) * keys[x]
    return O.rope(out, p, d_r, base, inverse=True)


def test_attend_matches_loops():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((3, 8))
    keys = rng.standard_normal((11, 8))
    got = O.attend(q, 77, keys, 0.35, 4, 10000.0)
    assert np.allclose(got, _attend_loops(q, 77, keys, 0.35, 4, 10000.0), atol=1e-12)


def test_window_only_attention_is_sdpa():
    """With no compressed entry visible (p < 8) and no rotation, the layer is textbook
    softmax attention over the window, checked against torch's SDPA in fp64."""
    w = wl.tiny_prefill(seed=10, L=8, d_r=0)
    L, spec = w.layers[0], w.layers[0].spec
    pools = _fresh_pools(w)
    _run_compress(w, pools)
    qs = w.queries
    out = O.attention(spec, pools, qs.seq, qs.pos, qs.q, topk=np.full((8, spec.top_k), -1))
    keys = torch.tensor(w.batch.kv, dtype=torch.float64)              # SWA rows (d_r = 0)
    q = torch.tensor(qs.q, dtype=torch.float64).transpose(0, 1)       # [H, n, D]
    mask = torch.tensor([[t <= p for t in range(8)] for p in range(8)])
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, keys.expand(spec.H, 8, spec.D), keys.expand(spec.H, 8, spec.D), attn_mask=mask,
        scale=spec.scale).transpose(0, 1).numpy()
    assert np.allclose(out, ref, atol=1e-12)


def test_window_edge_is_sdpa_with_a_128_token_band():
    """The window's edge, pinned away from the oracle's own code: with no rotation and every
    top-k slot empty, the oracle's attention at each of 320 positions equals torch's fp64
    SDPA over all tokens with a band mask of the pages' 128 tokens ([notes] 四大核心技术 4,
    窗口大小 128): a query at p sees t with 0 <= p - t < 128, its own token included (the
    reading of the window range). A 127- or 129-token band gives a different output, so an
    off-by-one at either end of the window fails this test."""
    n = 320
    w = wl.tiny_prefill(seed=16, L=n, d_r=0)
    spec = w.layers[0].spec
    width = GOLD["swa_window"]["value"]
    pools = _fresh_pools(w)
    _run_compress(w, pools)
    qs = w.queries
    out = O.attention(spec, pools, qs.seq, qs.pos, qs.q, topk=np.full((n, spec.top_k), -1))
    keys = torch.tensor(w.batch.kv, dtype=torch.float64)              # window rows (d_r = 0)
    q = torch.tensor(qs.q, dtype=torch.float64).transpose(0, 1)       # [H, n, D]
    lag = torch.arange(n)[:, None] - torch.arange(n)[None, :]         # p - t

    def sdpa(band):
        mask = (lag >= 0) & (lag < band)
        return torch.nn.functional.scaled_dot_product_attention(
            q, keys.expand(spec.H, n, spec.D), keys.expand(spec.H, n, spec.D),
            attn_mask=mask, scale=spec.scale).transpose(0, 1).numpy()

    assert np.allclose(out, sdpa(width), atol=1e-12)
    for wrong in (width - 1, width + 1):
        d = np.abs(out - sdpa(wrong)).max(axis=(1, 2))
        assert (d[:wrong - 1] < 1e-12).all() and d[width:].min() > 1e-6


def _pipeline(w, permute=False):
    """Whole layer from raw tokens: insert, index + top-k, attention. With permute, every
    pool's pages are shuffled (contents moved, block tables rewritten to match)."""
    L, spec = w.layers[0], w.layers[0].spec
    pools = _fresh_pools(w)
    if permute:
        rng = np.random.default_rng(0)
        for pool in (pools.attn, pools.idx, pools.swa, pools.state):
            R = pool.R
            n_pages = len(pool.data) // R
            perm = rng.permutation(n_pages)
            old = pool.data.copy()
            for pg in range(n_pages):
                pool.data[perm[pg] * R:(perm[pg] + 1) * R] = old[pg * R:(pg + 1) * R]
            pool.bt = np.where(pool.bt >= 0, perm[np.maximum(pool.bt, 0)], -1)
    O.compress_insert(spec, L.bias, L.gamma, L.ibias, pools, w.batch.cu, w.batch.start,
                      w.batch.kv, w.batch.s, w.batch.ik, w.batch.is_)
    qs = w.queries
    top, _ = O.index_topk(spec, pools, qs.seq, qs.pos, qs.q_idx, qs.w, spec.top_k)
    out = O.attention(spec, pools, qs.seq, qs.pos, qs.q, top)
    return top, out


def _shift_pair(c, L=300):
    """The same tokens inserted at positions [0, L) and at [c, c+L), c a multiple of 256."""
    w = wl.tiny_prefill(seed=11, L=L, top_k=16)
    L0, spec = w.layers[0], w.layers[0].spec
    a = _fresh_pools(w)
    O.compress_insert(spec, L0.bias, L0.gamma, L0.ibias, a, w.batch.cu, w.batch.start,
                      w.batch.kv, w.batch.s, w.batch.ik, w.batch.is_)
    lay = wl.make_layer(np.random.default_rng(3), spec, [c], [L], prefill_cache=False)
    b = O.Pools(spec, lay.attn, lay.idx, lay.swa, lay.state)
    O.compress_insert(spec, L0.bias, L0.gamma, L0.ibias, b, w.batch.cu, w.batch.start + c,
                      w.batch.kv, w.batch.s, w.batch.ik, w.batch.is_)
    return w, spec, a, b


def test_shift_invariance():
    """Adding a constant c to every position leaves the output unchanged: the inverse RoPE
    at the query position removes the absolute position ([notes] Inverse RoPE 的数学原理).
    Moving the sequence by c moves entry j to j + c/S and rotates every stored row by c
    more; attention over the moved lists at p + c then equals attention at p."""
    c = 12288
    w, spec, a, b = _shift_pair(c)
    dj = c // spec.S
    n_e = O.visible_entries(spec.S, spec.W, spec.win_off, 300)
    for j in range(n_e):
        assert np.allclose(b.attn.read(0, j + dj, False),
                           O.rope(a.attn.read(0, j, False), c, spec.d_r, spec.rope_base),
                           atol=1e-9)
        assert np.allclose(b.idx.read(0, j + dj, False), a.idx.read(0, j, False), atol=1e-12)
    qs = w.queries
    keep = qs.pos >= spec.swa - 1                  # whole window inside the sequence
    ta, _ = O.index_topk(spec, a, qs.seq[keep], qs.pos[keep], qs.q_idx[keep], qs.w[keep], 16)
    tb = np.where(ta >= 0, ta + dj, -1)
    oa = O.attention(spec, a, qs.seq[keep], qs.pos[keep], qs.q[keep], ta)
    ob = O.attention(spec, b, qs.seq[keep], qs.pos[keep] + c, qs.q[keep], tb)
    assert np.allclose(oa, ob, atol=1e-9)


def test_shift_invariance_catches_a_missing_inverse_rope(monkeypatch):
    """The shift pin has teeth: an oracle without the inverse rotation fails it."""
    c = 12288
    w, spec, a, b = _shift_pair(c)
    real = O.rope

    def no_inverse(x, pos, d_r, base, inverse=False):
        return np.array(x, dtype=np.float64) if inverse else real(x, pos, d_r, base)
    monkeypatch.setattr(O, "rope", no_inverse)
    qs = w.queries
    keep = qs.pos >= spec.swa - 1
    ta, _ = O.index_topk(spec, a, qs.seq[keep], qs.pos[keep], qs.q_idx[keep], qs.w[keep], 16)
    tb = np.where(ta >= 0, ta + c // spec.S, -1)
    oa = O.attention(spec, a, qs.seq[keep], qs.pos[keep], qs.q[keep], ta)
    ob = O.attention(spec, b, qs.seq[keep], qs.pos[keep] + c, qs.q[keep], tb)
    assert not np.allclose(oa, ob, atol=1e-3)


def test_topk_all_visible_equals_dense():
    """k >= number of visible entries: the top-k list is every visible entry and the
    c4a attention equals dense attention over them."""
    w = wl.tiny_prefill(seed=12, L=160, top_k=64)
    L, spec = w.layers[0], w.layers[0].spec
    pools = _fresh_pools(w)
    _run_compress(w, pools)
    qs = w.queries
    top, _ = O.index_topk(spec, pools, qs.seq, qs.pos, qs.q_idx, qs.w, 64)
    for i, p in enumerate(qs.pos):
        n = O.visible_entries(spec.S, spec.W, spec.win_off, int(p))
        assert n <= 64 and list(top[i][:n]) == list(range(n))
    assert np.allclose(O.attention(spec, pools, qs.seq, qs.pos, qs.q, top),
                       O.attention(spec, pools, qs.seq, qs.pos, qs.q, None), atol=1e-13)


def test_causality_scan_and_brute_force_attention():
    """Every selected entry covers only positions < p, and the oracle's attention equals
    the loop implementation over the selected entries and the window."""
    w = wl.tiny_prefill(seed=13, L=96, top_k=8, D=16, d_r=4, H=2, d_I=8)
    L, spec = w.layers[0], w.layers[0].spec
    pools = _fresh_pools(w)
    _run_compress(w, pools)
    qs = w.queries
    top, _ = O.index_topk(spec, pools, qs.seq, qs.pos, qs.q_idx, qs.w, spec.top_k)
    out = O.attention(spec, pools, qs.seq, qs.pos, qs.q, top)
    for i in range(0, 96, 7):
        p = int(qs.pos[i])
        for j in top[i]:
            if j >= 0:
                assert max(O.entry_positions(spec.S, spec.W, spec.win_off, int(j))) < p
        keys = [pools.attn.read(0, int(j), False) for j in top[i] if j >= 0]
        keys += [pools.swa.read(0, t, False) for t in range(max(0, p - 127), p + 1)]
        want = _attend_loops(qs.q[i].astype(np.float64), p, np.stack(keys), spec.scale, 4,
                             spec.rope_base)
        assert np.allclose(out[i], want, atol=1e-12)


def test_block_permutation_invariance():
    w = wl.tiny_prefill(seed=14, L=300, top_k=16)
    t0, o0 = _pipeline(w)
    t1, o1 = _pipeline(w, permute=True)
    assert np.array_equal(t0, t1) and np.array_equal(o0, o1)


# ------------------------------------------------------------------------- footprint
def test_kv_footprint_matches_pages():
    """The pages' 9.62 GiB (V4) and 83.9 GiB (V3.2-style, 61 layers) per 1M-token bf16
    sequence, from entry sizes D=512 + d_I=128 (V4) and 576 + 128 elements (V3.2)."""
    GiB = float(1 << 30)
    v4 = O.kv_bytes_per_sequence(1 << 20, GOLD["c4a_layers"]["value"],
                                 GOLD["c128a_layers"]["value"], 512, 128, 2) / GiB
    v32 = O.kv_bytes_per_sequence_v32(1 << 20, 61, 576, 128, 2) / GiB
    assert round(v4, 2) == GOLD["kv_gib_per_1m_seq_v4_bf16"]["value"]
    assert round(v32, 1) == GOLD["kv_gib_per_1m_seq_v32_61_layers_bf16"]["value"]
    assert round(v32 / v4, 1) == GOLD["v4_over_v32_ratio"]["value"]
