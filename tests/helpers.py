"""Shared pieces of the GPU parity tests: moving generated inputs to the device, running
the layer through the C ABI, and the acceptance rules.

Acceptance rules:
  * integers (slots, entry indices, top-k lists where no tie band is involved): exact;
  * top-k sets: identical except entries whose oracle score lies within 1e-3 (relative)
    of the oracle's k-th score;
  * fp8 cache rows: scales within 1e-6 relative; codes equal except a one-step rounding
    difference where the oracle's y/scale lies near a rounding midpoint: within 1e-3 of a
    grid step, or within 448 x 2^-20 in code units. The second bound is the kernel's own
    error: it evaluates y in fp32 (a chain of about sixteen operations, each within 2^-24
    of the row's largest value), so |y_gpu - y| <= 2^-20 amax, i.e. 448 x 2^-20 after the
    division by scale = amax / 448. It matters only near zero, where an e4m3 step is 2^-9
    (subnormal codes); fp4 rows use 6 x 2^-20 the same way;
  * fp32 cache rows: within 1e-5 absolute;
  * attention output: max-abs 1e-4 (fp32 layer), max-abs 3e-2 and mean-abs 3e-3
    (bf16 / fp8 layers), against the oracle run on the same stored values.
"""
from __future__ import annotations

import numpy as np
import torch

from compressed_sparse_long_gb300.layer import Layer
from oracle import v4a_oracle as O

TIE_BAND = 1e-3
FP32_Y_ERR = 2.0 ** -20      # bound on the kernel's fp32 error in y, relative to the row amax
FP32_OUT_TOL = 1e-4
BF16_MAX_TOL = 3e-2
BF16_MEAN_TOL = 3e-3


def T(x, dt, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev, dt)


class DevInputs:
    """Device copies of a workload's new tokens and queries."""

    def __init__(self, w, dev="cuda"):
        fp8 = w.layers[0].spec.fp8
        dt = torch.bfloat16 if fp8 else torch.float32
        b, q = w.batch, w.queries
        self.cu = T(b.cu, torch.int32, dev)
        self.start = T(b.start, torch.int64, dev)
        self.kv, self.s = T(b.kv, dt, dev), T(b.s, dt, dev)
        self.ik = None if b.ik is None else T(b.ik, dt, dev)
        self.is_ = None if b.is_ is None else T(b.is_, dt, dev)
        self.q_seq, self.q_pos = T(q.seq, torch.int32, dev), T(q.pos, torch.int64, dev)
        self.q = T(q.q, dt, dev)
        self.q_idx = None if q.q_idx is None else T(q.q_idx, dt, dev)
        self.w = None if q.w is None else T(q.w, torch.float32, dev)
        self.max_pos = int(q.pos.max()) if len(q.pos) else 0


def oracle_pools(layer):
    return O.Pools(layer.spec, layer.attn, layer.idx, layer.swa, layer.state)


class _HostPool:
    """Host copy of one device pool, in the shape the oracle's Pools reads."""

    def __init__(self, pool):
        d = pool.data.cpu()
        self.data = d.float().numpy() if d.dtype in (torch.bfloat16, torch.float32) else d.numpy()
        self.scale = None if pool.scale is None else pool.scale.cpu().numpy()
        self.bt = pool.block_table.cpu().numpy()
        self.rows_per_block = pool.rows_per_block


def device_pools(lay, spec):
    """The oracle's view of the pools as the GPU left them: indexer and attention parity
    run on the GPU-written codes and scales (the same dequantised values on both sides)."""
    return O.Pools(spec, _HostPool(lay.attn), None if lay.idx is None else _HostPool(lay.idx),
                   _HostPool(lay.swa), _HostPool(lay.state))


def oracle_insert(w, layer, pools):
    b = w.batch
    return O.compress_insert(layer.spec, layer.bias, layer.gamma, layer.ibias, pools, b.cu,
                             b.start, b.kv, b.s, b.ik, b.is_)


def check_topk(got, ref, scores, k):
    """Top-k acceptance; returns the indices of the rows whose sets are identical."""
    same = []
    for i in range(len(ref)):
        g, r = got[i], ref[i]
        gv = g[g >= 0]
        assert np.all(g[len(gv):] == -1), "padding must trail"
        assert np.all(np.diff(gv) > 0), "entries must be ascending and distinct"
        n = len(scores[i])
        assert len(gv) == min(k, n)
        assert np.all((gv >= 0) & (gv < n)), "an index outside the visible entries"
        if np.array_equal(g, r):
            same.append(i)
            continue
        kth = np.sort(scores[i])[::-1][k - 1]
        for j in set(gv.tolist()) ^ set(r[r >= 0].tolist()):
            assert abs(scores[i][j] - kth) <= TIE_BAND * abs(kth), \
                "row %d: entry %d score %.9g outside the tie band of %.9g" % (i, j, scores[i][j], kth)
    return same


def check_fp8_rows(gpu_data, gpu_scale, ref_pool, slots):
    """Compare GPU-written fp8 rows with the oracle's at the given pool rows."""
    n_close = 0
    for s in slots:
        y = ref_pool.raw[s]
        so = float(ref_pool.scale[s])
        sg = float(gpu_scale[s])
        assert abs(sg - so) <= 1e-6 * so, (s, sg, so)
        cg, co = gpu_data[s], ref_pool.data[s]
        bad = np.nonzero(cg != co)[0]
        if len(bad) == 0:
            continue
        v = y[bad] / so
        dg = O.e4m3_decode(cg[bad])
        do = O.e4m3_decode(co[bad])
        same_value = dg == do                           # +0 / -0
        # the GPU picked the other grid neighbour of y/scale, and y/scale sits at a tie
        grid = O.e4m3_values()
        a = np.minimum(np.abs(v), 448.0)
        hi = np.minimum(np.searchsorted(grid, a, side="left"), 126)
        lo = np.maximum(hi - 1, 0)
        sgn = np.where(np.signbit(v), -1.0, 1.0)
        neighbour = (dg == sgn * grid[lo]) | (dg == sgn * grid[hi])
        dist = O.e4m3_midpoint_distance(v)                  # in grid steps
        near = (dist < 1e-3) | (dist * (grid[hi] - grid[lo]) <= 448.0 * FP32_Y_ERR)
        ok = same_value | (neighbour & near)
        assert ok.all(), "row %d: codes %s vs %s at y/scale %s" % (s, cg[bad][~ok], co[bad][~ok],
                                                                   v[~ok])
        n_close += int((~same_value).sum())
    return n_close


def check_fp4_rows(gpu_data, gpu_scale, ref_pool, slots):
    """Compare GPU-written packed fp4 rows with the oracle's at the given pool rows: scales
    within 1e-6 relative; codes equal except the other grid neighbour of y/scale where it
    lies within 1e-3 of a rounding midpoint (in grid-step units)."""
    n_close = 0
    for s in slots:
        y = ref_pool.raw[s]
        so = float(ref_pool.scale[s])
        sg = float(gpu_scale[s])
        assert abs(sg - so) <= 1e-6 * so, (s, sg, so)
        cg, co = O.unpack_e2m1(gpu_data[s]), O.unpack_e2m1(ref_pool.data[s])
        bad = np.nonzero(cg != co)[0]
        if len(bad) == 0:
            continue
        v = y[bad] / so
        dg, do = O.e2m1_decode(cg[bad]), O.e2m1_decode(co[bad])
        same_value = dg == do                           # +0 / -0
        grid = O.e2m1_values()
        a = np.minimum(np.abs(v), 6.0)
        hi = np.minimum(np.searchsorted(grid, a, side="left"), 7)
        lo = np.maximum(hi - 1, 0)
        sgn = np.where(np.signbit(v), -1.0, 1.0)
        neighbour = (dg == sgn * grid[lo]) | (dg == sgn * grid[hi])
        dist = O.e2m1_midpoint_distance(v)                  # in grid steps
        near = (dist < 1e-3) | (dist * (grid[hi] - grid[lo]) <= 6.0 * FP32_Y_ERR)
        ok = same_value | (neighbour & near)
        assert ok.all(), "row %d: codes %s vs %s at y/scale %s" % (s, cg[bad][~ok], co[bad][~ok],
                                                                   v[~ok])
        n_close += int((~same_value).sum())
    return n_close


def check_out(got, ref, fp8):
    d = np.abs(got.astype(np.float64) - ref)
    if fp8:
        assert d.max() <= BF16_MAX_TOL and d.mean() <= BF16_MEAN_TOL, (d.max(), d.mean())
    else:
        assert d.max() <= FP32_OUT_TOL, d.max()
    return float(d.max()), float(d.mean())


def device_layer(layer, dev="cuda"):
    return Layer.from_host(layer, dev)
