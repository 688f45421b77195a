"""Plain fp64 CPU oracle for one layer of DeepSeek-V4-style hybrid compressed attention.

TEST INFRASTRUCTURE ONLY. This package exists to check the CUDA path. Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import it; the
product package never does, and the two share no code.

Everything here is written for a reader to check against the pages by eye: one
function per step, numpy fp64, no blocking or fusion. Citations name the page and its
section:

  [notes]  "DeepSeek V4 in vLLM 技术博客详尽笔记" (vllm-deepseek-v4-notes.pages.dev)
  [blog]   "vLLM DeepSeek V4 支援：高效長上下文注意力" (agentlenshq.com)
  [serve]  "DeepSeek-V4服务：百万token上下文成为推理系统难题" (ai-pulse-lab.com)

Readings taken where the pages are silent or garbled (each is listed with its reason in
the design notes of the repository):
  R1  entry j of a layer with window W, stride S covers positions S*j+win_off .. +W-1,
      win_off = 0 (c4a: 4j..4j+7), RoPE at position S*j. Positions < 0 are absent.
  R2  an entry is visible to a query at p only if every position it covers is < p.
  R3  the sliding window of a query at p is the tokens [max(0, p-swa+1), p] (own token
      included), each stored as RoPE(kv_t, t) without normalisation.
  R4  entry weights: per-channel softmax over the window of s_t + b[offset]; b is
      [W, D]. RMSNorm eps = 1e-6; RoPE rotates adjacent pairs of the last d_r dims,
      theta_i = base^(-2i/d_r).
  R5  indexer keys are compressed with their own bias and get neither RMSNorm nor RoPE.
  R6  fp8 storage: one scale per row, scale = amax/448 (1 if amax = 0), code =
      e4m3 round-to-nearest-even of y/scale, saturated to +-448.
  R7  top-k: all visible entries if there are at most k, else the k largest scores,
      ties broken towards the smaller entry index; output ascending, -1 padded.
  R8  attention: one softmax over the selected entries and the window, logits
      scaled by 1/sqrt(D); the same stored vector is key and value; inverse RoPE at
      the query position on the output.
  R13 query norm: RMSNorm of each (query, head) row over its D dims, one gamma [D]
      shared by the heads, the entries' epsilon.
  R16 fp4 indexer cache: e2m1 codes (2 exponent bits, bias 1, 1 mantissa bit), two per
      byte with element 2i in the low nibble, one scale per 128-dim row = amax / 6 (1 if
      the row is zero), code = round-to-nearest-even of y / scale saturated to +-6.
"""
from __future__ import annotations

import math

import numpy as np

BLOCK = 256            # native positions per logical block ([notes] 解决方案一：统一逻辑块大小)
E4M3_MAX = 448.0


# --------------------------------------------------------------------------- RoPE
def rope_theta(d_r: int, base: float) -> np.ndarray:
    """theta_i = base^(-2i/d_r), i in [0, d_r/2) (R4)."""
    i = np.arange(d_r // 2, dtype=np.float64)
    return base ** (-2.0 * i / d_r)


def rope(x, pos, d_r: int, base: float, inverse: bool = False) -> np.ndarray:
    """Rotate the pairs (D-d_r+2i, D-d_r+2i+1) of the last axis by pos*theta_i.

    [notes] "Inverse RoPE 的数学原理": the output is multiplied by R^-1(theta_pos), the
    inverse rotation, which is this rotation with the angle negated.
    ``pos`` broadcasts against ``x[..., 0]``.
    """
    x = np.array(x, dtype=np.float64, copy=True)
    if d_r == 0:
        return x
    D = x.shape[-1]
    ang = np.asarray(pos, dtype=np.float64)[..., None] * rope_theta(d_r, base)
    if inverse:
        ang = -ang
    c, s = np.cos(ang), np.sin(ang)
    a = x[..., D - d_r::2].copy()
    b = x[..., D - d_r + 1::2].copy()
    x[..., D - d_r::2] = a * c - b * s
    x[..., D - d_r + 1::2] = a * s + b * c
    return x


# --------------------------------------------------------------------------- fp8
def e4m3_values() -> np.ndarray:
    """Magnitudes of the finite e4m3 codes 0..126, from the format's definition:
    4 exponent bits (bias 7), 3 mantissa bits, exponent 0 subnormal, code 127 NaN."""
    out = np.empty(127, dtype=np.float64)
    for code in range(127):
        e, m = code >> 3, code & 7
        out[code] = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


_E4M3 = e4m3_values()


def e4m3_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.int64)
    mag = _E4M3[np.minimum(c & 0x7F, 126)]
    return np.where(c & 0x80, -mag, mag)


def e4m3_encode(v) -> np.ndarray:
    """Round-to-nearest-even onto the e4m3 grid, saturating at +-448 (R6)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.searchsorted(_E4M3, a, side="left")          # first grid value >= a
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _E4M3[lo]
    d_hi = _E4M3[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a == _E4M3[hi], hi, code)
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def e4m3_midpoint_distance(v) -> np.ndarray:
    """Distance of |v| from the nearest rounding midpoint of the e4m3 grid, in units of
    the local grid step. Used by the tests to allow a one-code difference only where the
    rounding decision is within a hair of a tie."""
    a = np.minimum(np.abs(np.asarray(v, dtype=np.float64)), E4M3_MAX)
    hi = np.minimum(np.searchsorted(_E4M3, a, side="left"), 126)
    lo = np.maximum(hi - 1, 0)
    step = np.maximum(_E4M3[hi] - _E4M3[lo], 1e-300)
    mid = 0.5 * (_E4M3[hi] + _E4M3[lo])
    return np.abs(a - mid) / step


def quantize(y: np.ndarray):
    """Row-wise fp8 storage of y (R6): returns (codes uint8, scale fp64)."""
    y = np.asarray(y, dtype=np.float64)
    amax = np.abs(y).max(axis=-1)
    scale = np.where(amax > 0, amax / E4M3_MAX, 1.0)
    return e4m3_encode(y / scale[..., None]), scale


# --------------------------------------------------------------------------- fp4
E2M1_MAX = 6.0


def e2m1_values() -> np.ndarray:
    """Magnitudes of the e2m1 codes 0..7, from the format's definition: 2 exponent bits
    (bias 1), 1 mantissa bit, exponent 0 subnormal, no infinities or NaN."""
    out = np.empty(8, dtype=np.float64)
    for code in range(8):
        e, m = code >> 1, code & 1
        out[code] = (m / 2.0) if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return out


_E2M1 = e2m1_values()


def e2m1_decode(codes) -> np.ndarray:
    """Values of 4-bit codes (bit 3 the sign)."""
    c = np.asarray(codes, dtype=np.int64)
    mag = _E2M1[c & 7]
    return np.where(c & 8, -mag, mag)


def e2m1_encode(v) -> np.ndarray:
    """Round-to-nearest-even onto the e2m1 grid, saturating at +-6 (R16)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), E2M1_MAX)
    hi = np.minimum(np.searchsorted(_E2M1, a, side="left"), 7)   # first grid value >= a
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _E2M1[lo]
    d_hi = _E2M1[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a == _E2M1[hi], hi, code)
    return (code | np.where(np.signbit(v), 8, 0)).astype(np.uint8)


def e2m1_midpoint_distance(v) -> np.ndarray:
    """Distance of |v| from the nearest rounding midpoint of the e2m1 grid, in units of the
    local grid step (the tests allow a one-code difference only within a hair of a tie)."""
    a = np.minimum(np.abs(np.asarray(v, dtype=np.float64)), E2M1_MAX)
    hi = np.minimum(np.searchsorted(_E2M1, a, side="left"), 7)
    lo = np.maximum(hi - 1, 0)
    step = np.maximum(_E2M1[hi] - _E2M1[lo], 1e-300)
    return np.abs(a - 0.5 * (_E2M1[hi] + _E2M1[lo])) / step


def pack_e2m1(codes) -> np.ndarray:
    """Two codes per byte along the last axis: element 2i in the low nibble, 2i+1 high."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def quantize_fp4(y: np.ndarray):
    """Row-wise fp4 storage of y (R16): one scale per row, amax / 6 (1 if the row is
    zero); returns (packed codes uint8 [..., d/2], scale fp64)."""
    y = np.asarray(y, dtype=np.float64)
    amax = np.abs(y).max(axis=-1)
    scale = np.where(amax > 0, amax / E2M1_MAX, 1.0)
    return pack_e2m1(e2m1_encode(y / scale[..., None])), scale


# --------------------------------------------------------------------- paged layout
def slot(bt: np.ndarray, R: int, seq: int, r: int) -> int:
    """Pool row of logical row r (a token position or an entry index) of sequence seq.

    [notes] 解决方案一：统一逻辑块大小: one block is 256 native positions and stores
    256/ratio rows (64 c4a entries, 2 c128a entries, 256 tokens). Row r sits at native
    position r*256/R, so in logical block r // R, at row r % R of that block's page.
    Returns -1 when the block has no page.
    """
    blk = r // R
    if r < 0 or blk >= bt.shape[1]:
        return -1
    page = int(bt[seq, blk])
    return -1 if page < 0 else page * R + r % R


# ------------------------------------------------------------------------ compressor
def entry_positions(S: int, W: int, win_off: int, j: int) -> np.ndarray:
    """Positions covered by entry j (R1): S*j+win_off .. S*j+win_off+W-1.

    [notes] 四大核心技术 (C4A: 8 token -> 1, stride 4, neighbours overlap by 4;
    C128A: 128 -> 1, stride 128) and 数学附录精要 (C128A 的精确位置范围 [128i, 128i+127]).
    """
    return S * j + win_off + np.arange(W)


def compress_window(kv_win: np.ndarray, s_win: np.ndarray, b_win: np.ndarray) -> np.ndarray:
    """One compressed vector from a window of tokens (R4).

    [blog] DeepSeek V4 注意力架構: a compressed token is a weighted sum of the window's
    tokens. Weights: per channel, softmax over the window of s_t + b[offset].
    kv_win, s_win, b_win: [n_present, d].
    """
    z = s_win + b_win
    z = z - z.max(axis=0, keepdims=True)
    e = np.exp(z)
    w = e / e.sum(axis=0, keepdims=True)
    return (w * kv_win).sum(axis=0)


def rmsnorm(c: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """y = gamma * c / sqrt(mean(c^2) + eps) ([notes] 融合 1: 压缩后的 K 经过 RMSNorm)."""
    return gamma * c / np.sqrt(np.mean(c * c) + eps)


def q_norm(q: np.ndarray, gamma_q: np.ndarray, eps: float) -> np.ndarray:
    """Per-head query RMSNorm (R13): every (query, head) row of q [n_q, H, D] becomes
    gamma_q * q_h / sqrt(mean(q_h^2) + eps), gamma_q [D] shared by the heads.

    [notes] 优化一：三大内核融合, fusion 3 (Q Norm + KV RoPE + K Insert): each Q head is
    normalised on its own, with no communication between heads.
    """
    q = np.asarray(q, dtype=np.float64)
    out = np.empty_like(q)
    for i in range(q.shape[0]):
        for h in range(q.shape[1]):
            out[i, h] = rmsnorm(q[i, h], np.asarray(gamma_q, dtype=np.float64), eps)
    return out


def visible_entries(S: int, W: int, win_off: int, p: int) -> int:
    """Number of entries visible to a query at position p (R2).

    [notes] 因果性条件: a query at p may only use information from [0, p-1]; and
    C128A 的因果性约束: no c128a entry is usable before position 128. Entry j is visible
    iff its last covered position S*j+win_off+W-1 <= p-1.
    """
    n = (p - win_off - W) // S + 1
    return max(0, n)


class Pools:
    """The oracle's copy of a layer's caches (fp64 values, or fp8 codes + fp64 scales)."""

    def __init__(self, spec, attn, idx, swa, state):
        self.spec = spec
        self.attn = _own(attn)
        self.idx = _own(idx, getattr(spec, "idx_fp4", False)) if idx is not None else None
        self.swa = _own(swa)
        self.state = _own(state)


class _Pool:
    def __init__(self, data, scale, bt, R, fp4=False):
        self.data, self.scale, self.bt, self.R = data, scale, bt, R
        self.fp4 = fp4         # packed e2m1 rows (R16) instead of fp8 / raw values
        self.raw = {}          # pool row -> value before fp8 rounding (for the tests)

    def _decode(self, s):
        if self.fp4:
            return e2m1_decode(unpack_e2m1(self.data[s])) * np.asarray(self.scale[s])[..., None]
        return e4m3_decode(self.data[s]) * np.asarray(self.scale[s])[..., None]

    def slots(self, seq, rows) -> np.ndarray:
        """slot() of many logical rows of one sequence."""
        rows = np.asarray(rows, dtype=np.int64)
        blk = rows // self.R
        inside = (rows >= 0) & (blk < self.bt.shape[1])
        page = np.where(inside, self.bt[seq, np.where(inside, blk, 0)], -1).astype(np.int64)
        return np.where(page >= 0, page * self.R + rows % self.R, -1)

    def read_many(self, seq, rows, fp8):
        s = self.slots(seq, rows)
        if (s < 0).any():
            raise ValueError("a row of sequence %d has no page" % seq)
        if fp8 or self.fp4:
            return self._decode(s)
        return self.data[s].astype(np.float64)

    def read(self, seq, r, fp8):
        s = slot(self.bt, self.R, seq, r)
        if s < 0:
            raise ValueError("row %d of sequence %d has no page" % (r, seq))
        if fp8 or self.fp4:
            return self._decode(s)
        return self.data[s].astype(np.float64)

    def write(self, seq, r, y, fp8):
        s = slot(self.bt, self.R, seq, r)
        if s < 0:
            return -1
        if self.fp4:
            codes, sc = quantize_fp4(y[None, :])
            self.data[s] = codes[0]
            self.scale[s] = sc[0]
        elif fp8:
            codes, sc = quantize(y[None, :])
            self.data[s] = codes[0]
            self.scale[s] = sc[0]
        else:
            self.data[s] = y
        self.raw[s] = np.array(y, dtype=np.float64)
        return s


def _own(p, fp4=False):
    data = np.array(p.data, copy=True)
    if data.dtype != np.uint8:
        data = data.astype(np.float64)
    scale = None if p.scale is None else np.asarray(p.scale, dtype=np.float64).copy()
    return _Pool(data, scale, np.array(p.bt, copy=True), p.rows_per_block, fp4)


def compress_insert(spec, bias, gamma, ibias, pools: Pools, cu, start, kv, s, ik=None, is_=None):
    """Insert the new tokens of every sequence (steps a1-a5).

    For sequence b the new tokens sit at positions start[b] .. start[b]+n_b-1.
      * every new token t: sliding-window row RoPE(kv_t, t) (R3; [blog] 短滑動窗口 and
        the "Q norm + KV RoPE + K insert" fusion of GPU 計算飽和度);
      * every entry whose window ends among the new tokens: compressed vector, RMSNorm,
        RoPE at S*j, stored ([notes] 融合 1); for c4a also the indexer key, compressed
        with its own bias (R5);
      * raw (kv, s, ik, is) of the last W new positions into the residual pool, which
        plays the part of the compressor state kept as sliding-window KV ([notes]
        解决方案二：压缩器状态滑动窗口化).
    Tokens of a window that precede start[b] are read from the residual pool.
    Returns the list of (kind, seq, logical row, pool row) writes, for slot checks.
    """
    fp8 = spec.fp8
    D, dI, W, S, off = spec.D, spec.d_I, spec.W, spec.S, spec.win_off
    writes = []
    for b in range(len(start)):
        P0 = int(start[b])
        a0, a1 = int(cu[b]), int(cu[b + 1])
        P1 = P0 + (a1 - a0)

        def token(t):
            if t >= P0:
                i = a0 + (t - P0)
                row = [kv[i], s[i]]
                if spec.has_indexer:
                    row += [ik[i], is_[i]]
                return np.concatenate(row).astype(np.float64)
            return pools.state.read(b, t, fp8=False)

        for t in range(P0, P1):
            key = rope(kv[a0 + t - P0], t, spec.d_r, spec.rope_base)
            writes.append(("swa", b, t, pools.swa.write(b, t, key, fp8)))

        last_off = off + W - 1
        j_lo = max(0, -((-(P0 - last_off)) // S))      # ceil((P0 - last_off) / S)
        j_hi = (P1 - 1 - last_off) // S
        for j in range(j_lo, j_hi + 1):
            pos = entry_positions(S, W, off, j)
            present = pos >= 0
            rows = np.stack([token(int(t)) for t in pos[present]])
            c = compress_window(rows[:, :D], rows[:, D:2 * D], bias[present])
            y = rope(rmsnorm(c, gamma, spec.eps), S * j, spec.d_r, spec.rope_base)
            writes.append(("attn", b, j, pools.attn.write(b, j, y, fp8)))
            if spec.has_indexer:
                ci = compress_window(rows[:, 2 * D:2 * D + dI], rows[:, 2 * D + dI:],
                                     ibias[present])
                writes.append(("idx", b, j, pools.idx.write(b, j, ci, fp8)))

        for t in range(max(P0, P1 - W), P1):
            i = a0 + (t - P0)
            row = [kv[i], s[i]] + ([ik[i], is_[i]] if spec.has_indexer else [])
            writes.append(("state", b, t,
                           pools.state.write(b, t, np.concatenate(row).astype(np.float64),
                                             fp8=False)))
    return writes


# ---------------------------------------------------------------------- indexer + top-k
def index_scores(q_idx: np.ndarray, w: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """score_j = sum_h w_h * ReLU(q_h . k_j) ([blog] DeepSeek Sparse Attention: only the
    top-k compressed tokens are attended; the score is the DSA indexer's head-weighted
    sum of ReLU dot products). q_idx [H_I, d_I], w [H_I], keys [n, d_I]."""
    dots = keys @ q_idx.T
    return (np.maximum(dots, 0.0) * w[None, :]).sum(axis=1)


def select_topk(scores: np.ndarray, k: int) -> np.ndarray:
    """R7: indices of the k largest scores (ties -> smaller index), ascending, -1 padded."""
    n = len(scores)
    if n <= k:
        sel = np.arange(n)
    else:
        order = np.lexsort((np.arange(n), -scores))
        sel = np.sort(order[:k])
    out = np.full(k, -1, dtype=np.int32)
    out[:len(sel)] = sel
    return out


def index_topk(spec, pools: Pools, q_seq, q_pos, q_idx, w, k: int):
    """Top-k entry lists and the full score rows of every query ([notes] 压缩参数细节:
    C4A keeps the top 512 compressed entries)."""
    n_q = len(q_pos)
    out = np.full((n_q, k), -1, dtype=np.int32)
    all_scores = []
    for i in range(n_q):
        b, p = int(q_seq[i]), int(q_pos[i])
        n = visible_entries(spec.S, spec.W, spec.win_off, p)
        keys = pools.idx.read_many(b, np.arange(n), spec.fp8) if n else np.zeros((0, spec.d_I))
        sc = index_scores(np.asarray(q_idx[i], np.float64), np.asarray(w[i], np.float64), keys)
        out[i] = select_topk(sc, k)
        all_scores.append(sc)
    return out, all_scores


# ---------------------------------------------------------------------------- attention
def attend(q_row: np.ndarray, p: int, keys: np.ndarray, scale: float, d_r: int,
           base: float) -> np.ndarray:
    """Shared-K=V attention of one query (R8).

    [notes] Inverse RoPE 的数学原理: AttentionOutput = sum(softmax(Q K^T) V) R^-1(theta_p).
    The query is rotated to its position; every stored vector is already rotated to its
    own position and serves as key and value.
    q_row [H, D]; keys [n, D] -> [H, D].
    """
    qr = rope(q_row, p, d_r, base)
    logits = scale * (qr @ keys.T)
    logits = logits - logits.max(axis=1, keepdims=True)
    pr = np.exp(logits)
    pr = pr / pr.sum(axis=1, keepdims=True)
    o = pr @ keys
    return rope(o, p, d_r, base, inverse=True)


def gather_keys(spec, pools: Pools, b: int, p: int, entries) -> np.ndarray:
    """Keys of a query at p: the listed compressed entries, then the window tokens
    [max(0, p-swa+1), p] (R3; [blog] 短滑動窗口)."""
    ent = pools.attn.read_many(b, np.asarray(list(entries), dtype=np.int64), spec.fp8)
    win = pools.swa.read_many(b, np.arange(max(0, p - spec.swa + 1), p + 1), spec.fp8)
    return np.concatenate([ent.reshape(-1, spec.D), win])


def attention(spec, pools: Pools, q_seq, q_pos, q, topk=None) -> np.ndarray:
    """Attention of every query: over its top-k list (c4a, [blog] DSA) or densely over all
    visible entries (topk None: c128a, [serve] HCA attends its ~8k entries densely)."""
    n_q = len(q_pos)
    out = np.zeros((n_q, spec.H, spec.D))
    for i in range(n_q):
        b, p = int(q_seq[i]), int(q_pos[i])
        if topk is None:
            entries = range(visible_entries(spec.S, spec.W, spec.win_off, p))
        else:
            entries = [int(j) for j in topk[i] if j >= 0]
        keys = gather_keys(spec, pools, b, p, entries)
        out[i] = attend(np.asarray(q[i], np.float64), p, keys, spec.scale, spec.d_r,
                        spec.rope_base)
    return out


# ------------------------------------------------------------------------- footprint
def kv_bytes_per_sequence(tokens: int, c4a_layers: int, c128a_layers: int, D: int,
                          d_I: int, elem_bytes: int) -> int:
    """KV bytes one sequence keeps across a V4 stack ([notes] 8.7x 节省的算术推导):
    c4a layers keep tokens/4 entries of (D + d_I) elements (shared KV + indexer key),
    c128a layers keep tokens/128 entries of D elements."""
    c4a = (tokens // 4) * (D + d_I) * elem_bytes * c4a_layers
    c128a = (tokens // 128) * D * elem_bytes * c128a_layers
    return c4a + c128a


def kv_bytes_per_sequence_v32(tokens: int, layers: int, mla_elems: int, idx_elems: int,
                              elem_bytes: int) -> int:
    """A V3.2-style stack keeps one MLA entry and one indexer entry per token per layer."""
    return tokens * (mla_elems + idx_elems) * elem_bytes * layers
