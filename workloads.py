"""Seeded synthetic inputs for one layer of hybrid compressed attention.

This module only draws random numbers and lays them out in the paged-cache shapes.
It holds none of the method's arithmetic: no compression, normalisation, rotation,
fp8 quantisation rule, scoring, selection or attention. Both the CUDA path and the
oracle consume what it returns; neither imports the other.

Draw order (numpy ``default_rng(seed)``, PCG64, fp64 draws, cast afterwards):
  1. layer parameters: compressor bias b[W, D] ~ N(0, 0.5) (0.5 read as the standard
     deviation), RMSNorm gamma[D] ~ N(1, 0.1), indexer-compressor bias ib[W, d_I] ~ N(0, 0.5);
  2. physical page permutation of each pool;
  3. pre-filled cache contents (random fp8 rows + scales, raw residual tokens);
  4. new-token inputs kv, s, ik, is ~ N(0, 1);
  5. queries q, q_idx ~ N(0, 1) and indexer head weights w (U(0,1) for the tiny fp32
     layer, N(0,1) otherwise).
bf16 workloads round every draw to bf16 (round-to-nearest-even, via torch's cast) so
both sides read identical values; fp32 workloads round to fp32.

Random fp8 cache rows: the stored (code, scale) pairs stand for already-quantised
cache entries. A row scale is drawn as U(0.5, 1.5)/64 and the codes as the e4m3
values nearest to N(0,1)/scale, clipped to the e4m3 range (torch's cast does not
saturate). The dequantised values code*scale are then close to N(0,1).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

BLOCK = 256          # native token positions per logical cache block
E4M3_MAX = 448.0


@dataclass(frozen=True)
class LayerSpec:
    """Numbers that define one attention layer (parameters only)."""
    kind: str                 # "c4a" (window 8, stride 4) or "c128a" (window 128, stride 128)
    fp8: bool                 # True: bf16 inputs + fp8 e4m3 caches; False: fp32 everywhere
    D: int = 512              # head dim of the single shared K=V head and of the query heads
    d_r: int = 64             # rotated tail dims
    H: int = 64               # query heads
    H_I: int = 64             # indexer heads (c4a only)
    d_I: int = 128            # indexer head dim (c4a only)
    swa: int = 128            # sliding-window length (tokens [p-swa+1, p])
    top_k: int = 512          # indexer top-k (c4a only)
    rope_base: float = 10000.0
    eps: float = 1e-6
    win_off: int = 0          # entry j covers S*j+win_off .. S*j+win_off+W-1
    sm_scale: float = 0.0     # 0 -> 1/sqrt(D)
    idx_fp4: bool = False     # indexer cache in packed 4-bit e2m1 codes + row scale (fp8 layers)

    @property
    def W(self) -> int:
        return 8 if self.kind == "c4a" else 128

    @property
    def S(self) -> int:
        return 4 if self.kind == "c4a" else 128

    @property
    def rows_per_block(self) -> int:
        return BLOCK // self.S

    @property
    def scale(self) -> float:
        return self.sm_scale if self.sm_scale > 0 else 1.0 / math.sqrt(self.D)

    @property
    def has_indexer(self) -> bool:
        return self.kind == "c4a"

    @property
    def state_width(self) -> int:
        # raw residual row per token: kv | s | ik | is (indexer half only for c4a)
        return 2 * self.D + (2 * self.d_I if self.has_indexer else 0)


@dataclass
class Paged:
    """One paged pool plus its block table.

    data:  [n_pages * rows_per_block, width]; uint8 e4m3 codes (fp8 pools), float32
           (fp32 pools) or bf16-valued float32 (residual-state pools of bf16 layers).
    scale: [n_pages * rows_per_block] float32 per-row scales (fp8 pools) or None.
    bt:    [n_seq, max_blocks] int32 physical page of each logical block, -1 = none.
    """
    data: np.ndarray
    scale: np.ndarray | None
    bt: np.ndarray
    rows_per_block: int

    def copy(self) -> "Paged":
        return Paged(self.data.copy(), None if self.scale is None else self.scale.copy(),
                     self.bt.copy(), self.rows_per_block)


@dataclass
class Batch:
    """New tokens of a step: sequence b owns rows cu[b]:cu[b+1] at positions start[b]+i."""
    cu: np.ndarray          # [n_seq+1] int32
    start: np.ndarray       # [n_seq] int64
    kv: np.ndarray          # [T, D]
    s: np.ndarray           # [T, D]
    ik: np.ndarray | None   # [T, d_I]
    is_: np.ndarray | None  # [T, d_I]


@dataclass
class Queries:
    seq: np.ndarray         # [n_q] int32
    pos: np.ndarray         # [n_q] int64
    q: np.ndarray           # [n_q, H, D]
    q_idx: np.ndarray | None  # [n_q, H_I, d_I]
    w: np.ndarray | None      # [n_q, H_I]


@dataclass
class Layer:
    spec: LayerSpec
    bias: np.ndarray        # [W, D] float32
    gamma: np.ndarray       # [D] float32
    ibias: np.ndarray | None  # [W, d_I] float32
    attn: Paged             # compressed entries (64 or 2 per block)
    idx: Paged | None       # indexer keys (c4a)
    swa: Paged              # token-granular sliding-window keys
    state: Paged            # token-granular raw residual (kv, s, ik, is)


@dataclass
class Workload:
    name: str
    layers: list            # [Layer] (two for the mixed workload)
    batch: Batch            # new tokens (shared by all layers)
    queries: Queries
    meta: dict = field(default_factory=dict)


# ----------------------------------------------------------------------------- draws

def _round(x: np.ndarray, fp8: bool) -> np.ndarray:
    """Round fp64 draws to the storage dtype of the inputs (bf16 or fp32), kept as float32."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if fp8:
        t = t.to(torch.bfloat16).to(torch.float32)
    return t.numpy()


def random_fp8_rows(rng: np.random.Generator, n: int, width: int):
    """n random fp8 rows: (codes uint8 [n, width], scales float32 [n])."""
    scale = (rng.uniform(0.5, 1.5, size=n) / 64.0).astype(np.float32)
    codes = np.empty((n, width), dtype=np.uint8)
    chunk = max(1, (1 << 24) // max(width, 1))
    for a in range(0, n, chunk):
        b = min(n, a + chunk)
        v = rng.standard_normal((b - a, width)) / scale[a:b, None].astype(np.float64)
        v = np.clip(v, -E4M3_MAX, E4M3_MAX).astype(np.float32)
        codes[a:b] = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return codes, scale


def random_fp4_rows(rng: np.random.Generator, n: int, width: int):
    """n random rows of 4-bit codes, two per byte (element 2i in the low nibble):
    (packed uint8 [n, width / 2], scales float32 [n]). Magnitude codes 0..7 are drawn
    with weights that roughly follow a rounded normal, signs uniformly."""
    scale = (rng.uniform(0.5, 1.5, size=n) / 3.0).astype(np.float32)
    w = np.array([0.10, 0.18, 0.17, 0.15, 0.13, 0.14, 0.08, 0.05])
    mag = rng.choice(8, size=(n, width), p=w / w.sum()).astype(np.uint8)
    codes = mag | (rng.integers(0, 2, size=(n, width), dtype=np.uint8) << 3)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8), scale


def block_table(rng: np.random.Generator, need: list, max_blocks: int):
    """Assign physical pages to the logical blocks listed in need[b] (a set of block ids).

    Pages are a seeded permutation of 0..n_pages-1, so consecutive logical blocks land
    at scattered physical pages. Returns (bt [n_seq, max_blocks] int32, n_pages).
    """
    n_pages = sum(len(x) for x in need)
    perm = rng.permutation(n_pages).astype(np.int32)
    bt = np.full((len(need), max_blocks), -1, dtype=np.int32)
    k = 0
    for b, blocks in enumerate(need):
        for blk in sorted(blocks):
            bt[b, blk] = perm[k]
            k += 1
    return bt, n_pages


def _empty_pool(spec: LayerSpec, rows: int, width: int, fp8_codes: bool):
    if fp8_codes:
        return np.zeros((rows, width), np.uint8), np.ones(rows, np.float32)
    return np.zeros((rows, width), np.float32), None


def layer_params(rng, spec: LayerSpec):
    bias = rng.normal(0.0, 0.5, size=(spec.W, spec.D)).astype(np.float32)
    gamma = rng.normal(1.0, 0.1, size=spec.D).astype(np.float32)
    ibias = (rng.normal(0.0, 0.5, size=(spec.W, spec.d_I)).astype(np.float32)
             if spec.has_indexer else None)
    return bias, gamma, ibias


def entries_complete(spec: LayerSpec, n_tokens: int) -> int:
    """Number of entries whose whole window lies in positions [0, n_tokens).

    Pure counting of the layout (entry j's last covered position is S*j+win_off+W-1);
    used only to size pre-filled pools.
    """
    last = n_tokens - 1 - (spec.win_off + spec.W - 1)
    return 0 if last < 0 else last // spec.S + 1


# ------------------------------------------------------------------------ workloads

def make_layer(rng, spec: LayerSpec, ctx: list, new: list, prefill_cache: bool,
               extra_entry_blocks: int = 1) -> Layer:
    """Pools and block tables for n_seq sequences.

    ctx[b]:  tokens already processed before this step (positions 0..ctx[b]-1).
    new[b]:  tokens arriving in this step (positions ctx[b]..ctx[b]+new[b]-1).
    prefill_cache: fill entries / SWA / residual of the context with random contents.
    """
    n_seq = len(ctx)
    R = spec.rows_per_block
    ends = [c + n for c, n in zip(ctx, new)]
    max_blocks = max(1, max((e + BLOCK - 1) // BLOCK for e in ends) + extra_entry_blocks)
    # compressed-entry blocks: every block up to the one holding the last native position
    need_e = [set(range((e + BLOCK - 1) // BLOCK + 1)) & set(range(max_blocks)) for e in ends]
    # token-granular pools: only blocks touching the SWA / residual windows
    lo_t = [max(0, c - max(spec.swa, spec.W)) for c in ctx]
    need_t = [set(range(l // BLOCK, (e - 1) // BLOCK + 1)) if e > 0 else set()
              for l, e in zip(lo_t, ends)]
    bt_e, np_e = block_table(rng, need_e, max_blocks)
    bt_t, np_t = block_table(rng, need_t, max_blocks)
    attn_d, attn_s = _empty_pool(spec, np_e * R, spec.D, spec.fp8)
    idx_d = idx_s = None
    if spec.has_indexer:
        idx_d, idx_s = _empty_pool(spec, np_e * R, spec.d_I // 2 if spec.idx_fp4 else spec.d_I,
                                   spec.fp8)
    swa_d, swa_s = _empty_pool(spec, np_t * BLOCK, spec.D, spec.fp8)
    st_d = np.zeros((np_t * BLOCK, spec.state_width), np.float32)
    bias, gamma, ibias = (None, None, None)
    layer = Layer(spec, bias, gamma, ibias,
                  Paged(attn_d, attn_s, bt_e, R),
                  Paged(idx_d, idx_s, bt_e.copy(), R) if spec.has_indexer else None,
                  Paged(swa_d, swa_s, bt_t, BLOCK),
                  Paged(st_d, None, bt_t.copy(), BLOCK))
    if prefill_cache:
        for b in range(n_seq):
            ne = entries_complete(spec, ctx[b])
            rows = _rows(bt_e[b], R, np.arange(ne))
            if spec.fp8:
                c, s = random_fp8_rows(rng, ne, spec.D)
                layer.attn.data[rows], layer.attn.scale[rows] = c, s
                if spec.has_indexer:
                    c, s = (random_fp4_rows if spec.idx_fp4 else random_fp8_rows)(rng, ne, spec.d_I)
                    layer.idx.data[rows], layer.idx.scale[rows] = c, s
            else:
                layer.attn.data[rows] = rng.standard_normal((ne, spec.D))
                if spec.has_indexer:
                    layer.idx.data[rows] = rng.standard_normal((ne, spec.d_I))
            # SWA rows of the last swa-1 context tokens, residual rows of the last W
            t_swa = np.arange(max(0, ctx[b] - spec.swa + 1), ctx[b])
            rows = _rows(bt_t[b], BLOCK, t_swa)
            if spec.fp8:
                c, s = random_fp8_rows(rng, len(t_swa), spec.D)
                layer.swa.data[rows], layer.swa.scale[rows] = c, s
            else:
                layer.swa.data[rows] = rng.standard_normal((len(t_swa), spec.D))
            t_st = np.arange(max(0, ctx[b] - spec.W), ctx[b])
            rows = _rows(bt_t[b], BLOCK, t_st)
            layer.state.data[rows] = _round(rng.standard_normal((len(t_st), spec.state_width)),
                                            spec.fp8)
    return layer


def _rows(bt_row: np.ndarray, R: int, idx: np.ndarray) -> np.ndarray:
    """Pool rows of logical rows idx (generator-side bookkeeping for pre-filling)."""
    pages = bt_row[idx // R]
    assert (pages >= 0).all(), "pre-fill needs allocated blocks"
    return pages.astype(np.int64) * R + idx % R


def make_batch(rng, spec: LayerSpec, ctx: list, new: list) -> Batch:
    T = int(sum(new))
    cu = np.zeros(len(new) + 1, np.int32)
    cu[1:] = np.cumsum(new)
    kv = _round(rng.standard_normal((T, spec.D)), spec.fp8)
    s = _round(rng.standard_normal((T, spec.D)), spec.fp8)
    ik = is_ = None
    if spec.has_indexer:
        ik = _round(rng.standard_normal((T, spec.d_I)), spec.fp8)
        is_ = _round(rng.standard_normal((T, spec.d_I)), spec.fp8)
    return Batch(cu, np.asarray(ctx, np.int64), kv, s, ik, is_)


def make_queries(rng, spec: LayerSpec, seq: np.ndarray, pos: np.ndarray,
                 w_uniform: bool, idx_spec: LayerSpec | None = None) -> Queries:
    n = len(seq)
    q = _round(rng.standard_normal((n, spec.H, spec.D)), spec.fp8).reshape(n, spec.H, spec.D)
    ispec = idx_spec or spec
    q_idx = w = None
    if ispec.has_indexer:
        q_idx = _round(rng.standard_normal((n, ispec.H_I, ispec.d_I)), ispec.fp8)
        q_idx = q_idx.reshape(n, ispec.H_I, ispec.d_I)
        w = (rng.uniform(0.0, 1.0, size=(n, ispec.H_I)) if w_uniform
             else rng.standard_normal((n, ispec.H_I))).astype(np.float32)
    return Queries(np.asarray(seq, np.int32), np.asarray(pos, np.int64), q, q_idx, w)


def tiny_prefill(seed: int = 0, L: int = 1024, **over) -> Workload:
    """Tiny fp32 c4a layer, one sequence of L tokens, every position queried.

    H=8, D=128 (32 rotated), indexer 4 heads x 32, top-64, SWA 128, w ~ U(0,1).
    """
    spec = replace(LayerSpec("c4a", False, D=128, d_r=32, H=8, H_I=4, d_I=32, top_k=64), **over)
    rng = np.random.default_rng(seed)
    bias, gamma, ibias = layer_params(rng, spec)
    layer = make_layer(rng, spec, [0], [L], prefill_cache=False)
    layer.bias, layer.gamma, layer.ibias = bias, gamma, ibias
    batch = make_batch(rng, spec, [0], [L])
    qs = make_queries(rng, spec, np.zeros(L, np.int32), np.arange(L), w_uniform=True)
    return Workload("tiny fp32 c4a prefill L=%d" % L, [layer], batch, qs)


def c4a_decode(seed: int = 1, B: int = 32, L: int = 32768, **over) -> Workload:
    """c4a decode: B sequences of L context tokens, one new token + query at position L."""
    spec = replace(LayerSpec("c4a", True), **over)
    rng = np.random.default_rng(seed)
    bias, gamma, ibias = layer_params(rng, spec)
    layer = make_layer(rng, spec, [L] * B, [1] * B, prefill_cache=True)
    layer.bias, layer.gamma, layer.ibias = bias, gamma, ibias
    batch = make_batch(rng, spec, [L] * B, [1] * B)
    qs = make_queries(rng, spec, np.arange(B), np.full(B, L), w_uniform=False)
    return Workload("c4a decode B=%d L=%d" % (B, L), [layer], batch, qs)


def c128a_decode(seed: int = 2, B: int = 8, L: int = 1 << 20, **over) -> Workload:
    """c128a dense decode: B sequences of L context tokens, one new token + query at L."""
    spec = replace(LayerSpec("c128a", True), **over)
    rng = np.random.default_rng(seed)
    bias, gamma, _ = layer_params(rng, spec)
    layer = make_layer(rng, spec, [L] * B, [1] * B, prefill_cache=True)
    layer.bias, layer.gamma = bias, gamma
    batch = make_batch(rng, spec, [L] * B, [1] * B)
    qs = make_queries(rng, spec, np.arange(B), np.full(B, L), w_uniform=False)
    return Workload("c128a decode B=%d L=%d" % (B, L), [layer], batch, qs)


def c4a_prefill(seed: int = 3, cached: int = 122880, chunk: int = 8192, **over) -> Workload:
    """c4a chunked prefill: one sequence with `cached` tokens, a new chunk of `chunk` tokens,
    every chunk position queried."""
    spec = replace(LayerSpec("c4a", True), **over)
    rng = np.random.default_rng(seed)
    bias, gamma, ibias = layer_params(rng, spec)
    layer = make_layer(rng, spec, [cached], [chunk], prefill_cache=True)
    layer.bias, layer.gamma, layer.ibias = bias, gamma, ibias
    batch = make_batch(rng, spec, [cached], [chunk])
    qs = make_queries(rng, spec, np.zeros(chunk, np.int32), cached + np.arange(chunk),
                      w_uniform=False)
    return Workload("c4a prefill cached=%d chunk=%d" % (cached, chunk), [layer], batch, qs)


def mixed_lengths(seed: int, B: int, lo: int = 4096, span: float = 256.0):
    """Context lengths L_b = floor(lo * span**u), u ~ U[0,1) (log-uniform in [lo, lo*span))."""
    rng = np.random.default_rng(seed)
    u = rng.uniform(0.0, 1.0, size=B)
    return [int(math.floor(lo * span ** x)) for x in u], rng


def mixed_decode(seed: int = 4, B: int = 64, lo: int = 4096, span: float = 256.0,
                 **over) -> Workload:
    """Mixed variable-length decode through one c4a and one c128a layer.

    Lengths are log-uniform in [lo, lo*span); each sequence gets one new token and one
    query at its length. Each layer keeps its own pools; the partial compressor window
    of every sequence sits in the residual pool.
    """
    lens, rng = mixed_lengths(seed, B, lo, span)
    s4 = replace(LayerSpec("c4a", True), **over)
    s128 = replace(LayerSpec("c128a", True), **over)
    layers = []
    for spec in (s4, s128):
        bias, gamma, ibias = layer_params(rng, spec)
        layer = make_layer(rng, spec, lens, [1] * B, prefill_cache=True)
        layer.bias, layer.gamma, layer.ibias = bias, gamma, ibias
        layers.append(layer)
    batch = make_batch(rng, s4, lens, [1] * B)
    qs = make_queries(rng, s4, np.arange(B), np.asarray(lens), w_uniform=False)
    return Workload("mixed decode B=%d" % B, layers, batch, qs, meta={"lens": lens})
