"""Device-resident layer state and the per-step call sequence, on top of the C ABI.

torch owns the device memory (pools, block tables, workspaces) and the stream; every
computation is one of the four library calls. ``from_host`` copies host arrays (numpy)
describing a layer's parameters and pools to the device.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import (BF16_FP8, C4A, C128A, FP32, IDX_DEFAULT, IDX_FP4, cache, layer_cfg,
               v4a_attn_decode,
               v4a_attn_decode_q8, v4a_attn_q8_workspace_size,
               v4a_attn_prefill, v4a_attn_workspace_size, v4a_compress_insert,
               v4a_compress_insert_qnorm,
               v4a_index_scores, v4a_index_scores_row_stride, v4a_index_topk,
               v4a_index_topk_workspace_size)


def _t(x, dtype, device):
    return torch.from_numpy(np.ascontiguousarray(x)).to(device=device, dtype=dtype)


@dataclass
class PagedPool:
    data: torch.Tensor
    scale: torch.Tensor | None
    block_table: torch.Tensor
    rows_per_block: int
    elems_per_byte: int = 1      # 2 for packed fp4 rows

    @property
    def c(self):
        return cache(self.data, self.scale, self.block_table, self.rows_per_block,
                     self.elems_per_byte)

    def clone(self) -> "PagedPool":
        return PagedPool(self.data.clone(), None if self.scale is None else self.scale.clone(),
                         self.block_table.clone(), self.rows_per_block, self.elems_per_byte)


def pool_from_host(p, elem_dtype, device, elems_per_byte=1) -> PagedPool:
    if p.data.dtype == np.uint8:
        data = torch.from_numpy(np.ascontiguousarray(p.data)).to(device)
    else:
        data = _t(p.data, elem_dtype, device)
    scale = None if p.scale is None else _t(p.scale, torch.float32, device)
    return PagedPool(data, scale, _t(p.bt, torch.int32, device), p.rows_per_block,
                     elems_per_byte)


class Layer:
    """One attention layer on the device: config, compressor parameters, four pools."""

    def __init__(self, cfg, bias, gamma, ibias, attn: PagedPool, idx: PagedPool | None,
                 swa: PagedPool, state: PagedPool, top_k: int = 0):
        self.cfg, self.bias, self.gamma, self.ibias = cfg, bias, gamma, ibias
        self.attn, self.idx, self.swa, self.state = attn, idx, swa, state
        self.top_k = top_k
        self.in_dtype = torch.bfloat16 if cfg.dtype == BF16_FP8 else torch.float32
        self._ws = {}

    @staticmethod
    def from_host(h, device="cuda") -> "Layer":
        """h: object with spec (kind, fp8, D, d_r, H, H_I, d_I, W, S, win_off, swa, rope_base,
        eps, scale, top_k), bias, gamma, ibias and paged pools attn, idx, swa, state."""
        s = h.spec
        fp4 = bool(getattr(s, "idx_fp4", False))
        cfg = layer_cfg(C4A if s.kind == "c4a" else C128A, BF16_FP8 if s.fp8 else FP32, s.D,
                        s.d_r, s.H, s.H_I, s.d_I, s.W, s.S, s.win_off, s.swa, s.rope_base,
                        s.eps, s.scale, IDX_FP4 if fp4 else IDX_DEFAULT)
        in_dt = torch.bfloat16 if s.fp8 else torch.float32
        ib = None if h.ibias is None else _t(h.ibias, torch.float32, device)
        return Layer(cfg, _t(h.bias, torch.float32, device), _t(h.gamma, torch.float32, device),
                     ib, pool_from_host(h.attn, torch.float32, device),
                     None if h.idx is None else pool_from_host(h.idx, torch.float32, device,
                                                               2 if fp4 else 1),
                     pool_from_host(h.swa, torch.float32, device),
                     pool_from_host(h.state, in_dt, device),
                     s.top_k if s.kind == "c4a" else 0)

    def clone_pools(self) -> "Layer":
        return Layer(self.cfg, self.bias, self.gamma, self.ibias, self.attn.clone(),
                     None if self.idx is None else self.idx.clone(), self.swa.clone(),
                     self.state.clone(), self.top_k)

    def workspace(self, key, nbytes, device) -> torch.Tensor:
        ws = self._ws.get(key)
        if ws is None or ws.numel() < nbytes:
            ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
            self._ws[key] = ws
        return ws

    # -------------------------------------------------------------- library calls
    def compress_insert(self, cu, start, kv, s, ik=None, is_=None, dev_err=None, stream=None):
        idx_c = None if self.idx is None else self.idx.c
        v4a_compress_insert(self.cfg, cu.numel() - 1, kv.shape[0], cu, start, kv, s, self.bias,
                            self.gamma, ik, is_, self.ibias, self.attn.c, idx_c, self.swa.c,
                            self.state.c, dev_err, stream)

    def compress_insert_qnorm(self, cu, start, kv, s, ik, is_, q, q_gamma, q_out=None,
                              dev_err=None, stream=None):
        """Insert the new tokens and RMSNorm every query head row of q [n_q, H, D] in the
        same launch; returns q_out (a new tensor unless given; q itself normalises in place)."""
        if q_out is None:
            q_out = torch.empty_like(q)
        idx_c = None if self.idx is None else self.idx.c
        v4a_compress_insert_qnorm(self.cfg, cu.numel() - 1, kv.shape[0], cu, start, kv, s,
                                  self.bias, self.gamma, ik, is_, self.ibias, self.attn.c, idx_c,
                                  self.swa.c, self.state.c, q.shape[0], q, q_gamma, q_out,
                                  dev_err, stream)
        return q_out

    def index_topk(self, q_seq, q_pos, max_pos, q_idx, w, out=None, k=None, dev_err=None,
                   stream=None):
        k = k or self.top_k
        n_q = q_seq.numel()
        if out is None:
            out = torch.empty((n_q, k), dtype=torch.int32, device=q_seq.device)
        nb = v4a_index_topk_workspace_size(self.cfg, n_q, max_pos)
        ws = self.workspace("index", nb, q_seq.device)
        v4a_index_topk(self.cfg, n_q, q_seq, q_pos, max_pos, q_idx, w, self.idx.c, k, out, ws,
                       dev_err, stream)
        return out

    def index_scores(self, q_seq, q_pos, max_pos, q_idx, w, dev_err=None, stream=None):
        """Indexer score rows alone: fp32 [n_q, row stride]; row i is valid up to the
        number of entries visible at q_pos[i]."""
        n_q = q_seq.numel()
        stride = v4a_index_scores_row_stride(self.cfg, max_pos)
        out = torch.empty((n_q, max(stride, 4)), dtype=torch.float32, device=q_seq.device)
        v4a_index_scores(self.cfg, n_q, q_seq, q_pos, max_pos, q_idx, w, self.idx.c, out,
                         dev_err, stream)
        return out

    def attention(self, q_seq, q_pos, max_pos, q, topk=None, k=0, out=None, prefill=False,
                  dev_err=None, stream=None):
        n_q = q_seq.numel()
        if out is None:
            out = torch.empty_like(q)
        k = k if topk is None else topk.shape[1]
        nb = v4a_attn_workspace_size(self.cfg, n_q, max_pos, k if topk is not None else 0,
                                     prefill)
        ws = self.workspace("attn_p" if prefill else "attn_d", nb, q_seq.device)
        fn = v4a_attn_prefill if prefill else v4a_attn_decode
        fn(self.cfg, n_q, q_seq, q_pos, max_pos, q, topk, k, self.attn.c, self.swa.c, out, ws,
           dev_err, stream)
        return out

    def attention_q8(self, q_seq, q_pos, max_pos, q, topk=None, k=0, dev_err=None, stream=None):
        """Decode attention with an fp8 output: (e4m3 codes [n_q, H, D] uint8, scales [n_q, H])."""
        n_q = q_seq.numel()
        k = k if topk is None else topk.shape[1]
        codes = torch.empty(q.shape, dtype=torch.uint8, device=q.device)
        scale = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
        nb = v4a_attn_q8_workspace_size(self.cfg, n_q, max_pos, k if topk is not None else 0)
        ws = self.workspace("attn_q8", nb, q_seq.device)
        v4a_attn_decode_q8(self.cfg, n_q, q_seq, q_pos, max_pos, q, topk, k, self.attn.c,
                           self.swa.c, codes, scale, ws, dev_err, stream)
        return codes, scale

    def step(self, cu, start, kv, s, ik, is_, q_seq, q_pos, max_pos, q, q_idx=None, w=None,
             out=None, prefill=False, dev_err=None, stream=None, side_stream=None,
             topk_out=None):
        """One pass of the layer: insert the new tokens, select (c4a), attend.

        side_stream (c4a decode): the insert runs there while the indexer and top-k run on
        `stream`; attention waits for both. This is valid only when no query of the call can
        see an entry completed by the call's own tokens, i.e. every new token of a sequence
        sits at or after the positions of that sequence's queries (decode: one token at the
        query's own position). An entry completed by the token at t covers t, and a query
        at p sees only entries whose positions are all below p.
        """
        main = stream if stream is not None else torch.cuda.current_stream()
        topk = None
        if side_stream is not None and self.cfg.kind == C4A and not prefill:
            side_stream.wait_stream(main)
            topk = self.index_topk(q_seq, q_pos, max_pos, q_idx, w, out=topk_out,
                                   dev_err=dev_err, stream=main)
            self.compress_insert(cu, start, kv, s, ik, is_, dev_err, side_stream)
            main.wait_stream(side_stream)
        else:
            self.compress_insert(cu, start, kv, s, ik, is_, dev_err, main)
            if self.cfg.kind == C4A:
                topk = self.index_topk(q_seq, q_pos, max_pos, q_idx, w, out=topk_out,
                                       dev_err=dev_err, stream=main)
        return self.attention(q_seq, q_pos, max_pos, q, topk, out=out, prefill=prefill,
                              dev_err=dev_err, stream=main), topk
