"""v4a: one layer of DeepSeek-V4-style hybrid compressed attention on GB300 (sm_103a).

Python binding of ``libv4a.so`` (the C ABI declared in ``include/v4a.h``). The functions
below carry the C names and only marshal arguments: torch tensors become device
pointers, the current torch stream becomes the CUDA stream. Every step of the layer runs
in the library's CUDA kernels; there is no other implementation to fall back to, and
importing this package fails if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "V4AError", "LayerCfg", "Cache", "library", "layer_cfg", "cache",
    "v4a_compress_insert", "v4a_compress_insert_qnorm", "v4a_index_topk", "v4a_index_topk_workspace_size",
    "v4a_index_scores", "v4a_index_scores_row_stride", "v4a_index_topk_noalloc",
    "v4a_index_topk_noalloc_capacity",
    "v4a_attn_decode", "v4a_attn_prefill", "v4a_attn_workspace_size", "v4a_slot_mapping",
    "v4a_attn_decode_q8", "v4a_attn_q8_workspace_size", "v4a_attn_plan",
    "v4a_get_error", "v4a_version",
    "C4A", "C128A", "FP32", "BF16_FP8", "IDX_DEFAULT", "IDX_FP4", "DEV_MISSING_PAGE", "DEV_BAD_PAGE", "DEV_BAD_INDEX", "DEV_BAD_POS",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libv4a.so")

C4A, C128A = 0, 1
FP32, BF16_FP8 = 0, 1
IDX_DEFAULT, IDX_FP4 = 0, 1
OK, ERR_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE, ERR_TOO_LARGE = 0, -1, -2, -3, -4, -5
DEV_MISSING_PAGE, DEV_BAD_PAGE, DEV_BAD_INDEX, DEV_BAD_POS = 1, 2, 4, 8
_NAMES = {ERR_ARG: "V4A_ERR_ARG", ERR_UNSUPPORTED: "V4A_ERR_UNSUPPORTED",
          ERR_CUDA: "V4A_ERR_CUDA", ERR_DEVICE: "V4A_ERR_DEVICE",
          ERR_TOO_LARGE: "V4A_ERR_TOO_LARGE"}


class V4AError(RuntimeError):
    def __init__(self, fn: str, code: int, flags: int = 0):
        super().__init__("%s returned %s (%d)%s" % (fn, _NAMES.get(code, "?"), code,
                                                    " flags=0x%x" % flags if flags else ""))
        self.code, self.flags = code, flags


class LayerCfg(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("rope_dim", ctypes.c_int32),
                ("n_heads", ctypes.c_int32), ("idx_heads", ctypes.c_int32),
                ("idx_dim", ctypes.c_int32), ("window", ctypes.c_int32),
                ("stride", ctypes.c_int32), ("win_off", ctypes.c_int32),
                ("swa", ctypes.c_int32), ("rope_base", ctypes.c_float),
                ("rms_eps", ctypes.c_float), ("softmax_scale", ctypes.c_float),
                ("idx_format", ctypes.c_int32)]


class Cache(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("max_blocks", ctypes.c_int32),
                ("rows_per_block", ctypes.c_int32), ("n_pages", ctypes.c_int64),
                ("row_width", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_P = ctypes.c_void_p
_I32, _I64, _SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_CFG, _CACHE = ctypes.POINTER(LayerCfg), ctypes.POINTER(Cache)

_SIGS = {
    "v4a_version": (_I32, []),
    "v4a_compress_insert": (ctypes.c_int, [_CFG, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                                           _CACHE, _CACHE, _CACHE, _CACHE, _P, _P]),
    "v4a_compress_insert_qnorm": (ctypes.c_int, [_CFG, _I32, _I32, _P, _P, _P, _P, _P, _P, _P,
                                                 _P, _P, _CACHE, _CACHE, _CACHE, _CACHE, _I32,
                                                 _P, _P, _P, _P, _P]),
    "v4a_index_topk_workspace_size": (_SZ, [_CFG, _I32, _I64]),
    "v4a_index_topk": (ctypes.c_int, [_CFG, _I32, _P, _P, _I64, _P, _P, _CACHE, _I32, _P, _P,
                                      _SZ, _P, _P]),
    "v4a_attn_workspace_size": (_SZ, [_CFG, _I32, _I64, _I32, _I32]),
    "v4a_attn_plan": (ctypes.c_int, [_CFG, _I32, _I64, _I32, _I32, ctypes.POINTER(_I32),
                                     ctypes.POINTER(_I32)]),
    "v4a_attn_decode": (ctypes.c_int, [_CFG, _I32, _P, _P, _I64, _P, _P, _I32, _CACHE, _CACHE,
                                       _P, _P, _SZ, _P, _P]),
    "v4a_attn_prefill": (ctypes.c_int, [_CFG, _I32, _P, _P, _I64, _P, _P, _I32, _CACHE, _CACHE,
                                        _P, _P, _SZ, _P, _P]),
    "v4a_slot_mapping": (ctypes.c_int, [_CACHE, _I32, _P, _P, _P, _P, _P]),
    "v4a_attn_q8_workspace_size": (_SZ, [_CFG, _I32, _I64, _I32]),
    "v4a_attn_decode_q8": (ctypes.c_int, [_CFG, _I32, _P, _P, _I64, _P, _P, _I32, _CACHE, _CACHE,
                                          _P, _P, _P, _SZ, _P, _P]),
    "v4a_index_scores_row_stride": (_I64, [_CFG, _I64]),
    "v4a_index_scores": (ctypes.c_int, [_CFG, _I32, _P, _P, _I64, _P, _P, _CACHE, _P, _SZ, _P,
                                        _P]),
    "v4a_index_topk_noalloc_capacity": (_SZ, []),
    "v4a_index_topk_noalloc": (ctypes.c_int, [_CFG, _I32, _P, _P, _I64, _P, _P, _CACHE, _I32,
                                              _P, _P, _P]),
    "v4a_get_error": (ctypes.c_int, [_P, _P, ctypes.POINTER(_I32)]),
}

_lib = None


def library() -> ctypes.CDLL:
    """Load libv4a.so (built in-tree by ``compressed_sparse_long_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libv4a.so is not built (%s); run "
                              "`python -m compressed_sparse_long_gb300.build`. There is no "
                              "fallback implementation." % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
    return _lib


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if t.numel() and not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _check(fn: str, rc: int):
    if rc != OK:
        raise V4AError(fn, rc)


def layer_cfg(kind: int, dtype: int, head_dim: int, rope_dim: int, n_heads: int,
              idx_heads: int, idx_dim: int, window: int, stride: int, win_off: int = 0,
              swa: int = 128, rope_base: float = 10000.0, rms_eps: float = 1e-6,
              softmax_scale: float | None = None, idx_format: int = 0) -> LayerCfg:
    return LayerCfg(kind, dtype, head_dim, rope_dim, n_heads, idx_heads, idx_dim, window,
                    stride, win_off, swa, rope_base, rms_eps,
                    softmax_scale if softmax_scale else head_dim ** -0.5, idx_format)


def cache(data: torch.Tensor, scale: torch.Tensor | None, block_table: torch.Tensor,
          rows_per_block: int, elems_per_byte: int = 1) -> Cache:
    """Describe a paged pool. The tensors must stay alive while the library uses them.
    elems_per_byte = 2 for a pool of packed fp4 rows (uint8 data, two elements a byte)."""
    assert data.dim() == 2 and block_table.dim() == 2 and block_table.dtype == torch.int32
    return Cache(data.data_ptr(), None if scale is None else scale.data_ptr(),
                 block_table.data_ptr(), block_table.shape[1], rows_per_block,
                 data.shape[0] // rows_per_block, data.shape[1] * elems_per_byte, 0)


def v4a_version() -> int:
    return library().v4a_version()


def v4a_compress_insert(cfg, n_seq, n_tokens, cu_tokens, start_pos, kv, score, bias, gamma,
                        ikv, iscore, ibias, attn, idx, swa, state, dev_err=None, stream=None):
    _check("v4a_compress_insert", library().v4a_compress_insert(
        ctypes.byref(cfg), n_seq, n_tokens, _ptr(cu_tokens), _ptr(start_pos), _ptr(kv),
        _ptr(score), _ptr(bias), _ptr(gamma), _ptr(ikv), _ptr(iscore), _ptr(ibias),
        ctypes.byref(attn), None if idx is None else ctypes.byref(idx), ctypes.byref(swa),
        ctypes.byref(state), _ptr(dev_err), _stream(stream)))


def _cref(c):
    return None if c is None else ctypes.byref(c)


def v4a_compress_insert_qnorm(cfg, n_seq, n_tokens, cu_tokens, start_pos, kv, score, bias,
                              gamma, ikv, iscore, ibias, attn, idx, swa, state, n_q, q, q_gamma,
                              q_out, dev_err=None, stream=None):
    _check("v4a_compress_insert_qnorm", library().v4a_compress_insert_qnorm(
        ctypes.byref(cfg), n_seq, n_tokens, _ptr(cu_tokens), _ptr(start_pos), _ptr(kv),
        _ptr(score), _ptr(bias), _ptr(gamma), _ptr(ikv), _ptr(iscore), _ptr(ibias),
        _cref(attn), _cref(idx), _cref(swa), _cref(state), n_q, _ptr(q), _ptr(q_gamma),
        _ptr(q_out), _ptr(dev_err), _stream(stream)))


def v4a_index_topk_workspace_size(cfg, n_q, max_pos) -> int:
    return library().v4a_index_topk_workspace_size(ctypes.byref(cfg), n_q, max_pos)


def v4a_index_topk(cfg, n_q, q_seq, q_pos, max_pos, q_idx, w, idx, k, topk_out, workspace,
                   dev_err=None, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("v4a_index_topk", library().v4a_index_topk(
        ctypes.byref(cfg), n_q, _ptr(q_seq), _ptr(q_pos), max_pos, _ptr(q_idx), _ptr(w),
        ctypes.byref(idx), k, _ptr(topk_out), _ptr(workspace), ws_bytes, _ptr(dev_err),
        _stream(stream)))


def v4a_index_scores_row_stride(cfg, max_pos) -> int:
    return library().v4a_index_scores_row_stride(ctypes.byref(cfg), max_pos)


def v4a_index_scores(cfg, n_q, q_seq, q_pos, max_pos, q_idx, w, idx, scores, dev_err=None,
                     stream=None):
    """Indexer score rows alone: scores [n_q, v4a_index_scores_row_stride(cfg, max_pos)] fp32."""
    nb = 0 if scores is None else scores.numel() * scores.element_size()
    _check("v4a_index_scores", library().v4a_index_scores(
        ctypes.byref(cfg), n_q, _ptr(q_seq), _ptr(q_pos), max_pos, _ptr(q_idx), _ptr(w),
        ctypes.byref(idx), _ptr(scores), nb, _ptr(dev_err), _stream(stream)))


def v4a_index_topk_noalloc_capacity() -> int:
    return library().v4a_index_topk_noalloc_capacity()


def v4a_index_topk_noalloc(cfg, n_q, q_seq, q_pos, max_pos, q_idx, w, idx, k, topk_out,
                           dev_err=None, stream=None):
    """v4a_index_topk for callers that cannot provide or allocate a workspace: the scores
    go to the library's fixed device scratch (see include/v4a.h for its limit and rules)."""
    _check("v4a_index_topk_noalloc", library().v4a_index_topk_noalloc(
        ctypes.byref(cfg), n_q, _ptr(q_seq), _ptr(q_pos), max_pos, _ptr(q_idx), _ptr(w),
        ctypes.byref(idx), k, _ptr(topk_out), _ptr(dev_err), _stream(stream)))


def v4a_attn_workspace_size(cfg, n_q, max_pos, k, prefill) -> int:
    return library().v4a_attn_workspace_size(ctypes.byref(cfg), n_q, max_pos, k, int(prefill))


def _attn(name, cfg, n_q, q_seq, q_pos, max_pos, q, topk, k, attn, swa, out, workspace,
          dev_err, stream):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(name, getattr(library(), name)(
        ctypes.byref(cfg), n_q, _ptr(q_seq), _ptr(q_pos), max_pos, _ptr(q), _ptr(topk), k,
        ctypes.byref(attn), ctypes.byref(swa), _ptr(out), _ptr(workspace), ws_bytes,
        _ptr(dev_err), _stream(stream)))


def v4a_attn_decode(cfg, n_q, q_seq, q_pos, max_pos, q, topk, k, attn, swa, out, workspace,
                    dev_err=None, stream=None):
    _attn("v4a_attn_decode", cfg, n_q, q_seq, q_pos, max_pos, q, topk, k, attn, swa, out,
          workspace, dev_err, stream)


def v4a_attn_q8_workspace_size(cfg, n_q, max_pos, k) -> int:
    return library().v4a_attn_q8_workspace_size(ctypes.byref(cfg), n_q, max_pos, k)


def v4a_attn_plan(cfg, n_q, max_pos, k, prefill=False):
    """(key ranges per query, kernels per call) of an attention call of this shape."""
    ns, nk = ctypes.c_int32(0), ctypes.c_int32(0)
    _check("v4a_attn_plan", library().v4a_attn_plan(ctypes.byref(cfg), n_q, max_pos, k,
                                                     int(prefill), ctypes.byref(ns),
                                                     ctypes.byref(nk)))
    return ns.value, nk.value


def v4a_attn_decode_q8(cfg, n_q, q_seq, q_pos, max_pos, q, topk, k, attn, swa, out_codes,
                       out_scale, workspace, dev_err=None, stream=None):
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("v4a_attn_decode_q8", library().v4a_attn_decode_q8(
        ctypes.byref(cfg), n_q, _ptr(q_seq), _ptr(q_pos), max_pos, _ptr(q), _ptr(topk), k,
        ctypes.byref(attn), ctypes.byref(swa), _ptr(out_codes), _ptr(out_scale), _ptr(workspace),
        ws_bytes, _ptr(dev_err), _stream(stream)))


def v4a_attn_prefill(cfg, n_q, q_seq, q_pos, max_pos, q, topk, k, attn, swa, out, workspace,
                     dev_err=None, stream=None):
    _attn("v4a_attn_prefill", cfg, n_q, q_seq, q_pos, max_pos, q, topk, k, attn, swa, out,
          workspace, dev_err, stream)


def v4a_slot_mapping(c, n, seq, row, slots, dev_err=None, stream=None):
    _check("v4a_slot_mapping", library().v4a_slot_mapping(
        ctypes.byref(c), n, _ptr(seq), _ptr(row), _ptr(slots), _ptr(dev_err), _stream(stream)))


def v4a_get_error(dev_err, stream=None) -> int:
    """Synchronise the stream, return and clear the device error bits."""
    flags = _I32(0)
    rc = library().v4a_get_error(_ptr(dev_err), _stream(stream), ctypes.byref(flags))
    if rc not in (OK, ERR_DEVICE):
        raise V4AError("v4a_get_error", rc)
    return flags.value
