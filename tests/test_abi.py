"""CPU-side checks of the C ABI: the library loads, exports every declared symbol, the
ctypes structs match the C layout, and host-side validation rejects bad arguments
without touching a GPU."""
import ctypes
import os
import re
import subprocess

import pytest

import compressed_sparse_long_gb300 as v4a

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "v4a.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(v4a_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(v4a.LIB_PATH):
        from compressed_sparse_long_gb300 import build
        build.build()
    return v4a.library()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "v4a_compress_insert" in names and "v4a_attn_prefill" in names
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", v4a.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r"\bT (v4a_\w+)", out))
    assert set(names) <= exported
    assert v4a.v4a_version() >= 1


def test_struct_layout_matches_c(tmp_path):
    prog = tmp_path / "layout.c"
    prog.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "v4a.h"\n'
                    'int main(void){printf("%zu %zu %zu %zu %zu %zu\\n", sizeof(v4a_layer_cfg),'
                    ' offsetof(v4a_layer_cfg, softmax_scale), sizeof(v4a_cache),'
                    ' offsetof(v4a_cache, n_pages), offsetof(v4a_cache, row_width),'
                    ' offsetof(v4a_cache, max_blocks)); return 0;}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(prog), "-o",
                    str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    want = [ctypes.sizeof(v4a.LayerCfg), v4a.LayerCfg.softmax_scale.offset,
            ctypes.sizeof(v4a.Cache), v4a.Cache.n_pages.offset, v4a.Cache.row_width.offset,
            v4a.Cache.max_blocks.offset]
    assert got == want


def _cfg(**kw):
    base = dict(kind=v4a.C4A, dtype=v4a.BF16_FP8, head_dim=512, rope_dim=64, n_heads=64,
                idx_heads=64, idx_dim=128, window=8, stride=4)
    base.update(kw)
    return v4a.layer_cfg(**base)


def test_host_validation_rejects_bad_arguments(lib):
    cfg = _cfg()
    c = v4a.Cache()
    null = ctypes.POINTER(v4a.LayerCfg)()
    # no config
    assert lib.v4a_compress_insert(null, 1, 1, 8, 8, 8, 8, 8, 8, 8, 8, 8, None, None, None, None,
                                   None, None) == v4a.ERR_ARG
    # zero tokens / queries: nothing to do
    assert lib.v4a_compress_insert(ctypes.byref(cfg), 1, 0, None, None, None, None, None, None,
                                   None, None, None, None, None, None, None, None, None) == v4a.OK
    assert lib.v4a_index_topk(ctypes.byref(cfg), 0, None, None, 0, None, None, ctypes.byref(c),
                              512, None, None, 0, None, None) == v4a.OK
    # missing pointers
    assert lib.v4a_attn_decode(ctypes.byref(cfg), 4, None, None, 100, None, None, 0,
                               ctypes.byref(c), ctypes.byref(c), None, None, 0, None,
                               None) == v4a.ERR_ARG
    # unsupported kind / odd rope dim / positive window offset
    assert lib.v4a_index_topk(ctypes.byref(_cfg(kind=7)), 1, 8, 8, 0, 16, 16, ctypes.byref(c),
                              1, 16, None, 0, None, None) == v4a.ERR_UNSUPPORTED
    assert lib.v4a_index_topk(ctypes.byref(_cfg(rope_dim=3)), 1, 8, 8, 0, 16, 16,
                              ctypes.byref(c), 1, 16, None, 0, None, None) == v4a.ERR_UNSUPPORTED
    assert lib.v4a_index_topk(ctypes.byref(_cfg(win_off=1)), 1, 8, 8, 0, 16, 16, ctypes.byref(c),
                              1, 16, None, 0, None, None) == v4a.ERR_ARG
    # fp8 output: bf16 layers only, and it needs the scale array
    assert lib.v4a_attn_decode_q8(ctypes.byref(_cfg(dtype=v4a.FP32)), 4, 8, 8, 100, 16, 16, 512,
                                  ctypes.byref(c), ctypes.byref(c), 16, 16, None, 0, None,
                                  None) == v4a.ERR_UNSUPPORTED
    assert lib.v4a_attn_decode_q8(ctypes.byref(_cfg(dtype=v4a.BF16_FP8)), 4, 8, 8, 100, 16, 16,
                                  512, ctypes.byref(c), ctypes.byref(c), 16, None, None, 0, None,
                                  None) == v4a.ERR_ARG
    assert v4a.v4a_attn_q8_workspace_size(_cfg(dtype=v4a.BF16_FP8), 4, 1000, 512) > 256
    # query norm: negative count, missing or misaligned buffers, partial overlap of q_out
    # and q (every case returns before anything is enqueued)
    qn = lib.v4a_compress_insert_qnorm
    n13 = [None] * 13
    assert qn(ctypes.byref(cfg), 0, 0, *n13, -1, 4096, 4096, 4096, None, None) == v4a.ERR_ARG
    assert qn(ctypes.byref(cfg), 0, 0, *n13, 1, None, 4096, 4096, None, None) == v4a.ERR_ARG
    assert qn(ctypes.byref(cfg), 0, 0, *n13, 1, 4104, 4096, 4104, None, None) == v4a.ERR_ARG
    assert qn(ctypes.byref(cfg), 0, 0, *n13, 1, 4096, 4100, 4096, None, None) == v4a.ERR_ARG
    assert qn(ctypes.byref(cfg), 0, 0, *n13, 1, 1 << 20, 4096, (1 << 20) + 1024, None,
              None) == v4a.ERR_ARG
    assert qn(ctypes.byref(cfg), 0, 0, *n13, 0, None, None, None, None, None) == v4a.OK
    # fp4 indexer cache: bf16/fp8 c4a layers with d_I = 128 only; unknown formats refused
    for bad in (_cfg(dtype=v4a.FP32, idx_format=v4a.IDX_FP4), _cfg(idx_format=v4a.IDX_FP4, idx_dim=64),
                _cfg(idx_format=7)):
        assert lib.v4a_index_topk(ctypes.byref(bad), 1, 8, 8, 0, 16, 16, ctypes.byref(c), 1, 16,
                                  None, 0, None, None) == v4a.ERR_UNSUPPORTED
    # the indexer exists only for c4a layers
    assert lib.v4a_index_topk(ctypes.byref(_cfg(kind=v4a.C128A, window=128, stride=128)), 1, 8,
                              8, 0, 16, 16, ctypes.byref(c), 1, 16, None, 0, None,
                              None) == v4a.ERR_UNSUPPORTED


def test_cache_descriptor_checks(lib):
    cfg = _cfg()
    bt = 256
    good = v4a.Cache(4096, 8192, bt, 4, 64, 10, 128, 0)
    bad_width = v4a.Cache(4096, 8192, bt, 4, 64, 10, 96, 0)
    misaligned = v4a.Cache(4100, 8192, bt, 4, 64, 10, 128, 0)
    no_scale = v4a.Cache(4096, None, bt, 4, 64, 10, 128, 0)
    for c, want in ((bad_width, v4a.ERR_ARG), (misaligned, v4a.ERR_ARG), (no_scale, v4a.ERR_ARG)):
        assert lib.v4a_index_topk(ctypes.byref(cfg), 1, 16, 16, 100, 4096, 16, ctypes.byref(c),
                                  4, 16, 4096, 1 << 20, None, None) == want
    # workspace too small is refused before any launch
    assert lib.v4a_index_topk(ctypes.byref(cfg), 1, 16, 16, 100, 4096, 16, ctypes.byref(good),
                              4, 16, 4096, 8, None, None) == v4a.ERR_ARG
    assert v4a.v4a_index_topk_workspace_size(cfg, 32, 32768) >= 32 * 8191 * 4


def test_workspace_sizes_are_monotone():
    cfg = _cfg()
    a = v4a.v4a_index_topk_workspace_size(cfg, 8, 4096)
    b = v4a.v4a_index_topk_workspace_size(cfg, 8, 8192)
    assert 0 < a < b
    assert v4a.v4a_attn_workspace_size(cfg, 8192, 131072, 512, 1) >= 256


def test_attention_split_plan_on_a_152_sm_gpu():
    """Host planning of decode attention (no device here: the planner assumes 152 SMs). A
    query's 512 selected rows + 128 window rows are 5 tiles of 128 keys; a plan costs
    waves x (tiles per range + 1) with one CTA per SM, the smallest split of least cost wins,
    and a split needs the merge kernel."""
    c4a = _cfg()
    assert v4a.v4a_attn_plan(c4a, 32, 32768, 512) == (3, 2)    # 5 ranges = 160 CTAs: 2 waves
    assert v4a.v4a_attn_plan(c4a, 64, 4096, 512) == (2, 2)     # 3 ranges = 192 CTAs: 2 waves
    assert v4a.v4a_attn_plan(c4a, 16, 4096, 512) == (5, 2)     # 80 CTAs: one tile each
    assert v4a.v4a_attn_plan(c4a, 160, 4096, 512) == (1, 1)    # more queries than SMs
    assert v4a.v4a_attn_plan(c4a, 0, 4096, 512) == (1, 0)      # nothing to launch
    assert v4a.v4a_attn_plan(c4a, 32, 32768, 512, True) == (1, 1)   # prefill never splits
    c128a = _cfg(kind=v4a.C128A, window=128, stride=128)
    # dense: 2^20 / 128 = 8192 compressed rows + 128 window rows = 65 tiles; with one wave
    # (up to 19 ranges for 8 queries) the cost is ceil(65 / r) + 1, least (5) first at r = 17:
    # 4 tiles (512 keys) a range, 17 ranges
    assert v4a.v4a_attn_plan(c128a, 8, 1 << 20, 0) == (17, 2)
    assert v4a.v4a_attn_plan(c128a, 8, 1 << 20, 0, True) == (1, 1)


def test_indexer_entry_points_share_their_host_checks(lib):
    """v4a_index_topk, v4a_index_topk_noalloc and v4a_index_scores run the same host checks:
    for each invalid configuration or cache descriptor they return the same code, and none
    of them enqueues anything (no GPU is touched here)."""
    c = v4a.Cache(4096, 8192, 256, 4, 64, 10, 128, 0)
    bad_cfgs = [_cfg(kind=7), _cfg(rope_dim=3), _cfg(win_off=1), _cfg(window=512),
                _cfg(head_dim=100), _cfg(swa=0), _cfg(rms_eps=-1.0),
                _cfg(rope_base=0.0), _cfg(idx_format=7), _cfg(dtype=v4a.FP32, idx_format=1),
                _cfg(kind=v4a.C128A, window=128, stride=128)]
    bad_caches = [v4a.Cache(4096, 8192, 256, 4, 64, 10, 96, 0),      # row width
                  v4a.Cache(4100, 8192, 256, 4, 64, 10, 128, 0),     # misaligned pool
                  v4a.Cache(4096, None, 256, 4, 64, 10, 128, 0),     # fp8 pool without scales
                  v4a.Cache(4096, 8192, 256, 4, 32, 10, 128, 0),     # rows per block
                  v4a.Cache(4096, 8192, 256, 4, 64, 10, 128, 1)]     # reserved field
    cases = [(cfg, c) for cfg in bad_cfgs] + [(_cfg(), bc) for bc in bad_caches]
    for cfg, cc in cases:
        a = lib.v4a_index_topk(ctypes.byref(cfg), 1, 16, 16, 100, 4096, 16, ctypes.byref(cc), 4,
                               16, 4096, 1 << 20, None, None)
        b = lib.v4a_index_topk_noalloc(ctypes.byref(cfg), 1, 16, 16, 100, 4096, 16,
                                       ctypes.byref(cc), 4, 16, None, None)
        s = lib.v4a_index_scores(ctypes.byref(cfg), 1, 16, 16, 100, 4096, 16, ctypes.byref(cc),
                                 4096, 1 << 20, None, None)
        assert a != v4a.OK and a == b == s, (cfg.kind, cfg.rope_dim, a, b, s)
    # misaligned query operands, and a non-positive k where the call selects
    for args in ((4100, 16, 4), (4096, 20, 4)):
        a = lib.v4a_index_topk(ctypes.byref(_cfg()), 1, 16, 16, 100, args[0], args[1],
                               ctypes.byref(c), args[2], 16, 4096, 1 << 20, None, None)
        b = lib.v4a_index_topk_noalloc(ctypes.byref(_cfg()), 1, 16, 16, 100, args[0], args[1],
                                       ctypes.byref(c), args[2], 16, None, None)
        assert a == b == v4a.ERR_ARG
    assert lib.v4a_index_topk_noalloc(ctypes.byref(_cfg()), 1, 16, 16, 100, 4096, 16,
                                      ctypes.byref(c), 0, 16, None, None) == v4a.ERR_ARG
    # the scores call checks the size of its output rows
    assert v4a.v4a_index_scores_row_stride(_cfg(), 32768) == 8192
    assert v4a.v4a_index_scores_row_stride(_cfg(), 100) == 24
    assert lib.v4a_index_scores(ctypes.byref(_cfg()), 2, 16, 16, 100, 4096, 16, ctypes.byref(c),
                                4096, 2 * 24 * 4 - 4, None, None) == v4a.ERR_ARG
    assert lib.v4a_index_scores(ctypes.byref(_cfg()), 2, 16, 16, 100, 4096, 16, ctypes.byref(c),
                                4100, 2 * 24 * 4, None, None) == v4a.ERR_ARG
