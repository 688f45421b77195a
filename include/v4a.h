/*
 * v4a — one layer of DeepSeek-V4-style hybrid compressed attention on one GB300 (sm_103a).
 *
 * C ABI of the library. Every call is asynchronous on the caller's CUDA stream, allocates
 * nothing, keeps no state between calls and may be called from several host threads.
 * All pointers named "device" point to device memory owned by the caller; the library
 * never frees or retains them after the call returns (the kernels it enqueued may still
 * be reading them until the stream reaches that point). Structs passed by pointer
 * (v4a_layer_cfg, v4a_cache) live in host memory and are copied during the call.
 *
 * Sources (page title, section):
 *   [notes] "DeepSeek V4 in vLLM 技术博客详尽笔记" (vllm-deepseek-v4-notes.pages.dev)
 *   [blog]  "vLLM DeepSeek V4 支援：高效長上下文注意力" (agentlenshq.com)
 *   [serve] "DeepSeek-V4服务：百万token上下文成为推理系统难题" (ai-pulse-lab.com)
 *
 * Paged layout ([notes] 解决方案一：统一逻辑块大小): every cache is split into logical
 * blocks of 256 native token positions. A block of a c4a entry cache holds 64 entries,
 * a block of a c128a entry cache holds 2 entries, a block of a token cache (sliding
 * window, compressor residual) holds 256 tokens. Row r of sequence b (a token position or
 * an entry index) lives in logical block r / R (R = rows per block), whose physical page
 * is block_table[b * max_blocks + r / R]; its pool row ("slot") is page * R + r % R.
 * A page of -1 means the block is not allocated.
 *
 * Error behaviour: every call first validates its host-visible arguments and returns
 * V4A_ERR_ARG or V4A_ERR_UNSUPPORTED without enqueuing anything. A failed launch returns
 * V4A_ERR_CUDA. Problems only the device can see (a needed row whose block has no page, a
 * page id outside the pool, a top-k entry that is not visible to its query) are OR-ed
 * into the caller's device error word `dev_err` (may be NULL to ignore them); the affected
 * row or query is skipped or zeroed, never read out of bounds. v4a_get_error() reads and
 * clears that word.
 */
#ifndef V4A_H
#define V4A_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* v4a_stream_t; /* a cudaStream_t; NULL = legacy default stream */

/* return codes */
#define V4A_OK 0
#define V4A_ERR_ARG (-1)          /* NULL pointer, misaligned pointer, inconsistent sizes */
#define V4A_ERR_UNSUPPORTED (-2)  /* dims / dtype / kind without a kernel */
#define V4A_ERR_CUDA (-3)         /* a CUDA launch or runtime call failed */
#define V4A_ERR_DEVICE (-4)       /* v4a_get_error found device-side error bits */
#define V4A_ERR_TOO_LARGE (-5)    /* the request exceeds the fixed scratch of v4a_index_topk_noalloc */

/* device error word bits */
#define V4A_DEV_MISSING_PAGE 1u   /* a row the computation needs is in a block with no page */
#define V4A_DEV_BAD_PAGE 2u       /* a block table names a page >= n_pages */
#define V4A_DEV_BAD_INDEX 4u      /* a top-k list names an entry its query may not see */
#define V4A_DEV_BAD_POS 8u        /* a query position above the max_pos the call was sized for;
                                     the query's rows beyond that bound are ignored */
#define V4A_DEV_TIMEOUT 16u       /* a bounded wait inside a kernel gave up (about 1 s); the
                                     kernel drained its copies, released its tensor memory and
                                     returned; its outputs are incomplete */

/* layer kinds ([notes] 四大核心技术; 数学附录精要) */
#define V4A_C4A 0                 /* entry = weighted sum of 8 tokens at stride 4 */
#define V4A_C128A 1               /* entry = weighted sum of 128 tokens at stride 128 */

/* arithmetic / storage */
#define V4A_FP32 0                /* fp32 inputs, fp32 caches, fp32 output */
#define V4A_BF16_FP8 1            /* bf16 inputs, fp8 e4m3 caches + fp32 row scale, bf16 output */

/* indexer-cache formats (v4a_layer_cfg.idx_format) */
#define V4A_IDX_DEFAULT 0         /* the layer's cache type: fp8 e4m3 (BF16_FP8) or fp32 (FP32) */
#define V4A_IDX_FP4 1             /* e2m1 codes, two per byte (element 2i in the low nibble), and
                                     one fp32 scale per row: scale = max|y| / 6 (1 for a zero row),
                                     code = round-to-nearest-even of y / scale saturated to +-6
                                     ([notes] 四大核心技术 and [blog] KV 快取記憶體管理: the fp4
                                     indexer cache; the block of one scale is the whole row).
                                     BF16_FP8 layers with d_I = 128 only. */

typedef struct v4a_layer_cfg {
  int32_t kind;          /* V4A_C4A or V4A_C128A */
  int32_t dtype;         /* V4A_FP32 or V4A_BF16_FP8 */
  int32_t head_dim;      /* D: dim of the shared K=V head and of each query head */
  int32_t rope_dim;      /* d_r: the last d_r dims are rotated, as adjacent pairs */
  int32_t n_heads;       /* H: query heads */
  int32_t idx_heads;     /* H_I: indexer heads (c4a) */
  int32_t idx_dim;       /* d_I: indexer head dim (c4a) */
  int32_t window;        /* W: tokens per entry (8 for c4a, 128 for c128a) */
  int32_t stride;        /* S: tokens between entries (4 / 128) */
  int32_t win_off;       /* entry j covers S*j+win_off .. S*j+win_off+W-1, win_off in (-W, 0] */
  int32_t swa;           /* sliding window: a query at p sees tokens [p-swa+1, p] */
  float rope_base;       /* theta_i = rope_base^(-2i/d_r) */
  float rms_eps;         /* RMSNorm epsilon of compressed entries */
  float softmax_scale;   /* logit scale, usually 1/sqrt(D) */
  int32_t idx_format;    /* V4A_IDX_DEFAULT or V4A_IDX_FP4 (c4a indexer cache) */
} v4a_layer_cfg;

typedef struct v4a_cache {
  void* data;                  /* device: [n_pages*rows_per_block, row_width] elements; e4m3
                                  bytes for fp8 pools, fp32 or bf16 for the others */
  float* scale;                /* device: [n_pages*rows_per_block] row scales (fp8 pools), else NULL */
  const int32_t* block_table;  /* device: [n_seq, max_blocks] physical page per logical block, -1 = none */
  int32_t max_blocks;          /* columns of block_table */
  int32_t rows_per_block;      /* 64 (c4a entries), 2 (c128a entries), 256 (token caches) */
  int64_t n_pages;             /* pages in the pool (bounds check of block-table values) */
  int32_t row_width;           /* elements per row (an fp4 row holds two per byte) */
  int32_t reserved;            /* must be 0 */
} v4a_cache;

/*
 * v4a_compress_insert — insert one step's new tokens of every sequence (steps a1-a5).
 *
 * [blog] GPU 計算飽和度 / [notes] 优化一：三大内核融合 (fusion 1: compressor + RMSNorm +
 * RoPE + cache insert; fusion 3's KV RoPE + K insert) and [notes] 解决方案二 (the compressor
 * state kept as sliding-window KV).
 *
 * Sequence b owns input rows cu_tokens[b] .. cu_tokens[b+1]-1 at positions
 * start_pos[b] + (row - cu_tokens[b]). For every new token t:
 *   - swa row t      = RoPE(kv_t, t), stored (fp8: per-row scale amax/448, e4m3 RNE);
 *   - state row t    = raw (kv_t | s_t | ik_t | is_t) if t is among the last W positions of
 *                      the sequence's new tokens (what later calls can still need);
 *   - if t completes entry j (t = S*j + win_off + W - 1, j >= 0):
 *       attn row j   = RoPE(RMSNorm(sum_o softmax_o(s + bias[o]) * kv) * gamma, S*j),
 *       idx row j    = sum_o softmax_o(is + ibias[o]) * ik (c4a only; no norm, no RoPE),
 *     where the window's tokens before start_pos[b] are read from the state cache.
 * Rows whose block has no page are not written (a needed state row without a page sets
 * V4A_DEV_MISSING_PAGE and the entry is skipped).
 *
 * kv, score:    device [n_tokens, D]    (fp32 or bf16 per cfg->dtype)
 * ikv, iscore:  device [n_tokens, d_I]  (c4a; NULL for c128a)
 * bias:         device fp32 [W, D];  gamma: device fp32 [D];  ibias: device fp32 [W, d_I] (c4a)
 * cu_tokens:    device int32 [n_seq+1], non-decreasing, cu_tokens[n_seq] == n_tokens
 * start_pos:    device int64 [n_seq]
 * attn:  entry cache (rows_per_block = 256/S, row_width = D)
 * idx:   indexer-key cache (c4a: rows_per_block 64, row_width d_I; NULL for c128a)
 * swa:   token cache (rows_per_block 256, row_width D)
 * state: token cache of raw rows (rows_per_block 256, row_width 2D (+2 d_I for c4a)),
 *        element type of the inputs.
 * Pool data pointers and kv, score, ikv, iscore, bias, gamma, ibias must be 16-byte
 * aligned (V4A_ERR_ARG otherwise).
 */
int v4a_compress_insert(const v4a_layer_cfg* cfg, int32_t n_seq, int32_t n_tokens,
                        const int32_t* cu_tokens, const int64_t* start_pos,
                        const void* kv, const void* score, const float* bias,
                        const float* gamma, const void* ikv, const void* iscore,
                        const float* ibias, const v4a_cache* attn, const v4a_cache* idx,
                        const v4a_cache* swa, const v4a_cache* state, int32_t* dev_err,
                        v4a_stream_t stream);

/*
 * v4a_compress_insert_qnorm — v4a_compress_insert plus the per-head query RMSNorm of the
 * step's queries, in the same launch.
 *
 * [notes] 优化一：三大内核融合, fusion 3 (Q Norm + KV RoPE + K Insert, static warp-ID
 * dispatch: every warp handles one Q head or one K row on its own). The launch's first
 * n_tokens warps do exactly what v4a_compress_insert does; each of the next n_q * H warps
 * takes one (query, head) row:
 *   q_out[i, h, :] = q_gamma * q[i, h, :] / sqrt(mean(q[i, h, :]^2) + cfg->rms_eps),
 * computed in fp32 and stored in the input type (bf16 round-to-nearest-even or fp32).
 *
 * n_q:      queries (>= 0); n_q = 0 makes the call v4a_compress_insert
 * q:        device [n_q, H, D] (fp32 or bf16 per cfg->dtype), 16-byte aligned
 * q_gamma:  device fp32 [D], 16-byte aligned, shared by the heads
 * q_out:    device [n_q, H, D], same type, 16-byte aligned; q_out == q normalises in place,
 *           any other overlap with q returns V4A_ERR_ARG
 * The insert arguments are checked only when n_tokens > 0, so n_tokens = 0 runs the norm
 * alone. Errors: as v4a_compress_insert, plus V4A_ERR_ARG for a NULL, misaligned or
 * partially overlapping query buffer.
 */
int v4a_compress_insert_qnorm(const v4a_layer_cfg* cfg, int32_t n_seq, int32_t n_tokens,
                              const int32_t* cu_tokens, const int64_t* start_pos,
                              const void* kv, const void* score, const float* bias,
                              const float* gamma, const void* ikv, const void* iscore,
                              const float* ibias, const v4a_cache* attn, const v4a_cache* idx,
                              const v4a_cache* swa, const v4a_cache* state, int32_t n_q,
                              const void* q, const float* q_gamma, void* q_out,
                              int32_t* dev_err, v4a_stream_t stream);

/*
 * v4a_index_topk — indexer scores and top-k selection of c4a entries (steps a6, a7).
 *
 * [blog] DeepSeek Sparse Attention (DSA) and [notes] 压缩参数细节 (C4A top-k 512).
 * For query i of sequence q_seq[i] at position p = q_pos[i], over the visible entries
 * j (every position S*j+win_off+o they cover is < p; [notes] 因果性条件):
 *   score_j = sum_h w[i,h] * max(0, q_idx[i,h,:] . k_j)
 * with k_j the dequantised indexer key. If at most k entries are visible, all are kept;
 * otherwise the k largest scores, ties to the smaller j. topk_out[i, :] lists the kept j
 * in ascending order, padded with -1.
 *
 * q_idx:    device [n_q, H_I, d_I] (fp32 or bf16)
 * w:        device fp32 [n_q, H_I]
 * q_seq:    device int32 [n_q];  q_pos: device int64 [n_q], every q_pos <= max_pos
 * topk_out: device int32 [n_q, k]
 * workspace: device, >= v4a_index_topk_workspace_size(...) bytes, 256-byte aligned.
 */
size_t v4a_index_topk_workspace_size(const v4a_layer_cfg* cfg, int32_t n_q, int64_t max_pos);
int v4a_index_topk(const v4a_layer_cfg* cfg, int32_t n_q, const int32_t* q_seq,
                   const int64_t* q_pos, int64_t max_pos, const void* q_idx, const float* w,
                   const v4a_cache* idx, int32_t k, int32_t* topk_out, void* workspace,
                   size_t workspace_bytes, int32_t* dev_err, v4a_stream_t stream);

/*
 * v4a_index_scores — the indexer scores alone (step a6), as v4a_index_topk computes them
 * before its selection ([blog] DeepSeek Sparse Attention: score_j = sum_h w_h ReLU(q_h . k_j)).
 * Same arguments and checks as v4a_index_topk without k and the output list. Row i of
 * `scores` holds score_j of query i in column j for every visible j (j < visible(q_pos[i]));
 * the other columns of the row are not written.
 *
 * scores:       device fp32 [n_q, v4a_index_scores_row_stride(cfg, max_pos)], 16-byte
 *               aligned, caller-owned; scores_bytes its size (V4A_ERR_ARG if too small)
 * row stride:   visible(max_pos) rounded up to a multiple of 4 floats (0 for a bad cfg)
 */
int64_t v4a_index_scores_row_stride(const v4a_layer_cfg* cfg, int64_t max_pos);
int v4a_index_scores(const v4a_layer_cfg* cfg, int32_t n_q, const int32_t* q_seq,
                     const int64_t* q_pos, int64_t max_pos, const void* q_idx, const float* w,
                     const v4a_cache* idx, float* scores, size_t scores_bytes, int32_t* dev_err,
                     v4a_stream_t stream);

/*
 * v4a_index_topk_noalloc — v4a_index_topk without a workspace argument, for callers that
 * cannot allocate device memory and have none to lend: for example a library embedded in
 * a framework or serving runtime that owns all device memory and gives its kernels no
 * scratch, or a code path where an allocation would synchronise the device or exceed a
 * memory budget fixed in advance. The pages have no counterpart to this call; it exists
 * for such callers only.
 *
 * Same arguments, meaning and results as v4a_index_topk, minus workspace and
 * workspace_bytes. The score rows live in a fixed 8 MiB array inside the library's device
 * image (held by every GPU that loads the library until the process exits), so
 * n_q * visible(max_pos), with visible(max_pos) rounded up to a multiple of 4 (score rows
 * start on 16-byte boundaries), must not exceed v4a_index_topk_noalloc_capacity() floats
 * (2,097,152; e.g. 64 queries at positions up to 131,072); larger requests return
 * V4A_ERR_TOO_LARGE without enqueuing anything. The call itself allocates nothing.
 * The first call on each device looks up the array's device address while that device
 * is current and keeps it for the life of the process; make that first call before any
 * stream capture. A device reset (cudaDeviceReset) unloads the library's device image and
 * makes the kept address invalid: do not call this entry point on a device after resetting
 * it. The host checks and their return codes are those of v4a_index_topk. All calls share the array
 * and it keeps the previous call's contents (each call writes every score it reads, so no
 * clearing is needed); calls that overlap on the GPU, e.g. on two unordered streams, race
 * on it and must be serialised by the caller.
 */
size_t v4a_index_topk_noalloc_capacity(void);
int v4a_index_topk_noalloc(const v4a_layer_cfg* cfg, int32_t n_q, const int32_t* q_seq,
                           const int64_t* q_pos, int64_t max_pos, const void* q_idx,
                           const float* w, const v4a_cache* idx, int32_t k, int32_t* topk_out,
                           int32_t* dev_err, v4a_stream_t stream);

/*
 * v4a_attn_decode / v4a_attn_prefill — shared-K=V attention with inverse RoPE (a8, a9).
 *
 * [notes] Inverse RoPE 的数学原理: out = (sum softmax(q K^T) V) R^-1(theta_p), K = V;
 * [blog] 短滑動窗口 (window of 128 uncompressed tokens).
 * For query i at p = q_pos[i] of sequence b = q_seq[i]:
 *   keys  = { attn row j : j in topk[i, :], j >= 0 }   (topk != NULL, c4a)
 *         | { attn row j : j visible at p }             (topk == NULL, dense, c128a)
 *         + { swa row t : max(0, p-swa+1) <= t <= p }
 *   out_h = R^-1(p) * sum_x softmax_x(scale * RoPE(q_h, p) . key_x) * key_x
 * Both calls compute the same function; decode splits each query's keys over several
 * CTAs (few queries, one per sequence), prefill gives each query one CTA (many queries).
 *
 * q:    device [n_q, H, D] (fp32 or bf16);  out: device [n_q, H, D] (fp32 or bf16)
 * topk: device int32 [n_q, k] or NULL
 * attn: entry cache;  swa: token cache
 * workspace: device, >= v4a_attn_workspace_size(...) bytes, 256-byte aligned.
 */
size_t v4a_attn_workspace_size(const v4a_layer_cfg* cfg, int32_t n_q, int64_t max_pos,
                               int32_t k, int32_t prefill);
int v4a_attn_decode(const v4a_layer_cfg* cfg, int32_t n_q, const int32_t* q_seq,
                    const int64_t* q_pos, int64_t max_pos, const void* q, const int32_t* topk,
                    int32_t k, const v4a_cache* attn, const v4a_cache* swa, void* out,
                    void* workspace, size_t workspace_bytes, int32_t* dev_err,
                    v4a_stream_t stream);
/* v4a_attn_plan — how v4a_attn_decode (prefill = 0) or v4a_attn_prefill (prefill = 1) of
 * this shape runs on the current device: *n_split = key ranges per query (1 = no split),
 * *n_kernels = kernels the call launches (0 for n_q = 0; 1, or 2 when a split is combined
 * by the merge kernel). Host only, enqueues nothing. Returns V4A_ERR_ARG for NULL outputs
 * or negative sizes. */
int v4a_attn_plan(const v4a_layer_cfg* cfg, int32_t n_q, int64_t max_pos, int32_t k,
                  int32_t prefill, int32_t* n_split, int32_t* n_kernels);

/* v4a_attn_decode_q8 — v4a_attn_decode whose epilogue also quantises the output for an fp8
 * output projection ([notes] 优化一, 融合 2：Inverse RoPE + FP8 Quant: the attention output goes
 * through the inverse RoPE and straight into an fp8 batched matmul; [blog] GPU 計算飽和度).
 *   out_codes  [n_q, H, D] e4m3 bytes, 16-byte aligned (caller-owned)
 *   out_scale  [n_q, H] fp32 (caller-owned)
 * Per (query, head) row y of R^-1(p) o_h: scale = max|y| / 448 (1 for a zero row) and
 * code = e4m3 round-to-nearest-even, saturating, of y / scale: the rule of the fp8 caches.
 * bf16 layers (V4A_BF16_FP8) only, else V4A_ERR_UNSUPPORTED. The keys of a query are always
 * split into at least two ranges (the quantisation runs where the ranges are merged), so the
 * workspace is v4a_attn_q8_workspace_size(cfg, n_q, max_pos, k), 256-byte aligned. Other
 * arguments, errors and the device error word as for v4a_attn_decode. */
size_t v4a_attn_q8_workspace_size(const v4a_layer_cfg* cfg, int32_t n_q, int64_t max_pos, int32_t k);
int v4a_attn_decode_q8(const v4a_layer_cfg* cfg, int32_t n_q, const int32_t* q_seq,
                       const int64_t* q_pos, int64_t max_pos, const void* q, const int32_t* topk,
                       int32_t k, const v4a_cache* attn, const v4a_cache* swa, uint8_t* out_codes,
                       float* out_scale, void* workspace, size_t workspace_bytes, int32_t* dev_err,
                       v4a_stream_t stream);
int v4a_attn_prefill(const v4a_layer_cfg* cfg, int32_t n_q, const int32_t* q_seq,
                     const int64_t* q_pos, int64_t max_pos, const void* q,
                     const int32_t* topk, int32_t k, const v4a_cache* attn,
                     const v4a_cache* swa, void* out, void* workspace, size_t workspace_bytes,
                     int32_t* dev_err, v4a_stream_t stream);

/*
 * v4a_slot_mapping — pool rows of logical rows ([notes] 解决方案一: slot mapping in the
 * unit of the 256-position block). slots[i] = page * R + row[i] % R with
 * page = block_table[seq[i], row[i] / R], or -1 if the block has no page or lies beyond
 * max_blocks (a page >= n_pages also gives -1 and sets V4A_DEV_BAD_PAGE).
 * seq: device int32 [n]; row: device int64 [n]; slots: device int32 [n].
 */
int v4a_slot_mapping(const v4a_cache* cache, int32_t n, const int32_t* seq,
                     const int64_t* row, int32_t* slots, int32_t* dev_err,
                     v4a_stream_t stream);

/* Synchronise `stream`, read the device error word, clear it. *flags_out (may be NULL)
 * receives the bits. Returns V4A_OK, V4A_ERR_DEVICE if any bit was set, or V4A_ERR_CUDA. */
int v4a_get_error(int32_t* dev_err, v4a_stream_t stream, int32_t* flags_out);

/* Library version, raised whenever an entry point or a kernel changes (profiles and the
 * binding compare against it). */
int32_t v4a_version(void);

#ifdef __cplusplus
}
#endif
#endif /* V4A_H */
