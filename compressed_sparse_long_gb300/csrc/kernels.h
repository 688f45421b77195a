// Launch parameters and launchers of the v4a kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace v4a {

struct CompressParams {
  int64_t n_tokens;
  int32_t n_seq;
  int32_t D, DI, W, S, win_off;
  float eps;
  const int32_t* cu;
  const int64_t* start;
  const void* kv;
  const void* score;
  const void* ikv;
  const void* iscore;
  const float* bias;
  const float* gamma;
  const float* ibias;
  CacheView attn, idx, swa, state;
  Rope rope;
  int32_t* err;
  int32_t idx_fp4;             // indexer rows as packed e2m1 + row scale (idx.width in bytes)
  // query RMSNorm rows handled by the warps after the n_tokens insert warps (0: none)
  int64_t n_qrows;             // n_q * H rows of D elements
  const void* q;               // [n_qrows, D] input type
  const float* q_gamma;        // [D]
  void* q_out;                 // [n_qrows, D] input type; equal to q or disjoint from it
};

struct IndexParams {
  int32_t n_q;
  int32_t H_I, d_I, W, S, win_off;
  int32_t k;
  int64_t row_stride;          // floats between consecutive score rows in the workspace
                               // (the visible count rounded up to a multiple of 4)
  const int32_t* q_seq;
  const int64_t* q_pos;
  const void* q_idx;
  const float* w;
  CacheView idx;
  int32_t idx_fp4;             // indexer rows as packed e2m1 + row scale (idx.width in bytes)
  float* scores;               // workspace [n_q, row_stride]
  int32_t* topk;               // [n_q, k]
  int32_t* err;
};

struct AttnParams {
  int32_t n_q;
  int32_t H, D, W, S, win_off, swa_len;
  int32_t k;                   // top-k list width (0 with topk == nullptr: dense)
  int32_t n_split;             // CTAs per query
  int32_t keys_per_split;      // keys handled by one split (multiple of the key tile)
  float scale;                 // softmax scale
  const int32_t* q_seq;
  const int64_t* q_pos;
  const void* q;
  const int32_t* topk;
  CacheView attn, swa;
  void* out;                   // bf16 / fp32 [n_q, H, D], or e4m3 codes when out_scale is set
  float* out_scale;            // [n_q, H] row scales of an fp8 output (nullptr: no quantisation)
  float* part_o;               // [n_q, n_split, H, D]   (n_split > 1)
  float* part_ml;              // [n_q, n_split, H, 2]   (n_split > 1)
  Rope rope;
  int32_t* err;
};

// Host-side checks shared by the entry points (V4A_OK or the code the call returns).
int check_cfg(const v4a_layer_cfg* cfg);
int check_cache(const v4a_cache* c, int rows_per_block, int width, bool fp8);
// Validation and parameters of the indexer calls; p->scores is set by the caller.
int prepare_index(const v4a_layer_cfg* cfg, int32_t n_q, const int32_t* q_seq,
                  const int64_t* q_pos, int64_t max_pos, const void* q_idx, const float* w,
                  const v4a_cache* idx, int32_t k, int32_t* topk_out, bool with_topk,
                  int32_t* dev_err, IndexParams* p, int64_t* max_vis);
// The indexer pool as the kernels see it (width in bytes for packed fp4 rows).
CacheView idx_view(const v4a_layer_cfg* cfg, const v4a_cache* idx);
int launch_compress_insert(const CompressParams& p, int dtype, cudaStream_t st);
int launch_index_scores(const IndexParams& p, int dtype, int64_t max_vis, cudaStream_t st);
cudaError_t launch_index_scores_tc(const IndexParams& p, int64_t max_vis, cudaStream_t st);
int launch_topk(const IndexParams& p, int64_t max_vis, cudaStream_t st);
int launch_attention(const AttnParams& p, int dtype, cudaStream_t st);
cudaError_t launch_attention_tc(const AttnParams& p, cudaStream_t st);
// A 2-D byte tensor map over n_rows rows of row_bytes at base (16-byte aligned), boxes of
// box_rows x box_bytes, 128-byte swizzle, elements outside the tensor read as zero. False
// when the driver entry point is missing or the driver refuses the map.
bool encode_byte_rows_map(CUtensorMap* map, const void* base, uint64_t n_rows, uint32_t row_bytes,
                          uint32_t box_bytes, uint32_t box_rows);
int launch_slot_mapping(const CacheView& c, int32_t n, const int32_t* seq, const int64_t* row,
                        int32_t* slots, int32_t* err, cudaStream_t st);

}  // namespace v4a
