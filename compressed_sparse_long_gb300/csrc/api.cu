// extern "C" entry points of libv4a: host-side validation, workspace layout, dispatch.
#include <cmath>
#include <cstring>
#include <cstdint>

#include "common.cuh"
#include "kernels.h"

using namespace v4a;

namespace {

constexpr int32_t kVersion = 21;

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Turns per position phi_i = theta_i / (2 pi) and psi_i = frac(4096 phi_i), as fp32 hi/lo.
Rope make_rope(const v4a_layer_cfg* c) {
  Rope r{};
  r.d_r = c->rope_dim;
  r.D = c->head_dim;
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < c->rope_dim / 2 && i < kMaxRopePairs; ++i) {
    const double theta = std::pow((double)c->rope_base, -2.0 * i / (double)c->rope_dim);
    const double phi = theta / two_pi;
    double psi = 4096.0 * phi;
    psi -= std::floor(psi);
    r.phi_hi[i] = (float)phi;
    r.phi_lo[i] = (float)(phi - (double)r.phi_hi[i]);
    r.psi_hi[i] = (float)psi;
    r.psi_lo[i] = (float)(psi - (double)r.psi_hi[i]);
  }
  return r;
}

}  // namespace

// Layer-level checks shared by every call.
int v4a::check_cfg(const v4a_layer_cfg* c) {
  if (!c) return V4A_ERR_ARG;
  if (c->kind != V4A_C4A && c->kind != V4A_C128A) return V4A_ERR_UNSUPPORTED;
  if (c->dtype != V4A_FP32 && c->dtype != V4A_BF16_FP8) return V4A_ERR_UNSUPPORTED;
  if (c->head_dim <= 0 || c->head_dim % 32 != 0) return V4A_ERR_UNSUPPORTED;
  if (c->rope_dim < 0 || c->rope_dim % 2 != 0 || c->rope_dim > 2 * kMaxRopePairs ||
      c->rope_dim > c->head_dim)
    return V4A_ERR_UNSUPPORTED;
  if (c->window <= 0 || c->stride <= 0 || c->window > 256 || kBlock % c->stride != 0)
    return V4A_ERR_UNSUPPORTED;
  if (c->win_off > 0 || c->win_off <= -c->window) return V4A_ERR_ARG;
  if (c->swa <= 0) return V4A_ERR_ARG;
  if (!(c->rms_eps >= 0.f) || !(c->softmax_scale > 0.f) || !(c->rope_base > 0.f)) return V4A_ERR_ARG;
  if (c->idx_format != V4A_IDX_DEFAULT && c->idx_format != V4A_IDX_FP4) return V4A_ERR_UNSUPPORTED;
  if (c->idx_format == V4A_IDX_FP4 &&
      (c->dtype != V4A_BF16_FP8 || c->kind != V4A_C4A || c->idx_dim != 128))
    return V4A_ERR_UNSUPPORTED;
  return V4A_OK;
}

// Checks of a cache descriptor: geometry, alignment, scales of fp8 pools.
int v4a::check_cache(const v4a_cache* c, int rows_per_block, int width, bool fp8) {
  if (!c || !c->data || !c->block_table) return V4A_ERR_ARG;
  if (c->rows_per_block != rows_per_block || c->row_width != width) return V4A_ERR_ARG;
  if (c->max_blocks <= 0 || c->n_pages < 0 || c->reserved != 0) return V4A_ERR_ARG;
  if (!aligned(c->data, 16)) return V4A_ERR_ARG;
  if (fp8 && (!c->scale || !aligned(c->scale, 16))) return V4A_ERR_ARG;
  return V4A_OK;
}

// The indexer pool as the kernels see it: width in bytes for packed fp4 rows.
CacheView v4a::idx_view(const v4a_layer_cfg* cfg, const v4a_cache* idx) {
  CacheView v = view_of(idx);
  if (cfg->idx_format == V4A_IDX_FP4) v.width = idx->row_width / 2;
  return v;
}

// Host-side validation and parameters of the indexer calls (v4a_index_topk,
// v4a_index_topk_noalloc, v4a_index_scores): every one of them returns the same code for
// the same arguments. with_topk: k and topk_out are part of the call. p->scores is left for
// the caller to set.
int v4a::prepare_index(const v4a_layer_cfg* cfg, int32_t n_q, const int32_t* q_seq,
                       const int64_t* q_pos, int64_t max_pos, const void* q_idx, const float* w,
                       const v4a_cache* idx, int32_t k, int32_t* topk_out, bool with_topk,
                       int32_t* dev_err, IndexParams* p, int64_t* max_vis) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (cfg->kind != V4A_C4A) return V4A_ERR_UNSUPPORTED;
  if (n_q < 0 || (with_topk && k <= 0) || max_pos < 0) return V4A_ERR_ARG;
  if (n_q == 0) return V4A_OK;
  if (!q_seq || !q_pos || !q_idx || !w || (with_topk && !topk_out)) return V4A_ERR_ARG;
  const bool fp8 = cfg->dtype == V4A_BF16_FP8;
  if ((rc = check_cache(idx, kBlock / cfg->stride, cfg->idx_dim, fp8))) return rc;
  if (!aligned(q_idx, 16) || !aligned(w, 16)) return V4A_ERR_ARG;
  *max_vis = visible_entries(max_pos, cfg->stride, cfg->window, cfg->win_off);
  *p = IndexParams{};
  p->n_q = n_q;
  p->H_I = cfg->idx_heads;
  p->d_I = cfg->idx_dim;
  p->W = cfg->window;
  p->S = cfg->stride;
  p->win_off = cfg->win_off;
  p->k = with_topk ? k : 0;
  p->row_stride = score_row_stride(*max_vis);
  p->q_seq = q_seq;
  p->q_pos = q_pos;
  p->q_idx = q_idx;
  p->w = w;
  p->idx = idx_view(cfg, idx);
  p->idx_fp4 = cfg->idx_format == V4A_IDX_FP4;
  p->topk = with_topk ? topk_out : nullptr;
  p->err = dev_err;
  return V4A_OK;
}

namespace {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

extern "C" {

int32_t v4a_version(void) { return kVersion; }

namespace {

// v4a_compress_insert and v4a_compress_insert_qnorm: one launch, n_tokens insert warps
// followed by n_q * H query-norm warps.
int compress_common(const v4a_layer_cfg* cfg, int32_t n_seq, int32_t n_tokens,
                    const int32_t* cu_tokens, const int64_t* start_pos, const void* kv,
                    const void* score, const float* bias, const float* gamma, const void* ikv,
                    const void* iscore, const float* ibias, const v4a_cache* attn,
                    const v4a_cache* idx, const v4a_cache* swa, const v4a_cache* state,
                    int32_t n_q, const void* q, const float* q_gamma, void* q_out,
                    int32_t* dev_err, v4a_stream_t stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (n_seq < 0 || n_tokens < 0 || n_q < 0) return V4A_ERR_ARG;
  const bool fp8 = cfg->dtype == V4A_BF16_FP8;
  const bool c4a = cfg->kind == V4A_C4A;
  const int D = cfg->head_dim, DI = c4a ? cfg->idx_dim : 0;
  const size_t es = fp8 ? 2 : 4;
  const int64_t n_qrows = (int64_t)n_q * cfg->n_heads;
  if (n_q > 0) {
    if (!q || !q_gamma || !q_out || !aligned(q, 16) || !aligned(q_gamma, 16) ||
        !aligned(q_out, 16))
      return V4A_ERR_ARG;
    // q_out is q itself or does not overlap it
    const uintptr_t a = (uintptr_t)q, b = (uintptr_t)q_out, n = (uintptr_t)(n_qrows * D * es);
    if (a != b && a < b + n && b < a + n) return V4A_ERR_ARG;
    if ((int64_t)n_tokens + n_qrows > ((int64_t)1 << 33)) return V4A_ERR_ARG;   // grid limit
  }
  if (n_tokens > 0) {
    if (n_seq == 0) return V4A_ERR_ARG;
    if (!cu_tokens || !start_pos || !kv || !score || !bias || !gamma) return V4A_ERR_ARG;
    if (!aligned(kv, 16) || !aligned(score, 16) || !aligned(bias, 16) || !aligned(gamma, 16))
      return V4A_ERR_ARG;
    if (c4a && (!ikv || !iscore || !ibias || !aligned(ikv, 16) || !aligned(iscore, 16) ||
                !aligned(ibias, 16)))
      return V4A_ERR_ARG;
    const int R = kBlock / cfg->stride;
    if ((rc = check_cache(attn, R, D, fp8))) return rc;
    if (c4a && (rc = check_cache(idx, R, DI, fp8))) return rc;
    if ((rc = check_cache(swa, kBlock, D, fp8))) return rc;
    if ((rc = check_cache(state, kBlock, 2 * D + 2 * DI, false))) return rc;
  }
  if (n_tokens == 0 && n_qrows == 0) return V4A_OK;

  CompressParams p{};
  p.n_tokens = n_tokens;
  p.n_seq = n_seq;
  p.D = D;
  p.DI = DI;
  p.W = cfg->window;
  p.S = cfg->stride;
  p.win_off = cfg->win_off;
  p.eps = cfg->rms_eps;
  p.cu = cu_tokens;
  p.start = start_pos;
  p.kv = kv;
  p.score = score;
  p.ikv = c4a ? ikv : nullptr;
  p.iscore = c4a ? iscore : nullptr;
  p.bias = bias;
  p.gamma = gamma;
  p.ibias = c4a ? ibias : nullptr;
  if (n_tokens > 0) {
    p.attn = view_of(attn);
    p.idx = c4a ? idx_view(cfg, idx) : CacheView{};
    p.idx_fp4 = cfg->idx_format == V4A_IDX_FP4;
    p.swa = view_of(swa);
    p.state = view_of(state);
  }
  p.rope = make_rope(cfg);
  p.err = dev_err;
  p.n_qrows = n_qrows;
  p.q = n_q > 0 ? q : nullptr;
  p.q_gamma = n_q > 0 ? q_gamma : nullptr;
  p.q_out = n_q > 0 ? q_out : nullptr;
  return launch_compress_insert(p, cfg->dtype, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

int v4a_compress_insert(const v4a_layer_cfg* cfg, int32_t n_seq, int32_t n_tokens,
                        const int32_t* cu_tokens, const int64_t* start_pos, const void* kv,
                        const void* score, const float* bias, const float* gamma,
                        const void* ikv, const void* iscore, const float* ibias,
                        const v4a_cache* attn, const v4a_cache* idx, const v4a_cache* swa,
                        const v4a_cache* state, int32_t* dev_err, v4a_stream_t stream) {
  return compress_common(cfg, n_seq, n_tokens, cu_tokens, start_pos, kv, score, bias, gamma,
                         ikv, iscore, ibias, attn, idx, swa, state, 0, nullptr, nullptr,
                         nullptr, dev_err, stream);
}

int v4a_compress_insert_qnorm(const v4a_layer_cfg* cfg, int32_t n_seq, int32_t n_tokens,
                              const int32_t* cu_tokens, const int64_t* start_pos,
                              const void* kv, const void* score, const float* bias,
                              const float* gamma, const void* ikv, const void* iscore,
                              const float* ibias, const v4a_cache* attn, const v4a_cache* idx,
                              const v4a_cache* swa, const v4a_cache* state, int32_t n_q,
                              const void* q, const float* q_gamma, void* q_out,
                              int32_t* dev_err, v4a_stream_t stream) {
  return compress_common(cfg, n_seq, n_tokens, cu_tokens, start_pos, kv, score, bias, gamma,
                         ikv, iscore, ibias, attn, idx, swa, state, n_q, q, q_gamma, q_out,
                         dev_err, stream);
}

size_t v4a_index_topk_workspace_size(const v4a_layer_cfg* cfg, int32_t n_q, int64_t max_pos) {
  if (check_cfg(cfg) || n_q < 0 || max_pos < 0) return 0;
  const int64_t max_vis = visible_entries(max_pos, cfg->stride, cfg->window, cfg->win_off);
  return align_up((size_t)n_q * (size_t)score_row_stride(max_vis) * sizeof(float), 256) + 256;
}

int v4a_index_topk(const v4a_layer_cfg* cfg, int32_t n_q, const int32_t* q_seq,
                   const int64_t* q_pos, int64_t max_pos, const void* q_idx, const float* w,
                   const v4a_cache* idx, int32_t k, int32_t* topk_out, void* workspace,
                   size_t workspace_bytes, int32_t* dev_err, v4a_stream_t stream) {
  IndexParams p{};
  int64_t max_vis = 0;
  int rc = prepare_index(cfg, n_q, q_seq, q_pos, max_pos, q_idx, w, idx, k, topk_out, true,
                         dev_err, &p, &max_vis);
  if (rc || n_q == 0) return rc;
  if (max_vis > 0) {
    if (!workspace || !aligned(workspace, 256)) return V4A_ERR_ARG;
    if (workspace_bytes < v4a_index_topk_workspace_size(cfg, n_q, max_pos)) return V4A_ERR_ARG;
  }
  p.scores = reinterpret_cast<float*>(workspace);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((rc = launch_index_scores(p, cfg->dtype, max_vis, st))) return rc;
  return launch_topk(p, max_vis, st);
}

int64_t v4a_index_scores_row_stride(const v4a_layer_cfg* cfg, int64_t max_pos) {
  if (check_cfg(cfg) || max_pos < 0) return 0;
  return score_row_stride(visible_entries(max_pos, cfg->stride, cfg->window, cfg->win_off));
}

int v4a_index_scores(const v4a_layer_cfg* cfg, int32_t n_q, const int32_t* q_seq,
                     const int64_t* q_pos, int64_t max_pos, const void* q_idx, const float* w,
                     const v4a_cache* idx, float* scores, size_t scores_bytes, int32_t* dev_err,
                     v4a_stream_t stream) {
  IndexParams p{};
  int64_t max_vis = 0;
  int rc = prepare_index(cfg, n_q, q_seq, q_pos, max_pos, q_idx, w, idx, 0, nullptr, false,
                         dev_err, &p, &max_vis);
  if (rc || n_q == 0 || max_vis == 0) return rc;
  if (!scores || !aligned(scores, 16)) return V4A_ERR_ARG;
  if (scores_bytes < (size_t)n_q * (size_t)p.row_stride * sizeof(float)) return V4A_ERR_ARG;
  p.scores = scores;
  return launch_index_scores(p, cfg->dtype, max_vis, reinterpret_cast<cudaStream_t>(stream));
}

namespace {

struct SplitPlan {
  int32_t n_split;
  int32_t keys_per_split;
};

SplitPlan plan_split(const v4a_layer_cfg* cfg, int32_t n_q, int64_t max_pos, int32_t k,
                     bool dense, bool prefill, bool at_least_two = false) {
  const int64_t max_keys =
      (dense ? visible_entries(max_pos, cfg->stride, cfg->window, cfg->win_off) : k) + cfg->swa;
  SplitPlan s{1, (int32_t)max_keys};
  if (prefill || n_q == 0) return s;
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) sms = v;
  }
  // Split each query's keys into k ranges (whole key tiles). With one CTA per SM, a choice
  // costs waves * (tiles per range + 1), the +1 standing for the per-range query setup;
  // take the smallest k of least cost (the merge handles k <= 64).
  const int64_t tile = cfg->dtype == V4A_BF16_FP8 ? 128 : 32;   // key tile of the kernel
  const int64_t tiles = (max_keys + tile - 1) / tile;
  int64_t best_k = 1, best_cost = INT64_MAX;
  for (int64_t k = 1; k <= tiles && k <= 64; ++k) {
    const int64_t waves = (n_q * k + sms - 1) / sms;
    const int64_t cost = waves * ((tiles + k - 1) / k + 1);
    if (cost < best_cost) {
      best_cost = cost;
      best_k = k;
    }
  }
  if (at_least_two && best_k < 2) best_k = 2;
  const int64_t per = ((tiles + best_k - 1) / best_k) * tile;
  s.keys_per_split = (int32_t)per;
  s.n_split = (int32_t)((max_keys + per - 1) / per);
  if (at_least_two && s.n_split < 2) s.n_split = 2;   // the second range may hold no key
  return s;
}

size_t attn_ws(const v4a_layer_cfg* cfg, int32_t n_q, const SplitPlan& s) {
  if (s.n_split <= 1) return 256;
  const size_t o = (size_t)n_q * s.n_split * cfg->n_heads * cfg->head_dim * sizeof(float);
  const size_t ml = (size_t)n_q * s.n_split * cfg->n_heads * 2 * sizeof(float);
  return align_up(o, 256) + align_up(ml, 256) + 256;
}

int attn_common(const v4a_layer_cfg* cfg, int32_t n_q, const int32_t* q_seq, const int64_t* q_pos,
                int64_t max_pos, const void* q, const int32_t* topk, int32_t k,
                const v4a_cache* attn, const v4a_cache* swa, void* out, void* workspace,
                size_t workspace_bytes, int32_t* dev_err, v4a_stream_t stream, bool prefill,
                float* out_scale = nullptr) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (n_q < 0 || max_pos < 0) return V4A_ERR_ARG;
  if (n_q == 0) return V4A_OK;
  if (!q_seq || !q_pos || !q || !out) return V4A_ERR_ARG;
  if (topk && k <= 0) return V4A_ERR_ARG;
  if (!aligned(q, 16) || !aligned(out, 16)) return V4A_ERR_ARG;
  const bool fp8 = cfg->dtype == V4A_BF16_FP8;
  if ((rc = check_cache(attn, kBlock / cfg->stride, cfg->head_dim, fp8))) return rc;
  if ((rc = check_cache(swa, kBlock, cfg->head_dim, fp8))) return rc;
  const SplitPlan s = plan_split(cfg, n_q, max_pos, topk ? k : 0, topk == nullptr, prefill,
                                 out_scale != nullptr);
  const size_t need = attn_ws(cfg, n_q, s);
  if (s.n_split > 1) {
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return V4A_ERR_ARG;
  }
  AttnParams p{};
  p.n_q = n_q;
  p.H = cfg->n_heads;
  p.D = cfg->head_dim;
  p.W = cfg->window;
  p.S = cfg->stride;
  p.win_off = cfg->win_off;
  p.swa_len = cfg->swa;
  p.k = topk ? k : 0;
  p.n_split = s.n_split;
  p.keys_per_split = s.keys_per_split;
  p.out_scale = out_scale;
  p.scale = cfg->softmax_scale;
  p.q_seq = q_seq;
  p.q_pos = q_pos;
  p.q = q;
  p.topk = topk;
  p.attn = view_of(attn);
  p.swa = view_of(swa);
  p.out = out;
  if (s.n_split > 1) {
    const size_t o = (size_t)n_q * s.n_split * cfg->n_heads * cfg->head_dim * sizeof(float);
    p.part_o = reinterpret_cast<float*>(workspace);
    p.part_ml = reinterpret_cast<float*>(reinterpret_cast<char*>(workspace) + align_up(o, 256));
  }
  p.rope = make_rope(cfg);
  p.err = dev_err;
  return launch_attention(p, cfg->dtype, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

size_t v4a_attn_workspace_size(const v4a_layer_cfg* cfg, int32_t n_q, int64_t max_pos, int32_t k,
                               int32_t prefill) {
  if (check_cfg(cfg) || n_q < 0 || max_pos < 0) return 0;
  const SplitPlan s = plan_split(cfg, n_q, max_pos, k, k <= 0, prefill != 0);
  return attn_ws(cfg, n_q, s);
}

int v4a_attn_plan(const v4a_layer_cfg* cfg, int32_t n_q, int64_t max_pos, int32_t k,
                  int32_t prefill, int32_t* n_split, int32_t* n_kernels) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (n_q < 0 || max_pos < 0 || !n_split || !n_kernels) return V4A_ERR_ARG;
  const SplitPlan s = plan_split(cfg, n_q, max_pos, k, k <= 0, prefill != 0);
  *n_split = s.n_split;
  *n_kernels = n_q == 0 ? 0 : (s.n_split > 1 ? 2 : 1);   // attention (+ the split merge)
  return V4A_OK;
}

int v4a_attn_decode(const v4a_layer_cfg* cfg, int32_t n_q, const int32_t* q_seq,
                    const int64_t* q_pos, int64_t max_pos, const void* q, const int32_t* topk,
                    int32_t k, const v4a_cache* attn, const v4a_cache* swa, void* out,
                    void* workspace, size_t workspace_bytes, int32_t* dev_err,
                    v4a_stream_t stream) {
  return attn_common(cfg, n_q, q_seq, q_pos, max_pos, q, topk, k, attn, swa, out, workspace,
                     workspace_bytes, dev_err, stream, false);
}

size_t v4a_attn_q8_workspace_size(const v4a_layer_cfg* cfg, int32_t n_q, int64_t max_pos, int32_t k) {
  if (check_cfg(cfg) || n_q < 0 || max_pos < 0) return 0;
  const SplitPlan s = plan_split(cfg, n_q, max_pos, k, k <= 0, false, true);
  return attn_ws(cfg, n_q, s);
}

int v4a_attn_decode_q8(const v4a_layer_cfg* cfg, int32_t n_q, const int32_t* q_seq,
                       const int64_t* q_pos, int64_t max_pos, const void* q, const int32_t* topk,
                       int32_t k, const v4a_cache* attn, const v4a_cache* swa, uint8_t* out_codes,
                       float* out_scale, void* workspace, size_t workspace_bytes, int32_t* dev_err,
                       v4a_stream_t stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (cfg->dtype != V4A_BF16_FP8) return V4A_ERR_UNSUPPORTED;
  if (n_q > 0 && (!out_scale || !aligned(out_scale, 4))) return V4A_ERR_ARG;
  return attn_common(cfg, n_q, q_seq, q_pos, max_pos, q, topk, k, attn, swa, out_codes, workspace,
                     workspace_bytes, dev_err, stream, false, out_scale);
}

int v4a_attn_prefill(const v4a_layer_cfg* cfg, int32_t n_q, const int32_t* q_seq,
                     const int64_t* q_pos, int64_t max_pos, const void* q, const int32_t* topk,
                     int32_t k, const v4a_cache* attn, const v4a_cache* swa, void* out,
                     void* workspace, size_t workspace_bytes, int32_t* dev_err,
                     v4a_stream_t stream) {
  return attn_common(cfg, n_q, q_seq, q_pos, max_pos, q, topk, k, attn, swa, out, workspace,
                     workspace_bytes, dev_err, stream, true);
}

int v4a_slot_mapping(const v4a_cache* cache, int32_t n, const int32_t* seq, const int64_t* row,
                     int32_t* slots, int32_t* dev_err, v4a_stream_t stream) {
  if (!cache || !cache->block_table || cache->rows_per_block <= 0 || cache->max_blocks <= 0)
    return V4A_ERR_ARG;
  if (n < 0) return V4A_ERR_ARG;
  if (n == 0) return V4A_OK;
  if (!seq || !row || !slots) return V4A_ERR_ARG;
  return launch_slot_mapping(view_of(cache), n, seq, row, slots, dev_err,
                             reinterpret_cast<cudaStream_t>(stream));
}

int v4a_get_error(int32_t* dev_err, v4a_stream_t stream, int32_t* flags_out) {
  if (!dev_err) return V4A_ERR_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, dev_err, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return V4A_ERR_CUDA;
  if (cudaMemsetAsync(dev_err, 0, sizeof(int32_t), st) != cudaSuccess) return V4A_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return V4A_ERR_CUDA;
  if (flags_out) *flags_out = h;
  return h ? V4A_ERR_DEVICE : V4A_OK;
}

}  // extern "C"

namespace v4a {

namespace {
__global__ void slot_mapping_kernel(CacheView c, int32_t n, const int32_t* seq, const int64_t* row,
                                    int32_t* slots, int32_t* err) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int64_t s = slot_of(c, __ldg(seq + i), __ldg(row + i));
  if (s == -2) raise_err(err, V4A_DEV_BAD_PAGE);
  slots[i] = s >= 0 ? (int32_t)s : -1;
}
}  // namespace

int launch_slot_mapping(const CacheView& c, int32_t n, const int32_t* seq, const int64_t* row,
                        int32_t* slots, int32_t* err, cudaStream_t st) {
  if (launch_pdl(slot_mapping_kernel, dim3((n + 255) / 256), dim3(256), 0, st, c, n, seq, row, slots, err) !=
      cudaSuccess)
    return V4A_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? V4A_OK : V4A_ERR_CUDA;
}

}  // namespace v4a
