// compress_insert: the token-axis KV compressor with RMSNorm, RoPE, fp8 quantisation and
// paged insert, plus the sliding-window insert and the residual-state insert, in one
// launch (steps a1-a5).
//
// [notes] "DeepSeek V4 in vLLM 技术博客详尽笔记", 优化一：三大内核融合 (fusion 1: compressor +
// RMSNorm + RoPE + cache insert; the K RoPE + K insert half of fusion 3) and 解决方案二
// (compressor state kept as sliding-window KV); 数学附录精要 for the window positions.
//
// Work decomposition: one warp per new token (and, in the call with the query norm, one
// warp per query head row after them: fusion 3's static warp dispatch). The warp writes the token's sliding-window
// row and, if the token is among the last W of its sequence's new tokens, its raw residual
// row. If the token is the last position of entry j's window, the same warp also builds
// entry j (attention row and, for c4a, indexer row). Lane l owns channels
// [l*CPL, (l+1)*CPL) of the D-wide vectors and [l*ICPL, (l+1)*ICPL) of the d_I-wide ones,
// so every load and store is a contiguous 16-64 byte vector per lane.
//
// Inputs are read once per (token, entry using it): with W = 2S (c4a) each token feeds two
// entries and is re-read from L2 by the neighbouring warp. The kernel is HBM-bound.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace v4a {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxWindow = 256;   // the largest window a layer may have (host-checked)

template <typename TIn, int CPL, int ICPL, bool kFp8>
struct CompressKernel {
  static constexpr int D = CPL * 32;
  static constexpr int DI = ICPL * 32;

  // fp8 row store: per-row scale amax/448 (1 if the row is zero), e4m3 RNE satfinite of
  // y * (1/scale) in fp32; fp32 rows are stored as they are.
  template <int N>
  static __device__ __forceinline__ void store_row(const CacheView& c, int64_t slot, float (&y)[N],
                                                   int lane) {
    if constexpr (kFp8) {
      float amax = 0.f;
#pragma unroll
      for (int k = 0; k < N; ++k) amax = fmaxf(amax, fabsf(y[k]));
      amax = warp_max(amax);
      float scale = amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.0f;
      // y / scale as y * (1 / scale): two fp32 roundings (a relative error below 2^-23),
      // against one per element for a division
      const float inv = __frcp_rn(scale);
      uint8_t* dst = reinterpret_cast<uint8_t*>(c.data) + slot * (int64_t)c.width + lane * N;
      if constexpr (N % 4 == 0) {
        uint32_t words[N / 4];
#pragma unroll
        for (int k = 0; k < N / 4; ++k) {
          uint32_t lo = e4m3x2_encode(y[4 * k] * inv, y[4 * k + 1] * inv);
          uint32_t hi = e4m3x2_encode(y[4 * k + 2] * inv, y[4 * k + 3] * inv);
          words[k] = lo | (hi << 16);
        }
        if constexpr (N == 16) {
          *reinterpret_cast<uint4*>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
        } else if constexpr (N == 8) {
          *reinterpret_cast<uint2*>(dst) = make_uint2(words[0], words[1]);
        } else {
#pragma unroll
          for (int k = 0; k < N / 4; ++k) reinterpret_cast<uint32_t*>(dst)[k] = words[k];
        }
      } else {
#pragma unroll
        for (int k = 0; k < N; ++k) dst[k] = (uint8_t)(e4m3x2_encode(y[k] * inv, 0.f) & 0xFF);
      }
      if (lane == 0) c.scale[slot] = scale;
    } else {
      float* dst = reinterpret_cast<float*>(c.data) + slot * (int64_t)c.width + lane * N;
      store_f<float, N>(dst, y);
    }
  }

  // fp4 row store: per-row scale amax/6 (1 if the row is zero), e2m1 round-to-nearest-even
  // of y/scale; lane l owns elements [N l, N l + N), i.e. bytes [N l / 2, N l / 2 + N / 2)
  // of the packed row (element 2i in the low nibble).
  template <int N>
  static __device__ __forceinline__ void store_row_fp4(const CacheView& c, int64_t slot, float (&y)[N],
                                                       int lane) {
    static_assert(N == 4, "one 16-bit group of four codes per lane");
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < N; ++k) amax = fmaxf(amax, fabsf(y[k]));
    amax = warp_max(amax);
    const float scale = amax > 0.f ? __fdiv_rn(amax, kE2m1Max) : 1.0f;
    const float inv = __frcp_rn(scale);
    uint32_t packed = 0;
#pragma unroll
    for (int k = 0; k < N; ++k) packed |= e2m1_encode(y[k] * inv) << (4 * k);
    uint8_t* dst = reinterpret_cast<uint8_t*>(c.data) + slot * (int64_t)c.width + lane * (N / 2);
    *reinterpret_cast<uint16_t*>(dst) = (uint16_t)packed;
    if (lane == 0) c.scale[slot] = scale;
  }

  // Rotate the lane's channels that fall in the rotated tail (adjacent pairs). Lane i
  // evaluates the angle of pair i (d_r / 2 <= 32 pairs) and the lanes owning the tail take
  // theirs by shuffle, so the warp evaluates each angle once and in parallel.
  // tab: the angle constants staged in shared memory (stage_rope), or nullptr.
  template <int N>
  static __device__ __forceinline__ void rope_lane(const Rope& rp, float (&y)[N], int lane,
                                                   int64_t pos, const float* tab = nullptr) {
    const int tail0 = rp.D - rp.d_r;
    float c_l = 1.f, s_l = 0.f;
    if (lane < (rp.d_r >> 1)) {
      if (tab) rope_cs_tab(tab, pos, lane, c_l, s_l);
      else rope_cs(rp, pos, lane, c_l, s_l);
    }
#pragma unroll
    for (int k = 0; k < N; k += 2) {
      const int d = lane * N + k;
      const int pi = (d - tail0) >> 1;
      const float c = __shfl_sync(0xffffffffu, c_l, pi & 31);
      const float s = __shfl_sync(0xffffffffu, s_l, pi & 31);
      if (d >= tail0) {
        const float a = y[k], b = y[k + 1];
        y[k] = a * c - b * s;
        y[k + 1] = a * s + b * c;
      }
    }
  }

  // One (query, head) row of the query RMSNorm: y = gamma_q * q / sqrt(mean(q^2) + eps),
  // stored in the input type. The row is in registers before the first store, so q_out may
  // be q itself.
  static __device__ void q_norm_row(const CompressParams& p, int64_t r, int lane) {
    float x[CPL], g[CPL];
    load_f<TIn, CPL>(reinterpret_cast<const TIn*>(p.q) + r * D + lane * CPL, x);
    load_f<float, CPL>(p.q_gamma + lane * CPL, g);
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < CPL; ++k) ss = fmaf(x[k], x[k], ss);
    ss = warp_sum(ss);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fdiv_rn(ss, (float)D) + p.eps));
#pragma unroll
    for (int k = 0; k < CPL; ++k) x[k] = x[k] * inv * g[k];
    pdl_wait();   // q_out may still be read by the kernel before this one
    store_f<TIn, CPL>(reinterpret_cast<TIn*>(p.q_out) + r * D + lane * CPL, x);
  }

  // Pointers to the four parts of one window token's row (inputs, residual pool or a
  // staged copy in shared memory: the loads go through generic addresses).
  struct WindowRow {
    const TIn* kv;
    const TIn* s;
    const TIn* ik;
    const TIn* is;
  };

  template <typename T, int N>
  static __device__ __forceinline__ void load_g(const T* __restrict__ ptr, float (&out)[N]) {
    constexpr int kBytes = N * (int)sizeof(T);
    if constexpr (kBytes % 16 == 0) {
      constexpr int kPer = 16 / sizeof(T);
#pragma unroll
      for (int v = 0; v < kBytes / 16; ++v) {
        const uint4 u = reinterpret_cast<const uint4*>(ptr)[v];
        const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
        for (int k = 0; k < kPer; ++k) out[v * kPer + k] = Elem<T>::to_f(e[k]);
      }
    } else {
#pragma unroll
      for (int k = 0; k < N; ++k) out[k] = Elem<T>::to_f(ptr[k]);
    }
  }

  // 2^x by the hardware approximation (ex2.approx.ftz: relative error ~2^-22, 0 for -inf).
  static __device__ __forceinline__ float exp2_approx(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
  }

  // Weighted sum of one window with per-channel softmax weights, as the pages' compressor
  // defines it: z_o = s_o + bias[o], w_o = exp(z_o - max_o z_o) / sum_o exp(z_o - max_o z_o),
  // c = sum_o w_o kv_o (max first, then the exponentials, tokens in window order; the
  // exponentials in base 2 of z log2(e)). N
  // channels per lane; fetch(o, row) fills token o's row pointers and returns its status
  // (1 present, 0 absent: a position before the sequence, -1 / -2 a residual row without a
  // page or with a page outside the pool); kIdx selects the (ik, is) halves instead of
  // (kv, s). Returns false, after raising the error bit, if a row is missing (the caller
  // skips the entry).
  template <int N, bool kIdx, class Fetch>
  static __device__ __forceinline__ bool window_sum(const CompressParams& p, int lane,
                                                    const Fetch& fetch, float (&c)[N]) {
    const int width = kIdx ? DI : D;
    const float* bias = kIdx ? p.ibias : p.bias;
    float m[N];
#pragma unroll
    for (int k = 0; k < N; ++k) m[k] = -INFINITY;
#pragma unroll 8
    for (int o = 0; o < p.W; ++o) {
      WindowRow w;
      const int st = fetch(o, w);
      if (st == 0) continue;
      if (st < 0) {
        raise_err(p.err, st == -2 ? V4A_DEV_BAD_PAGE : V4A_DEV_MISSING_PAGE);
        return false;
      }
      float sv[N], bv[N];
      load_g<TIn, N>((kIdx ? w.is : w.s) + lane * N, sv);
      load_f<float, N>(bias + (int64_t)o * width + lane * N, bv);
#pragma unroll
      for (int k = 0; k < N; ++k) m[k] = fmaxf(m[k], (sv[k] + bv[k]) * kLog2e);
    }
    float l[N], acc[N];
#pragma unroll
    for (int k = 0; k < N; ++k) { l[k] = 0.f; acc[k] = 0.f; }
#pragma unroll 8
    for (int o = 0; o < p.W; ++o) {
      WindowRow w;
      if (fetch(o, w) <= 0) continue;
      float sv[N], bv[N], xv[N];
      load_g<TIn, N>((kIdx ? w.is : w.s) + lane * N, sv);
      load_g<TIn, N>((kIdx ? w.ik : w.kv) + lane * N, xv);
      load_f<float, N>(bias + (int64_t)o * width + lane * N, bv);
#pragma unroll
      for (int k = 0; k < N; ++k) {
        const float e = exp2_approx((sv[k] + bv[k]) * kLog2e - m[k]);
        l[k] += e;
        acc[k] = fmaf(e, xv[k], acc[k]);
      }
    }
    // l >= 1 (the window's largest weight is 2^0): an approximate division (~2 ulp)
#pragma unroll
    for (int k = 0; k < N; ++k) c[k] = __fdividef(acc[k], l[k]);
    return true;
  }

  // Entry j of sequence b: attention row RoPE(gamma * c / rms(c), S*j) and, for c4a, the
  // indexer row (no norm, no RoPE), each quantised and stored at its slot. Both insert
  // kernels build entries here, so they write identical bytes.
  template <class Fetch>
  static __device__ void build_entry(const CompressParams& p, int b, int64_t j, int lane,
                                     const Fetch& fetch, const float* rope_tab = nullptr) {
    const int64_t e_slot = slot_of(p.attn, b, j);
    const int64_t i_slot = ICPL > 0 ? slot_of(p.idx, b, j) : -1;
    if (e_slot == -2 || i_slot == -2) raise_err(p.err, V4A_DEV_BAD_PAGE);
    if (e_slot >= 0) {
      float c[CPL], g[CPL];
      if (!window_sum<CPL, false>(p, lane, fetch, c)) return;
      float ss = 0.f;
#pragma unroll
      for (int k = 0; k < CPL; ++k) ss = fmaf(c[k], c[k], ss);
      ss = warp_sum(ss);
      const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fdiv_rn(ss, (float)D) + p.eps));
      load_f<float, CPL>(p.gamma + lane * CPL, g);
#pragma unroll
      for (int k = 0; k < CPL; ++k) c[k] = c[k] * inv * g[k];
      rope_lane<CPL>(p.rope, c, lane, j * p.S, rope_tab);
      store_row<CPL>(p.attn, e_slot, c, lane);
    }
    if constexpr (ICPL > 0) {
      if (i_slot >= 0) {
        float c[ICPL];
        if (!window_sum<ICPL, true>(p, lane, fetch, c)) return;
        if constexpr (kFp8 && ICPL == 4) {
          if (p.idx_fp4) store_row_fp4<ICPL>(p.idx, i_slot, c, lane);
          else store_row<ICPL>(p.idx, i_slot, c, lane);
        } else {
          store_row<ICPL>(p.idx, i_slot, c, lane);
        }
      }
    }
  }

  // Long windows (c128a: 128 tokens), attention entry only: the kWideWarps warps of the
  // token's block each take a contiguous quarter of the window. The same two passes as
  // window_sum (the window's max first, then the exponentials against it), with the max and
  // the partial sums exchanged through shared memory and the partial sums added in warp
  // order; every warp returns the same decision, warp 0 the sums.
  static constexpr int kWideWarps = 4;
  struct WideSmem {
    float m[kWideWarps][CPL][32];
    float l[kWideWarps][CPL][32];
    float a[kWideWarps][CPL][32];
  };
  template <class Fetch>
  static __device__ __forceinline__ bool window_sum_wide(const CompressParams& p, int lane, int w,
                                                         const Fetch& fetch, float (&c)[CPL], WideSmem& sm) {
    constexpr int N = CPL;
    for (int o = 0; o < p.W; ++o) {                // a missing row stops every warp
      WindowRow r;
      const int st = fetch(o, r);
      if (st < 0) {
        if (w == 0) raise_err(p.err, st == -2 ? V4A_DEV_BAD_PAGE : V4A_DEV_MISSING_PAGE);
        return false;
      }
    }
    const int per = (p.W + kWideWarps - 1) / kWideWarps;
    const int o0 = w * per, o1 = min(p.W, o0 + per);
    float m[N];
#pragma unroll
    for (int k = 0; k < N; ++k) m[k] = -INFINITY;
#pragma unroll 8
    for (int o = o0; o < o1; ++o) {
      WindowRow r;
      if (fetch(o, r) == 0) continue;
      float sv[N], bv[N];
      load_g<TIn, N>(r.s + lane * N, sv);
      load_f<float, N>(p.bias + (int64_t)o * D + lane * N, bv);
#pragma unroll
      for (int k = 0; k < N; ++k) m[k] = fmaxf(m[k], (sv[k] + bv[k]) * kLog2e);
    }
#pragma unroll
    for (int k = 0; k < N; ++k) sm.m[w][k][lane] = m[k];
    __syncthreads();
#pragma unroll
    for (int k = 0; k < N; ++k) {
      float mx = sm.m[0][k][lane];
#pragma unroll
      for (int v = 1; v < kWideWarps; ++v) mx = fmaxf(mx, sm.m[v][k][lane]);
      m[k] = mx;
    }
    float l[N], acc[N];
#pragma unroll
    for (int k = 0; k < N; ++k) { l[k] = 0.f; acc[k] = 0.f; }
#pragma unroll 8
    for (int o = o0; o < o1; ++o) {
      WindowRow r;
      if (fetch(o, r) <= 0) continue;
      float sv[N], bv[N], xv[N];
      load_g<TIn, N>(r.s + lane * N, sv);
      load_g<TIn, N>(r.kv + lane * N, xv);
      load_f<float, N>(p.bias + (int64_t)o * D + lane * N, bv);
#pragma unroll
      for (int k = 0; k < N; ++k) {
        const float e = exp2_approx((sv[k] + bv[k]) * kLog2e - m[k]);
        l[k] += e;
        acc[k] = fmaf(e, xv[k], acc[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < N; ++k) {
      sm.l[w][k][lane] = l[k];
      sm.a[w][k][lane] = acc[k];
    }
    __syncthreads();
    if (w == 0) {
#pragma unroll
      for (int k = 0; k < N; ++k) {
        float lt = sm.l[0][k][lane], at = sm.a[0][k][lane];
#pragma unroll
        for (int v = 1; v < kWideWarps; ++v) {
          lt += sm.l[v][k][lane];
          at += sm.a[v][k][lane];
        }
        c[k] = __fdividef(at, lt);   // lt >= 1: the window's largest weight is 2^0
      }
    }
    return true;
  }

  // build_entry for a long window and no indexer row, the whole block taking part
  template <class Fetch>
  static __device__ void build_entry_wide(const CompressParams& p, int b, int64_t j, int lane, int w,
                                          const Fetch& fetch) {
    __shared__ WideSmem sm;
    const int64_t e_slot = slot_of(p.attn, b, j);
    if (e_slot == -2 && w == 0) raise_err(p.err, V4A_DEV_BAD_PAGE);
    if (e_slot < 0) return;
    float c[CPL], g[CPL];
    if (!window_sum_wide(p, lane, w, fetch, c, sm)) return;
    if (w != 0) return;
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < CPL; ++k) ss = fmaf(c[k], c[k], ss);
    ss = warp_sum(ss);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fdiv_rn(ss, (float)D) + p.eps));
    load_f<float, CPL>(p.gamma + lane * CPL, g);
#pragma unroll
    for (int k = 0; k < CPL; ++k) c[k] = c[k] * inv * g[k];
    rope_lane<CPL>(p.rope, c, lane, j * p.S);
    store_row<CPL>(p.attn, e_slot, c, lane);
  }

  // kWide: blocks of kWideWarps warps, one token each (warp 0 writes its rows, all warps
  // build an entry its window completes); otherwise one warp per token or query row.
  template <bool kWide>
  static __device__ void run(const CompressParams& p) {
    const int lane = threadIdx.x & 31;
    const int wb = kWide ? (int)(threadIdx.x >> 5) : 0;   // warp of the token's block
    const int64_t i = kWide ? (int64_t)blockIdx.x : ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    // static warp dispatch: warps [0, n_tokens) insert tokens, the next n_qrows warps
    // normalise query head rows; no warp depends on another
    if (i >= p.n_tokens) {
      if (i < p.n_tokens + p.n_qrows) q_norm_row(p, i - p.n_tokens, lane);
      return;
    }

    // sequence of row i: the largest b with cu[b] <= i, 32 candidates per warp load; the
    // candidates' cu[k], cu[k+1] and start[k] come in the same round and the hit's values
    // are taken by shuffle
    int b = -1;
    int64_t row0 = 0, n_new = 0, P0 = 0;
    for (int base = 0; base < p.n_seq && b < 0; base += 32) {
      const int k = base + lane;
      const int64_t c0 = k < p.n_seq ? (int64_t)__ldg(p.cu + k) : INT64_MAX;
      const int64_t c1 = k < p.n_seq ? (int64_t)__ldg(p.cu + k + 1) : INT64_MAX;
      const int64_t st = k < p.n_seq ? __ldg(p.start + k) : 0;
      const bool hit_k = c0 <= i && !(k + 1 < p.n_seq && c1 <= i);
      const uint32_t hit = __ballot_sync(0xffffffffu, k < p.n_seq && hit_k);
      if (hit) {
        const int src = __ffs(hit) - 1;
        b = base + src;
        row0 = __shfl_sync(0xffffffffu, c0, src);
        n_new = __shfl_sync(0xffffffffu, c1, src) - row0;
        P0 = __shfl_sync(0xffffffffu, st, src);
      }
    }
    if (b < 0) return;
    const int64_t P1 = P0 + n_new;
    const int64_t t = P0 + (i - row0);

    const TIn* kv_t = reinterpret_cast<const TIn*>(p.kv) + i * D;
    float x[CPL], sv_t[CPL];
    float ik_t[ICPL > 0 ? ICPL : 1], is_t[ICPL > 0 ? ICPL : 1];
    const bool keep_state = t >= P1 - p.W;
    load_f<TIn, CPL>(kv_t + lane * CPL, x);
    if (keep_state) {
      load_f<TIn, CPL>(reinterpret_cast<const TIn*>(p.score) + i * D + lane * CPL, sv_t);
      if constexpr (ICPL > 0) {
        load_f<TIn, ICPL>(reinterpret_cast<const TIn*>(p.ikv) + i * DI + lane * ICPL, ik_t);
        load_f<TIn, ICPL>(reinterpret_cast<const TIn*>(p.iscore) + i * DI + lane * ICPL, is_t);
      }
    }

    // Everything above read only this call's inputs (and so did the slot lookups below):
    // it ran while the previous kernel finished. Pool writes, and the residual reads of
    // the window loop, wait for it.
    const int64_t swa_slot = slot_of(p.swa, b, t);
    const int64_t state_slot = keep_state ? slot_of(p.state, b, t) : -1;
    pdl_wait();

    // (1) sliding-window row: RoPE(kv_t, t)
    if (wb == 0) {
      const int64_t s = swa_slot;
      if (s >= 0) {
        float y[CPL];
#pragma unroll
        for (int k = 0; k < CPL; ++k) y[k] = x[k];
        rope_lane<CPL>(p.rope, y, lane, t);
        store_row<CPL>(p.swa, s, y, lane);
      } else if (s == -2) {
        raise_err(p.err, V4A_DEV_BAD_PAGE);
      }
    }

    // (2) raw residual row for the last W new positions
    if (keep_state && wb == 0) {
      const int64_t s = state_slot;
      if (s >= 0) {
        TIn* dst = reinterpret_cast<TIn*>(p.state.data) + s * (int64_t)p.state.width;
        store_f<TIn, CPL>(dst + lane * CPL, x);
        store_f<TIn, CPL>(dst + D + lane * CPL, sv_t);
        if constexpr (ICPL > 0) {
          store_f<TIn, ICPL>(dst + 2 * D + lane * ICPL, ik_t);
          store_f<TIn, ICPL>(dst + 2 * D + DI + lane * ICPL, is_t);
        }
      } else if (s == -2) {
        raise_err(p.err, V4A_DEV_BAD_PAGE);
      }
    }

    // (3) entry j whose window ends at t: window token o at position S*j + win_off + o is a
    // row of this call's inputs (position >= P0) or of the residual pool (before P0)
    const int64_t first = t - p.win_off - (p.W - 1);   // = S*j
    if (first < 0 || first % p.S != 0) return;
    const int64_t j = first / p.S;
    const TIn* kv_in = reinterpret_cast<const TIn*>(p.kv);
    const TIn* s_in = reinterpret_cast<const TIn*>(p.score);
    const TIn* ik_in = reinterpret_cast<const TIn*>(p.ikv);
    const TIn* is_in = reinterpret_cast<const TIn*>(p.iscore);
    // the window's rows are resolved once, lane o taking tokens o, o + 32, ... (the residual
    // rows' block-table lookups in parallel): status 0 absent, 1 an input row, 2 a residual
    // row, < 0 a residual row without a usable page; ref = input row or pool row
    __shared__ int64_t s_ref[kMaxWindow];
    __shared__ int8_t s_st[kMaxWindow];
    for (int o = (int)threadIdx.x; o < p.W; o += (int)blockDim.x) {
      const int64_t pos = j * p.S + p.win_off + o;
      int st = 0;
      int64_t ref = 0;
      if (pos >= P0) {
        st = 1;
        ref = row0 + (pos - P0);
      } else if (pos >= 0) {
        ref = slot_of(p.state, b, pos);
        st = ref >= 0 ? 2 : (int)ref;
      }
      s_st[o] = (int8_t)st;
      s_ref[o] = ref;
    }
    if constexpr (kWide) __syncthreads();
    else __syncwarp();
    auto fetch = [&](int o, WindowRow& w) -> int {
      const int st = s_st[o];
      if (st <= 0) return st;                      // absent, or -1 / -2 (page errors)
      const int64_t ref = s_ref[o];
      if (st == 1) {
        w.kv = kv_in + ref * D;
        w.s = s_in + ref * D;
        if constexpr (ICPL > 0) {
          w.ik = ik_in + ref * DI;
          w.is = is_in + ref * DI;
        }
      } else {
        const TIn* base = reinterpret_cast<const TIn*>(p.state.data) + ref * (int64_t)p.state.width;
        w.kv = base;
        w.s = base + D;
        if constexpr (ICPL > 0) {
          w.ik = base + 2 * D;
          w.is = base + 2 * D + DI;
        }
      }
      return 1;
    };
    if constexpr (kWide) build_entry_wide(p, b, j, lane, wb, fetch);
    else build_entry(p, b, j, lane, fetch);
  }
};

// Large calls (many new tokens per sequence, windows of at most 8 tokens): one persistent
// CTA per SM walks tiles of kTT consecutive new tokens of one sequence. A tile's rows and the
// W - 1 window tokens before them are staged in shared memory by bulk copies (a tile's input
// rows are contiguous in kv, s, ik and is: one copy per array; rows before the call's first
// position come from the residual pool, one copy per part of the row), double-buffered so
// the next tile streams in while this one is computed. Every row is read from memory once
// per tile (the window overlap between tiles, W - 1 rows, is read twice). The window rows,
// residual rows and entries are then computed from shared memory: warp w takes tokens
// w, w + 8, ... and entries w, w + 8, ... of the tile, with the same entry routine as the
// warp-per-token kernel, so both write identical bytes.
template <typename TIn, int CPL, int ICPL, bool kFp8>
struct CompressTile {
  using K = CompressKernel<TIn, CPL, ICPL, kFp8>;
  using WindowRow = typename K::WindowRow;
  static constexpr int D = CPL * 32, DI = ICPL * 32;
  static constexpr int kTT = 32;                    // new tokens per tile
  static constexpr int kMaxW = 8;                   // window tokens the staging holds
  static constexpr int kRows = kTT + kMaxW - 1;     // staged rows
  // Two groups of 8 warps, each with its own staging buffer: while one group computes a
  // tile the other computes the next (or waits for its copy), so each SM issues from 16
  // warps; group g takes the CTA's tiles j = g, g + 2, ...
  static constexpr int kWarps = 8, kGroups = 2, kThreads = kGroups * kWarps * 32;
  static constexpr int kMaxSeq = 1023;              // sequences of a call on this path (the
                                                    // 256 threads write prefix[0 .. kMaxSeq])
  static constexpr int kRowBytes = (2 * D + 2 * DI) * (int)sizeof(TIn);
  // one stage: kv, s [kRows][D] and ik, is [kRows][DI] (input type), row status [kRows]
  static constexpr int kKv = kRows * D * (int)sizeof(TIn);
  static constexpr int kIk = kRows * DI * (int)sizeof(TIn);
  static constexpr int kOffS = kKv, kOffIk = 2 * kKv, kOffIs = 2 * kKv + kIk;
  static constexpr int kOffSt = 2 * kKv + 2 * kIk;
  static constexpr int kStage = (kOffSt + kRows * 4 + 127) / 128 * 128;
  static constexpr int kOffPrefix = 2 * kStage;     // int32 [kMaxSeq + 1] tiles before sequence b
  static constexpr int kOffBar = (kOffPrefix + (kMaxSeq + 1) * 4 + 7) / 8 * 8;
  static constexpr int kOffMisc = kOffBar + 2 * 8;
  static constexpr int kSmem = kOffMisc + 16 + 128;   // + alignment slack
  static constexpr bool kFits = kSmem <= 227 * 1024;   // fp32 rows of 512 do not fit

  struct Tile {
    int b;
    int64_t r0, n, pa, P0, P1;   // input rows [r0, r0 + n) at positions pa .. pa + n - 1
  };

  static __device__ __forceinline__ bool tile_of(const CompressParams& p, const int* prefix, int k,
                                                 Tile& t) {
    if (k >= prefix[p.n_seq]) return false;
    int lo = 0, hi = p.n_seq - 1;                   // largest b with prefix[b] <= k
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= k) lo = mid;
      else hi = mid - 1;
    }
    const int64_t c = k - prefix[lo];
    const int64_t cu0 = __ldg(p.cu + lo), cu1 = __ldg(p.cu + lo + 1);
    t.b = lo;
    t.P0 = __ldg(p.start + lo);
    t.P1 = t.P0 + (cu1 - cu0);
    t.r0 = cu0 + c * kTT;
    t.n = min((int64_t)kTT, cu1 - t.r0);
    t.pa = t.P0 + c * kTT;
    return true;
  }

  // Warp 0: stage tile t (its rows and the W - 1 window tokens before them). Row status:
  // 1 staged, 0 a position before the sequence (absent), -1 / -2 a residual row without a
  // page or with a page outside the pool.
  static __device__ void issue(const CompressParams& p, const Tile& t, uint8_t* st, uint64_t* bar,
                               int lane) {
    const int W = p.W;
    const int64_t base = t.pa - (W - 1);
    const int n_rows = (int)t.n + W - 1;
    int* status = reinterpret_cast<int*>(st + kOffSt);
    const int64_t q_in = max(base, t.P0);          // first position read from the inputs
    const int k_in = (int)(q_in - base);           // < W: rows before it are residual rows
    const int n_in = n_rows - k_in;
    const int64_t r_in = t.r0 - (t.pa - q_in);
    int64_t slot = -1;
    int stt = 0;
    if (lane < k_in) {
      const int64_t q = base + lane;
      if (q >= 0) {
        slot = slot_of(p.state, t.b, q);
        stt = slot >= 0 ? 1 : (int)slot;
      }
      status[lane] = stt;
    }
    for (int k = k_in + lane; k < n_rows; k += 32) status[k] = 1;
    const uint32_t n_state = __popc(__ballot_sync(0xffffffffu, stt > 0));
    __syncwarp();
    if (lane == 0) tc::mbar_arrive_tx(bar, (uint32_t)(n_in + n_state) * kRowBytes);
    __syncwarp();
    constexpr int es = (int)sizeof(TIn);
    if (lane == 0) {
      tc::bulk_g2s(st + (size_t)k_in * D * es, reinterpret_cast<const TIn*>(p.kv) + r_in * D,
                   (uint32_t)(n_in * D * es), bar);
      tc::bulk_g2s(st + kOffS + (size_t)k_in * D * es, reinterpret_cast<const TIn*>(p.score) + r_in * D,
                   (uint32_t)(n_in * D * es), bar);
      if constexpr (ICPL > 0) {
        tc::bulk_g2s(st + kOffIk + (size_t)k_in * DI * es, reinterpret_cast<const TIn*>(p.ikv) + r_in * DI,
                     (uint32_t)(n_in * DI * es), bar);
        tc::bulk_g2s(st + kOffIs + (size_t)k_in * DI * es,
                     reinterpret_cast<const TIn*>(p.iscore) + r_in * DI, (uint32_t)(n_in * DI * es), bar);
      }
    }
    if (stt > 0) {
      const TIn* row = reinterpret_cast<const TIn*>(p.state.data) + slot * (int64_t)p.state.width;
      tc::bulk_g2s(st + (size_t)lane * D * es, row, (uint32_t)(D * es), bar);
      tc::bulk_g2s(st + kOffS + (size_t)lane * D * es, row + D, (uint32_t)(D * es), bar);
      if constexpr (ICPL > 0) {
        tc::bulk_g2s(st + kOffIk + (size_t)lane * DI * es, row + 2 * D, (uint32_t)(DI * es), bar);
        tc::bulk_g2s(st + kOffIs + (size_t)lane * DI * es, row + 2 * D + DI, (uint32_t)(DI * es), bar);
      }
    }
  }

  // All warps: the window and residual rows of the tile's tokens, then its entries.
  static __device__ void compute(const CompressParams& p, const Tile& t, const uint8_t* st, int warp,
                                 int lane, const float* rope_tab) {
    const int W = p.W, S = p.S;
    const TIn* kv_s = reinterpret_cast<const TIn*>(st);
    const TIn* s_s = reinterpret_cast<const TIn*>(st + kOffS);
    const TIn* ik_s = reinterpret_cast<const TIn*>(st + kOffIk);
    const TIn* is_s = reinterpret_cast<const TIn*>(st + kOffIs);
    const int* status = reinterpret_cast<const int*>(st + kOffSt);
    for (int i = warp; i < t.n; i += kWarps) {
      const int64_t pos = t.pa + i;
      const int k = i + W - 1;
      const int64_t sw = slot_of(p.swa, t.b, pos);
      if (sw >= 0) {
        float y[CPL];
        K::template load_g<TIn, CPL>(kv_s + k * D + lane * CPL, y);
        K::template rope_lane<CPL>(p.rope, y, lane, pos, rope_tab);
        K::template store_row<CPL>(p.swa, sw, y, lane);
      } else if (sw == -2) {
        raise_err(p.err, V4A_DEV_BAD_PAGE);
      }
      if (pos >= t.P1 - W) {                       // raw residual row for the last W positions
        const int64_t ss = slot_of(p.state, t.b, pos);
        if (ss >= 0) {
          TIn* dst = reinterpret_cast<TIn*>(p.state.data) + ss * (int64_t)p.state.width;
          constexpr int kV = CPL * (int)sizeof(TIn) / 16;   // 16-byte vectors per lane
          static_assert(CPL * sizeof(TIn) % 16 == 0, "whole vectors per lane");
#pragma unroll
          for (int v = 0; v < kV; ++v) {
            reinterpret_cast<uint4*>(dst + lane * CPL)[v] =
                reinterpret_cast<const uint4*>(kv_s + k * D + lane * CPL)[v];
            reinterpret_cast<uint4*>(dst + D + lane * CPL)[v] =
                reinterpret_cast<const uint4*>(s_s + k * D + lane * CPL)[v];
          }
          if constexpr (ICPL > 0) {
#pragma unroll
            for (int e = 0; e < ICPL; ++e) {
              dst[2 * D + lane * ICPL + e] = ik_s[k * DI + lane * ICPL + e];
              dst[2 * D + DI + lane * ICPL + e] = is_s[k * DI + lane * ICPL + e];
            }
          }
        } else if (ss == -2) {
          raise_err(p.err, V4A_DEV_BAD_PAGE);
        }
      }
    }
    // entries completed by the tile's tokens: position tt completes entry (tt - c0) / S
    const int64_t c0 = p.win_off + W - 1;
    int64_t tt0 = max(t.pa, c0);
    tt0 += (S - (tt0 - c0) % S) % S;
    const int64_t j0 = (tt0 - c0) / S;            // entry completed at tt0 (one division a tile)
    int64_t j = j0 + warp;
    for (int64_t tt = tt0 + (int64_t)warp * S; tt < t.pa + t.n; tt += (int64_t)kWarps * S, j += kWarps) {
      const int ko = (int)(tt - t.pa);            // staged row of the window's first token
      K::build_entry(p, t.b, j, lane, [&](int o, WindowRow& w) -> int {
        const int k = ko + o;
        const int sk = status[k];
        if (sk <= 0) return sk;
        w.kv = kv_s + k * D;
        w.s = s_s + k * D;
        if constexpr (ICPL > 0) {
          w.ik = ik_s + k * DI;
          w.is = is_s + k * DI;
        }
        return 1;
      }, rope_tab);
    }
  }

  static __device__ void run(const CompressParams& p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = tc::smem_u32(smem_raw);
    uint8_t* sm = smem_raw + ((128u - (raw_addr & 127u)) & 127u);
    int* prefix = reinterpret_cast<int*>(sm + kOffPrefix);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + kOffBar);
    volatile int* abort_flag = reinterpret_cast<int*>(sm + kOffMisc);
    __shared__ int warp_tot[kGroups * kWarps];
    __shared__ float rope_tab[4 * kMaxRopePairs];
    stage_rope(p.rope, rope_tab, threadIdx.x, kThreads);   // read after the barriers below
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
      tc::mbar_init(full, 1);
      tc::mbar_init(full + 1, 1);
      *abort_flag = 0;
      tc::fence_mbar_init();
    }
    // tiles before each sequence: thread tid counts sequences 4 tid .. 4 tid + 3 (inputs
    // only, before waiting for the previous kernel)
    int cnt[4], sum = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int b = 4 * tid + u;
      cnt[u] = 0;
      if (b < p.n_seq) {
        const int64_t n = (int64_t)__ldg(p.cu + b + 1) - __ldg(p.cu + b);
        cnt[u] = n > 0 ? (int)((n + kTT - 1) / kTT) : 0;
      }
      sum += cnt[u];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int before = 0;
#pragma unroll
    for (int w = 0; w < kGroups * kWarps; ++w) before += w < warp ? warp_tot[w] : 0;
    int run_sum = before + incl - sum;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int b = 4 * tid + u;
      if (b <= p.n_seq) prefix[b] = run_sum;      // prefix[n_seq] is the total
      run_sum += cnt[u];
    }
    __syncthreads();
    const int total = prefix[p.n_seq];
    pdl_wait();   // residual rows may come from the previous kernel; every pool write waits

    const int grp = warp / kWarps, gw = warp % kWarps;
    uint8_t* stage = sm + grp * kStage;
    uint64_t* bar = full + grp;
    // barrier of the group's 256 threads (ids 1 and 2; 0 is __syncthreads); reports whether
    // every thread of the group passed `pred`
    auto group_sync_and = [&](bool pred) -> bool {
      uint32_t r;
      asm volatile("{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.and.pred q, %2, %3, p; selp.u32 %0, 1, 0, q; }"
                   : "=r"(r)
                   : "r"((uint32_t)pred), "r"(1 + grp), "r"(kWarps * 32)
                   : "memory");
      return r != 0;
    };
    Tile t;
    if (gw == 0) {
      const int k = blockIdx.x + grp * gridDim.x;
      if (tile_of(p, prefix, k, t)) issue(p, t, stage, bar, lane);
    }
    int i = 0;                                     // tiles of this group so far
    bool ok = true;
    for (int k = blockIdx.x + grp * gridDim.x; k < total; k += kGroups * gridDim.x, ++i) {
      tile_of(p, prefix, k, t);
      // every thread of the group takes the same decision, so its barriers always pair up
      const bool got = tc::mbar_wait(bar, i & 1, abort_flag, p.err);
      if (!group_sync_and(got)) { ok = false; break; }
      compute(p, t, stage, gw, lane, rope_tab);
      group_sync_and(true);                        // every warp of the group is done with the stage
      if (gw == 0) {
        const int k2 = k + kGroups * gridDim.x;
        tc::fence_proxy_async();                  // reads of the stage before the next copy
        if (tile_of(p, prefix, k2, t)) issue(p, t, stage, bar, lane);
      }
    }
    if (!ok && gw == 0 && lane == 0) {             // a copy still in flight lands before exit
      if (blockIdx.x + (int64_t)(grp + kGroups * i) * gridDim.x < total) tc::mbar_wait_drain(bar, i & 1);
    }
    __syncthreads();
  }
};

template <typename TIn, int CPL, int ICPL, bool kFp8>
__global__ void __launch_bounds__(512, 1) compress_tile_kernel(const __grid_constant__ CompressParams p) {
  pdl_trigger();
  CompressTile<TIn, CPL, ICPL, kFp8>::run(p);
}

template <typename TIn, int CPL, int ICPL, bool kFp8, bool kWide>
__global__ void __launch_bounds__(256) compress_insert_kernel(const __grid_constant__ CompressParams p) {
  pdl_trigger();   // the kernel waits (pdl_wait) after loading its inputs
  CompressKernel<TIn, CPL, ICPL, kFp8>::template run<kWide>(p);
}

template <typename TIn, int CPL, int ICPL, bool kFp8>
cudaError_t launch(const CompressParams& p, cudaStream_t st) {
  using Tile = CompressTile<TIn, CPL, ICPL, kFp8>;
  // Many tokens per sequence, small windows, no query rows: the tile kernel (one persistent
  // CTA per SM, rows staged in shared memory).
  if constexpr (Tile::kFits) {
  if (p.n_qrows == 0 && p.W <= Tile::kMaxW && p.n_tokens >= 256 && p.n_seq <= Tile::kMaxSeq &&
      p.n_tokens >= 8 * (int64_t)p.n_seq) {
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t max_tiles = p.n_tokens / Tile::kTT + p.n_seq;   // bound on the tile count
    const int grid = (int)(max_tiles < sms ? max_tiles : sms);
    cudaError_t e = cudaFuncSetAttribute(compress_tile_kernel<TIn, CPL, ICPL, kFp8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Tile::kSmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(compress_tile_kernel<TIn, CPL, ICPL, kFp8>, dim3(grid), dim3(Tile::kThreads), Tile::kSmem,
                   st, p);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  }
  // One warp per block (the c4a bf16 kernel compiles to 128 registers a thread): such a
  // block fits on an SM beside a persistent indexer CTA, so a small insert never holds
  // an SM the indexer is waiting for.
  // Windows longer than a warp (c128a) and no indexer rows or query rows: blocks of four
  // warps, one token each, so that an entry's 128-token window is summed by four warps.
  if constexpr (ICPL == 0) {
    using K = CompressKernel<TIn, CPL, ICPL, kFp8>;
    if (p.W > 32 && p.n_qrows == 0) {
      const cudaError_t e = launch_pdl(compress_insert_kernel<TIn, CPL, ICPL, kFp8, true>, dim3((unsigned)p.n_tokens),
                                       dim3(32 * K::kWideWarps), 0, st, p);
      return e != cudaSuccess ? e : cudaGetLastError();
    }
  }
  const int threads = 32;
  const int64_t blocks = p.n_tokens + p.n_qrows;
  const cudaError_t e = launch_pdl(compress_insert_kernel<TIn, CPL, ICPL, kFp8, false>, dim3((unsigned)blocks), dim3(threads), 0, st, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

int launch_compress_insert(const CompressParams& p, int dtype, cudaStream_t st) {
  if (p.n_tokens == 0 && p.n_qrows == 0) return V4A_OK;
  const int D = p.D, DI = p.DI;
  cudaError_t e = cudaErrorInvalidValue;
  bool done = false;
  if (dtype == V4A_BF16_FP8) {
    if (D == 512 && DI == 128) { e = launch<__nv_bfloat16, 16, 4, true>(p, st); done = true; }
    else if (D == 512 && DI == 0) { e = launch<__nv_bfloat16, 16, 0, true>(p, st); done = true; }
  } else {
    if (D == 128 && DI == 32) { e = launch<float, 4, 1, false>(p, st); done = true; }
    else if (D == 128 && DI == 0) { e = launch<float, 4, 0, false>(p, st); done = true; }
    else if (D == 512 && DI == 128) { e = launch<float, 16, 4, false>(p, st); done = true; }
    else if (D == 512 && DI == 0) { e = launch<float, 16, 0, false>(p, st); done = true; }
  }
  if (!done) return V4A_ERR_UNSUPPORTED;
  return e == cudaSuccess ? V4A_OK : V4A_ERR_CUDA;
}

}  // namespace v4a
