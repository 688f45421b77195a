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

namespace v4a {

namespace {

template <typename TIn, int CPL, int ICPL, bool kFp8>
struct CompressKernel {
  static constexpr int D = CPL * 32;
  static constexpr int DI = ICPL * 32;

  struct Row {
    const TIn* kv;
    const TIn* s;
    const TIn* ik;
    const TIn* is;
    bool ok;
  };

  // fp8 row store: per-row scale amax/448 (1 if the row is zero), e4m3 RNE satfinite of
  // y/scale; fp32 rows are stored as they are.
  template <int N>
  static __device__ __forceinline__ void store_row(const CacheView& c, int64_t slot, float (&y)[N],
                                                   int lane) {
    if constexpr (kFp8) {
      float amax = 0.f;
#pragma unroll
      for (int k = 0; k < N; ++k) amax = fmaxf(amax, fabsf(y[k]));
      amax = warp_max(amax);
      float scale = amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.0f;
      uint8_t* dst = reinterpret_cast<uint8_t*>(c.data) + slot * (int64_t)c.width + lane * N;
      if constexpr (N % 4 == 0) {
        uint32_t words[N / 4];
#pragma unroll
        for (int k = 0; k < N / 4; ++k) {
          uint32_t lo = e4m3x2_encode(__fdiv_rn(y[4 * k], scale), __fdiv_rn(y[4 * k + 1], scale));
          uint32_t hi = e4m3x2_encode(__fdiv_rn(y[4 * k + 2], scale), __fdiv_rn(y[4 * k + 3], scale));
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
        for (int k = 0; k < N; ++k) {
          float v = __fdiv_rn(y[k], scale);
          dst[k] = (uint8_t)(e4m3x2_encode(v, 0.f) & 0xFF);
        }
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
    uint32_t packed = 0;
#pragma unroll
    for (int k = 0; k < N; ++k) packed |= e2m1_encode(__fdiv_rn(y[k], scale)) << (4 * k);
    uint8_t* dst = reinterpret_cast<uint8_t*>(c.data) + slot * (int64_t)c.width + lane * (N / 2);
    *reinterpret_cast<uint16_t*>(dst) = (uint16_t)packed;
    if (lane == 0) c.scale[slot] = scale;
  }

  // Rotate the lane's channels that fall in the rotated tail (adjacent pairs).
  template <int N>
  static __device__ __forceinline__ void rope_lane(const Rope& rp, float (&y)[N], int lane,
                                                   int64_t pos) {
    const int tail0 = rp.D - rp.d_r;
#pragma unroll
    for (int k = 0; k < N; k += 2) {
      int d = lane * N + k;
      if (d >= tail0) {
        float c, s;
        rope_cs(rp, pos, (d - tail0) >> 1, c, s);
        float a = y[k], b = y[k + 1];
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

  static __device__ void run(const CompressParams& p) {
    const int lane = threadIdx.x & 31;
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
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
    {
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
    if (keep_state) {
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

    // (3) entry j whose window ends at t
    const int64_t first = t - p.win_off - (p.W - 1);   // = S*j
    if (first < 0 || first % p.S != 0) return;
    const int64_t j = first / p.S;
    const int64_t e_slot = slot_of(p.attn, b, j);
    const int64_t i_slot = ICPL > 0 ? slot_of(p.idx, b, j) : -1;
    if (e_slot == -2 || i_slot == -2) raise_err(p.err, V4A_DEV_BAD_PAGE);
    if (e_slot < 0 && i_slot < 0) return;

    // online per-channel softmax over the window's present tokens
    float m[CPL], l[CPL], acc[CPL];
    float im[ICPL > 0 ? ICPL : 1], il[ICPL > 0 ? ICPL : 1], iacc[ICPL > 0 ? ICPL : 1];
#pragma unroll
    for (int k = 0; k < CPL; ++k) { m[k] = -INFINITY; l[k] = 0.f; acc[k] = 0.f; }
#pragma unroll
    for (int k = 0; k < (ICPL > 0 ? ICPL : 1); ++k) { im[k] = -INFINITY; il[k] = 0.f; iacc[k] = 0.f; }

#pragma unroll 8
    for (int o = 0; o < p.W; ++o) {
      const int64_t pos = j * p.S + p.win_off + o;
      if (pos < 0) continue;                       // before the sequence: absent
      const TIn *kvp, *sp, *ikp = nullptr, *isp = nullptr;
      if (pos >= P0) {
        const int64_t r = row0 + (pos - P0);
        kvp = reinterpret_cast<const TIn*>(p.kv) + r * D;
        sp = reinterpret_cast<const TIn*>(p.score) + r * D;
        if constexpr (ICPL > 0) {
          ikp = reinterpret_cast<const TIn*>(p.ikv) + r * DI;
          isp = reinterpret_cast<const TIn*>(p.iscore) + r * DI;
        }
      } else {
        const int64_t s = slot_of(p.state, b, pos);
        if (!slot_ok(s, p.err)) return;            // residual row missing: skip the entry
        const TIn* base = reinterpret_cast<const TIn*>(p.state.data) + s * (int64_t)p.state.width;
        kvp = base;
        sp = base + D;
        if constexpr (ICPL > 0) {
          ikp = base + 2 * D;
          isp = base + 2 * D + DI;
        }
      }
      float kvv[CPL], sv[CPL], bv[CPL];
      load_f<TIn, CPL>(kvp + lane * CPL, kvv);
      load_f<TIn, CPL>(sp + lane * CPL, sv);
      load_f<float, CPL>(p.bias + (int64_t)o * D + lane * CPL, bv);
#pragma unroll
      for (int k = 0; k < CPL; ++k) {
        float z = sv[k] + bv[k];
        float mn = fmaxf(m[k], z);
        float corr = expf(m[k] - mn);
        float e = expf(z - mn);
        l[k] = l[k] * corr + e;
        acc[k] = acc[k] * corr + e * kvv[k];
        m[k] = mn;
      }
      if constexpr (ICPL > 0) {
        float a[ICPL], sc[ICPL], bb[ICPL];
        load_f<TIn, ICPL>(ikp + lane * ICPL, a);
        load_f<TIn, ICPL>(isp + lane * ICPL, sc);
        load_f<float, ICPL>(p.ibias + (int64_t)o * DI + lane * ICPL, bb);
#pragma unroll
        for (int k = 0; k < ICPL; ++k) {
          float z = sc[k] + bb[k];
          float mn = fmaxf(im[k], z);
          float corr = expf(im[k] - mn);
          float e = expf(z - mn);
          il[k] = il[k] * corr + e;
          iacc[k] = iacc[k] * corr + e * a[k];
          im[k] = mn;
        }
      }
    }

    if (e_slot >= 0) {
      float c[CPL], g[CPL];
      float ss = 0.f;
#pragma unroll
      for (int k = 0; k < CPL; ++k) {
        c[k] = __fdiv_rn(acc[k], l[k]);
        ss = fmaf(c[k], c[k], ss);
      }
      ss = warp_sum(ss);
      const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fdiv_rn(ss, (float)D) + p.eps));
      load_f<float, CPL>(p.gamma + lane * CPL, g);
#pragma unroll
      for (int k = 0; k < CPL; ++k) c[k] = c[k] * inv * g[k];
      rope_lane<CPL>(p.rope, c, lane, j * p.S);
      store_row<CPL>(p.attn, e_slot, c, lane);
    }
    if constexpr (ICPL > 0) {
      if (i_slot >= 0) {
        float c[ICPL];
#pragma unroll
        for (int k = 0; k < ICPL; ++k) c[k] = __fdiv_rn(iacc[k], il[k]);
        if constexpr (kFp8 && ICPL == 4) {
          if (p.idx_fp4) store_row_fp4<ICPL>(p.idx, i_slot, c, lane);
          else store_row<ICPL>(p.idx, i_slot, c, lane);
        } else {
          store_row<ICPL>(p.idx, i_slot, c, lane);
        }
      }
    }
  }
};

template <typename TIn, int CPL, int ICPL, bool kFp8>
__global__ void __launch_bounds__(256) compress_insert_kernel(const __grid_constant__ CompressParams p) {
  pdl_trigger();   // the kernel waits (pdl_wait) after loading its inputs
  CompressKernel<TIn, CPL, ICPL, kFp8>::run(p);
}

template <typename TIn, int CPL, int ICPL, bool kFp8>
cudaError_t launch(const CompressParams& p, cudaStream_t st) {
  // One warp per block (the c4a bf16 kernel compiles to 128 registers a thread): such a
  // block fits on an SM beside a persistent indexer CTA, so a small insert never holds
  // an SM the indexer is waiting for.
  const int threads = 32;
  const int64_t blocks = p.n_tokens + p.n_qrows;
  const cudaError_t e = launch_pdl(compress_insert_kernel<TIn, CPL, ICPL, kFp8>, dim3((unsigned)blocks), dim3(threads), 0, st, p);
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
