// Shared-K=V attention over the selected (c4a) or all visible (c128a) compressed entries
// plus the sliding window, with inverse RoPE on the output (steps a8, a9).
//
// [notes] "DeepSeek V4 in vLLM 技术博客详尽笔记", Inverse RoPE 的数学原理:
//   out = (sum_x softmax_x(q~ . key_x) key_x) R^-1(theta_p),
// one stored vector per entry serving as key and value (共享 Key-Value 向量), and
// [blog] 短滑動窗口 for the 128 uncompressed local tokens.
//
// Key list of a query at p: positions [0, n_ent) are compressed entries (top-k list slots,
// -1 slots masked; or entries 0..n_vis-1 when dense), positions [n_ent, n_ent + n_swa) the
// window tokens max(0, p-swa+1) .. p. Split s of a query handles keys
// [s*keys_per_split, (s+1)*keys_per_split); splits > 1 write (m, l, o) partials that
// attn_merge combines.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace v4a {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kChunk = 32;        // keys per shared-memory chunk
constexpr int kThreads = 256;     // 8 warps

struct KeyRef {
  int64_t slot;                   // pool row, or < 0 when masked
  bool is_swa;
};

// Resolve key x of query (seq, p): entry or window token, its pool row, visibility.
__device__ __forceinline__ KeyRef key_ref(const AttnParams& p, int qi, int seq, int64_t pos,
                                          int64_t n_ent, int64_t n_vis, int64_t t0, int64_t x) {
  KeyRef r{-1, false};
  if (x < n_ent) {
    int64_t j = p.topk ? (int64_t)__ldg(p.topk + (int64_t)qi * p.k + x) : x;
    if (j < 0) return r;                         // padding slot of the top-k list
    if (j >= n_vis) { raise_err(p.err, V4A_DEV_BAD_INDEX); return r; }
    int64_t s = slot_of(p.attn, seq, j);
    if (!slot_ok(s, p.err)) return r;
    r.slot = s;
  } else {
    int64_t t = t0 + (x - n_ent);
    int64_t s = slot_of(p.swa, seq, t);
    if (!slot_ok(s, p.err)) return r;
    r.slot = s;
    r.is_swa = true;
  }
  return r;
}

// CUDA-core kernel: fp32 queries in shared memory, keys dequantised into a padded chunk.
// Warp w owns heads w*HPW .. w*HPW+HPW-1; lane l owns dims l, l+32, ... of every head.
template <typename QT, bool kFp8, typename OT, int H, int D>
__global__ void __launch_bounds__(kThreads) attn_simt(const __grid_constant__ AttnParams p) {
  pdl_trigger();
  pdl_wait();
  constexpr int HPW = H / 8;
  constexpr int DPL = D / 32;
  constexpr int KS = D + 1;                      // padded key row (conflict-free columns)
  extern __shared__ float smem[];
  float* qs = smem;                              // [H][D]
  float* kb = smem + H * D;                      // [kChunk][KS]
  __shared__ int64_t kslot[kChunk];
  __shared__ int kswa[kChunk];
  __shared__ float csn[kMaxRopePairs][2];

  const int qi = blockIdx.y, split = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seq = __ldg(p.q_seq + qi);
  const int64_t pos = __ldg(p.q_pos + qi);
  const int64_t n_vis = visible_entries(pos, p.S, p.W, p.win_off);
  const int64_t n_ent = p.topk ? p.k : n_vis;
  const int64_t t0 = pos - p.swa_len + 1 > 0 ? pos - p.swa_len + 1 : 0;
  const int64_t n_keys = n_ent + (pos - t0 + 1);
  if (split == 0 && tid == 0 && n_keys > (int64_t)p.n_split * p.keys_per_split)
    raise_err(p.err, V4A_DEV_BAD_POS);
  const int64_t x_begin = (int64_t)split * p.keys_per_split;
  const int64_t x_end = min(n_keys, x_begin + p.keys_per_split);

  // RoPE(q, p) * scale * log2(e) into shared memory
  const int n_pairs = p.rope.d_r / 2;
  for (int i = tid; i < n_pairs; i += kThreads) {
    float c, s;
    rope_cs(p.rope, pos, i, c, s);
    csn[i][0] = c;
    csn[i][1] = s;
  }
  __syncthreads();
  const QT* q = reinterpret_cast<const QT*>(p.q) + (int64_t)qi * H * D;
  const float qscale = p.scale * kLog2e;
  const int tail0 = D - p.rope.d_r;
  for (int e = tid * 2; e < H * D; e += kThreads * 2) {
    const int d = e % D;
    float a = Elem<QT>::to_f(q[e]), b = Elem<QT>::to_f(q[e + 1]);
    if (d >= tail0) {
      const int i = (d - tail0) >> 1;
      const float c = csn[i][0], s = csn[i][1];
      const float ra = a * c - b * s, rb = a * s + b * c;
      a = ra;
      b = rb;
    }
    qs[e] = a * qscale;
    qs[e + 1] = b * qscale;
  }

  float o[HPW][DPL];
  float m[HPW], l[HPW];
#pragma unroll
  for (int hh = 0; hh < HPW; ++hh) {
    m[hh] = -INFINITY;
    l[hh] = 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) o[hh][i] = 0.f;
  }

  for (int64_t c0 = x_begin; c0 < x_end; c0 += kChunk) {
    const int n_here = (int)min((int64_t)kChunk, x_end - c0);
    __syncthreads();
    if (tid < kChunk) {
      KeyRef r{-1, false};
      if (tid < n_here) r = key_ref(p, qi, seq, pos, n_ent, n_vis, t0, c0 + tid);
      kslot[tid] = r.slot;
      kswa[tid] = r.is_swa;
    }
    __syncthreads();
    // dequantise the chunk: 8 threads per row, 16-byte segments
    for (int task = tid; task < kChunk * (D / 16); task += kThreads) {
      const int row = task / (D / 16), seg = task % (D / 16);
      float* dst = kb + row * KS + seg * 16;
      const int64_t s = kslot[row];
      if (s < 0) {
#pragma unroll
        for (int k = 0; k < 16; ++k) dst[k] = 0.f;
        continue;
      }
      const CacheView& cv = kswa[row] ? p.swa : p.attn;
      if constexpr (kFp8) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(
            reinterpret_cast<const uint8_t*>(cv.data) + s * (int64_t)cv.width + seg * 16));
        const float sc = __ldg(cv.scale + s);
        const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          float f[4];
          e4m3x4_decode(w4[v], f);
#pragma unroll
          for (int k = 0; k < 4; ++k) dst[4 * v + k] = f[k] * sc;
        }
      } else {
        const float* src = reinterpret_cast<const float*>(cv.data) + s * (int64_t)cv.width + seg * 16;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const float4 f = __ldg(reinterpret_cast<const float4*>(src) + v);
          dst[4 * v] = f.x; dst[4 * v + 1] = f.y; dst[4 * v + 2] = f.z; dst[4 * v + 3] = f.w;
        }
      }
    }
    __syncthreads();

    // logits: lane = key of the chunk
    float lg[HPW];
#pragma unroll
    for (int hh = 0; hh < HPW; ++hh) lg[hh] = 0.f;
    const float* krow = kb + lane * KS;
    for (int d = 0; d < D; ++d) {
      const float kv = krow[d];
#pragma unroll
      for (int hh = 0; hh < HPW; ++hh) lg[hh] = fmaf(qs[(warp * HPW + hh) * D + d], kv, lg[hh]);
    }
    const bool valid = lane < n_here && kslot[lane] >= 0;
#pragma unroll
    for (int hh = 0; hh < HPW; ++hh) {
      const float x = valid ? lg[hh] : -INFINITY;
      const float cm = warp_max(x);
      const float mn = fmaxf(m[hh], cm);
      const float corr = mn == -INFINITY ? 1.f : exp2f(m[hh] - mn);
      const float pr = valid ? exp2f(x - mn) : 0.f;
      l[hh] = l[hh] * corr + warp_sum(pr);
      m[hh] = mn;
      lg[hh] = pr;
#pragma unroll
      for (int i = 0; i < DPL; ++i) o[hh][i] *= corr;
    }
    for (int x = 0; x < n_here; ++x) {
      const float* kr = kb + x * KS;
      float kv[DPL];
#pragma unroll
      for (int i = 0; i < DPL; ++i) kv[i] = kr[lane + 32 * i];
#pragma unroll
      for (int hh = 0; hh < HPW; ++hh) {
        const float px = __shfl_sync(0xffffffffu, lg[hh], x);
#pragma unroll
        for (int i = 0; i < DPL; ++i) o[hh][i] = fmaf(px, kv[i], o[hh][i]);
      }
    }
  }

  if (p.n_split > 1) {
    const int64_t base = ((int64_t)qi * p.n_split + split) * H;
#pragma unroll
    for (int hh = 0; hh < HPW; ++hh) {
      const int h = warp * HPW + hh;
      float* po = p.part_o + (base + h) * D;
#pragma unroll
      for (int i = 0; i < DPL; ++i) po[lane + 32 * i] = o[hh][i];
      if (lane == 0) {
        p.part_ml[(base + h) * 2] = m[hh];
        p.part_ml[(base + h) * 2 + 1] = l[hh];
      }
    }
    return;
  }
  // single split: normalise, inverse RoPE at p, store
  OT* out = reinterpret_cast<OT*>(p.out) + (int64_t)qi * H * D;
#pragma unroll
  for (int hh = 0; hh < HPW; ++hh) {
    const int h = warp * HPW + hh;
    const float inv = l[hh] > 0.f ? 1.f / l[hh] : 0.f;
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
      const int d = lane + 32 * i;
      float v = o[hh][i] * inv;
      const float partner = __shfl_xor_sync(0xffffffffu, v, 1);
      if (d >= tail0) {
        const int pi = (d - tail0) >> 1;
        const float c = csn[pi][0], s = csn[pi][1];
        // inverse rotation: (a, b) -> (a c + b s, -a s + b c)
        v = (d & 1) ? (-partner * s + v * c) : (v * c + partner * s);
      }
      out[(int64_t)h * D + d] = Elem<OT>::from_f(v);
    }
  }
}

// Combine split partials, normalise, inverse RoPE, store. One warp per (query, head): the
// lanes first reduce the split maxima and denominators (split s on lane s % 32), then lane
// l owns the rotation pairs (d, d+1), d = 2l + 64i, of that head; all partial loads of a
// group of splits are issued before they are used.
// The combine is sum_s w_s o_s / sum_s w_s l_s with w_s = 2^(m_s - max): o_s is the range's
// unnormalised numerator in the scale its (m_s, l_s) state (kBf16: stored as bf16 pairs,
// the tensor-core kernel's; else fp32).
template <typename OT, int kPairs, bool kBf16 = false>
__global__ void __launch_bounds__(256) attn_merge(const __grid_constant__ AttnParams p) {
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qi = blockIdx.x, h = blockIdx.y * 8 + warp;
  const int64_t pos = __ldg(p.q_pos + qi);
  // the query's rotation angles, once for the block's eight heads (inputs only)
  __shared__ float2 cs[kMaxRopePairs];
  if (threadIdx.x < (p.rope.d_r >> 1)) {
    float c, sn;
    rope_cs(p.rope, pos, threadIdx.x, c, sn);
    cs[threadIdx.x] = make_float2(c, sn);
  }
  __syncthreads();
  if (h >= p.H) return;
  const int H = p.H, D = p.D, tail0 = D - p.rope.d_r;
  const int64_t row0 = (int64_t)qi * p.n_split * H + h;          // (qi, split 0, h)
  pdl_wait();
  // One round of loads: every split's (m, l) (lane s holds split s, s < 32) and the first
  // four splits' partial rows; the weights are formed from registers afterwards.
  float m_l = -INFINITY, l_l = 0.f;
  if (lane < p.n_split) {
    m_l = p.part_ml[(row0 + (int64_t)lane * H) * 2];
    l_l = p.part_ml[(row0 + (int64_t)lane * H) * 2 + 1];
  }
  // bf16 partials stay packed (one 32-bit word per pair) until they are used, which halves
  // the registers and lets more warps keep loads in flight
  using VT = typename std::conditional<kBf16, uint32_t, float2>::type;
  VT v[4][kPairs];
  auto pair_of = [](const VT& x) -> float2 {
    if constexpr (kBf16) return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
    else return x;
  };
  auto load4 = [&](int s0) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int s = s0 + u;
      if constexpr (kBf16) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(p.part_o) + ((row0 + (int64_t)s * H) * D >> 1);
#pragma unroll
        for (int i = 0; i < kPairs; ++i) v[u][i] = s < p.n_split ? src[lane + 32 * i] : 0u;
      } else {
        const float* src = p.part_o + (row0 + (int64_t)s * H) * D;
#pragma unroll
        for (int i = 0; i < kPairs; ++i)
          v[u][i] = s < p.n_split ? *reinterpret_cast<const float2*>(src + 2 * lane + 64 * i)
                                  : make_float2(0.f, 0.f);
      }
    }
  };
  load4(0);
  float mx = m_l;
  for (int s = lane + 32; s < p.n_split; s += 32) mx = fmaxf(mx, p.part_ml[(row0 + (int64_t)s * H) * 2]);
  mx = warp_max(mx);
  float L = (mx != -INFINITY && m_l != -INFINITY) ? l_l * exp2f(m_l - mx) : 0.f;
  for (int s = lane + 32; s < p.n_split; s += 32) {
    const float ms = p.part_ml[(row0 + (int64_t)s * H) * 2];
    if (mx != -INFINITY && ms != -INFINITY) L += p.part_ml[(row0 + (int64_t)s * H) * 2 + 1] * exp2f(ms - mx);
  }
  L = warp_sum(L);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  float a[kPairs], b[kPairs];
#pragma unroll
  for (int i = 0; i < kPairs; ++i) a[i] = b[i] = 0.f;
  for (int s0 = 0; s0 < p.n_split; s0 += 4) {
    if (s0 > 0) load4(s0);
    float wg[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int s = s0 + u;
      float ms = -INFINITY;
      if (s < p.n_split) ms = s < 32 ? __shfl_sync(0xffffffffu, m_l, s) : p.part_ml[(row0 + (int64_t)s * H) * 2];
      wg[u] = (s < p.n_split && mx != -INFINITY && ms != -INFINITY) ? exp2f(ms - mx) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (wg[u] == 0.f) continue;   // a range without keys wrote no partial: never multiply it
#pragma unroll
      for (int i = 0; i < kPairs; ++i) {
        const float2 f = pair_of(v[u][i]);
        a[i] = fmaf(f.x, wg[u], a[i]);
        b[i] = fmaf(f.y, wg[u], b[i]);
      }
    }
  }
  float x[kPairs], y[kPairs];
#pragma unroll
  for (int i = 0; i < kPairs; ++i) {
    const int d = 2 * lane + 64 * i;
    x[i] = a[i] * inv;
    y[i] = b[i] * inv;
    if (d >= tail0) {
      const float2 r = cs[(d - tail0) >> 1];
      const float c = r.x, sn = r.y;
      const float rx = x[i] * c + y[i] * sn, ry = -x[i] * sn + y[i] * c;
      x[i] = rx;
      y[i] = ry;
    }
  }
  if (p.out_scale) {
    // fp8 output ([notes] 融合 2：Inverse RoPE + FP8 Quant): per (query, head) row,
    // scale = amax/448 (1 for a zero row), code = e4m3 RNE satfinite of value/scale
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kPairs; ++i) amax = fmaxf(amax, fmaxf(fabsf(x[i]), fabsf(y[i])));
    amax = warp_max(amax);
    const float scale = amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.0f;
    uint8_t* codes = reinterpret_cast<uint8_t*>(p.out) + ((int64_t)qi * H + h) * D;
#pragma unroll
    for (int i = 0; i < kPairs; ++i)
      *reinterpret_cast<uint16_t*>(codes + 2 * lane + 64 * i) =
          e4m3x2_encode(__fdiv_rn(x[i], scale), __fdiv_rn(y[i], scale));
    if (lane == 0) p.out_scale[(int64_t)qi * H + h] = scale;
    return;
  }
  OT* out = reinterpret_cast<OT*>(p.out) + ((int64_t)qi * H + h) * D;
#pragma unroll
  for (int i = 0; i < kPairs; ++i) {
    const int d = 2 * lane + 64 * i;
    if constexpr (std::is_same<OT, __nv_bfloat16>::value) {   // the pair as one 32-bit store
      *reinterpret_cast<__nv_bfloat162*>(out + d) = __floats2bfloat162_rn(x[i], y[i]);
    } else {
      out[d] = Elem<OT>::from_f(x[i]);
      out[d + 1] = Elem<OT>::from_f(y[i]);
    }
  }
}

template <typename QT, bool kFp8, typename OT, int H, int D>
cudaError_t launch_simt(const AttnParams& p, cudaStream_t st) {
  const size_t smem = (size_t)(H * D + kChunk * (D + 1)) * sizeof(float);
  cudaFuncSetAttribute(attn_simt<QT, kFp8, OT, H, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)smem);
  dim3 grid((unsigned)p.n_split, (unsigned)p.n_q);
  cudaError_t e = launch_pdl(attn_simt<QT, kFp8, OT, H, D>, grid, dim3(kThreads), smem, st, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess || p.n_split == 1) return e;
  e = launch_pdl(attn_merge<OT, D / 64>, dim3((unsigned)p.n_q, (unsigned)((p.H + 7) / 8)), dim3(256), 0, st, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

int launch_attention(const AttnParams& p, int dtype, cudaStream_t st) {
  if (p.n_q == 0) return V4A_OK;
  cudaError_t e;
  if (dtype == V4A_BF16_FP8 && p.H == 64 && p.D == 512)
  {
    e = launch_attention_tc(p, st);
    if (e == cudaSuccess && p.n_split > 1) {
      // A plain launch (full dependency on the attention kernel): launched early through
      // programmatic dependent launch, the merge's waiting CTAs held SMs during attention
      // and the next kernels started later (decode step 49.2 -> 47.0 us without it); with
      // the attention CTAs releasing it only as they leave, the step measured 3 us slower.
      attn_merge<__nv_bfloat16, 8, true><<<dim3((unsigned)p.n_q, (unsigned)((p.H + 7) / 8)), dim3(256), 0, st>>>(p);
      e = cudaGetLastError();
    }
  }
  else if (dtype == V4A_FP32 && p.H == 8 && p.D == 128)
    e = launch_simt<float, false, float, 8, 128>(p, st);
  else if (dtype == V4A_FP32 && p.H == 64 && p.D == 512)
    e = launch_simt<float, false, float, 64, 512>(p, st);
  else
    return V4A_ERR_UNSUPPORTED;
  return e == cudaSuccess ? V4A_OK : V4A_ERR_CUDA;
}

}  // namespace v4a
