// DSA-style indexer scores and top-k selection of c4a entries (steps a6, a7).
//
// [blog] "vLLM DeepSeek V4 支援：高效長上下文注意力", DeepSeek Sparse Attention bullet: after
// compression a query still only attends to its top-k compressed tokens; [notes] 压缩参数细节
// (C4A top-k = 512) and 因果性条件 (only entries covering positions < p are candidates).
//
//   score_j = sum_h w_h * max(0, q_h . k_j),  k_j = e4m3 code * row scale (fp8 layers)
//
// The per-row scale is applied after the head sum: ReLU is positively homogeneous and the
// scale is positive, so sum_h w_h ReLU(q_h . (c*k)) = c * sum_h w_h ReLU(q_h . k).
//
// Top-k, on the order-preserving uint32 image of the fp32 scores: rows of up to 8192 entries
// in registers (topk_reg_kernel), longer rows in three streaming passes (topk_stream_kernel);
// both find the k-th largest key from score-linear buckets and the exact key inside the
// boundary bucket, with radix passes for rows whose scores cannot be bucketed, and emit
// every entry above it plus the lowest-index entries equal to it, in ascending index order.
#include "common.cuh"
#include "kernels.h"

namespace v4a {

namespace {

// ------------------------------------------------------------------ fp32 indexer scores
// One thread per entry, the query's heads in shared memory (broadcast reads).
template <typename T, bool kFp8, int HI, int DI>
__global__ void __launch_bounds__(128) index_scores_simt(const __grid_constant__ IndexParams p) {
  pdl_trigger();
  pdl_wait();
  __shared__ float qs[HI * DI];
  __shared__ float ws[HI];
  const int qi = blockIdx.y;
  const int64_t pos = __ldg(p.q_pos + qi);
  int64_t n_vis = visible_entries(pos, p.S, p.W, p.win_off);
  if (n_vis > p.row_stride) {
    if (blockIdx.x == 0 && threadIdx.x == 0) raise_err(p.err, V4A_DEV_BAD_POS);
    n_vis = p.row_stride;
  }
  if ((int64_t)blockIdx.x * 128 >= n_vis) return;
  const T* q = reinterpret_cast<const T*>(p.q_idx) + (int64_t)qi * HI * DI;
  for (int i = threadIdx.x; i < HI * DI; i += 128) qs[i] = Elem<T>::to_f(q[i]);
  for (int i = threadIdx.x; i < HI; i += 128) ws[i] = __ldg(p.w + (int64_t)qi * HI + i);
  __syncthreads();
  const int64_t j = (int64_t)blockIdx.x * 128 + threadIdx.x;
  if (j >= n_vis) return;
  const int seq = __ldg(p.q_seq + qi);
  const int64_t s = slot_of(p.idx, seq, j);
  float* out = p.scores + (int64_t)qi * p.row_stride + j;
  if (!slot_ok(s, p.err)) { *out = -INFINITY; return; }

  float acc[HI];
#pragma unroll
  for (int h = 0; h < HI; ++h) acc[h] = 0.f;
  for (int c = 0; c < DI; c += 32) {
    float key[32];
    if constexpr (kFp8) {
      const uint32_t* src = reinterpret_cast<const uint32_t*>(
          reinterpret_cast<const uint8_t*>(p.idx.data) + s * (int64_t)p.idx.width + c);
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        float f[4];
        e4m3x4_decode(__ldg(src + v), f);
#pragma unroll
        for (int k = 0; k < 4; ++k) key[4 * v + k] = f[k];
      }
    } else {
      load_f<float, 32>(reinterpret_cast<const float*>(p.idx.data) + s * (int64_t)p.idx.width + c, key);
    }
#pragma unroll
    for (int h = 0; h < HI; ++h) {
      float a = acc[h];
#pragma unroll
      for (int d = 0; d < 32; ++d) a = fmaf(qs[h * DI + c + d], key[d], a);
      acc[h] = a;
    }
  }
  float sc = 0.f;
#pragma unroll
  for (int h = 0; h < HI; ++h) sc = fmaf(ws[h], fmaxf(acc[h], 0.f), sc);
  if constexpr (kFp8) sc *= __ldg(p.idx.scale + s);
  *out = sc + 0.0f;   // canonical +0 for an all-zero sum
}

// ------------------------------------------------------------------------------ top-k
__device__ __forceinline__ float warp_min_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t b = __float_as_uint(x + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t u) {   // inverse of order_key
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// Register-resident variant for rows of up to ITEMS * THREADS entries: thread tid holds
// entries tid*ITEMS .. tid*ITEMS + ITEMS-1 as u[0..ITEMS-1] (16-byte loads).
// Threshold: 1024 buckets linear in the score between the row's min and max (a monotone
// map, so every entry of a higher bucket scores strictly higher); a block-wide scan with one
// bucket per thread finds the bucket where the count from the top reaches k, which holds
// the k-th score, and the exact k-th key is found among that bucket's entries alone (a
// handful for spread-out scores). When the bucket is large (many equal or clustered
// scores) or the range is not finite, four 8-bit radix passes find it instead (one atomic
// per distinct digit per warp, two histograms, two barriers a pass). The output places
// entries in index order from one block scan of each thread's packed (above, equal) counts.
template <int ITEMS, int THREADS>
__global__ void __launch_bounds__(THREADS, 1) topk_reg_kernel(const __grid_constant__ IndexParams p) {
  pdl_trigger();
  pdl_wait();
  constexpr int kWarps = THREADS / 32;
  constexpr int kCnt = kWarps;      // per-warp scan totals
  static_assert(kWarps <= 32, "one scan total per lane");
  static_assert(ITEMS * THREADS <= 65535, "packed 16-bit counts");
  constexpr int kBuckets = 1024, kCandMax = 512;
  __shared__ uint32_t hist[2][256];
  __shared__ uint32_t cnt[kCnt];
  __shared__ uint32_t bhist[kBuckets];
  __shared__ uint32_t cand[kCandMax];
  __shared__ float s_min[kWarps], s_max[kWarps];
  __shared__ uint32_t s_digit, s_remaining, s_bucket, s_above, s_ncand, s_kth;
  const int qi = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t pos = __ldg(p.q_pos + qi);
  const int64_t n = min(visible_entries(pos, p.S, p.W, p.win_off), p.row_stride);
  int32_t* out = p.topk + (int64_t)qi * p.k;
  if (n <= p.k) {
    for (int i = tid; i < p.k; i += THREADS) out[i] = i < n ? i : -1;
    return;
  }
  const float* row = p.scores + (int64_t)qi * p.row_stride;
  const int nn = (int)n;   // <= ITEMS * THREADS (the launcher's choice)
  // thread t holds entries t*ITEMS .. t*ITEMS + ITEMS-1 (rows start on 16-byte boundaries
  // and their stride is a multiple of 4, so a group of 4 starting below nn is in the row)
  static_assert(ITEMS % 4 == 0, "whole float4 groups");
  const int i0 = tid * ITEMS;
  uint32_t u[ITEMS];
#pragma unroll
  for (int r = 0; r < ITEMS; r += 4) {
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i0 + r < nn) x = __ldg(reinterpret_cast<const float4*>(row + i0 + r));
    u[r] = i0 + r < nn ? order_key(x.x) : 0u;
    u[r + 1] = i0 + r + 1 < nn ? order_key(x.y) : 0u;
    u[r + 2] = i0 + r + 2 < nn ? order_key(x.z) : 0u;
    u[r + 3] = i0 + r + 3 < nn ? order_key(x.w) : 0u;
  }
  for (int i = tid; i < 512; i += THREADS) (&hist[0][0])[i] = 0u;
  for (int i = tid; i < kBuckets; i += THREADS) bhist[i] = 0u;
  if (tid == 0) s_ncand = 0u;
  {
    float lo = INFINITY, hi = -INFINITY;
#pragma unroll
    for (int r = 0; r < ITEMS; ++r) {
      if (i0 + r < nn) {
        const float x = key_value(u[r]);
        lo = fminf(lo, x);
        hi = x != x ? INFINITY : fmaxf(hi, x);   // a NaN score sends the row to the radix path
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
      s_min[warp] = lo;
      s_max[warp] = hi;
    }
  }
  __syncthreads();
  // every warp reduces the per-warp extremes itself (lane l reads warp l's)
  float lo = lane < kWarps ? s_min[lane] : INFINITY, hi = lane < kWarps ? s_max[lane] : -INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  uint32_t kth = 0, remaining = 0;
  bool found = false;
  const float span = hi - lo;
  if (span > 0.f && span <= 3.0e38f) {           // finite, not all equal (block-uniform)
    const float inv = (float)kBuckets / span;
    auto bucket = [&](uint32_t key) -> int {
      return max(0, min((int)((key_value(key) - lo) * inv), kBuckets - 1));
    };
#pragma unroll
    for (int r = 0; r < ITEMS; ++r)
      if (i0 + r < nn) atomicAdd(&bhist[bucket(u[r])], 1u);
    __syncthreads();
    // block-wide scan from the top bucket down: thread t owns bucket 1023 - t, a warp scan,
    // then each warp adds the totals of the warps before it; exactly one thread holds the
    // bucket where the running count reaches k
    {
      static_assert(THREADS == kBuckets, "one bucket per thread");
      uint32_t* wsum = cnt;   // free until the compaction below
      const uint32_t c = bhist[kBuckets - 1 - tid];
      uint32_t incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) wsum[warp] = incl;
      __syncthreads();
      uint32_t off = lane < warp ? wsum[lane] : 0u;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) off += __shfl_xor_sync(0xffffffffu, off, o);
      incl += off;
      const uint32_t before = incl - c, kk = (uint32_t)p.k;
      if (before < kk && incl >= kk) {
        s_bucket = (uint32_t)(kBuckets - 1 - tid);
        s_above = before;
      }
    }
    __syncthreads();
    const int bstar = (int)s_bucket;
    const uint32_t r_need = (uint32_t)p.k - s_above;   // entries still to take from bstar
    if (bhist[bstar] <= (uint32_t)kCandMax) {          // block-uniform
#pragma unroll
      for (int r = 0; r < ITEMS; ++r)
        if (i0 + r < nn && bucket(u[r]) == bstar) cand[atomicAdd(&s_ncand, 1u)] = u[r];
      __syncthreads();
      const int nc = (int)s_ncand;
      // the candidate whose key has fewer than r_need keys above it and at least r_need at
      // or above it holds the k-th key (all such candidates hold the same key)
      for (int c = tid; c < nc; c += THREADS) {
        const uint32_t uc = cand[c];
        uint32_t gt = 0, ge = 0;
        for (int j = 0; j < nc; ++j) {
          const uint32_t v = cand[j];
          gt += v > uc;
          ge += v >= uc;
        }
        if (gt < r_need && r_need <= ge) {
          s_kth = uc;
          s_remaining = r_need - gt;
        }
      }
      __syncthreads();
      kth = s_kth;
      remaining = s_remaining;
      found = true;
    }
  }
  if (!found) {
    uint32_t prefix = 0, mask = 0;
    remaining = (uint32_t)p.k;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      uint32_t* h = hist[pass & 1];
      // the other histogram was last read before the previous pass's second barrier
      if (pass > 0)
        for (int i = tid; i < 256; i += THREADS) hist[(pass + 1) & 1][i] = 0u;
#pragma unroll
      for (int r = 0; r < ITEMS; ++r) {
        const bool in = i0 + r < nn && (u[r] & mask) == prefix;
        const uint32_t bin = in ? (u[r] >> shift) & 0xFFu : 0x100u;
        const uint32_t peers = __match_any_sync(0xffffffffu, bin);
        if (in && lane == __ffs(peers) - 1) atomicAdd(&h[bin], (uint32_t)__popc(peers));
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns digits 255-8l-7 .. 255-8l, scanned from the top; exactly one lane holds
        // the digit where the running count reaches `remaining`
        uint32_t c[8], sum = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          c[k] = h[255 - 8 * lane - k];
          sum += c[k];
        }
        uint32_t incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t before = incl - sum;
        if (before < remaining && incl >= remaining) {
          uint32_t cum = before;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            if (cum + c[k] >= remaining) {
              s_digit = 255 - 8 * lane - k;
              s_remaining = remaining - cum;
              break;
            }
            cum += c[k];
          }
        }
      }
      __syncthreads();
      prefix |= s_digit << shift;
      mask |= 0xFFu << shift;
      remaining = s_remaining;
    }
    kth = prefix;
  }

  // kth is the key of the k-th largest score: take every key above it and the first
  // `remaining` keys equal to it, in index order. A block-wide exclusive scan of each
  // thread's (above, equal) counts, packed 16 | 16 bits, gives its first output position.
  uint32_t g = 0, e = 0;
#pragma unroll
  for (int r = 0; r < ITEMS; ++r) {
    const bool v = i0 + r < nn;
    g += (v && u[r] > kth) ? 1u : 0u;
    e += (v && u[r] == kth) ? 1u : 0u;
  }
  const uint32_t packed = (g << 16) | e;
  uint32_t incl = packed;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) cnt[warp] = incl;
  __syncthreads();
  uint32_t off = lane < kWarps && lane < warp ? cnt[lane] : 0u;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) off += __shfl_xor_sync(0xffffffffu, off, o);
  const uint32_t ex = off + incl - packed;
  uint32_t n_gt = ex >> 16, n_eq = ex & 0xFFFFu;
#pragma unroll
  for (int r = 0; r < ITEMS; ++r) {
    if (i0 + r >= nn) continue;
    if (u[r] > kth) {
      const uint32_t at = n_gt + min(n_eq, remaining);
      if (at < (uint32_t)p.k) out[at] = i0 + r;
      ++n_gt;
    } else if (u[r] == kth) {
      if (n_eq < remaining && n_gt + n_eq < (uint32_t)p.k) out[n_gt + n_eq] = i0 + r;
      ++n_eq;
    }
  }
}

// ---------------------------------------------------------------------- streaming top-k
// Every row of a call whose rows may exceed what the register-resident kernel holds: 256
// threads a row, several rows per SM. Three coalesced passes over the row: its extremes; a
// histogram of 2048 buckets linear in the score between them (a monotone map, so every
// entry of a higher bucket scores strictly higher); the entries of the buckets at and above
// the one where the count from the top reaches k, collected with their indices in shared
// memory (at most kStreamCap). The exact k-th key among the boundary bucket's entries comes
// from 8-bit radix passes over shared memory; the selected entries (those above it and the
// smallest-index ties equal to it) are placed by their index rank. A row with non-finite or
// constant scores, or too many collected entries, takes radix passes over the whole row
// instead (four histogram passes, then an ordered compaction of per-thread chunks).
constexpr int kStreamMaxThreads = 1024;
constexpr int kStreamBuckets = 2048;
constexpr int kStreamCap = 2048;

// Exclusive block-wide sum of one value per thread (WARPS warps); the total through *total.
template <int WARPS>
__device__ __forceinline__ uint32_t stream_excl_sum(uint32_t v, uint32_t* warp_tot, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  uint32_t before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < WARPS; ++w) {
    const uint32_t t = warp_tot[w];
    before += w < warp ? t : 0u;
    all += t;
  }
  __syncthreads();
  if (total) *total = all;
  return before + incl - v;
}

// The digit (scanning from the top) where the running count of h[] reaches `need`, and the
// count still needed inside it; warp 0 only (lane l owns digits 255-8l-7 .. 255-8l).
__device__ __forceinline__ void top_digit(const uint32_t* h, uint32_t need, uint32_t* s_digit,
                                          uint32_t* s_need) {
  const int lane = threadIdx.x & 31;
  uint32_t c[8], sum = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    c[k] = h[255 - 8 * lane - k];
    sum += c[k];
  }
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t before = incl - sum;
  if (before < need && incl >= need) {
    uint32_t cum = before;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (cum + c[k] >= need) {
        *s_digit = 255 - 8 * lane - k;
        *s_need = need - cum;
        break;
      }
      cum += c[k];
    }
  }
}

template <int kStreamThreads>
__global__ void __launch_bounds__(kStreamThreads, 1024 / kStreamThreads)
    topk_stream_kernel(const __grid_constant__ IndexParams p) {
  constexpr int kStreamWarps = kStreamThreads / 32;
  constexpr int kBpt = kStreamBuckets / kStreamThreads;   // histogram buckets a thread scans
  pdl_trigger();
  pdl_wait();
  __shared__ uint32_t bh[kStreamBuckets];           // bucket histogram; radix histograms after
  __shared__ uint32_t ckey[kStreamCap];             // collected entries: order key,
  __shared__ int32_t cidx[kStreamCap];              // entry index,
  __shared__ uint8_t cin[kStreamCap];               // 1 = in the boundary bucket
  __shared__ int32_t sel[kStreamCap];               // selected entry indices
  __shared__ float s_lo[kStreamWarps], s_hi[kStreamWarps], s_fl[kStreamWarps];
  __shared__ uint32_t warp_tot[kStreamWarps];
  __shared__ uint32_t s_bucket, s_above, s_nc, s_digit, s_need, s_total;
  const int qi = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t pos = __ldg(p.q_pos + qi);
  const int64_t n = min(visible_entries(pos, p.S, p.W, p.win_off), p.row_stride);
  int32_t* out = p.topk + (int64_t)qi * p.k;
  const uint32_t k = (uint32_t)p.k;
  if (n <= p.k) {
    for (int i = tid; i < p.k; i += kStreamThreads) out[i] = i < n ? i : -1;
    return;
  }
  const float* row = p.scores + (int64_t)qi * p.row_stride;
  // row starts are 16-byte aligned and the stride is a multiple of 4: whole float4 groups
  // are inside the row's allocation; entries >= n are masked. Each thread keeps kUnroll
  // 16-byte loads in flight (they are issued before any is used).
  constexpr int kUnroll = 8;
  constexpr int64_t kStep = 4 * kStreamThreads;
  {
    // the whole row is requested into L2 at once (16 KB per copy), so the first pass's
    // loads wait on fills already in flight rather than on their own DRAM round trips
    const int64_t bytes = ((n + 3) & ~(int64_t)3) * 4;
    const int64_t off = (int64_t)tid * 16384;
    if (off < bytes) {
      const uint32_t len = (uint32_t)min((int64_t)16384, bytes - off);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<const char*>(row) + off),
                   "r"(len)
                   : "memory");
    }
  }
  auto for_each4 = [&](auto&& f) {
    for (int64_t i0 = (int64_t)tid * 4; i0 < n; i0 += kStep * kUnroll) {
      float4 x[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = i0 + u * kStep;
        x[u] = i < n ? __ldg(reinterpret_cast<const float4*>(row + i)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = i0 + u * kStep;
        if (i < n) f(i, x[u].x);
        if (i + 1 < n) f(i + 1, x[u].y);
        if (i + 2 < n) f(i + 2, x[u].z);
        if (i + 3 < n) f(i + 3, x[u].w);
      }
    }
  };
  // ---- pass 1: extremes (a NaN score sends the row to the radix passes), and the four
  // largest of each thread's group maxima (each group of four loaded entries gives one,
  // a distinct entry). Warp w's candidates (four per lane) give its key T_w: the
  // ceil(k / warps)-th largest among them; the warp has that many entries at or above T_w,
  // so at least k entries of the row score at or above the floor min_w T_w, and the k
  // largest are among them (usually a few hundred beyond k; needs k <= 4 x 256).
  float lo = INFINITY, hi = -INFINITY;
  float t0 = -INFINITY, t1 = -INFINITY, t2 = -INFINITY, t3 = -INFINITY;
  auto top4 = [&](float x) {
    if (x > t3) {
      if (x > t1) {
        t3 = t2;
        t2 = t1;
        if (x > t0) {
          t1 = t0;
          t0 = x;
        } else {
          t1 = x;
        }
      } else if (x > t2) {
        t3 = t2;
        t2 = x;
      } else {
        t3 = x;
      }
    }
  };
  bool nan = false;
  for (int64_t i0 = (int64_t)tid * 4; i0 < n; i0 += kStep * kUnroll) {
    float4 x[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = i0 + u * kStep;
      x[u] = i < n ? __ldg(reinterpret_cast<const float4*>(row + i))
                   : make_float4(INFINITY, INFINITY, INFINITY, INFINITY);
      // entries past n within the last group take a value that changes neither extreme
      if (i < n && i + 3 >= n) {
        if (i + 1 >= n) x[u].y = x[u].x;
        if (i + 2 >= n) x[u].z = x[u].x;
        x[u].w = x[u].x;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t i = i0 + u * kStep;
      if (i >= n) continue;
      lo = fminf(lo, fminf(fminf(x[u].x, x[u].y), fminf(x[u].z, x[u].w)));
      const float m4 = fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w));
      hi = fmaxf(hi, m4);
      // a NaN makes the sum NaN (so can +inf beside -inf: such a row takes the radix passes,
      // which are exact for it too)
      const float sum4 = (x[u].x + x[u].y) + (x[u].z + x[u].w);
      nan |= sum4 != sum4;
      top4(m4);   // one entry of each group of four (the copies past n repeat its first)
    }
  }
  float fl = -INFINITY;
  if (k <= 4u * kStreamThreads && k <= (uint32_t)kStreamCap) {
    const uint32_t need_w = (k + kStreamWarps - 1) / kStreamWarps;
    const uint32_t u0 = order_key(t0), u1 = order_key(t1), u2 = order_key(t2), u3 = order_key(t3);
    uint32_t T = 0;                                 // bitwise search from the top bit
#pragma unroll 1
    for (int b = 31; b >= 0; --b) {
      const uint32_t c = T | (1u << b);
      const uint32_t cnt = __popc(__ballot_sync(0xffffffffu, u0 >= c)) + __popc(__ballot_sync(0xffffffffu, u1 >= c)) +
                           __popc(__ballot_sync(0xffffffffu, u2 >= c)) + __popc(__ballot_sync(0xffffffffu, u3 >= c));
      if (cnt >= need_w) T = c;
    }
    fl = key_value(T);                              // -inf when the warp lacks candidates
  }
  if (nan) hi = INFINITY;
  lo = warp_min_f(lo);
  hi = warp_max_f(hi);
  if (lane == 0) { s_lo[warp] = lo; s_hi[warp] = hi; s_fl[warp] = fl; }
  for (int i = tid; i < kStreamBuckets; i += kStreamThreads) bh[i] = 0u;
  if (tid == 0) s_nc = 0u;
  __syncthreads();
  lo = INFINITY;
  hi = -INFINITY;
  fl = INFINITY;
#pragma unroll
  for (int w = 0; w < kStreamWarps; ++w) {
    lo = fminf(lo, s_lo[w]);
    hi = fmaxf(hi, s_hi[w]);
    fl = fminf(fl, s_fl[w]);
  }
  const float span = hi - lo;
  bool bucketed = span > 0.f && span <= 3.0e38f;   // block-uniform
  uint32_t kth = 0, remaining = 0, above = 0;
  int bstar = 0;
  // ---- pass 2: collect every entry at or above the floor (usually a few percent of the
  // row) with warp-aggregated appends, one shared-memory atomic per warp and iteration
  bool have = false;                                // candidates collected (block-uniform)
  if (!nan && fl > -INFINITY) {
    constexpr int kU2 = 8;                          // 16-byte loads in flight per thread
    for (int64_t i0 = (int64_t)tid * 4; i0 - (int64_t)lane * 4 < n; i0 += kStep * kU2) {
      float4 x[kU2];
#pragma unroll
      for (int u = 0; u < kU2; ++u) {
        const int64_t i = i0 + u * kStep;
        x[u] = i < n ? __ldg(reinterpret_cast<const float4*>(row + i))
                     : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
      uint32_t cnt = 0;
      if (i0 + (kU2 - 1) * kStep + 3 < n) {         // every group of this iteration is whole
#pragma unroll
        for (int u = 0; u < kU2; ++u)
          cnt += (x[u].x >= fl) + (x[u].y >= fl) + (x[u].z >= fl) + (x[u].w >= fl);
      } else {                                      // (groups past n were loaded as -inf)
#pragma unroll
        for (int u = 0; u < kU2; ++u) {
          const int64_t i = i0 + u * kStep;
          cnt += (i < n && x[u].x >= fl) + (i + 1 < n && x[u].y >= fl) + (i + 2 < n && x[u].z >= fl) +
                 (i + 3 < n && x[u].w >= fl);
        }
      }
      uint32_t incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      uint32_t base = 0;
      if (lane == 31 && incl) base = atomicAdd(&s_nc, incl);
      uint32_t at = __shfl_sync(0xffffffffu, base, 31) + incl - cnt;
      if (cnt) {
#pragma unroll
        for (int u = 0; u < kU2; ++u) {
          const float v[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int64_t i = i0 + u * kStep + e;
            if (i < n && v[e] >= fl) {
              if (at < (uint32_t)kStreamCap) {
                ckey[at] = order_key(v[e]);
                cidx[at] = (int32_t)i;
                cin[at] = 1;
              }
              ++at;
            }
          }
        }
      }
    }
    __syncthreads();
    have = s_nc <= (uint32_t)kStreamCap;
    __syncthreads();
    if (!have && tid == 0) s_nc = 0u;               // ordered before pass 4 by its barriers
  }
  if (!have && bucketed) {
    const float inv = (float)kStreamBuckets / span;
    auto bucket = [&](float x) -> int {
      return max(0, min((int)((x - lo) * inv), kStreamBuckets - 1));
    };
    // ---- pass 2: histogram
    for_each4([&](int64_t, float x) { atomicAdd(&bh[bucket(x)], 1u); });
    __syncthreads();
    // boundary bucket: thread t owns the kBpt buckets below 2047 - kBpt t, from the top
    {
      uint32_t c[kBpt], sum = 0;
#pragma unroll
      for (int j = 0; j < kBpt; ++j) {
        c[j] = bh[kStreamBuckets - 1 - kBpt * tid - j];
        sum += c[j];
      }
      const uint32_t before = stream_excl_sum<kStreamWarps>(sum, warp_tot, nullptr);
      if (before < k && before + sum >= k) {
        uint32_t cum = before;
#pragma unroll
        for (int j = 0; j < kBpt; ++j) {
          if (cum + c[j] >= k) {
            s_bucket = (uint32_t)(kStreamBuckets - 1 - kBpt * tid - j);
            s_above = cum;
            break;
          }
          cum += c[j];
        }
      }
    }
    __syncthreads();
    bstar = (int)s_bucket;
    above = s_above;
    bucketed = above + bh[bstar] <= (uint32_t)kStreamCap;   // block-uniform
    if (bucketed) {
      // ---- pass 4: collect the entries of buckets >= bstar (warp-aggregated appends)
      // (the loop bound is the warp's first index, so every lane of a warp runs the same
      // iterations and the ballots are warp-wide)
      for (int64_t i0 = (int64_t)tid * 4; i0 - (int64_t)lane * 4 < n; i0 += kStep * kUnroll) {
        float4 x[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int64_t i = i0 + u * kStep;
          x[u] = i < n ? __ldg(reinterpret_cast<const float4*>(row + i))
                       : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const float v[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
          // (masked entries are -inf: bucket 0 < bstar unless bstar is 0, checked below)
          const bool any4 = bucket(fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]))) >= bstar;
          if (!__any_sync(0xffffffffu, any4)) continue;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int64_t i = i0 + u * kStep + e;
            const bool in = i < n && bucket(v[e]) >= bstar;
            const uint32_t m = __ballot_sync(0xffffffffu, in);
            uint32_t base = 0;
            if (lane == 0 && m) base = atomicAdd(&s_nc, (uint32_t)__popc(m));
            base = __shfl_sync(0xffffffffu, base, 0);
            if (in) {
              const uint32_t at = base + __popc(m & ((1u << lane) - 1u));
              ckey[at] = order_key(v[e]);
              cidx[at] = (int32_t)i;
              cin[at] = bucket(v[e]) == bstar ? 1 : 0;
            }
          }
        }
      }
      __syncthreads();
      have = true;
    }
  }
  if (have) {
    const int nc = (int)s_nc;
    // ---- exact k-th key among the collected entries flagged in cin (pass 2: all of them;
    // pass 4: the boundary bucket's, those above it being selected already): 8-bit radix
    uint32_t prefix = 0, mask = 0, need = k - above;
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
      const int shift = 24 - 8 * pass;
      for (int i = tid; i < 256; i += kStreamThreads) bh[i] = 0u;
      __syncthreads();
      for (int c = tid; c < nc; c += kStreamThreads)
        if (cin[c] && (ckey[c] & mask) == prefix) atomicAdd(&bh[(ckey[c] >> shift) & 0xFFu], 1u);
      __syncthreads();
      if (warp == 0) top_digit(bh, need, &s_digit, &s_need);
      __syncthreads();
      prefix |= s_digit << shift;
      mask |= 0xFFu << shift;
      need = s_need;
    }
    kth = prefix;
    remaining = need;              // ties equal to kth still to take, smallest indices first
    // entries equal to kth: when all of them are taken (the usual case, one entry), no
    // tie needs its index rank
    uint32_t n_tie = 0;
    for (int c = tid; c < nc; c += kStreamThreads) n_tie += (cin[c] && ckey[c] == kth) ? 1u : 0u;
    stream_excl_sum<kStreamWarps>(n_tie, warp_tot, &s_total);
    const bool all_ties = s_total <= remaining;
    // ---- selection: contiguous chunks of the collected entries, one block scan
    const int per = (nc + kStreamThreads - 1) / kStreamThreads;
    const int c0 = tid * per, c1 = min(nc, c0 + per);
    auto selected = [&](int c) -> bool {
      const uint32_t key = ckey[c];
      if (!cin[c] || key > kth) return true;
      if (key != kth) return false;
      if (all_ties) return true;
      uint32_t rank = 0;           // ties equal to kth with a smaller index
      for (int d = 0; d < nc; ++d) rank += (cin[d] && ckey[d] == kth && cidx[d] < cidx[c]) ? 1u : 0u;
      return rank < remaining;
    };
    uint32_t cnt = 0;
    for (int c = c0; c < c1; ++c) cnt += selected(c) ? 1u : 0u;
    uint32_t at = stream_excl_sum<kStreamWarps>(cnt, warp_tot, &s_total);
    for (int c = c0; c < c1; ++c)
      if (selected(c)) sel[at++] = cidx[c];
    __syncthreads();
    // ---- output in ascending index order: a bitonic sort of the selected indices, padded
    // to a power of two with INT32_MAX
    const int ns = (int)s_total;   // == k
    if (ns <= 2 * kStreamThreads) {
      // n2 = the power of two >= ns (at least 64) slots, thread t < n2 / 2 holding slots 2t
      // and 2t + 1 in registers (the others only pass the barriers): strides below 64 pair
      // threads of one warp (shuffles), the longer ones exchange through shared memory.
      int n2 = 64;
      while (n2 < ns) n2 <<= 1;
      const bool act = 2 * tid < n2;                // warp-uniform (n2 >= 64)
      int32_t a0 = act && 2 * tid < ns ? sel[2 * tid] : INT32_MAX;
      int32_t a1 = act && 2 * tid + 1 < ns ? sel[2 * tid + 1] : INT32_MAX;
#pragma unroll 1
      for (int size = 2; size <= n2; size <<= 1) {
        const bool asc = ((2 * tid) & size) == 0;
#pragma unroll 1
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
          if (stride == 1) {
            const int32_t lo2 = min(a0, a1), hi2 = max(a0, a1);
            a0 = asc ? lo2 : hi2;
            a1 = asc ? hi2 : lo2;
            continue;
          }
          const int tp = stride >> 1;                 // partner thread: tid ^ tp
          int32_t w0 = a0, w1 = a1;
          if (tp < 32) {
            if (act) {
              w0 = __shfl_xor_sync(0xffffffffu, a0, tp);
              w1 = __shfl_xor_sync(0xffffffffu, a1, tp);
            }
          } else {
            __syncthreads();                          // the previous exchange was read
            if (act) {
              sel[2 * tid] = a0;
              sel[2 * tid + 1] = a1;
            }
            __syncthreads();
            if (act) {
              w0 = sel[(2 * tid) ^ stride];
              w1 = sel[(2 * tid + 1) ^ stride];
            }
          }
          const bool lower = (tid & tp) == 0;         // this thread's slots are the pairs' lower
          a0 = lower == asc ? min(a0, w0) : max(a0, w0);
          a1 = lower == asc ? min(a1, w1) : max(a1, w1);
        }
      }
      if (act && 2 * tid < ns) out[2 * tid] = a0;
      if (act && 2 * tid + 1 < ns) out[2 * tid + 1] = a1;
      return;
    }
    int np2 = 1;
    while (np2 < ns) np2 <<= 1;
    for (int i = ns + tid; i < np2; i += kStreamThreads) sel[i] = INT32_MAX;
    __syncthreads();
    for (int size = 2; size <= np2; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int t = tid; t < (np2 >> 1); t += kStreamThreads) {
          const int a = 2 * t - (t & (stride - 1)), b = a + stride;
          const int32_t x0 = sel[a], x1 = sel[b];
          if ((x0 > x1) == ((a & size) == 0)) {
            sel[a] = x1;
            sel[b] = x0;
          }
        }
        __syncthreads();
      }
    }
    for (int i = tid; i < ns && i < p.k; i += kStreamThreads) out[i] = sel[i];
    return;
  }
  // ---- radix passes over the whole row: the k-th key, then an ordered compaction
  uint32_t* h = bh;
  uint32_t prefix = 0, mask = 0, need = k;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kStreamThreads) h[i] = 0u;
    __syncthreads();
    for_each4([&](int64_t, float x) {
      const uint32_t u = order_key(x);
      if ((u & mask) == prefix) atomicAdd(&h[(u >> shift) & 0xFFu], 1u);
    });
    __syncthreads();
    if (warp == 0) top_digit(h, need, &s_digit, &s_need);
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= 0xFFu << shift;
    need = s_need;
  }
  kth = prefix;
  remaining = need;
  // thread t owns the contiguous chunk [t C, (t+1) C): one block scan of its (above, equal)
  // counts places its selected entries
  const int64_t C = (n + kStreamThreads - 1) / kStreamThreads;
  const int64_t r0 = (int64_t)tid * C, r1 = min(n, r0 + C);
  uint32_t n_gt = 0, n_eq = 0;
  for (int64_t i = r0; i < r1; ++i) {
    const uint32_t u = order_key(__ldg(row + i));
    n_gt += u > kth;
    n_eq += u == kth;
  }
  const uint32_t ex_gt = stream_excl_sum<kStreamWarps>(n_gt, warp_tot, nullptr);
  const uint32_t ex_eq = stream_excl_sum<kStreamWarps>(n_eq, warp_tot, nullptr);
  uint32_t at = ex_gt + min(ex_eq, remaining);
  uint32_t tie = ex_eq;
  for (int64_t i = r0; i < r1; ++i) {
    const uint32_t u = order_key(__ldg(row + i));
    if (u > kth || (u == kth && tie < remaining)) {
      if (at < k) out[at] = (int32_t)i;
      ++at;
    }
    tie += u == kth;
  }
}

template <typename T, bool kFp8, int HI, int DI>
cudaError_t launch_simt(const IndexParams& p, int64_t max_vis, cudaStream_t st) {
  dim3 grid((unsigned)((max_vis + 127) / 128), (unsigned)p.n_q);
  const cudaError_t e = launch_pdl(index_scores_simt<T, kFp8, HI, DI>, grid, dim3(128), 0, st, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

int launch_index_scores(const IndexParams& p, int dtype, int64_t max_vis, cudaStream_t st) {
  if (p.n_q == 0 || max_vis == 0) return V4A_OK;
  cudaError_t e;
  if (dtype == V4A_BF16_FP8 && p.H_I == 64 && p.d_I == 128)
    e = launch_index_scores_tc(p, max_vis, st);
  else if (dtype == V4A_FP32 && p.H_I == 4 && p.d_I == 32)
    e = launch_simt<float, false, 4, 32>(p, max_vis, st);
  else if (dtype == V4A_FP32 && p.H_I == 64 && p.d_I == 128)
    e = launch_simt<float, false, 64, 128>(p, max_vis, st);
  else
    return V4A_ERR_UNSUPPORTED;
  return e == cudaSuccess ? V4A_OK : V4A_ERR_CUDA;
}

int launch_topk(const IndexParams& p, int64_t max_vis, cudaStream_t st) {
  if (p.n_q == 0) return V4A_OK;
  cudaError_t e;
  if (max_vis <= 8 * 1024)   // decode-sized rows: register-resident, one CTA of 1024 threads a row
    e = launch_pdl(topk_reg_kernel<8, 1024>, dim3(p.n_q), dim3(1024), 0, st, p);
  else {                     // longer rows: streaming passes, 256 threads a row (four rows an
    int dev = 0, sms = 152;    // SM), or 1024 when the call has too few rows to fill the SMs
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (p.n_q <= 2 * (int64_t)sms)
      e = launch_pdl(topk_stream_kernel<kStreamMaxThreads>, dim3(p.n_q), dim3(kStreamMaxThreads), 0, st, p);
    else
      e = launch_pdl(topk_stream_kernel<256>, dim3(p.n_q), dim3(256), 0, st, p);
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? V4A_OK : V4A_ERR_CUDA;
}

}  // namespace v4a
