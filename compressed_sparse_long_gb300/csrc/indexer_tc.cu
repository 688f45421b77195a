// Indexer scores on the 5th-generation tensor cores (tcgen05), bf16 x bf16 -> fp32.
//
//   score[q, j] = scale_j * sum_h w[q,h] * max(0, q_idx[q,h,:] . code_j)
//
// ([blog] "vLLM DeepSeek V4 支援：高效長上下文注意力", DeepSeek Sparse Attention bullet; the
// scale is applied after the head sum because ReLU is positively homogeneous.)
//
// Tile: M = 128 consecutive c4a entries of one sequence (two 64-entry pages of the paged
// cache), N = 64 heads x NQ queries of the same sequence, K = d_I = 128. Entries sit on
// the M axis so each TMEM lane holds one entry's head dot products and the head sum is a
// per-thread loop in the epilogue.
//
// One persistent CTA per SM, warp-specialised, every hand-off an mbarrier:
//   warp 0      producer: per tile two 8 KB cp.async.bulk copies of fp8 pages plus their
//               row scales into one ring stage (6 stages for one query per group, 4 for four)
//   warp 1      MMA: allocates TMEM, one thread issues 8 x tcgen05.mma (K = 16) per tile
//               into one of two TMEM accumulators, commits to the barriers
//   warps 2-9   converters: fp8 e4m3 -> bf16 (exact) into the 128B-swizzled K-major A
//               operand (two buffers); load the group's queries into the B operand
//   warps 10-13 epilogue: tcgen05.ld of the accumulator, ReLU, head-weighted sum, row
//               scale, store of the fp32 scores
// Work: units = (query group, sequence sub-pass, tile); each CTA takes a contiguous slice
// of the units of all groups (found with a block scan), so long and short rows balance.
// Every wait is bounded (~1 s): on expiry the CTA sets V4A_DEV_TIMEOUT, drains its copies
// and MMAs, frees its TMEM and returns.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace v4a {
namespace {

constexpr int kHI = 64;
constexpr int kDI = 128;
constexpr int kTile = 128;                  // entries per tile
constexpr int kStageBytes = kTile * kDI;    // fp8 codes of one tile (two 64-entry pages)
// a stage: codes, then the two pages' 64 row scales, then two page-status words
constexpr int kStageScaleOff = kStageBytes;
constexpr int kStageMetaOff = kStageBytes + 2 * 64 * 4;
constexpr int kStageStride = kStageBytes + 1024;
constexpr int kABytes = kTile * kDI * 2;    // bf16, two 64-wide K blocks of 16 KB
constexpr int kThreads = 448;              // 14 warps
constexpr int kConv0 = 2, kEpi0 = 10;       // first converter / epilogue warp
constexpr int kConvThreads = (kEpi0 - kConv0) * 32;

template <int NQ>
struct Layout {
  static constexpr int N = NQ * kHI;
  static constexpr int kStages = NQ == 1 ? 6 : 4;
  static constexpr int kBBytes = N * kDI * 2;
  static constexpr int kTmemCols = 2 * N;   // two accumulators
  static constexpr int off_stage = 0;
  static constexpr int off_a = off_stage + kStages * kStageStride;
  static constexpr int off_b = off_a + 2 * kABytes;
  static constexpr int off_w = off_b + kBBytes;
  static constexpr int off_bar = off_w + N * 4;
  static constexpr int n_bar = 2 * kStages + 8 + 3;
  static constexpr int off_misc = off_bar + n_bar * 8;
  static constexpr int bytes = off_misc + 128 + 1024;  // + alignment slack
};

struct Group {
  int n_sub;
  int units;
  int seq[4];          // per query of the group (-1: beyond n_q)
  int64_t nvis[4];     // per query, clamped to the score row length
  int sub_seq[4];
  int sub_tiles[4];
};

template <int NQ>
__device__ __forceinline__ Group load_group(const IndexParams& p, int g, bool flag_pos) {
  Group G;
  G.n_sub = 0;
  G.units = 0;
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    const int qi = g * NQ + q;
    if (qi < p.n_q) {
      G.seq[q] = __ldg(p.q_seq + qi);
      int64_t nv = visible_entries(__ldg(p.q_pos + qi), p.S, p.W, p.win_off);
      if (nv > p.row_stride) {
        if (flag_pos) raise_err(p.err, V4A_DEV_BAD_POS);
        nv = p.row_stride;
      }
      G.nvis[q] = nv;
    } else {
      G.seq[q] = -1;
      G.nvis[q] = 0;
    }
  }
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    if (G.seq[q] < 0) continue;
    int k = -1;
    for (int s = 0; s < G.n_sub; ++s)
      if (G.sub_seq[s] == G.seq[q]) k = s;
    if (k < 0) {
      k = G.n_sub++;
      G.sub_seq[k] = G.seq[q];
      G.sub_tiles[k] = 0;
    }
    const int tiles = (int)((G.nvis[q] + kTile - 1) / kTile);
    if (tiles > G.sub_tiles[k]) G.sub_tiles[k] = tiles;
  }
  for (int s = 0; s < G.n_sub; ++s) G.units += G.sub_tiles[s];
  return G;
}

// Position in the CTA's unit sequence: group, sub-pass, tile.
template <int NQ>
struct Walk {
  int g, s, t;
  Group G;
  __device__ void settle(const IndexParams& p, int n_groups) {
    // move forward to the first existing unit at or after (g, s, t)
    while (g < n_groups) {
      while (s < G.n_sub && t >= G.sub_tiles[s]) {
        ++s;
        t = 0;
      }
      if (s < G.n_sub) return;
      ++g;
      s = 0;
      t = 0;
      if (g < n_groups) G = load_group<NQ>(p, g, false);
    }
  }
  __device__ void next(const IndexParams& p, int n_groups) {
    ++t;
    settle(p, n_groups);
  }
};

// Inclusive block-wide scan of one int per thread (kThreads threads); returns the
// inclusive value, the chunk total in *total.
__device__ __forceinline__ int block_scan(int v, int* warp_buf, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_buf[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kThreads / 32 ? warp_buf[lane] : 0;
    int z = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, z, o);
      if (lane >= o) z += y;
    }
    if (lane < kThreads / 32) warp_buf[lane] = z - w;
    if (lane == kThreads / 32 - 1) *total = z;
  }
  __syncthreads();
  const int r = x + warp_buf[warp];
  __syncthreads();
  return r;
}

template <int NQ>
__global__ void __launch_bounds__(kThreads, 1) index_scores_tc(const __grid_constant__ IndexParams p) {
  using Lay = Layout<NQ>;
  constexpr int N = Lay::N;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = tc::smem_u32(smem_raw);
  uint8_t* sm = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* stage = sm + Lay::off_stage;
  uint8_t* abuf = sm + Lay::off_a;
  uint8_t* bbuf = sm + Lay::off_b;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::off_bar);
  uint64_t* full = bars;
  uint64_t* empty = bars + Lay::kStages;
  uint64_t* afull = bars + 2 * Lay::kStages;
  uint64_t* aempty = afull + 2;
  uint64_t* tfull = afull + 4;
  uint64_t* tempty = afull + 6;
  uint64_t* bfull = afull + 8;
  uint64_t* bempty = afull + 9;
  uint64_t* done = afull + 10;
  int* misc = reinterpret_cast<int*>(sm + Lay::off_misc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = misc + 1;
  int* scan_buf = misc + 4;          // one int per warp (kThreads / 32 <= 24)
  int* scan_tot = misc + 28;
  static_assert(kThreads / 32 <= 24, "scan buffer holds 24 warps");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_groups = (p.n_q + NQ - 1) / NQ;

  if (tid == 0) {
    for (int i = 0; i < Lay::kStages; ++i) {
      tc::mbar_init(full + i, 1);
      tc::mbar_init(empty + i, 12);         // 8 converter + 4 epilogue warps
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(afull + i, 8);
      tc::mbar_init(aempty + i, 1);
      tc::mbar_init(tfull + i, 1);
      tc::mbar_init(tempty + i, 4);
    }
    tc::mbar_init(bfull, 8);
    tc::mbar_init(bempty, 1);
    tc::mbar_init(done, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, Lay::kTmemCols);
    tc::tmem_relinquish();
  }

  // ---- this CTA's slice of the units (one block scan when the groups fit the block)
  __shared__ int s_g0, s_off;
  int total_units = 0;
  if (n_groups <= kThreads) {
    const int g = tid;
    const int u = g < n_groups ? load_group<NQ>(p, g, true).units : 0;
    const int incl = block_scan(u, scan_buf, scan_tot);
    total_units = *scan_tot;
    const int64_t ub = (int64_t)total_units * blockIdx.x / gridDim.x;
    if (tid == 0) { s_g0 = n_groups; s_off = 0; }
    __syncthreads();
    if (u > 0 && incl - u <= ub && ub < incl) {
      s_g0 = g;
      s_off = (int)(ub - (incl - u));
    }
  } else {
  for (int base = 0; base < n_groups; base += kThreads) {
    const int g = base + tid;
    const int u = g < n_groups ? load_group<NQ>(p, g, true).units : 0;
    int tot;
    block_scan(u, scan_buf, scan_tot);
    tot = *scan_tot;
    total_units += tot;
    __syncthreads();
  }
  const int64_t u_begin = (int64_t)total_units * blockIdx.x / gridDim.x;
  // locate u_begin: group g0 and the offset inside it
  if (tid == 0) { s_g0 = n_groups; s_off = 0; }
  __syncthreads();
  {
    int run = 0;
    for (int base = 0; base < n_groups; base += kThreads) {
      const int g = base + tid;
      const int u = g < n_groups ? load_group<NQ>(p, g, false).units : 0;
      const int incl = block_scan(u, scan_buf, scan_tot) + run;
      const int excl = incl - u;
      if (u > 0 && excl <= u_begin && u_begin < incl) {
        s_g0 = g;
        s_off = (int)(u_begin - excl);
      }
      run += *scan_tot;
      __syncthreads();
    }
  }
  }
  const int64_t u_begin = (int64_t)total_units * blockIdx.x / gridDim.x;
  const int64_t u_end = (int64_t)total_units * (blockIdx.x + 1) / gridDim.x;
  const int n_units = (int)(u_end - u_begin);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  Walk<NQ> start;
  start.g = s_g0;
  start.s = 0;
  start.t = 0;
  if (n_units > 0 && start.g < n_groups) {
    start.G = load_group<NQ>(p, start.g, false);
    int off = s_off;
    start.settle(p, n_groups);
    // offset inside the group: walk its sub-passes (each step consumes at least one unit;
    // the walk stops at the end of the groups)
    while (off > 0 && start.g < n_groups) {
      const int left = start.G.sub_tiles[start.s] - start.t;
      if (left <= 0) break;
      if (off < left) {
        start.t += off;
        off = 0;
      } else {
        off -= left;
        start.t = start.G.sub_tiles[start.s];
        start.settle(p, n_groups);
      }
    }
  }

  constexpr uint32_t idesc = tc::idesc_bf16(kTile, N);
  const int8_t* idx_data = reinterpret_cast<const int8_t*>(p.idx.data);

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    // The whole warp keeps the page ids of 32 consecutive blocks (16 tiles) of the current
    // sequence in registers, one per lane; lane 0 waits on the ring and issues the copies.
    if (n_units > 0) {
      Walk<NQ> w = start;
      int issued = 0;
      uint32_t had_copy = 0;
      int cache_seq = -1;
      int64_t cache_blk0 = 0;
      int32_t cache_page = -1;
      bool ok = true;
      for (int i = 0; i < n_units; ++i) {
        if (w.g >= n_groups) break;                    // every role stops at the same tile
        const int st = i % Lay::kStages;
        const int seq = w.G.sub_seq[w.s];
        const int64_t blk0 = 2 * (int64_t)w.t;
        if (seq != cache_seq || blk0 < cache_blk0 || blk0 + 1 >= cache_blk0 + 32) {   // warp-uniform
          cache_seq = seq;
          cache_blk0 = blk0;
          const int64_t b = blk0 + lane;
          cache_page = b < p.idx.max_blocks ? __ldg(p.idx.bt + (int64_t)seq * p.idx.max_blocks + b) : -1;
        }
        const int32_t pg0 = __shfl_sync(0xffffffffu, cache_page, (int)(blk0 - cache_blk0));
        const int32_t pg1 = __shfl_sync(0xffffffffu, cache_page, (int)(blk0 + 1 - cache_blk0));
        if (lane == 0) {
          if (!tc::mbar_wait(empty + st, ((i / Lay::kStages) & 1) ^ 1, abort_flag, p.err)) ok = false;
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
        uint8_t* sb = stage + st * kStageStride;
        int64_t src[2];
        int nv = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int32_t page = h ? pg1 : pg0;
          src[h] = -1;
          int status = -1;                              // no page
          if (page >= p.idx.n_pages) status = -2;       // page id outside the pool
          if (page >= 0 && page < p.idx.n_pages) {
            src[h] = page;
            status = 0;
            ++nv;
          }
          reinterpret_cast<int*>(sb + kStageMetaOff)[h] = status;
        }
        if (nv) {
          tc::mbar_arrive_tx(full + st, (uint32_t)(nv * (64 * kDI + 64 * 4)));
          for (int h = 0; h < 2; ++h)
            if (src[h] >= 0) {
              tc::bulk_g2s(sb + h * 64 * kDI, idx_data + src[h] * 64 * kDI, 64 * kDI, full + st);
              tc::bulk_g2s(sb + kStageScaleOff + h * 256, p.idx.scale + src[h] * 64, 256, full + st);
            }
          had_copy |= 1u << st;
        } else {
          tc::mbar_arrive(full + st);
          had_copy &= ~(1u << st);
        }
        }
        issued = i + 1;
        w.next(p, n_groups);
      }
      if (lane == 0 && *abort_flag) {   // drain copies still in flight
        for (int i = issued > Lay::kStages ? issued - Lay::kStages : 0; i < issued; ++i)
          if (had_copy & (1u << (i % Lay::kStages)))
            tc::mbar_wait_drain(full + i % Lay::kStages, (i / Lay::kStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_units > 0) {
      Walk<NQ> w = start;
      int prev_g = -1, gc = 0;
      const uint32_t a0 = tc::smem_u32(abuf), b0 = tc::smem_u32(bbuf);
      for (int i = 0; i < n_units; ++i) {
        if (w.g >= n_groups) break;
        if (w.g != prev_g) {
          if (!tc::mbar_wait(bfull, gc & 1, abort_flag, p.err)) break;
          ++gc;
          prev_g = w.g;
        }
        const int ab = i & 1;
        if (!tc::mbar_wait(afull + ab, (i >> 1) & 1, abort_flag, p.err)) break;
        if (!tc::mbar_wait(tempty + ab, ((i >> 1) & 1) ^ 1, abort_flag, p.err)) break;
        tc::fence_after_sync();
        const uint32_t d = tmem + ab * N;
#pragma unroll
        for (int k = 0; k < kDI / 16; ++k) {
          const uint32_t koff = (k & 3) * 32u;   // 16 bf16 = 32 bytes inside the swizzle row
          const uint64_t ad = tc::sdesc_sw128(a0 + ab * kABytes + (k >> 2) * (kTile * 128) + koff, 16, 1024);
          const uint64_t bd = tc::sdesc_sw128(b0 + (k >> 2) * (N * 128) + koff, 16, 1024);
          tc::mma_bf16(d, ad, bd, idesc, k > 0 ? 1u : 0u);
        }
        tc::mma_commit(aempty + ab);
        tc::mma_commit(tfull + ab);
        const int g_here = w.g;
        w.next(p, n_groups);
        if (w.g != g_here || i == n_units - 1) tc::mma_commit(bempty);
      }
      tc::mma_commit(done);
      tc::mbar_wait_drain(done, 0);
    }
    __syncwarp();
  } else if (warp >= kConv0 && warp < kEpi0) {
    // ------------------------------------------------------------------ converters
    const int ct = tid - kConv0 * 32;
    Walk<NQ> w = start;
    int prev_g = -1, gc = 0;
    for (int i = 0; i < n_units; ++i) {
      if (w.g >= n_groups) break;
      if (w.g != prev_g) {
        if (gc > 0 && !tc::mbar_wait(bempty, (gc - 1) & 1, abort_flag, p.err)) break;
        // the group's queries -> B operand [N rows = query*64 + head][128 dims]
        const __nv_bfloat16* qsrc = reinterpret_cast<const __nv_bfloat16*>(p.q_idx);
#pragma unroll 1
        for (int base = 0; base < N * 16; base += kConvThreads * 8) {   // 8 loads in flight per thread
          uint4 v[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int item = base + k * kConvThreads + ct;
            const int n = item >> 4, c = item & 15;
            const int qi = w.g * NQ + n / kHI;
            v[k] = (item < N * 16 && qi < p.n_q)
                       ? __ldg(reinterpret_cast<const uint4*>(qsrc + ((int64_t)qi * kHI + (n % kHI)) * kDI) + c)
                       : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int item = base + k * kConvThreads + ct;
            const int n = item >> 4, c = item & 15;
            if (item < N * 16)                           // N rows x 16 chunks of 16 bytes
              *reinterpret_cast<uint4*>(bbuf + (c >> 3) * (N * 128) + tc::sw128_off(n, c & 7)) = v[k];
          }
        }
        tc::fence_proxy_async();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bfull);
        ++gc;
        prev_g = w.g;
      }
      const int st = i % Lay::kStages, ab = i & 1;
      if (!tc::mbar_wait(full + st, (i / Lay::kStages) & 1, abort_flag, p.err)) break;
      if (!tc::mbar_wait(aempty + ab, ((i >> 1) & 1) ^ 1, abort_flag, p.err)) break;
      const uint8_t* src = stage + st * kStageStride;
      uint8_t* dst = abuf + ab * kABytes;
      uint4 raw[kTile * 8 / kConvThreads];
#pragma unroll
      for (int k = 0; k < kTile * 8 / kConvThreads; ++k)
        raw[k] = *reinterpret_cast<const uint4*>(src + (ct + k * kConvThreads) * 16);
#pragma unroll
      for (int k = 0; k < kTile * 8 / kConvThreads; ++k) {
        const int item = ct + k * kConvThreads;
        const int r = item >> 3, v = item & 7;      // 16 codes = dims 16v .. 16v+15
        uint4 lo, hi;
        e4m3x16_to_bf16x16(raw[k], lo, hi);
        const int c0 = 2 * v;                        // bf16 chunk index over 128 dims
        *reinterpret_cast<uint4*>(dst + (c0 >> 3) * (kTile * 128) + tc::sw128_off(r, c0 & 7)) = lo;
        *reinterpret_cast<uint4*>(dst + ((c0 + 1) >> 3) * (kTile * 128) + tc::sw128_off(r, (c0 + 1) & 7)) = hi;
      }
      tc::fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(afull + ab);
        tc::mbar_arrive(empty + st);
      }
      w.next(p, n_groups);
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    Walk<NQ> w = start;
    for (int i = 0; i < n_units; ++i) {
      if (w.g >= n_groups) break;
      const int ab = i & 1, st = i % Lay::kStages;
      // the tile's page status and row scales arrive with its codes in the stage
      if (!tc::mbar_wait(full + st, (i / Lay::kStages) & 1, abort_flag, p.err)) break;
      const uint8_t* sb = stage + st * kStageStride;
      const int status = reinterpret_cast<const int*>(sb + kStageMetaOff)[row >> 6];
      const float sc = status == 0 ? reinterpret_cast<const float*>(sb + kStageScaleOff)[row] : 0.f;
      if (!tc::mbar_wait(tfull + ab, (i >> 1) & 1, abort_flag, p.err)) break;
      tc::fence_after_sync();
      const int seq = w.G.sub_seq[w.s];
      const int64_t j = (int64_t)w.t * kTile + row;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (w.G.seq[q] != seq) continue;            // warp-uniform
        float s = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float acc[32];
          tc::tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + ab * N + q * kHI + half * 32, acc);
          tc::tmem_wait_ld();
          const float4* wv = reinterpret_cast<const float4*>(p.w + (int64_t)(w.g * NQ + q) * kHI + half * 32);
#pragma unroll
          for (int h4 = 0; h4 < 8; ++h4) {
            const float4 ww = __ldg(wv + h4);
            s = fmaf(ww.x, fmaxf(acc[4 * h4], 0.f), s);
            s = fmaf(ww.y, fmaxf(acc[4 * h4 + 1], 0.f), s);
            s = fmaf(ww.z, fmaxf(acc[4 * h4 + 2], 0.f), s);
            s = fmaf(ww.w, fmaxf(acc[4 * h4 + 3], 0.f), s);
          }
        }
        if (j < w.G.nvis[q] && w.g * NQ + q < p.n_q) {
          float out;
          if (status == 0) {
            out = s * sc + 0.0f;
          } else {
            raise_err(p.err, status == -2 ? V4A_DEV_BAD_PAGE : V4A_DEV_MISSING_PAGE);
            out = -INFINITY;
          }
          p.scores[(int64_t)(w.g * NQ + q) * p.row_stride + j] = out;
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(tempty + ab);
        tc::mbar_arrive(empty + st);
      }
      w.next(p, n_groups);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, Lay::kTmemCols);
  }
}

template <int NQ>
cudaError_t launch_tc(const IndexParams& p, int64_t max_vis, cudaStream_t st) {
  using Lay = Layout<NQ>;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t n_groups = (p.n_q + NQ - 1) / NQ;
  const int64_t max_units = n_groups * NQ * ((max_vis + kTile - 1) / kTile);
  const int grid = (int)(max_units < sms ? (max_units > 0 ? max_units : 1) : sms);
  cudaError_t e = cudaFuncSetAttribute(index_scores_tc<NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Lay::bytes);
  if (e != cudaSuccess) return e;
  index_scores_tc<NQ><<<grid, kThreads, Lay::bytes, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

// Tensor-core path for bf16 queries and fp8 keys with 64 heads of dim 128. Many queries
// (prefill) are taken four at a time (N = 256) so each key tile feeds four queries.
cudaError_t launch_index_scores_tc(const IndexParams& p, int64_t max_vis, cudaStream_t st) {
  if (p.n_q >= 1024) return launch_tc<4>(p, max_vis, st);
  return launch_tc<1>(p, max_vis, st);
}

}  // namespace v4a
