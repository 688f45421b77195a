// Indexer scores on the 5th-generation tensor cores (tcgen05), fp8 x fp8 -> fp32.
//
//   score[q, j] = scale_j * sum_h w[q,h] * max(0, q_idx[q,h,:] . code_j)
//
// ([blog] "vLLM DeepSeek V4 支援：高效長上下文注意力", DeepSeek Sparse Attention bullet; the
// row scale is applied after the head sum because ReLU is positively homogeneous.)
//
// Keys stay in their fp8 e4m3 codes: a page (64 entries x 128 bytes) is copied by a TMA
// tensor copy with 128-byte swizzle straight into the K-major operand layout, so nothing is
// converted or rewritten on chip. The bf16 query row of head h is split exactly into two
// e4m3 terms, q*s = hi + lo with s = 2^(7 - exponent(max|q_h|)): hi is q*s rounded to e4m3
// and the remainder lo = q*s - hi has at most four significant bits, so it is an e4m3 value
// too (up to the e4m3 subnormal step, 2^-9, for elements below 2^-2 after scaling). Both
// terms sit on the N axis of one product (kind::f8f6f4, fp32 accumulation); the epilogue
// adds them and applies w_h / s.
//
// Tile: M = 128 consecutive c4a entries of one sequence (two 64-entry pages), N = 128 rows
// per query (64 heads x {hi, lo}) x NQ queries of the same sequence, K = d_I = 128 (four
// MMAs of K = 32). With NQ = 4 the hi rows of the four queries and then their lo rows are
// two N = 256 products per K step accumulating into the same 256 columns (the epilogue's
// hi + lo is done by the accumulator). Entries sit on the M axis so each TMEM lane holds
// one entry's head dot products and the head sum is a per-thread loop in the epilogue.
//
// One persistent CTA per SM, warp-specialised, every hand-off an mbarrier:
//   warps 0,12-14 producers: a tile's two pages are copied into one ring stage by two
//               warps, one per page; even tiles go to warps 0 and 12, odd tiles to 13 and
//               14 (a warp serialises its bulk copies, ~0.3 us each). Each warp arms the
//               stage barrier with its own bytes and leaves its page id (or status) there.
//   warp 1      MMA: allocates TMEM, one thread issues 4 tcgen05.mma per tile (8 with four
//               queries) into one of four accumulators (two for two or four queries per
//               group); commits release the stage and hand the tile over
//   warps 2-9   epilogue, two sets of four (one per TMEM lane quadrant) taking even and
//               odd tiles (with four queries: both sets every tile, two queries each):
//               tcgen05.ld, hi + lo, ReLU, weighted head sum, row scale, store
//   warps 10-11 query preparation: the hi/lo B operand and w/s of each query group, double
//               buffered across groups
// fp4 indexer cache (packed e2m1 rows, one fp32 scale a row): warps 0 and 12 bulk-copy a
// tile's two 4 KB packed pages into the stage's packed area, and warps 13-15 (added to the
// block) take turns expanding them into the same swizzled e4m3 operand (every e2m1 value
// is an e4m3 value, so the product is unchanged); the product waits for the expansion.
// Work: units = (query group, sequence sub-pass, tile); each CTA takes a contiguous slice
// of the units of all groups (found with a block scan), so long and short rows balance.
// At kernel start each CTA prefetches its slice of the query operands into L2.
// Every wait is bounded (~1 s): on expiry the CTA sets V4A_DEV_TIMEOUT, drains its copies
// and MMAs, frees its TMEM and returns.
#include <cstring>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace v4a {
namespace {

constexpr int kHI = 64;
constexpr int kDI = 128;
constexpr int kTile = 128;                  // entries per tile
constexpr int kPageBytes = 64 * kDI;        // one 64-entry page of fp8 codes
constexpr int kPackedPageBytes = 64 * kDI / 2;   // one 64-entry page of packed fp4 codes
constexpr int kStageBytes = kTile * kDI;    // e4m3 operand of one tile (two pages)
constexpr int kEpi0 = 2, kPrep0 = 10;       // first epilogue / query-preparation warp
constexpr int kProd1 = 12;                  // producers: warp 0 and warps 12-14 (fp8) or 12 (fp4)
constexpr int kExp0 = 13;                   // fp4: expanders are warps 13-15

// Threads of the fp8 (15 warps) and fp4 (16 warps) kernels, 128 registers a thread.
template <bool kFp4>
constexpr int threads_of() { return kFp4 ? 512 : 480; }

// A stage: the e4m3 operand of a tile (swizzled, fed to the product), for fp4 the two
// packed pages it is expanded from, then the two pages' ids (-1: no page, -2: id outside
// the pool) and, from kScaleOff, the two pages' 64 row scales each (copied with the codes).
// Stages stay 1 KB aligned for the swizzled layout.
template <bool kFp4>
struct StageGeo {
  static constexpr int kPackOff = kStageBytes;                          // fp4 only
  static constexpr int kMetaOff = kFp4 ? kStageBytes + 2 * kPackedPageBytes : kStageBytes;
  static constexpr int kScaleOff = kMetaOff + 16;
  static constexpr int kStride = kMetaOff + 1024;
};

template <int NQ, bool kFp4>
struct Layout {
  static constexpr int N = NQ * 2 * kHI;    // B rows: hi and lo rows of each query
  // NQ = 4 (long prefill chunks): each query's hi and lo products accumulate into the same
  // 64 columns (B rows: the four queries' hi rows, then their lo rows; two N = 256 products
  // per K step), so a tile's accumulator is 256 columns and two fit in TMEM. A key tile then
  // feeds four queries: half the key copies of NQ = 2, whose tile period was set by the
  // copies (~0.77 us a tile with the 8-stage ring full and ~5 us from issue to landing).
  static constexpr bool kFused = NQ == 4;
  static constexpr int NC = kFused ? NQ * kHI : N;   // accumulator columns of a tile
  // fp8: even, tiles alternate producer pairs; fp4: the stage holds the packed pages too.
  // Shallow rings measured faster for the decode grid (a CTA streams only ~14 tiles and a
  // deep ring floods DRAM with requests that delay its first tiles): fp8 with one query
  // per group 4 stages (49.6 us per decode step against 51.0 with 10), fp4 6.
  // NQ = 4: two 64 KB query operands leave room for 4 stages (8 stages and one operand
  // buffer measured the same on long rows and stall at every group change on short ones).
  static constexpr int kStages = kFp4 ? 6 : (NQ == 1 || NQ == 4 ? 4 : 8);
  static constexpr int kBBuf = 2;   // query operand buffers (the next group's is built meanwhile)
  static constexpr int kBBytes = N * kDI;   // fp8 B operand of one group
  static constexpr int kAcc = kFused ? 512 / NC : (NQ == 1 ? 4 : 2);   // TMEM accumulators
  static constexpr int kTmemCols = kAcc * NC;
  static constexpr int off_stage = 0;
  static constexpr int off_b = kStages * StageGeo<kFp4>::kStride;  // 1 KB aligned
  static constexpr int off_w = off_b + kBBuf * kBBytes;           // w_h / s_h [kBBuf][NQ * 64]
  static constexpr int off_bar = off_w + 2 * NQ * kHI * 4;
  static constexpr int n_bar = (kFp4 ? 3 : 2) * kStages + 2 * kAcc + 6 + 1;
  static constexpr int off_misc = off_bar + n_bar * 8;
  static constexpr int bytes = off_misc + 128 + 1024;  // + alignment slack
  static_assert(off_b % 1024 == 0, "swizzled operands need 1 KB alignment");
  static_assert(bytes <= 227 * 1024, "shared memory of one CTA");
  static_assert(kFp4 || kStages % 2 == 0, "a stage's tiles keep one parity (producer pair, epilogue set)");
};

// tcgen05.mma kind::f8f6f4 instruction descriptor: fp32 accumulator, e4m3 A and B (format
// code 0), both K-major, shape M x N.
constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 2-D TMA tensor copy global -> shared (box given by the tensor map), completion on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          tc::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(tc::smem_u32(bar))
      : "memory");
}

struct Group {
  int n_sub;
  int units;
  int seq[4];          // per query of the group (-1: beyond n_q)
  int64_t nvis[4];     // per query, clamped to the score row length
  int sub_seq[4];
  int sub_tiles[4];
};

// Element i of a small array through unrolled selects, so the array stays in registers
// (dynamic indexing would place it in local memory).
template <typename T>
__device__ __forceinline__ T pick4(const T (&a)[4], int i) {
  T r = a[0];
#pragma unroll
  for (int k = 1; k < 4; ++k)
    if (i == k) r = a[k];
  return r;
}
template <typename T>
__device__ __forceinline__ void put4(T (&a)[4], int i, T v) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
    if (i == k) a[k] = v;
}

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
  for (int s = 0; s < 4; ++s) {
    G.sub_seq[s] = -1;
    G.sub_tiles[s] = 0;
  }
#pragma unroll
  for (int q = 0; q < NQ; ++q) {
    if (G.seq[q] < 0) continue;
    int k = -1;
#pragma unroll
    for (int s = 0; s < NQ; ++s)
      if (s < G.n_sub && G.sub_seq[s] == G.seq[q]) k = s;
    if (k < 0) {
      k = G.n_sub++;
      put4(G.sub_seq, k, G.seq[q]);
    }
    const int tiles = (int)((G.nvis[q] + kTile - 1) / kTile);
    if (tiles > pick4(G.sub_tiles, k)) put4(G.sub_tiles, k, tiles);
  }
#pragma unroll
  for (int s = 0; s < 4; ++s) G.units += G.sub_tiles[s];
  return G;
}

// Position in the CTA's unit sequence: group, sub-pass, tile.
template <int NQ>
// The sub-pass's tile count and sequence are cached so that the per-tile step is one
// increment and compare; the group state is consulted only when a sub-pass ends.
struct Walk {
  int g, s, t;
  int t_lim;   // tiles of sub-pass s
  int seq;     // sequence of sub-pass s
  Group G;
  __device__ __forceinline__ void settle(const IndexParams& p, int n_groups) {
    // move forward to the first existing unit at or after (g, s, t)
    while (g < n_groups) {
      while (s < G.n_sub && t >= pick4(G.sub_tiles, s)) {
        ++s;
        t = 0;
      }
      if (s < G.n_sub) {
        t_lim = pick4(G.sub_tiles, s);
        seq = pick4(G.sub_seq, s);
        return;
      }
      ++g;
      s = 0;
      t = 0;
      if (g < n_groups) G = load_group<NQ>(p, g, false);
    }
  }
  __device__ __forceinline__ void next(const IndexParams& p, int n_groups) {
    if (++t < t_lim) return;
    settle(p, n_groups);
  }
};

// Inclusive block-wide scan of one int per thread (kThreads threads); returns the
// inclusive value, the chunk total in *total.
template <int kThreads>
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

template <int NQ, bool kFp4>
__global__ void __launch_bounds__(threads_of<kFp4>(), 1) index_scores_tc(const __grid_constant__ IndexParams p,
                                                                          const __grid_constant__ CUtensorMap pages) {
  using Lay = Layout<NQ, kFp4>;
  using Geo = StageGeo<kFp4>;
  constexpr int kThreads = threads_of<kFp4>();
  constexpr int N = Lay::N;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = tc::smem_u32(smem_raw);
  uint8_t* sm = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* stage = sm + Lay::off_stage;
  uint8_t* bbuf = sm + Lay::off_b;                          // [2][N rows x 128 bytes]
  float* wsm = reinterpret_cast<float*>(sm + Lay::off_w);   // [2][NQ * 64]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Lay::off_bar);
  uint64_t* full = bars;
  uint64_t* empty = bars + Lay::kStages;
  uint64_t* tfull = bars + 2 * Lay::kStages;   // [kAcc]
  uint64_t* tempty = tfull + Lay::kAcc;
  uint64_t* bfull = tempty + Lay::kAcc;  // [2] query operand ready (by group parity)
  uint64_t* bempty = bfull + 2;    // [2] products of the group done
  uint64_t* egone = bempty + 2;    // [2] epilogue left the group
  uint64_t* done = egone + 2;
  uint64_t* xfull = done + 1;      // fp4: [kStages] the tile's operand expanded
  int* misc = reinterpret_cast<int*>(sm + Lay::off_misc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = misc + 1;
  int* scan_buf = misc + 4;          // one int per warp (kThreads / 32 <= 24)
  int* scan_tot = misc + 28;
  static_assert(kThreads / 32 <= 24, "scan buffer holds 24 warps");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_groups = (p.n_q + NQ - 1) / NQ;
  // The setup, the work partition and the query preparation read only this call's inputs
  // and run while the previous kernel finishes; the producers (pages the insert writes)
  // and the epilogue (row scales, scores) wait for it first.
  pdl_trigger();

  if (tid == 0) {
    for (int i = 0; i < Lay::kStages; ++i) {
      tc::mbar_init(full + i, 2);           // the tile's two page producers
      tc::mbar_init(empty + i, Lay::kFused ? 9 : 5);   // the tile's products + its epilogue warps
    }
    for (int i = 0; i < Lay::kAcc; ++i) {
      tc::mbar_init(tfull + i, 1);
      tc::mbar_init(tempty + i, Lay::kFused ? 8 : 4);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(bfull + i, kProd1 - kPrep0);   // the preparation warps
      tc::mbar_init(bempty + i, 1);
      tc::mbar_init(egone + i, 8);
    }
    tc::mbar_init(done, 1);
    if (kFp4)
      for (int i = 0; i < Lay::kStages; ++i) tc::mbar_init(xfull + i, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, Lay::kTmemCols);
    tc::tmem_relinquish();
  }
  // The query operands are read first by the preparation warps, right after the partition
  // below: when they are small, every CTA brings its slice of them (and of the positions
  // and sequence ids the partition reads) into L2 now, one 128-byte line per thread.
  {
    const int64_t qb = (int64_t)p.n_q * kHI * kDI * 2, wb = (int64_t)p.n_q * kHI * 4;
    if (qb + wb <= ((int64_t)4 << 20)) {
      const int64_t lines_q = (qb + 127) >> 7, lines_w = (wb + 127) >> 7;
      const int64_t lines = lines_q + lines_w;
      for (int64_t l = (int64_t)blockIdx.x * kThreads + tid; l < lines; l += (int64_t)gridDim.x * kThreads) {
        const char* a = l < lines_q ? reinterpret_cast<const char*>(p.q_idx) + (l << 7)
                                    : reinterpret_cast<const char*>(p.w) + ((l - lines_q) << 7);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
      }
    }
  }

  // ---- this CTA's slice of the units (one block scan when the groups fit the block)
  __shared__ int s_g0, s_off;
  int total_units = 0;
  if (n_groups <= kThreads) {
    const int g = tid;
    const int u = g < n_groups ? load_group<NQ>(p, g, true).units : 0;
    const int incl = block_scan<kThreads>(u, scan_buf, scan_tot);
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
    block_scan<kThreads>(u, scan_buf, scan_tot);
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
      const int incl = block_scan<kThreads>(u, scan_buf, scan_tot) + run;
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
      const int left = pick4(start.G.sub_tiles, start.s) - start.t;
      if (left <= 0) break;
      if (off < left) {
        start.t += off;
        off = 0;
      } else {
        off -= left;
        start.t = pick4(start.G.sub_tiles, start.s);
        start.settle(p, n_groups);
      }
    }
  }

  constexpr int NC = Lay::NC;
  constexpr uint32_t idesc = idesc_e4m3(kTile, Lay::kFused ? NQ * kHI : N);

  if (warp == 0 || (warp >= kProd1 && warp < (kFp4 ? kProd1 + 1 : kProd1 + 3))) {
    // ------------------------------------------------------------------ producers
    // fp8: four warps, page ph of the tiles i % 2 == parity; fp4: two warps, page ph of
    // every tile (a packed page is a 4 KB bulk copy into the stage's packed area)
    const int pw = warp == 0 ? 0 : warp - kProd1 + 1;
    const int ph = pw & 1, parity = kFp4 ? 0 : pw >> 1;
    // The whole warp keeps the page ids of 32 consecutive blocks (16 tiles) of the current
    // sequence in registers, one per lane; lane 0 waits on the ring and issues the copy.
    // Block tables are caller inputs that no kernel of this library writes: the first
    // slice is read before waiting for the previous kernel, the pages after.
    int cache_seq = -1;
    int64_t cache_blk0 = 0;
    int32_t cache_page = -1;
    // the pages' tensor map into the descriptor cache before the first copy needs it
    if (!kFp4 && lane == 0)
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&pages)) : "memory");
    if (n_units > 0 && start.g < n_groups) {
      cache_seq = start.seq;
      cache_blk0 = 2 * (int64_t)start.t;
      const int64_t b = cache_blk0 + lane;
      cache_page = b < p.idx.max_blocks ? __ldg(p.idx.bt + (int64_t)cache_seq * p.idx.max_blocks + b) : -1;
    }
    pdl_wait();
    if (n_units > 0) {
      Walk<NQ> w = start;
      int issued = 0;
      uint32_t had_copy = 0;
      bool ok = true;
      for (int i = 0; i < n_units; ++i) {
        if (w.g >= n_groups) break;                    // every role stops at the same tile
        if (!kFp4 && (i & 1) != parity) {              // the other pair's tile (stages of
          w.next(p, n_groups);                         // one parity: kStages is even)
          continue;
        }
        const int st = i % Lay::kStages;
        const int seq = w.seq;
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
        uint8_t* sb = stage + st * Geo::kStride;
        const int32_t page = ph ? pg1 : pg0;
        bool copied = false;
        if (lane == 0) {
          const bool valid = page >= 0 && page < p.idx.n_pages;
          reinterpret_cast<int*>(sb + Geo::kMetaOff)[ph] = valid ? page : (page >= p.idx.n_pages ? -2 : -1);
          if (valid) {
            // the page's codes, and its 64 row scales (256 bytes) beside them
            if constexpr (kFp4) {
              tc::mbar_arrive_tx(full + st, kPackedPageBytes + 256);
              tc::bulk_g2s(sb + Geo::kPackOff + ph * kPackedPageBytes,
                           reinterpret_cast<const uint8_t*>(p.idx.data) + (int64_t)page * kPackedPageBytes,
                           kPackedPageBytes, full + st);
            } else {
              tc::mbar_arrive_tx(full + st, kPageBytes + 256);
              tma_load_2d(sb + ph * kPageBytes, &pages, 0, page * 64, full + st);
            }
            tc::bulk_g2s(sb + Geo::kScaleOff + ph * 256, p.idx.scale + (int64_t)page * 64, 256, full + st);
            copied = true;
          } else {
            tc::mbar_arrive(full + st);
          }
        }
        if (copied) had_copy |= 1u << st;
        else had_copy &= ~(1u << st);
        issued = i + 1;
        w.next(p, n_groups);
      }
      if (lane == 0 && *abort_flag) {   // drain this warp's copies still in flight
        for (int i = issued > Lay::kStages ? issued - Lay::kStages : 0; i < issued; ++i)
          if ((kFp4 || (i & 1) == parity) && (had_copy & (1u << (i % Lay::kStages))))
            tc::mbar_wait_drain(full + i % Lay::kStages, (i / Lay::kStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp walks the units and waits (a converged warp); lane 0 issues.
    if (n_units > 0) {
      Walk<NQ> w = start;
      int prev_g = -1, gc = -1;
      const uint32_t s0 = tc::smem_u32(stage), b0 = tc::smem_u32(bbuf);
      for (int i = 0; i < n_units; ++i) {
        if (w.g >= n_groups) break;
        if (w.g != prev_g) {
          ++gc;
          if (!__all_sync(0xffffffffu, tc::mbar_wait(bfull + gc % Lay::kBBuf, (gc / Lay::kBBuf) & 1, abort_flag, p.err))) break;
          prev_g = w.g;
        }
        const int st = i % Lay::kStages, tb = i % Lay::kAcc;
        if (!__all_sync(0xffffffffu, tc::mbar_wait((kFp4 ? xfull : full) + st, (i / Lay::kStages) & 1,
                                                   abort_flag, p.err)))
          break;
        if (!__all_sync(0xffffffffu, tc::mbar_wait(tempty + tb, ((i / Lay::kAcc) & 1) ^ 1, abort_flag, p.err))) break;
        tc::fence_after_sync();
        const int g_here = w.g;
        w.next(p, n_groups);
        if (lane == 0) {
          const uint32_t d = tmem + tb * NC;
          const uint64_t ad0 = tc::sdesc_sw128(s0 + st * Geo::kStride, 16, 1024);
          const uint64_t bd0 = tc::sdesc_sw128(b0 + (gc % Lay::kBBuf) * Lay::kBBytes, 16, 1024);
          if constexpr (Lay::kFused) {
            // the hi rows then the lo rows (NQ * 64 rows each; 128-byte rows in 1 KB atoms of
            // 8, so row r starts 8 r descriptor units in), both into the same columns
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
              for (int k = 0; k < kDI / 32; ++k)
                mma_e4m3(d, ad0 + (uint64_t)(2 * k), bd0 + (uint64_t)(part * NQ * kHI * 8 + 2 * k), idesc,
                         (k > 0 || part > 0) ? 1u : 0u);
          } else {
#pragma unroll
            for (int k = 0; k < kDI / 32; ++k)   // K = 32 codes = 32 bytes = 2 descriptor units
              mma_e4m3(d, ad0 + (uint64_t)(2 * k), bd0 + (uint64_t)(2 * k), idesc, k > 0 ? 1u : 0u);
          }
          tc::mma_commit(empty + st);
          tc::mma_commit(tfull + tb);
          if (w.g != g_here || i == n_units - 1) tc::mma_commit(bempty + gc % Lay::kBBuf);
        }
        __syncwarp();
      }
      if (lane == 0) {
        tc::mma_commit(done);
        tc::mbar_wait_drain(done, 0);
      }
    }
    __syncwarp();
  } else if (kFp4 && warp >= kExp0) {
    // ------------------------------------------------------------------ fp4 expanders
    // Warp kExp0 + e takes the tiles i % 3 == e: once a tile's packed pages have landed,
    // row r's codes (64 bytes at r * 64 of the packed area) become its 128 e4m3 codes in
    // the swizzled operand layout, 16 bytes (8 packed bytes) per lane and step.
    const int e = warp - kExp0;
    Walk<NQ> w = start;
    for (int i = 0; i < n_units; ++i) {
      if (w.g >= n_groups) break;
      if (i % 3 != e) {
        w.next(p, n_groups);
        continue;
      }
      const int st = i % Lay::kStages;
      if (!__all_sync(0xffffffffu, tc::mbar_wait(full + st, (i / Lay::kStages) & 1, abort_flag, p.err))) break;
      uint8_t* sb = stage + st * Geo::kStride;
      const uint8_t* pk = sb + Geo::kPackOff;
#pragma unroll 4
      for (int it = 0; it < kTile * 8 / 32; ++it) {
        const int q = it * 32 + lane, r = q >> 3, c = q & 7;
        const uint2 v = *reinterpret_cast<const uint2*>(pk + r * 64 + c * 8);
        uint4 o;
        o.x = e2m1x4_to_e4m3x4(v.x & 0xFFFFu);
        o.y = e2m1x4_to_e4m3x4(v.x >> 16);
        o.z = e2m1x4_to_e4m3x4(v.y & 0xFFFFu);
        o.w = e2m1x4_to_e4m3x4(v.y >> 16);
        *reinterpret_cast<uint4*>(sb + tc::sw128_off(r, c)) = o;
      }
      tc::fence_proxy_async();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(xfull + st);
      w.next(p, n_groups);
    }
  } else if (warp >= kPrep0 && warp < kProd1) {
    // ------------------------------------------------------------------ query preparation
    // Per group: B rows qq*128 + h (hi) and qq*128 + 64 + h (lo), 128 bytes each, K-major
    // 128B-swizzled; wsm = w_h / s_h. Warp pw prepares heads pw*32 .. pw*32+31 of every
    // query of the group, 16 at a time: lane l takes head pw*32 + 16*pass + l/2, dims
    // 64*(l&1) .. +63 (the head's max needs one exchange with the neighbouring lane).
    const int pw = warp - kPrep0;
    const int dh = lane & 1;
    Walk<NQ> w = start;
    int prev_g = -1, gc = -1;
    const __nv_bfloat16* qsrc = reinterpret_cast<const __nv_bfloat16*>(p.q_idx);
    for (int i = 0; i < n_units; ++i) {
      if (w.g >= n_groups) break;
      if (w.g != prev_g) {
        ++gc;
        prev_g = w.g;
        const int b = gc % Lay::kBBuf;
        if (gc >= Lay::kBBuf) {   // the buffer's previous group: its products and epilogue are done
          const uint32_t par = ((gc / Lay::kBBuf) - 1) & 1;
          if (!tc::mbar_wait(bempty + b, par, abort_flag, p.err)) break;
          if (!tc::mbar_wait(egone + b, par, abort_flag, p.err)) break;
        }
        uint8_t* bb = bbuf + b * Lay::kBBytes;
#pragma unroll 1
        for (int pass = 0; pass < 2 * NQ; ++pass) {
          const int qq = pass >> 1;
          const int h = pw * 32 + (pass & 1) * 16 + (lane >> 1);
          const int qi = w.g * NQ + qq;
          uint4 v[8];                                  // 64 bf16
          const uint4* src = reinterpret_cast<const uint4*>(qsrc + ((int64_t)qi * kHI + h) * kDI + dh * 64);
#pragma unroll
          for (int c = 0; c < 8; ++c) v[c] = qi < p.n_q ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
          const float wh = qi < p.n_q ? __ldg(p.w + (int64_t)qi * kHI + h) : 0.f;
          float amax = 0.f;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&v[c]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 f = __bfloat1622float2(e[j]);
              amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
          }
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
          // s = 2^(7 - ex) with amax = f * 2^ex, f in [1, 2): max |q * s| < 256 <= 448
          int ex = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127;
          if (!(amax > 0.f) || ex < -100 || ex > 100) ex = 7;   // zero, tiny or huge row: s = 1
          const float sc = __uint_as_float((uint32_t)(127 + 7 - ex) << 23);
          const float inv_s = __uint_as_float((uint32_t)(127 - 7 + ex) << 23);
#pragma unroll
          for (int c = 0; c < 4; ++c) {               // 16 dims -> one 16-byte chunk each
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&v[2 * c + (k >> 1)]);
              uint32_t hp = 0, lp = 0;
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const float2 f = __bfloat1622float2(e[2 * (k & 1) + j]);
                const float a0 = f.x * sc, a1 = f.y * sc;   // exact (power of two)
                const __nv_fp8x2_storage_t h2 =
                    __nv_cvt_float2_to_fp8x2(make_float2(a0, a1), __NV_SATFINITE, __NV_E4M3);
                const __half2_raw hh = __nv_cvt_fp8x2_to_halfraw2(h2, __NV_E4M3);
                const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hh));
                const __nv_fp8x2_storage_t l2 =
                    __nv_cvt_float2_to_fp8x2(make_float2(a0 - hf.x, a1 - hf.y), __NV_SATFINITE, __NV_E4M3);
                hp |= (uint32_t)h2 << (16 * j);
                lp |= (uint32_t)l2 << (16 * j);
              }
              hw[k] = hp;
              lw[k] = lp;
            }
            const int chunk = dh * 4 + c;               // 16-byte chunk of the 128-byte row
            const int r_hi = Lay::kFused ? qq * kHI + h : qq * 128 + h;
            const int r_lo = Lay::kFused ? (NQ + qq) * kHI + h : qq * 128 + 64 + h;
            *reinterpret_cast<uint4*>(bb + tc::sw128_off(r_hi, chunk)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(bb + tc::sw128_off(r_lo, chunk)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
          if (dh == 0) wsm[b * NQ * kHI + qq * kHI + h] = wh * inv_s;
        }
        tc::fence_proxy_async();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bfull + b);
      }
      w.next(p, n_groups);
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    pdl_wait();
    const int es = (warp - kEpi0) >> 2;         // set: tiles i % 2 == es
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    Walk<NQ> w = start;
    int prev_g = -1, gc = -1;
    for (int i = 0; i < n_units; ++i) {
      if (w.g >= n_groups) break;
      if (w.g != prev_g) {
        if (gc >= 0 && lane == 0) tc::mbar_arrive(egone + gc % Lay::kBBuf);   // left the previous group
        ++gc;
        prev_g = w.g;
      }
      if (!Lay::kFused && (i & 1) != es) {
        w.next(p, n_groups);
        continue;
      }
      const int tb = i % Lay::kAcc, st = i % Lay::kStages, b = gc % Lay::kBBuf;
      // the tile's page ids and row scales arrive with its codes
      if (!tc::mbar_wait(full + st, (i / Lay::kStages) & 1, abort_flag, p.err)) break;
      const uint8_t* sb = stage + st * Geo::kStride;
      const int page = reinterpret_cast<const int*>(sb + Geo::kMetaOff)[row >> 6];
      const float sc = page >= 0 ? reinterpret_cast<const float*>(sb + Geo::kScaleOff)[row] : 0.f;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(empty + st);
      if (!tc::mbar_wait(bfull + b, (gc / Lay::kBBuf) & 1, abort_flag, p.err)) break;   // w / s of the group
      if (!tc::mbar_wait(tfull + tb, (i / Lay::kAcc) & 1, abort_flag, p.err)) break;
      tc::fence_after_sync();
      const int seq = w.seq;
      const int64_t j = (int64_t)w.t * kTile + row;
      const float* wq = wsm + b * NQ * kHI;
      if constexpr (Lay::kFused) {
        // Both sets take every tile, set es queries 2 es and 2 es + 1, so an accumulator is
        // free after half the epilogue time (the products of tile i + 2 wait for it), and
        // it is released as soon as its last columns are in registers. Queries of another
        // sequence are computed and dropped (their columns hold products with this
        // sequence's keys). Four chunks of 32 heads (query 2 es: chunks 0, 1; query 2 es + 1:
        // chunks 2, 3), each chunk's load in flight while the previous one is reduced.
        const uint32_t c0 = tmem + ((uint32_t)(quad * 32) << 16) + tb * NC + 2 * es * kHI;
        const float* wc = wq + 2 * es * kHI;
        // four chains (heads h mod 4) in two packed pairs: one paired FMA per two heads
        float2 s2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        float sq[2];
        auto reduce = [&](const float (&v)[32], int c) {
          const float4* w4 = reinterpret_cast<const float4*>(wc + c * 32);
#pragma unroll
          for (int h4 = 0; h4 < 8; ++h4) {
            const float4 ww = w4[h4];
            s2[0] = __ffma2_rn(make_float2(ww.x, ww.y),
                               make_float2(fmaxf(v[4 * h4], 0.f), fmaxf(v[4 * h4 + 1], 0.f)), s2[0]);
            s2[1] = __ffma2_rn(make_float2(ww.z, ww.w),
                               make_float2(fmaxf(v[4 * h4 + 2], 0.f), fmaxf(v[4 * h4 + 3], 0.f)), s2[1]);
          }
        };
        {
          float va[32], vb[32];
          tc::tmem_ld32(c0, va);
          tc::tmem_wait_ld();
          tc::tmem_ld32(c0 + 32, vb);
          reduce(va, 0);
          tc::tmem_wait_ld();
          tc::tmem_ld32(c0 + 64, va);
          reduce(vb, 1);
          sq[0] = (s2[0].x + s2[0].y) + (s2[1].x + s2[1].y);
          s2[0] = s2[1] = make_float2(0.f, 0.f);
          tc::tmem_wait_ld();
          tc::tmem_ld32(c0 + 96, vb);
          reduce(va, 2);
          tc::tmem_wait_ld();
          tc::fence_before_sync();                // every column of the tile is in registers
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(tempty + tb);
          reduce(vb, 3);
          sq[1] = (s2[0].x + s2[0].y) + (s2[1].x + s2[1].y);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int qq = 2 * es + u;
          if (pick4(w.G.seq, qq) == seq && j < pick4(w.G.nvis, qq) && w.g * NQ + qq < p.n_q) {
            float out;
            if (page >= 0) {
              out = sq[u] * sc + 0.0f;
            } else {
              raise_err(p.err, page == -2 ? V4A_DEV_BAD_PAGE : V4A_DEV_MISSING_PAGE);
              out = -INFINITY;
            }
            p.scores[(int64_t)(w.g * NQ + qq) * p.row_stride + j] = out;
          }
        }
      } else {
#pragma unroll
        for (int qq = 0; qq < NQ; ++qq) {
          if (w.G.seq[qq] != seq) continue;         // warp-uniform
          float s4[4] = {0.f, 0.f, 0.f, 0.f};     // four chains instead of one
#pragma unroll
          for (int qt = 0; qt < 4; ++qt) {        // 16 heads at a time (fewer live registers)
            float hi[16], lo[16];
            const uint32_t col = tmem + ((uint32_t)(quad * 32) << 16) + tb * NC + qq * 128 + qt * 16;
            tc::tmem_ld16(col, hi);
            tc::tmem_ld16(col + 64, lo);
            tc::tmem_wait_ld();
            const float4* w4 = reinterpret_cast<const float4*>(wq + qq * kHI + qt * 16);
#pragma unroll
            for (int h4 = 0; h4 < 4; ++h4) {
              const float4 ww = w4[h4];
              s4[0] = fmaf(ww.x, fmaxf(hi[4 * h4] + lo[4 * h4], 0.f), s4[0]);
              s4[1] = fmaf(ww.y, fmaxf(hi[4 * h4 + 1] + lo[4 * h4 + 1], 0.f), s4[1]);
              s4[2] = fmaf(ww.z, fmaxf(hi[4 * h4 + 2] + lo[4 * h4 + 2], 0.f), s4[2]);
              s4[3] = fmaf(ww.w, fmaxf(hi[4 * h4 + 3] + lo[4 * h4 + 3], 0.f), s4[3]);
            }
          }
          const float s = (s4[0] + s4[1]) + (s4[2] + s4[3]);
          if (j < w.G.nvis[qq] && w.g * NQ + qq < p.n_q) {
            float out;
            if (page >= 0) {
              out = s * sc + 0.0f;
            } else {
              raise_err(p.err, page == -2 ? V4A_DEV_BAD_PAGE : V4A_DEV_MISSING_PAGE);
              out = -INFINITY;
            }
            p.scores[(int64_t)(w.g * NQ + qq) * p.row_stride + j] = out;
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(tempty + tb);
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

// cuTensorMapEncodeTiled through the runtime's driver entry point (looked up once).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

}  // namespace

bool encode_byte_rows_map(CUtensorMap* map, const void* base, uint64_t n_rows, uint32_t row_bytes,
                          uint32_t box_bytes, uint32_t box_rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)n_rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {box_bytes, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <int NQ, bool kFp4>
cudaError_t launch_tc(const IndexParams& p, int64_t max_vis, cudaStream_t st) {
  using Lay = Layout<NQ, kFp4>;
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // fp8: the pool as a 2-D byte tensor [n_pages * 64 rows][128], one page per box, 128B
  // swizzle; fp4 pages are plain bulk copies (the map is unused)
  CUtensorMap map;
  memset(&map, 0, sizeof(map));
  if (!kFp4) {
    if (!encode_fn()) return cudaErrorNotSupported;
    if (!encode_byte_rows_map(&map, p.idx.data, (uint64_t)p.idx.n_pages * 64, kDI, kDI, 64))
      return cudaErrorInvalidValue;
  }
  const int64_t n_groups = (p.n_q + NQ - 1) / NQ;
  const int64_t max_units = n_groups * NQ * ((max_vis + kTile - 1) / kTile);
  const int grid = (int)(max_units < sms ? (max_units > 0 ? max_units : 1) : sms);
  cudaError_t e = cudaFuncSetAttribute(index_scores_tc<NQ, kFp4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Lay::bytes);
  if (e != cudaSuccess) return e;
  e = launch_pdl(index_scores_tc<NQ, kFp4>, dim3(grid), dim3(threads_of<kFp4>()), Lay::bytes, st, p, map);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

// Tensor-core path for bf16 queries and fp8 keys with 64 heads of dim 128. Many queries
// (prefill) are taken two at a time (N = 256), or four (two N = 256 products per K step,
// hi and lo terms summed in the accumulator), so that each key tile feeds several queries.
cudaError_t launch_index_scores_tc(const IndexParams& p, int64_t max_vis, cudaStream_t st) {
  if (p.idx.n_pages <= 0 || p.idx.n_pages * 64 > INT32_MAX) return cudaErrorInvalidValue;
  if (p.idx_fp4) {
    if (p.n_q >= 1024) return launch_tc<2, true>(p, max_vis, st);
    return launch_tc<1, true>(p, max_vis, st);
  }
  if (p.n_q >= 4096) return launch_tc<4, false>(p, max_vis, st);
  if (p.n_q >= 1024) return launch_tc<2, false>(p, max_vis, st);
  return launch_tc<1, false>(p, max_vis, st);
}

}  // namespace v4a
