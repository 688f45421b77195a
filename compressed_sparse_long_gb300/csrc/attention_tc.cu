// Shared-K=V attention on tcgen05 tensor cores with fp8 e4m3 operands, with the sliding
// window and inverse RoPE ([notes] "DeepSeek V4 in vLLM 技术博客详尽笔记", Inverse RoPE 的数学原理
// and 共享 Key-Value 向量; [blog] 短滑動窗口).
//
// Work item: one query (prefill) or one key range of one query (decode split). Keys come
// in tiles of 128 rows gathered from the paged pools (top-k entries or all visible
// entries, then the window tokens). The key tile is the pool's own e4m3 codes, copied
// row by row (16-byte cp.async) into a 128-byte-swizzled buffer, no conversion; per tile:
//   S^T = K Q~^T      M = 128 keys, N = 128 (64 heads x {hi, lo}), K = 512 dims
//                     (16 MMAs kind::f8f6f4, TMEM cols 0..127)
//   softmax over keys per head: logit = (hi + lo) / s * row scale; column max with
//     redux.sync.max.f32 and a 4-warp exchange; the running max is raised only when it
//     grows by more than 2^2 (then the O^T accumulator is rescaled); the per-row partial
//     denominators accumulate in TMEM (cols 384..447) and are summed over the keys once per
//     work item
//   O^T += V^T P'^T   M = 128 dims x 4 blocks, N = 64 heads, K = 128 keys, P' = hi + lo
//                     (32 MMAs, TMEM cols 128..383)
// K = V: the key tile is read K-major by the first product and MN-major by the second;
// P'^T is MN-major with a 64-byte swizzle (a thread writes its key's 64-byte row).
// Two key buffers: tile t+1 is copied while tile t is in use, and S^T of tile t+1 runs
// during the softmax of tile t (the softmax frees the S^T columns as soon as it has read
// them).
// e4m3 operands close to bf16 precision: Q~ = RoPE(q, p) * softmax_scale * log2(e) (logits
// in log2 units) is scaled by one power of two s per query (from sqrt(2) max |q|, which
// bounds |RoPE(q)|) and split into hi = e4m3(Q~ s) and lo = e4m3(Q~ s - hi), through f16,
// about 8 significant bits; P' = p * row scale * 2^A (A a per-range power of two that keeps
// P' below 2^8) is split the same way, and 2^-A is folded into the final 1/l. The row
// scales stay out of the codes.
//
// Warpgroups (setmaxnreg splits the 512 x 128 launch registers as 152 / 128 / 128 / 104):
// 0 = softmax and epilogue (warp w reads TMEM lanes 32w..32w+31), 1-2 = eight copy warps
// that also build Q~ (warps 4-7 fill key buffer 0 with the even tiles, warps 8-11 buffer 1
// with the odd tiles), 3 = warp 12 allocates TMEM, walks the items converged and issues
// the MMAs from lane 0 (warps 13-15 idle).
// Every hand-off is an mbarrier with a bounded wait (V4A_DEV_TIMEOUT on expiry).
// Decode split: each key range's CTA writes its unnormalised numerator O^T in bf16 plus its
// softmax state (m, l) in fp32, both in the scale of O^T; the merge kernel combines the
// ranges and applies R^-1.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace v4a {
namespace {

constexpr int kH = 64, kD = 512, kTile = 128;
constexpr int kThreads = 512;                  // 4 warpgroups
constexpr int kKBytes = kTile * kD;            // 64 KB e4m3 key tile, 4 K-blocks of 16 KB
constexpr int kQBytes = 2 * kH * kD;           // 64 KB Q~ hi (rows 0-63) and lo (64-127), 4 K-blocks
constexpr int kPBytes = kH * kTile;            // 8 KB per P' term, [128 keys][64 heads]
constexpr int kOffK = 0, kOffQ = 2 * kKBytes, kOffP = kOffQ + kQBytes;
// floats: l_fin[2][64] red_max[2][256] red_sum[256] sscale[2][128] mwarp[4][128] qamax[8]
// qinv[3] red_sc[2][4] rope_tab[4][kMaxRopePairs]
constexpr int kOffF = kOffP + 2 * kPBytes;
constexpr int kNFloats = 128 + 512 + 256 + 256 + 512 + 8 + 4 + 8 + 4 * kMaxRopePairs;
constexpr int kOffBar = kOffF + kNFloats * 4;
constexpr int kNBar = 15;
constexpr int kOffMisc = kOffBar + kNBar * 8;
constexpr int kSmemBytes = kOffMisc + 64 + 1024;
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kPBytes % 1024 == 0, "swizzled operands need 1 KB alignment");
static_assert(kOffBar % 8 == 0 && kSmemBytes <= 227 * 1024, "shared memory of one CTA");
constexpr uint32_t kTmemCols = 512;
// S^T (hi, lo), O^T (4 blocks of 64 heads), per-row partial denominators (64 heads)
constexpr uint32_t kSCol = 0, kOCol = 128, kLCol = 384;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 2.0f;      // log2 units: p <= 4 between rescales

struct Item {
  int qi, split, seq;
  int64_t pos, n_vis, n_ent, t0, x0, x1;
  int n_tiles;
};

__device__ __forceinline__ Item make_item(const AttnParams& p, int it) {
  Item I;
  I.qi = it / p.n_split;
  I.split = it % p.n_split;
  I.seq = __ldg(p.q_seq + I.qi);
  I.pos = __ldg(p.q_pos + I.qi);
  I.n_vis = visible_entries(I.pos, p.S, p.W, p.win_off);
  I.n_ent = p.topk ? p.k : I.n_vis;
  I.t0 = I.pos - p.swa_len + 1 > 0 ? I.pos - p.swa_len + 1 : 0;
  const int64_t n_keys = I.n_ent + (I.pos - I.t0 + 1);
  I.x0 = (int64_t)I.split * p.keys_per_split;
  I.x1 = min(n_keys, I.x0 + p.keys_per_split);
  I.n_tiles = I.x1 > I.x0 ? (int)((I.x1 - I.x0 + kTile - 1) / kTile) : 0;
  return I;
}

// Pool row of key x of an item (or -1 when masked), and whether it is a window token.
__device__ __forceinline__ int64_t key_slot(const AttnParams& p, const Item& I, int64_t x, bool& swa,
                                            bool report) {
  swa = false;
  if (x >= I.x1) return -1;
  if (x < I.n_ent) {
    const int64_t j = p.topk ? (int64_t)__ldg(p.topk + (int64_t)I.qi * p.k + x) : x;
    if (j < 0) return -1;
    if (j >= I.n_vis) {
      if (report) raise_err(p.err, V4A_DEV_BAD_INDEX);
      return -1;
    }
    const int64_t s = slot_of(p.attn, I.seq, j);
    if (s < 0 && report) raise_err(p.err, s == -2 ? V4A_DEV_BAD_PAGE : V4A_DEV_MISSING_PAGE);
    return s < 0 ? -1 : s;
  }
  swa = true;
  const int64_t s = slot_of(p.swa, I.seq, I.t0 + (x - I.n_ent));
  if (s < 0 && report) raise_err(p.err, s == -2 ? V4A_DEV_BAD_PAGE : V4A_DEV_MISSING_PAGE);
  return s < 0 ? -1 : s;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 2^x with the hardware approximation (relative error ~2^-22; the result is rounded to bf16).
__device__ __forceinline__ float fast_exp2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float redux_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "f"(v[8]),
      "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]),
      "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]),
      "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Sum of v[h] over the 32 lanes, scattered: lane l ends with heads 2l and 2l+1.
__device__ __forceinline__ float2 reduce_scatter_sum64(const float (&v)[64]) {
  const int lane = threadIdx.x & 31;
  float a[32];
  {
    const bool up = lane & 16;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float send = up ? v[j] : v[j + 32];
      const float keep = up ? v[j + 32] : v[j];
      a[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
  }
  float b[16];
  {
    const bool up = lane & 8;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float send = up ? a[j] : a[j + 16];
      const float keep = up ? a[j + 16] : a[j];
      b[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
  }
  float c[8];
  {
    const bool up = lane & 4;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float send = up ? b[j] : b[j + 8];
      const float keep = up ? b[j + 8] : b[j];
      c[j] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
  }
  float d[4];
  {
    const bool up = lane & 2;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float send = up ? c[j] : c[j + 4];
      const float keep = up ? c[j + 4] : c[j];
      d[j] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
  }
  float e[2];
  {
    const bool up = lane & 1;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float send = up ? d[j] : d[j + 2];
      const float keep = up ? d[j + 2] : d[j];
      e[j] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
    }
  }
  return make_float2(e[0], e[1]);
}

// tcgen05.mma kind::f8f6f4 instruction descriptor: fp32 accumulator, e4m3 A and B (format
// code 0), shape M x N; A and B read MN-major when asked (8-bit operands may be either
// major).
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, bool a_mn_major = false,
                                                  bool b_mn_major = false) {
  return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 16-byte global -> shared copy that bypasses registers; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// 2^a for an integer a in [-126, 127].
__device__ __forceinline__ float pow2i(int a) { return __uint_as_float((uint32_t)(127 + a) << 23); }

// Binary exponent of a positive normal float.
__device__ __forceinline__ int exponent_of(float x) { return (int)((__float_as_uint(x) >> 23) & 0xFFu) - 127; }

// Two values -> e4m3 codes hi (byte 0: a0, byte 1: a1) and the e4m3 codes of the
// remainders x - hi, where x is the pair rounded to f16 (11 significant bits; x - hi is
// exact in f16). hi + lo holds about 8 significant bits of each value.
__device__ __forceinline__ void split_e4m3x2(float a0, float a1, uint32_t& hi2, uint32_t& lo2) {
  const __half2 x = __floats2half2_rn(a0, a1);
  const __nv_fp8x2_storage_t h =
      __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&x), __NV_SATFINITE, __NV_E4M3);
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3);
  const __half2 r = __hsub2(x, *reinterpret_cast<const __half2*>(&hr));
  const __nv_fp8x2_storage_t l =
      __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&r), __NV_SATFINITE, __NV_E4M3);
  hi2 = (uint32_t)h;
  lo2 = (uint32_t)l;
}

// Shared-memory matrix descriptor, 64-byte swizzle (atoms of 8 rows x 64 bytes, 16-byte
// chunk c of row r stored at chunk c ^ ((r / 2) % 4)). Used for an MN-major operand whose
// M/N extent is one atom wide: rows are K indices, 8-row groups SBO bytes apart (LBO, the
// stride between atoms along M/N, is not needed and is given the same value).
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)4 << 61;
  return d;
}

template <bool kSplit>
__global__ void __launch_bounds__(kThreads, 1) attn_tc(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = tc::smem_u32(smem_raw);
  uint8_t* sm = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* kbuf = sm + kOffK;                             // [2][64 KB]
  uint8_t* qbuf = sm + kOffQ;
  uint8_t* pbuf = sm + kOffP;                             // hi, then lo
  float* l_fin = reinterpret_cast<float*>(sm + kOffF);   // [2][64] 2^-A / l by item parity
  float* red_max = l_fin + 128;                           // [2][64 heads][4 warps]
  float* red_sum = red_max + 512;                         // [64 heads][4 warps]
  float* sscale = red_sum + 256;                          // [2][128] row scales by key buffer
  float* mwarp = sscale + 256;                            // [4 warps][128] per-warp head broadcast
  float* qamax = mwarp + 512;                             // [8] raw |q| max of each build warp
  float* qinv = qamax + 8;                                // [3] 1 / s by item % 3 (+1 pad)
  float* red_sc = qinv + 4;                               // [2][4] tile max of the row scales
  float* rope_tab = red_sc + 8;                           // RoPE angle constants (stage_rope)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint64_t* kfull = bars;                                 // [2] by key buffer
  uint64_t* kempty = bars + 2;                            // [2]
  uint64_t* qfull = bars + 4;
  uint64_t* qempty = bars + 5;
  uint64_t* sfull = bars + 6;
  uint64_t* sempty = bars + 7;
  uint64_t* pfull = bars + 8;
  uint64_t* pvdone = bars + 9;
  uint64_t* ofull = bars + 10;
  uint64_t* oempty = bars + 11;
  uint64_t* redb = bars + 12;
  uint64_t* done = bars + 13;
  uint64_t* qmx = bars + 14;
  int* misc = reinterpret_cast<int*>(sm + kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = misc + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = p.n_q * p.n_split;
  // On-chip setup and the first query's Q~ read only this call's inputs and overlap the
  // previous kernel; the key gathers (top-k lists, pools) and every global write wait.
  pdl_trigger();

  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(kfull + b, 4);
      tc::mbar_init(kempty + b, 1);
    }
    tc::mbar_init(qfull, 8);
    tc::mbar_init(qempty, 1);
    tc::mbar_init(sfull, 1);
    tc::mbar_init(sempty, 4);
    tc::mbar_init(pfull, 4);
    tc::mbar_init(pvdone, 1);
    tc::mbar_init(ofull, 1);
    tc::mbar_init(oempty, 4);
    tc::mbar_init(redb, 4);
    tc::mbar_init(done, 1);
    tc::mbar_init(qmx, 8);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 12) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  stage_rope(p.rope, rope_tab, tid, kThreads);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 4 && warp < 12) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 128;");
    // ------------------------------------------------------------ Q~ build + key copies
    // Warp cw builds heads 8cw .. 8cw+7 of every item's Q~ (lane l: dims 16l .. 16l+15).
    // Copy group gb = cw / 4 fills key buffer gb with the tiles of parity gb; warp wg = cw % 4
    // of the group copies rows 32wg .. 32wg+31 (lane l resolves row 32wg + l, then each
    // row's 512 bytes go as 32 16-byte copies, lane l taking bytes 16l .. 16l+15).
    const int cw = warp - 4, gb = cw >> 2, wg = cw & 3;
    int gi = 0, ni = 0;   // global tile / item counters of this CTA
    bool ok = true, waited = false;
    const uint8_t* zsrc = reinterpret_cast<const uint8_t*>(p.attn.data);   // any valid address
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      // the item's query rows are loaded first, before its position (and whether the item
      // holds any key) is known: the two loads do not wait for one another
      uint4 u[16];
      {
        const uint4* q = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.q) +
                                                        ((int64_t)(it / p.n_split) * kH + 8 * cw) * kD) + 2 * lane;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          u[2 * i] = __ldg(q + i * (kD / 8));
          u[2 * i + 1] = __ldg(q + i * (kD / 8) + 1);
        }
      }
      const Item I = make_item(p, it);
      if (I.n_tiles == 0) continue;
      // ---- before the wait for the previous kernel (which the copies must await), the
      // window rows into L2: their slots need no top-k list. A prefetch only moves lines
      // into L2, where the insert's later writes to them land as well. (Prefetching the rows
      // of later tiles, or every row of a dense item, measured slower.)
      for (int t = 0; t < I.n_tiles && !waited; ++t) {
        if (((gi + t) & 1) != gb) continue;
        const int64_t x = I.x0 + (int64_t)t * kTile + wg * 32 + lane;
        if (x < I.n_ent) continue;
        bool is_swa;
        const int64_t slot = key_slot(p, I, x, is_swa, false);
        if (slot >= 0) {
          const CacheView& cv = is_swa ? p.swa : p.attn;
          const uint8_t* rowp = reinterpret_cast<const uint8_t*>(cv.data) + slot * (int64_t)cv.width;
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(rowp), "r"(kD) : "memory");
        }
      }
      // ---- Q~ of this item; the buffer is free once the previous item's S^T products are
      if (ni > 0 && !tc::mbar_wait(qempty, (ni - 1) & 1, abort_flag, p.err)) { ok = false; break; }
      {
        // RoPE of this lane's 8 dim pairs: lane i computes pair i, the tail lanes collect theirs
        const int tail0 = kD - p.rope.d_r;
        float c_l = 1.f, s_l = 0.f;
        if (lane < p.rope.d_r / 2) rope_cs_tab(rope_tab, I.pos, lane, c_l, s_l);
        float rc[8], rsn[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int d = 16 * lane + 2 * jj;
          const int pi = d >= tail0 ? ((d - tail0) >> 1) : 0;
          rc[jj] = __shfl_sync(0xffffffffu, c_l, pi & 31);
          rsn[jj] = __shfl_sync(0xffffffffu, s_l, pi & 31);
          if (d < tail0) {
            rc[jj] = 1.f;
            rsn[jj] = 0.f;
          }
        }
        // one power of two s per query: |RoPE(q)| <= sqrt(2) max |q|, so
        // s = 2^(7 - exponent(sqrt(2) |scale| max |q|)) keeps every |Q~ s| below 256 <= 448
        {
          __nv_bfloat162 m2 = __float2bfloat162_rn(0.f);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&u[k]);
#pragma unroll
            for (int j = 0; j < 4; ++j) m2 = __hmax2(m2, __habs2(e[j]));
          }
          const float2 mf = __bfloat1622float2(m2);
          const float am = redux_max(fmaxf(mf.x, mf.y));
          if (lane == 0) qamax[cw] = am;
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(qmx);
        }
        if (!tc::mbar_wait(qmx, ni & 1, abort_flag, p.err)) { ok = false; break; }
        const float4 qa = *reinterpret_cast<const float4*>(qamax);
        const float4 qb = *reinterpret_cast<const float4*>(qamax + 4);
        const float qs = p.scale * kLog2e;
        const float bound = fmaxf(fmaxf(fmaxf(qa.x, qa.y), fmaxf(qa.z, qa.w)),
                                  fmaxf(fmaxf(qb.x, qb.y), fmaxf(qb.z, qb.w))) * fabsf(qs) * 1.4142137f;
        int ex = exponent_of(bound);
        if (!(bound > 0.f) || ex < -100 || ex > 100) ex = 7;   // zero, tiny or huge query: s = 1
        const float kq = qs * pow2i(7 - ex);
        if (cw == 0 && lane == 0) qinv[ni % 3] = pow2i(ex - 7);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int h = 8 * cw + i;
          float f[16];
          {
            const __nv_bfloat162* e0 = reinterpret_cast<const __nv_bfloat162*>(&u[2 * i]);
            const __nv_bfloat162* e1 = reinterpret_cast<const __nv_bfloat162*>(&u[2 * i + 1]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float2 a = __bfloat1622float2(e0[j]);
              const float2 b = __bfloat1622float2(e1[j]);
              f[2 * j] = a.x;
              f[2 * j + 1] = a.y;
              f[8 + 2 * j] = b.x;
              f[8 + 2 * j + 1] = b.y;
            }
          }
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint32_t h0, l0, h1, l1;
            float x[4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const int jj = 2 * k + j;
              const float a0 = f[2 * jj], a1 = f[2 * jj + 1];
              x[2 * j] = (a0 * rc[jj] - a1 * rsn[jj]) * kq;
              x[2 * j + 1] = (a0 * rsn[jj] + a1 * rc[jj]) * kq;
            }
            split_e4m3x2(x[0], x[1], h0, l0);
            split_e4m3x2(x[2], x[3], h1, l1);
            hw[k] = h0 | (h1 << 16);
            lw[k] = l0 | (l1 << 16);
          }
          uint8_t* dst = qbuf + (lane >> 3) * 16384;
          *reinterpret_cast<uint4*>(dst + tc::sw128_off(h, lane & 7)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(dst + tc::sw128_off(kH + h, lane & 7)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        tc::fence_proxy_async();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(qfull);
      }
      if (!waited) {                                // first item: Q~ was built meanwhile
        pdl_wait();
        waited = true;
      }
      // every warp's Q~ part and 1 / s are complete (ordered before this group's kfull)
      if (!tc::mbar_wait(qfull, ni & 1, abort_flag, p.err)) { ok = false; break; }
      for (int t = 0; t < I.n_tiles; ++t) {
        const int g = gi + t;
        if ((g & 1) != gb) continue;
        // resolve the row first (top-k id, block table, scale), then wait for the buffer
        const int64_t x = I.x0 + (int64_t)t * kTile + wg * 32 + lane;
        bool is_swa;
        const int64_t slot = key_slot(p, I, x, is_swa, true);
        const uint8_t* rowp = nullptr;
        float sc = 0.f;
        if (slot >= 0) {
          const CacheView& cv = is_swa ? p.swa : p.attn;
          rowp = reinterpret_cast<const uint8_t*>(cv.data) + slot * (int64_t)cv.width;
          sc = __ldg(cv.scale + slot);
        }
        if (g >= 2 && !tc::mbar_wait(kempty + gb, ((g >> 1) - 1) & 1, abort_flag, p.err)) { ok = false; break; }
        uint8_t* kb = kbuf + gb * kKBytes + (lane >> 3) * 16384;
#pragma unroll 8
        for (int i = 0; i < 32; ++i) {
          const uint8_t* src = reinterpret_cast<const uint8_t*>(
              __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(rowp), i));
          cp_async16(tc::smem_u32(kb + tc::sw128_off(wg * 32 + i, lane & 7)), src ? src + 16 * lane : zsrc,
                     src ? 16u : 0u);
        }
        cp_async_commit();
        cp_async_wait_all();
        tc::fence_proxy_async();                    // the copied codes, for the tensor core
        sscale[gb * kTile + wg * 32 + lane] = sc;   // 0 for a masked key
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(kfull + gb);
      }
      gi += I.n_tiles;
      ++ni;
    }
  } else if (warp < 4) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 152;");
    pdl_wait();
    // ------------------------------------------------------------ softmax + epilogue
    // Thread `row` holds key `row` of the tile for all 64 heads. Every lane keeps the
    // running max of heads `lane` and `lane + 32` in registers (all four warps hold the same
    // copy) and publishes it in its warp's mwarp slice for the per-element exponentials.
    // The per-row partial denominators (sum over this thread's keys of p, per head) stay in
    // TMEM columns kLCol.. and are reduced over the keys once per item.
    const int quad = warp;
    const int row = quad * 32 + lane;             // TMEM lane: key (S^T) or dim (O^T)
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    float* mb = mwarp + quad * 128;               // [0,64): max; [64,128): rescale factors
    // this thread's P' row (key `row`, 64 bytes): 16-byte chunk c at c ^ ((row / 2) % 4)
    const uint32_t prow = (uint32_t)row * 64u, pswz = (uint32_t)((row >> 1) & 3);
    int gi = 0, ni = 0, ru = 0;
    bool ok = true;
    auto group_sync = [&]() -> bool {             // all four softmax warps
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(redb);
      const bool r = tc::mbar_wait(redb, ru & 1, abort_flag, p.err);
      ++ru;
      return r;
    };
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const Item I = make_item(p, it);
      if (I.n_tiles == 0) {
        if (kSplit) {
          const int64_t base = ((int64_t)I.qi * p.n_split + I.split) * kH;
          if (row < kH) {
            p.part_ml[(base + row) * 2] = -INFINITY;
            p.part_ml[(base + row) * 2 + 1] = 0.f;
          }
        }
        continue;
      }
      float mc0 = -INFINITY, mc1 = -INFINITY;     // running max of heads lane, lane + 32
      int A = 0;                                  // P' = p * row scale * 2^A
      bool a_set = false;                         // A chosen (a tile with an unmasked key seen)
      for (int t = 0; t < I.n_tiles; ++t, ++gi) {
        if (!tc::mbar_wait(sfull, gi & 1, abort_flag, p.err)) { ok = false; break; }
        tc::fence_after_sync();
        float s[64];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float a[32], b[32];
          tc::tmem_ld32(tmem + lane_base + kSCol + half * 32, a);        // hi
          tc::tmem_ld32(tmem + lane_base + kSCol + kH + half * 32, b);   // lo
          tc::tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 32; ++h) s[half * 32 + h] = a[h] + b[h];
        }
        // S^T is in registers: the next tile's product may overwrite it
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(sempty);
        // row scales of this tile (and the copy of its keys) are published with the buffer
        if (!tc::mbar_wait(kfull + (gi & 1), (gi >> 1) & 1, abort_flag, p.err)) { ok = false; break; }
        const float sc = sscale[(gi & 1) * kTile + row];   // 0 for a masked key
        {
          // 1 / s of this item's Q~ (written before the builders' qfull, which the copy
          // warps waited for before publishing this buffer)
          const float fq = sc * qinv[ni % 3];
#pragma unroll
          for (int h = 0; h < 64; ++h) s[h] *= fq;
          if (!(sc > 0.f)) {
#pragma unroll
            for (int h = 0; h < 64; ++h) s[h] = -INFINITY;
          }
        }
        // ---- per-head max over the tile's 128 keys, and the tile's largest row scale
        float* rb = red_max + (ru & 1) * 256;
#pragma unroll
        for (int h = 0; h < 64; ++h) {
          const float mh = redux_max(s[h]);
          if (lane == (h & 31)) rb[h * 4 + quad] = mh;
        }
        {
          const float scw = redux_max(sc);
          if (lane == 0) red_sc[(ru & 1) * 4 + quad] = scw;
        }
        const float* rsc = red_sc + (ru & 1) * 4;
        if (!group_sync()) { ok = false; break; }
        // new running max of heads lane and lane + 32 (raised only past the threshold) and
        // the correction factors exp2(old - new) of the accumulated O^T and denominators;
        // P' keeps the tile's largest row scale times 2^A below 64, so P' < 4 * 64 = 256
        float mn0, mn1, cr0 = 1.f, cr1 = 1.f;
        bool any_rescale = false;
        int a_new = A;
        {
          const float4 v0 = *reinterpret_cast<const float4*>(rb + lane * 4);
          const float4 v1 = *reinterpret_cast<const float4*>(rb + (lane + 32) * 4);
          const float mt0 = fmaxf(fmaxf(v0.x, v0.y), fmaxf(v0.z, v0.w));
          const float mt1 = fmaxf(fmaxf(v1.x, v1.y), fmaxf(v1.z, v1.w));
          const float scm = fmaxf(fmaxf(rsc[0], rsc[1]), fmaxf(rsc[2], rsc[3]));
          if (scm > 0.f) {
            // 2^A = 2^(4 - ex): the largest row scale times 2^A lands in [16, 32); chosen at
            // the range's first tile with an unmasked key (O^T is still zero when earlier
            // tiles were all masked) and lowered when a tile's scales outgrow it
            const int ex = max(-100, min(100, exponent_of(scm)));
            if (!a_set || scm * pow2i(A) >= 64.f) a_new = 4 - ex;
            a_set = true;
          }
          if (t == 0) {                          // nothing accumulated yet
            mn0 = mt0;
            mn1 = mt1;
          } else {
            mn0 = mt0 > mc0 + kRescaleThreshold ? mt0 : mc0;
            mn1 = mt1 > mc1 + kRescaleThreshold ? mt1 : mc1;
            if (mn0 != mc0) cr0 = fast_exp2(mc0 - mn0);   // 0 when the old max is -inf
            if (mn1 != mc1) cr1 = fast_exp2(mc1 - mn1);
            const bool grew = __any_sync(0xffffffffu, mn0 != mc0 || mn1 != mc1);
            any_rescale = grew || a_new != A;
          }
        }
        // broadcast the maxima (a head with no finite logit yet subtracts 0: its p are 0) and
        // the correction factors through this warp's slice
        mb[lane] = mn0 == -INFINITY ? 0.f : mn0;
        mb[32 + lane] = mn1 == -INFINITY ? 0.f : mn1;
        mb[64 + lane] = cr0;
        mb[96 + lane] = cr1;
        __syncwarp();
#pragma unroll
        for (int h4 = 0; h4 < 16; ++h4) {
          const float4 m = *reinterpret_cast<const float4*>(mb + 4 * h4);
          s[4 * h4 + 0] = fast_exp2(s[4 * h4 + 0] - m.x);   // exp2(-inf) = 0 for masked keys
          s[4 * h4 + 1] = fast_exp2(s[4 * h4 + 1] - m.y);
          s[4 * h4 + 2] = fast_exp2(s[4 * h4 + 2] - m.z);
          s[4 * h4 + 3] = fast_exp2(s[4 * h4 + 3] - m.w);
        }
        // ---- per-row partial denominators: l_row = l_row * cr + p (TMEM, 64 columns)
        {
          const uint32_t la = tmem + lane_base + kLCol;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float l[32];
            if (t > 0) {
              tc::tmem_ld32(la + half * 32, l);
              tc::tmem_wait_ld();
              if (any_rescale) {
#pragma unroll
                for (int h4 = 0; h4 < 8; ++h4) {
                  const float4 c = *reinterpret_cast<const float4*>(mb + 64 + half * 32 + 4 * h4);
                  l[4 * h4 + 0] = fmaf(l[4 * h4 + 0], c.x, s[half * 32 + 4 * h4 + 0]);
                  l[4 * h4 + 1] = fmaf(l[4 * h4 + 1], c.y, s[half * 32 + 4 * h4 + 1]);
                  l[4 * h4 + 2] = fmaf(l[4 * h4 + 2], c.z, s[half * 32 + 4 * h4 + 2]);
                  l[4 * h4 + 3] = fmaf(l[4 * h4 + 3], c.w, s[half * 32 + 4 * h4 + 3]);
                }
              } else {
#pragma unroll
                for (int h = 0; h < 32; ++h) l[h] += s[half * 32 + h];
              }
            } else {
#pragma unroll
              for (int h = 0; h < 32; ++h) l[h] = s[half * 32 + h];
            }
            tmem_st32(la + half * 32, l);
          }
          tmem_wait_st();
        }
        // ---- the P' buffers and O^T must be free of the previous tile's product
        if (gi > 0 && !tc::mbar_wait(pvdone, (gi - 1) & 1, abort_flag, p.err)) { ok = false; break; }
        if (any_rescale) {
          const float fa = pow2i(max(-126, min(127, a_new - A)));
          const float f0 = cr0 * fa, f1 = cr1 * fa;
          tc::fence_after_sync();
#pragma unroll 1
          for (int b = 0; b < 4; ++b) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              float o[32];
              const uint32_t addr = tmem + lane_base + kOCol + b * 64 + half * 32;
              tc::tmem_ld32(addr, o);
              tc::tmem_wait_ld();
#pragma unroll
              for (int h = 0; h < 32; ++h) o[h] *= __shfl_sync(0xffffffffu, half ? f1 : f0, h);
              tmem_st32(addr, o);
            }
          }
          tmem_wait_st();
        }
        A = a_new;
        // ---- P'^T = p * row scale * 2^A as e4m3 hi + lo, MN-major [128 keys][64 heads],
        // 64-byte swizzle: this thread writes its key's row, four 16-byte chunks per term
        {
          const float fp = sc * pow2i(A);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint32_t h0, l0, h1, l1;
              const int h = 16 * c + 4 * k;
              split_e4m3x2(s[h] * fp, s[h + 1] * fp, h0, l0);
              split_e4m3x2(s[h + 2] * fp, s[h + 3] * fp, h1, l1);
              hw[k] = h0 | (h1 << 16);
              lw[k] = l0 | (l1 << 16);
            }
            const uint32_t off = prow + (((uint32_t)c ^ pswz) << 4);
            *reinterpret_cast<uint4*>(pbuf + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(pbuf + kPBytes + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(pfull);
        mc0 = mn0;
        mc1 = mn1;
      }
      if (!ok) break;
      // ---- denominators: sum the per-row partials over the 128 rows (keys), owner thread h
      // (row < 64) gets head h's l and publishes 2^-A / l
      float l_own = 0.f;
      {
        float lv[64];
        tc::tmem_ld32(tmem + lane_base + kLCol, *reinterpret_cast<float(*)[32]>(&lv[0]));
        tc::tmem_ld32(tmem + lane_base + kLCol + 32, *reinterpret_cast<float(*)[32]>(&lv[32]));
        tc::tmem_wait_ld();
        const float2 part = reduce_scatter_sum64(lv);
        red_sum[(2 * lane) * 4 + quad] = part.x;
        red_sum[(2 * lane + 1) * 4 + quad] = part.y;
        if (!group_sync()) { ok = false; break; }
        if (row < 64) {
          const float4 v = *reinterpret_cast<const float4*>(red_sum + row * 4);
          l_own = (v.x + v.y) + (v.z + v.w);
          if (!kSplit) l_fin[(ni & 1) * 64 + row] = l_own > 0.f ? pow2i(-A) / l_own : 0.f;
        }
      }
      const float m_final = quad == 0 ? mc0 : mc1;   // used by the owners (row < 64)
      if (!kSplit && !group_sync()) { ok = false; break; }
      const float* linv = l_fin + (ni & 1) * 64;
      if (!tc::mbar_wait(ofull, ni & 1, abort_flag, p.err)) { ok = false; break; }
      tc::fence_after_sync();
      const bool even = (lane & 1) == 0;
      if (kSplit) {
        // the range's unnormalised numerator O^T in bf16, with its state (m - A, l 2^A) in
        // fp32 (O^T carries the factor 2^A of P'): lanes 2i and 2i+1 hold dims d, d+1; for
        // heads (h, h+1) the even lane stores head h's pair and the odd lane head h+1's, one
        // 32-bit store each
        const int64_t base = ((int64_t)I.qi * p.n_split + I.split) * kH;
        uint32_t* part = reinterpret_cast<uint32_t*>(p.part_o);
        for (int b = 0; b < 4; ++b) {
          const int d = b * 128 + row;
          float ob[2][32];                          // both halves of the block, one wait
          tc::tmem_ld32(tmem + lane_base + kOCol + b * 64, ob[0]);
          tc::tmem_ld32(tmem + lane_base + kOCol + b * 64 + 32, ob[1]);
          tc::tmem_wait_ld();
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const float (&o)[32] = ob[half];
#pragma unroll
            for (int h = 0; h < 32; h += 2) {
              const int hh = half * 32 + h;
              const float recv = __shfl_xor_sync(0xffffffffu, even ? o[h + 1] : o[h], 1);
              const uint32_t w = even ? pack_bf16(o[h], recv) : pack_bf16(recv, o[h + 1]);
              const int head = even ? hh : hh + 1, d0 = even ? d : d - 1;
              part[((base + head) * kD + d0) >> 1] = w;
            }
          }
        }
        if (row < 64) {
          p.part_ml[(base + row) * 2] = m_final - (float)A;
          p.part_ml[(base + row) * 2 + 1] = l_own * pow2i(A);
        }
      } else {
        // out = R^-1 (o / l) in bf16: the same pairing, the even lane rotating head h's pair
        // (d, d+1) and the odd lane head h+1's
        uint32_t* out = reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                                    (int64_t)I.qi * kH * kD);
        const int tail0 = kD - p.rope.d_r;
        for (int b = 0; b < 4; ++b) {
          const int d = b * 128 + row, d0 = even ? d : d - 1;
          float c = 1.f, sn = 0.f;
          if (d0 >= tail0) rope_cs_tab(rope_tab, I.pos, (d0 - tail0) >> 1, c, sn);
          float ob[2][32];
          tc::tmem_ld32(tmem + lane_base + kOCol + b * 64, ob[0]);
          tc::tmem_ld32(tmem + lane_base + kOCol + b * 64 + 32, ob[1]);
          tc::tmem_wait_ld();
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const float (&o)[32] = ob[half];
#pragma unroll
            for (int h = 0; h < 32; h += 2) {
              const int hh = half * 32 + h;
              const float2 li = *reinterpret_cast<const float2*>(linv + hh);
              const float a = o[h] * li.x, bb = o[h + 1] * li.y;
              const float recv = __shfl_xor_sync(0xffffffffu, even ? bb : a, 1);
              const float x0 = even ? a : recv, x1 = even ? recv : bb;   // dims d0, d0 + 1
              const int head = even ? hh : hh + 1;
              out[((int64_t)head * kD + d0) >> 1] = pack_bf16(x0 * c + x1 * sn, x1 * c - x0 * sn);
            }
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(oempty);
      ++ni;
    }
  } else {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 104;");
    // ------------------------------------------------------------ MMA issuer (warp 12)
    // The whole warp walks the items and waits (a converged warp); lane 0 issues. Order per
    // item: S(0); then for each tile t: S(t+1) as soon as the softmax has read S(t) and
    // tile t+1 is copied, then O += V P' of tile t once P'(t) is written.
    if (warp == 12) {
      constexpr uint32_t idesc_qk = idesc_e4m3(kTile, 2 * kH);
      constexpr uint32_t idesc_pv = idesc_e4m3(128, kH, true, true);
      const uint32_t k0 = tc::smem_u32(kbuf), q0 = tc::smem_u32(qbuf), p0 = tc::smem_u32(pbuf);
      const uint64_t dq = tc::sdesc_sw128(q0, 16, 1024);                   // Q~ hi/lo, K-major
      const uint64_t dph = sdesc_sw64(p0, 512);                            // P' hi, MN-major
      const uint64_t dpl = sdesc_sw64(p0 + kPBytes, 512);                  // P' lo, MN-major
      int gi = 0, ni = 0;
      bool ok = true;
      auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, tc::mbar_wait(bar, parity, abort_flag, p.err));
      };
      // S^T(g) = K Q~^T: 4 K-blocks x 4 steps of 32 dims
      auto issue_s = [&](int g, bool last) {
        tc::fence_after_sync();
        if (lane == 0) {
          const uint64_t dk = tc::sdesc_sw128(k0 + (uint32_t)(g & 1) * kKBytes, 16, 1024);
#pragma unroll
          for (int kb = 0; kb < 4; ++kb) {
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
              // descriptor start address field counts 16-byte units
              const uint64_t off = (uint64_t)((kb * 16384 + s4 * 32) >> 4);
              mma_e4m3(tmem + kSCol, dk + off, dq + off, idesc_qk, (kb | s4) ? 1u : 0u);
            }
          }
          tc::mma_commit(sfull);
          if (last) tc::mma_commit(qempty);
        }
        __syncwarp();
      };
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const Item I = make_item(p, it);
        if (I.n_tiles == 0) continue;
        if (!wait_all(qfull, ni & 1)) break;
        // S(first tile): the copy of its keys, and the softmax done reading the S^T columns
        if (!wait_all(kfull + (gi & 1), (gi >> 1) & 1)) break;
        if (gi > 0 && !wait_all(sempty, (gi - 1) & 1)) break;
        issue_s(gi, I.n_tiles == 1);
        for (int t = 0; t < I.n_tiles; ++t, ++gi) {
          if (t + 1 < I.n_tiles) {
            const int g1 = gi + 1;
            if (!wait_all(kfull + (g1 & 1), (g1 >> 1) & 1)) { ok = false; break; }
            if (!wait_all(sempty, gi & 1)) { ok = false; break; }
            issue_s(g1, t + 2 == I.n_tiles);
          }
          if (!wait_all(pfull, gi & 1)) { ok = false; break; }
          if (t == 0 && ni > 0 && !wait_all(oempty, (ni - 1) & 1)) { ok = false; break; }
          tc::fence_after_sync();
          if (lane == 0) {
            // O^T[dims of block b] += V^T (P'_hi + P'_lo)^T; V^T is the key tile read MN-major
            const uint64_t dv = tc::sdesc_sw128(k0 + (uint32_t)(gi & 1) * kKBytes, 16384, 1024);
            for (int b = 0; b < 4; ++b) {
#pragma unroll
              for (int s4 = 0; s4 < 4; ++s4) {
                const uint64_t ad = dv + (uint64_t)((b * 16384 + s4 * 4096) >> 4);
                const uint64_t boff = (uint64_t)((s4 * 32 * 64) >> 4);   // 32 keys of 64 bytes
                mma_e4m3(tmem + kOCol + b * 64, ad, dph + boff, idesc_pv, (t > 0 || s4 > 0) ? 1u : 0u);
                mma_e4m3(tmem + kOCol + b * 64, ad, dpl + boff, idesc_pv, 1u);
              }
            }
            tc::mma_commit(kempty + (gi & 1));
            tc::mma_commit(pvdone);
            if (t == I.n_tiles - 1) tc::mma_commit(ofull);
          }
          __syncwarp();
        }
        ++ni;
      }
      if (lane == 0) {
        tc::mma_commit(done);
        tc::mbar_wait_drain(done, 0);
      }
    }
    __syncwarp();
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 12) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_attention_tc(const AttnParams& p, cudaStream_t st) {
  int dev = 0, sms = 152;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t n_items = (int64_t)p.n_q * p.n_split;
  const int grid = (int)(n_items < sms ? n_items : sms);
  cudaError_t e;
  if (p.n_split > 1) {
    e = cudaFuncSetAttribute(attn_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    e = launch_pdl(attn_tc<true>, dim3(grid), dim3(kThreads), kSmemBytes, st, p);
    if (e != cudaSuccess) return e;
  } else {
    e = cudaFuncSetAttribute(attn_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    e = launch_pdl(attn_tc<false>, dim3(grid), dim3(kThreads), kSmemBytes, st, p);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace v4a
