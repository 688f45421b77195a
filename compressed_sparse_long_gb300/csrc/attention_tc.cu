// Shared-K=V attention on tcgen05 tensor cores (bf16 queries, fp8 e4m3 keys), with the
// sliding window and inverse RoPE ([notes] "DeepSeek V4 in vLLM 技术博客详尽笔记", Inverse
// RoPE 的数学原理 and 共享 Key-Value 向量; [blog] 短滑動窗口).
//
// Work item: one query (prefill) or one key range of one query (decode split). Keys come
// in tiles of 128 rows gathered from the paged pools (top-k entries or all visible
// entries, then the window tokens). Per tile:
//   S^T = K Q~^T      M = 128 keys, N = 64 heads, K = 512 dims   (32 MMAs, TMEM cols 0..63)
//   softmax over keys per head: column max with redux.sync.max.f32 across the warp and a
//     4-warp exchange, column sums with a butterfly reduce-scatter; the running max is
//     raised only when it grows by more than 2^8 (then the O^T accumulator is rescaled)
//   O^T += V^T P'^T   M = 128 dims x 4 blocks, N = 64 heads, K = 128 keys (32 MMAs,
//                     TMEM cols 64..319)
// K = V: the same shared-memory key tile (fp8 codes converted exactly to bf16, 128-byte
// swizzle) is read K-major by the first product and MN-major by the second. The fp8 row
// scale is applied to the logits after S^T and folded into P' = p * scale before the
// second product, so keys stay exact codes. Q~ = RoPE(q, p) * softmax_scale * log2(e) in
// bf16; logits are in log2 units.
//
// Warpgroups (setmaxnreg splits the 512 x 128 launch registers as 152 / 128 / 128 / 104):
// 0 = softmax and epilogue (warp w reads TMEM lanes 32w..32w+31), 1-2 = eight
// gather/convert warps that also build Q~, 3 = warp 12 allocates TMEM, walks the items
// converged and issues the MMAs from lane 0 (warps 13-15 idle).
// Every hand-off is an mbarrier with a bounded wait (V4A_DEV_TIMEOUT on expiry).
// Decode split: each key range's CTA writes its partial as o / l in bf16 plus (m, l) in
// fp32; the merge kernel combines the ranges and applies R^-1.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace v4a {
namespace {

constexpr int kH = 64, kD = 512, kTile = 128;
constexpr int kThreads = 512;                 // 4 warpgroups
constexpr int kKBytes = kTile * kD * 2;        // 128 KB key tile, 8 K-blocks of 16 KB
constexpr int kQBytes = kH * kD * 2;           // 64 KB Q~, 8 K-blocks of 8 KB
constexpr int kPBytes = kTile * kH * 2;        // 16 KB P'^T
constexpr int kOffK = 0, kOffQ = kKBytes, kOffP = kOffQ + kQBytes;
constexpr int kOffF = kOffP + kPBytes;         // floats: l_fin[2][64] red_max[2][256] red_sum[2][256] sscale[2][128]
constexpr int kOffBar = kOffF + (128 + 512 + 512 + 256) * 4;
constexpr int kNBar = 4 + 4 + 13;
constexpr int kOffMisc = kOffBar + kNBar * 8;
constexpr int kSmemBytes = kOffMisc + 64 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 0, kOCol = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;      // log2 units

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

template <bool kSplit>
__global__ void __launch_bounds__(kThreads, 1) attn_tc(const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = tc::smem_u32(smem_raw);
  uint8_t* sm = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  uint8_t* kbuf = sm + kOffK;
  uint8_t* qbuf = sm + kOffQ;
  uint8_t* pbuf = sm + kOffP;
  float* l_fin = reinterpret_cast<float*>(sm + kOffF);   // [2][64] 1 / l by item parity
  float* red_max = l_fin + 128;                           // [2][64 heads][4 warps]
  float* red_sum = red_max + 512;                         // [2][64 heads][4 warps]
  float* sscale = red_sum + 512;                          // [2][128] row scales by tile parity
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint64_t* kfull = bars;
  uint64_t* kempty = bars + 4;
  uint64_t* qfull = bars + 8;
  uint64_t* qempty = bars + 9;
  uint64_t* sfull = bars + 10;
  uint64_t* pfull = bars + 11;
  uint64_t* pvdone = bars + 12;
  uint64_t* ofull = bars + 13;
  uint64_t* oempty = bars + 14;
  uint64_t* redb = bars + 15;
  uint64_t* done = bars + 16;
  uint64_t* scfull = bars + 17;
  int* misc = reinterpret_cast<int*>(sm + kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
  volatile int* abort_flag = misc + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_items = p.n_q * p.n_split;
  // On-chip setup and the first query's Q~ read only this call's inputs and overlap the
  // previous kernel; the key gathers (top-k lists, pools) and every global write wait.
  pdl_trigger();

  if (tid == 0) {
    for (int b = 0; b < 4; ++b) {
      tc::mbar_init(kfull + b, 8);
      tc::mbar_init(kempty + b, 1);
    }
    tc::mbar_init(qfull, 8);
    tc::mbar_init(qempty, 1);
    tc::mbar_init(sfull, 1);
    tc::mbar_init(pfull, 4);
    tc::mbar_init(pvdone, 1);
    tc::mbar_init(ofull, 1);
    tc::mbar_init(oempty, 4);
    tc::mbar_init(redb, 4);
    tc::mbar_init(done, 1);
    tc::mbar_init(scfull, 8);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 12) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 4 && warp < 12) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 128;");
    // ------------------------------------------------------------ gather / convert
    // Eight warps; warp cw owns key rows 16cw .. 16cw+15 of every tile (lanes 0-15 resolve
    // them and publish their row scales). A lane holds 16 x 16 fp8 codes of a tile in
    // registers: for block b (128 dims) and j = 0..3, row 16cw + 4j + lane/8, codes
    // 128b + 16(lane%8) .. +15 (each warp load covers four 128-byte row segments). The
    // next tile's loads are issued as soon as the current tile is converted, so they are
    // in flight during the current tile's products and softmax.
    const int cw = warp - 4;
    int gi = 0, ni = 0;   // global tile / item counters of this CTA
    bool ok = true;
    uint4 d[4][4];        // [block][j]
    float sc_row = 0.f;   // scale of row 16cw + lane (lanes < 16)
    auto issue = [&](const Item& I, int t) {
      const int64_t x = I.x0 + (int64_t)t * kTile + cw * 16 + (lane & 15);
      bool is_swa;
      const int64_t slot = key_slot(p, I, x, is_swa, lane < 16);
      const uint8_t* rowp = nullptr;
      sc_row = 0.f;
      if (slot >= 0) {
        const CacheView& cv = is_swa ? p.swa : p.attn;
        rowp = reinterpret_cast<const uint8_t*>(cv.data) + slot * (int64_t)cv.width;
        sc_row = __ldg(cv.scale + slot);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(rowp), 4 * j + (lane >> 3)));
#pragma unroll
        for (int b = 0; b < 4; ++b)
          d[b][j] = src ? __ldg(reinterpret_cast<const uint4*>(src + b * 128 + (lane & 7) * 16))
                        : make_uint4(0, 0, 0, 0);
      }
    };
    bool waited = false;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const Item I = make_item(p, it);
      if (I.n_tiles == 0) continue;
      if (waited) issue(I, 0);                      // tile 0 of the item in flight
      // Q~ = RoPE(q, p) * scale * log2(e), bf16, K-major 128B-swizzled [64 heads][512]
      if (ni > 0 && !tc::mbar_wait(qempty, (ni - 1) & 1, abort_flag, p.err)) { ok = false; break; }
      {
        const int tail0 = kD - p.rope.d_r;
        float c = 1.f, s = 0.f;
        if (lane < p.rope.d_r / 2) rope_cs(p.rope, I.pos, lane, c, s);
        const float qs = p.scale * kLog2e;
        const uint4* q = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.q) +
                                                        (int64_t)I.qi * kH * kD);
        const int ct = cw * 32 + lane;              // 0..255
#pragma unroll 1
        for (int base = 0; base < kH * (kD / 8); base += 256 * 8) {
          uint4 u[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) u[k] = __ldg(q + base + k * 256 + ct);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int item = base + k * 256 + ct;
            const int h = item / (kD / 8), ch = item % (kD / 8);   // 8 dims per chunk
            const __nv_bfloat16* e = reinterpret_cast<const __nv_bfloat16*>(&u[k]);
            float f[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] = __bfloat162float(e[j]);
            const int d0 = ch * 8;
            const bool tail = d0 >= tail0;
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
              const int pi = tail ? (d0 + j - tail0) >> 1 : 0;
              const float cc = __shfl_sync(0xffffffffu, c, pi);
              const float ss = __shfl_sync(0xffffffffu, s, pi);
              if (tail) {
                const float a0 = f[j], a1 = f[j + 1];
                f[j] = a0 * cc - a1 * ss;
                f[j + 1] = a0 * ss + a1 * cc;
              }
            }
            uint4 o;
            o.x = pack_bf16(f[0] * qs, f[1] * qs);
            o.y = pack_bf16(f[2] * qs, f[3] * qs);
            o.z = pack_bf16(f[4] * qs, f[5] * qs);
            o.w = pack_bf16(f[6] * qs, f[7] * qs);
            *reinterpret_cast<uint4*>(qbuf + (ch >> 3) * 8192 + tc::sw128_off(h, ch & 7)) = o;
          }
        }
        tc::fence_proxy_async();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(qfull);
      }
      if (!waited) {                                // first item: Q~ was built meanwhile
        pdl_wait();
        waited = true;
        issue(I, 0);
      }
      for (int t = 0; t < I.n_tiles; ++t, ++gi) {
        for (int b = 0; b < 4; ++b) {
          if (!tc::mbar_wait(kempty + b, (gi & 1) ^ 1, abort_flag, p.err)) { ok = false; break; }
          if (b == 0) {
            // row scales for the softmax warps; the previous tile's product is done, so the
            // softmax warps have consumed the previous hand-off
            if (lane < 16) sscale[(gi & 1) * kTile + cw * 16 + lane] = sc_row;
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(scfull);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint4 lo, hi;
            e4m3x16_to_bf16x16(d[b][j], lo, hi);
            const int r = cw * 16 + 4 * j + (lane >> 3);
            const int c0 = 2 * (lane & 7);               // bf16 chunk within the 128-dim block
            const int kb = 2 * b + (c0 >> 3);
            *reinterpret_cast<uint4*>(kbuf + kb * 16384 + tc::sw128_off(r, c0 & 7)) = lo;
            *reinterpret_cast<uint4*>(kbuf + kb * 16384 + tc::sw128_off(r, (c0 + 1) & 7)) = hi;
          }
          tc::fence_proxy_async();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(kfull + b);
        }
        if (!ok) break;
        if (t + 1 < I.n_tiles) issue(I, t + 1);     // next tile in flight during this one
      }
      ++ni;
    }
  } else if (warp < 4) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 152;");
    pdl_wait();
    // ------------------------------------------------------------ softmax + epilogue
    // Every lane keeps the running max of heads `lane` and `lane + 32` in registers (all
    // four warps hold the same copy); the owner of head h (thread row h) keeps its
    // denominator in a register and publishes it in l_fin[item parity][64] for the epilogue.
    const int quad = warp;
    const int row = quad * 32 + lane;             // TMEM lane: key (S^T) or dim (O^T)
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
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
      float l_reg = 0.f;                          // owner threads (row < 64)
      float mc0 = -INFINITY, mc1 = -INFINITY;     // running max of heads lane, lane + 32
      for (int t = 0; t < I.n_tiles; ++t, ++gi) {
        if (!tc::mbar_wait(sfull, gi & 1, abort_flag, p.err)) { ok = false; break; }
        tc::fence_after_sync();
        float s[64];
        {
          float a[32];
          tc::tmem_ld32(tmem + lane_base + kSCol, a);
#pragma unroll
          for (int h = 0; h < 32; ++h) s[h] = a[h];
          tc::tmem_ld32(tmem + lane_base + kSCol + 32, a);
#pragma unroll
          for (int h = 0; h < 32; ++h) s[32 + h] = a[h];
          tc::tmem_wait_ld();
        }
        if (!tc::mbar_wait(scfull, gi & 1, abort_flag, p.err)) { ok = false; break; }
        const float sc = sscale[(gi & 1) * kTile + row];   // 0 for a masked key
#pragma unroll
        for (int h = 0; h < 64; ++h) s[h] = sc > 0.f ? s[h] * sc : -INFINITY;
        // ---- per-head max over the tile's 128 keys
        float* rb = red_max + (ru & 1) * 256;
#pragma unroll
        for (int h = 0; h < 64; ++h) {
          const float mh = redux_max(s[h]);
          if (lane == (h & 31)) rb[h * 4 + quad] = mh;
        }
        if (!group_sync()) { ok = false; break; }
        // new running max of heads lane and lane + 32 (raised only past the threshold) and
        // the correction factors exp2(old - new) of the accumulated O^T and denominators
        float mn0, mn1, cr0 = 1.f, cr1 = 1.f;
        bool any_rescale = false;
        {
          const float4 v0 = *reinterpret_cast<const float4*>(rb + lane * 4);
          const float4 v1 = *reinterpret_cast<const float4*>(rb + (lane + 32) * 4);
          const float mt0 = fmaxf(fmaxf(v0.x, v0.y), fmaxf(v0.z, v0.w));
          const float mt1 = fmaxf(fmaxf(v1.x, v1.y), fmaxf(v1.z, v1.w));
          if (t == 0) {                          // nothing accumulated yet
            mn0 = mt0;
            mn1 = mt1;
          } else {
            mn0 = mt0 > mc0 + kRescaleThreshold ? mt0 : mc0;
            mn1 = mt1 > mc1 + kRescaleThreshold ? mt1 : mc1;
            if (mn0 != mc0) cr0 = fast_exp2(mc0 - mn0);   // 0 when the old max is -inf
            if (mn1 != mc1) cr1 = fast_exp2(mc1 - mn1);
            any_rescale = __any_sync(0xffffffffu, mn0 != mc0 || mn1 != mc1);
          }
        }
#pragma unroll
        for (int h = 0; h < 64; ++h) {
          const float mn = __shfl_sync(0xffffffffu, h < 32 ? mn0 : mn1, h & 31);
          s[h] = (mn == -INFINITY || s[h] == -INFINITY) ? 0.f : fast_exp2(s[h] - mn);
        }
        // ---- the P' buffer and O^T must be free of the previous tile's product
        if (gi > 0 && !tc::mbar_wait(pvdone, (gi - 1) & 1, abort_flag, p.err)) { ok = false; break; }
        if (any_rescale) {
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
              for (int h = 0; h < 32; ++h) o[h] *= __shfl_sync(0xffffffffu, half ? cr1 : cr0, h);
              tmem_st32(addr, o);
            }
          }
          tmem_wait_st();
        }
        // ---- P'^T row of this key: p * row scale, bf16, MN-major swizzled [128 keys][64 heads]
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 v;
          v.x = pack_bf16(s[8 * c + 0] * sc, s[8 * c + 1] * sc);
          v.y = pack_bf16(s[8 * c + 2] * sc, s[8 * c + 3] * sc);
          v.z = pack_bf16(s[8 * c + 4] * sc, s[8 * c + 5] * sc);
          v.w = pack_bf16(s[8 * c + 6] * sc, s[8 * c + 7] * sc);
          *reinterpret_cast<uint4*>(pbuf + tc::sw128_off(row, c)) = v;
        }
        tc::fence_proxy_async();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(pfull);
        // ---- per-head sums of p over the tile's keys -> the owners' denominators (these
        // overlap the P'V product, which only needs P')
        float* rs = red_sum + (ru & 1) * 256;
        const float2 part = reduce_scatter_sum64(s);
        rs[(2 * lane) * 4 + quad] = part.x;
        rs[(2 * lane + 1) * 4 + quad] = part.y;
        if (!group_sync()) { ok = false; break; }
        mc0 = mn0;
        mc1 = mn1;
        if (row < 64) {
          const float4 v = *reinterpret_cast<const float4*>(rs + row * 4);
          l_reg = l_reg * (quad == 0 ? cr0 : cr1) + ((v.x + v.y) + (v.z + v.w));
        }
      }
      if (!ok) break;
      // ---- publish the denominators, then read O^T (lanes: dims 128b + row; cols: heads)
      if (row < 64) l_fin[(ni & 1) * 64 + row] = l_reg > 0.f ? 1.f / l_reg : 0.f;   // 1 / l
      const float m_final = quad == 0 ? mc0 : mc1;   // used by the owners (row < 64)
      if (!group_sync()) { ok = false; break; }
      const float* linv = l_fin + (ni & 1) * 64;
      if (!tc::mbar_wait(ofull, ni & 1, abort_flag, p.err)) { ok = false; break; }
      tc::fence_after_sync();
      if (kSplit) {
        // partial o / l in bf16 (the range's max and denominator go out in fp32): lanes 2i
        // and 2i+1 hold dims d, d+1; for heads (h, h+1) the even lane stores head h's pair
        // and the odd lane head h+1's, one 32-bit store each
        const int64_t base = ((int64_t)I.qi * p.n_split + I.split) * kH;
        uint32_t* part = reinterpret_cast<uint32_t*>(p.part_o);
        const bool even = (lane & 1) == 0;
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
              const float a = o[h] * linv[hh], bb = o[h + 1] * linv[hh + 1];
              const float recv = __shfl_xor_sync(0xffffffffu, even ? bb : a, 1);
              const uint32_t w = even ? pack_bf16(a, recv) : pack_bf16(recv, bb);
              const int head = even ? hh : hh + 1, d0 = even ? d : d - 1;
              part[((base + head) * kD + d0) >> 1] = w;
            }
          }
        }
        if (row < 64) {
          p.part_ml[(base + row) * 2] = m_final;
          p.part_ml[(base + row) * 2 + 1] = l_reg;
        }
      } else {
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + (int64_t)I.qi * kH * kD;
        const int tail0 = kD - p.rope.d_r;
        for (int b = 0; b < 4; ++b) {
          const int d = b * 128 + row;
          float c = 1.f, sn = 0.f;
          const bool tail = d >= tail0;
          if (tail) rope_cs(p.rope, I.pos, (d - tail0) >> 1, c, sn);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float o[32];
            tc::tmem_ld32(tmem + lane_base + kOCol + b * 64 + half * 32, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < 32; ++h) {
              float v = o[h] * linv[half * 32 + h];
              const float partner = __shfl_xor_sync(0xffffffffu, v, 1);
              if (tail) v = (d & 1) ? (-partner * sn + v * c) : (v * c + partner * sn);
              out[(int64_t)(half * 32 + h) * kD + d] = __float2bfloat16_rn(v);
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
    // The whole warp walks the items and waits (a converged warp); lane 0 issues.
    if (warp == 12) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16(kTile, kH);
      constexpr uint32_t idesc_pv = tc::idesc_bf16(128, kH, true, true);
      const uint32_t k0 = tc::smem_u32(kbuf), q0 = tc::smem_u32(qbuf), p0 = tc::smem_u32(pbuf);
      const uint64_t dk_k = tc::sdesc_sw128(k0, 16, 1024);        // key tile, K-major
      const uint64_t dq_k = tc::sdesc_sw128(q0, 16, 1024);        // Q~, K-major
      const uint64_t dk_mn = tc::sdesc_sw128(k0, 16384, 1024);    // key tile as V^T, MN-major
      const uint64_t dp_mn = tc::sdesc_sw128(p0, 8192, 1024);     // P'^T, MN-major
      int gi = 0, ni = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const Item I = make_item(p, it);
        if (I.n_tiles == 0) continue;
        if (!__all_sync(0xffffffffu, tc::mbar_wait(qfull, ni & 1, abort_flag, p.err))) break;
        for (int t = 0; t < I.n_tiles; ++t, ++gi) {
          // S^T = K Q~^T over the 8 K-blocks, block pair b as soon as it is converted
          for (int b = 0; b < 4; ++b) {
            if (!__all_sync(0xffffffffu, tc::mbar_wait(kfull + b, gi & 1, abort_flag, p.err))) { ok = false; break; }
            tc::fence_after_sync();
            if (lane == 0) {
#pragma unroll
              for (int kk = 0; kk < 2; ++kk) {
                const int kb = 2 * b + kk;
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                  // descriptor start address field counts 16-byte units
                  const uint64_t ad = dk_k + (uint64_t)((kb * 16384 + s4 * 32) >> 4);
                  const uint64_t bd = dq_k + (uint64_t)((kb * 8192 + s4 * 32) >> 4);
                  tc::mma_bf16(tmem + kSCol, ad, bd, idesc_qk, (kb | s4) ? 1u : 0u);
                }
              }
            }
            __syncwarp();
          }
          if (!ok) break;
          if (lane == 0) {
            tc::mma_commit(sfull);
            if (t == I.n_tiles - 1) tc::mma_commit(qempty);
          }
          __syncwarp();
          if (!__all_sync(0xffffffffu, tc::mbar_wait(pfull, gi & 1, abort_flag, p.err))) { ok = false; break; }
          if (t == 0 && ni > 0 &&
              !__all_sync(0xffffffffu, tc::mbar_wait(oempty, (ni - 1) & 1, abort_flag, p.err))) { ok = false; break; }
          tc::fence_after_sync();
          if (lane == 0) {
            // O^T[dims of block b] += V^T P'^T; V^T is the key tile read MN-major
            for (int b = 0; b < 4; ++b) {
#pragma unroll
              for (int s8 = 0; s8 < 8; ++s8) {
                const uint64_t ad = dk_mn + (uint64_t)(((2 * b) * 16384 + s8 * 2048) >> 4);
                const uint64_t bd = dp_mn + (uint64_t)((s8 * 2048) >> 4);
                tc::mma_bf16(tmem + kOCol + b * 64, ad, bd, idesc_pv, (t > 0 || s8 > 0) ? 1u : 0u);
              }
              tc::mma_commit(kempty + b);
            }
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
