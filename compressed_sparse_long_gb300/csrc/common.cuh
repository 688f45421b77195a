// Device helpers shared by the v4a kernels: paged-cache views, slot lookup, RoPE angles,
// fp8 e4m3 <-> fp32/bf16 conversion, warp reductions, the device error word.
#pragma once

#include <utility>

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/v4a.h"

namespace v4a {

constexpr int kBlock = 256;       // native positions per logical block
constexpr int kMaxRopePairs = 32; // d_r <= 64
constexpr float kE4m3Max = 448.0f;

// Kernel-parameter copy of a v4a_cache.
struct CacheView {
  void* data;
  float* scale;
  const int32_t* bt;
  int64_t n_pages;
  int32_t max_blocks;
  int32_t R;
  int32_t width;
  int32_t shift;     // log2(R) when R is a power of two (every layer pool), else -1
};

inline CacheView view_of(const v4a_cache* c) {
  CacheView v{};
  v.shift = -1;
  if (c) {
    v.data = c->data;
    v.scale = c->scale;
    v.bt = c->block_table;
    v.n_pages = c->n_pages;
    v.max_blocks = c->max_blocks;
    v.R = c->rows_per_block;
    v.width = c->row_width;
    if (v.R > 0 && (v.R & (v.R - 1)) == 0)
      for (v.shift = 0; (1 << v.shift) < v.R; ++v.shift) {}
  }
  return v;
}

// Pool row of logical row r of sequence seq: page * R + r % R, -1 if the block has no
// page (or r is out of the table), -2 if the page id is outside the pool.
__device__ __forceinline__ int64_t slot_of(const CacheView& c, int seq, int64_t r) {
  if (r < 0) return -1;
  const int64_t blk = c.shift >= 0 ? r >> c.shift : r / c.R;
  if (blk >= c.max_blocks) return -1;
  int32_t page = __ldg(c.bt + (int64_t)seq * c.max_blocks + blk);
  if (page < 0) return -1;
  if (page >= c.n_pages) return -2;
  const int64_t off = c.shift >= 0 ? (r & (int64_t)(c.R - 1)) : r % c.R;
  return (int64_t)page * c.R + off;
}

__device__ __forceinline__ void raise_err(int32_t* err, uint32_t bits) {
  if (err) atomicOr(reinterpret_cast<unsigned int*>(err), bits);
}

// Report a failed slot lookup; returns true when the slot is usable.
__device__ __forceinline__ bool slot_ok(int64_t s, int32_t* err) {
  if (s >= 0) return true;
  raise_err(err, s == -2 ? V4A_DEV_BAD_PAGE : V4A_DEV_MISSING_PAGE);
  return false;
}

// RoPE frequencies theta_i = base^(-2i/d_r), kept as turns per position
// phi_i = theta_i / (2 pi) and psi_i = frac(4096 phi_i), each split into fp32 hi + lo parts
// on the host (in double). The device never uses fp64.
struct Rope {
  int32_t d_r;
  int32_t D;
  float phi_hi[kMaxRopePairs], phi_lo[kMaxRopePairs];
  float psi_hi[kMaxRopePairs], psi_lo[kMaxRopePairs];
};

// Fractional part of x * (yh + yl), x an integer below 2^24: x*yh = p + e exactly (fma),
// p - rint(p) is exact, the remaining terms are tiny.
__device__ __forceinline__ float frac_prod(float x, float yh, float yl) {
  const float p = x * yh;
  const float e = fmaf(x, yh, -p);
  return (p - rintf(p)) + (e + x * yl);
}

// cos/sin of pos * theta_i. With pos = hi * 4096 + lo the angle in turns is
// frac(hi * psi_i + lo * phi_i), reduced exactly in fp32 (error ~1e-7 turn for positions up
// to 2^31); sincospif then evaluates the reduced angle.
// Pair i's four angle constants read with a per-thread index come from the constant bank
// one address at a time; kernels that evaluate many angles stage them in shared memory
// first ([4][kMaxRopePairs]: phi_hi, phi_lo, psi_hi, psi_lo) and use rope_cs_tab.
__device__ __forceinline__ void stage_rope(const Rope& rp, float* tab, int tid, int nthreads) {
  for (int k = tid; k < 4 * kMaxRopePairs; k += nthreads) {
    const int a = k / kMaxRopePairs, i = k % kMaxRopePairs;
    tab[k] = a == 0 ? rp.phi_hi[i] : a == 1 ? rp.phi_lo[i] : a == 2 ? rp.psi_hi[i] : rp.psi_lo[i];
  }
}
__device__ __forceinline__ void rope_cs_tab(const float* tab, int64_t pos, int i, float& c, float& s) {
  const float hi = (float)(int32_t)(pos >> 12), lo = (float)(int32_t)(pos & 4095);
  float a = frac_prod(hi, tab[2 * kMaxRopePairs + i], tab[3 * kMaxRopePairs + i]) +
            frac_prod(lo, tab[i], tab[kMaxRopePairs + i]);
  a -= rintf(a);
  sincospif(2.0f * a, &s, &c);
}

__device__ __forceinline__ void rope_cs(const Rope& rp, int64_t pos, int i, float& c, float& s) {
  // (positions below 2^43: both parts convert from 32-bit integers)
  const float hi = (float)(int32_t)(pos >> 12), lo = (float)(int32_t)(pos & 4095);
  float a = frac_prod(hi, rp.psi_hi[i], rp.psi_lo[i]) + frac_prod(lo, rp.phi_hi[i], rp.phi_lo[i]);
  a -= rintf(a);
  sincospif(2.0f * a, &s, &c);
}

// ---------------------------------------------------------------- warp reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ---------------------------------------------------------------- element access
template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float to_f(float x) { return x; }
  static __device__ __forceinline__ float from_f(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

// Load n contiguous elements (n * sizeof(T) a multiple of 4 bytes) into fp32 registers,
// using the widest aligned vector the byte count allows.
template <typename T, int N>
__device__ __forceinline__ void load_f(const T* __restrict__ p, float (&out)[N]) {
  constexpr int kBytes = N * (int)sizeof(T);
  if constexpr (kBytes % 16 == 0) {
    constexpr int kVec = kBytes / 16;
    constexpr int kPer = 16 / sizeof(T);
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      uint4 u = __ldg(reinterpret_cast<const uint4*>(p) + v);
      const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
      for (int k = 0; k < kPer; ++k) out[v * kPer + k] = Elem<T>::to_f(e[k]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < N; ++k) out[k] = Elem<T>::to_f(p[k]);
  }
}

template <typename T, int N>
__device__ __forceinline__ void store_f(T* __restrict__ p, const float (&in)[N]) {
  constexpr int kBytes = N * (int)sizeof(T);
  if constexpr (kBytes % 16 == 0) {
    constexpr int kVec = kBytes / 16;
    constexpr int kPer = 16 / sizeof(T);
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      uint4 u;
      T* e = reinterpret_cast<T*>(&u);
#pragma unroll
      for (int k = 0; k < kPer; ++k) e[k] = Elem<T>::from_f(in[v * kPer + k]);
      reinterpret_cast<uint4*>(p)[v] = u;
    }
  } else {
#pragma unroll
    for (int k = 0; k < N; ++k) p[k] = Elem<T>::from_f(in[k]);
  }
}

// ---------------------------------------------------------------- fp8 e4m3
// Encode: round-to-nearest-even, saturating to +-448 (cvt.rn.satfinite.e4m3x2.f32).
__device__ __forceinline__ uint16_t e4m3x2_encode(float lo, float hi) {
  __nv_fp8x2_storage_t r = __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
  return (uint16_t)r;
}

// ---------------------------------------------------------------- fp4 e2m1
constexpr float kE2m1Max = 6.0f;

// Encode: round-to-nearest-even onto the e2m1 magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6},
// saturating to +-6; bit 3 is the sign. Each comparison is a rounding midpoint, strict
// where the lower neighbour has the odd code (so a tie goes to the even code).
__device__ __forceinline__ uint32_t e2m1_encode(float v) {
  const float a = fminf(fabsf(v), kE2m1Max);
  const uint32_t m = (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
                     (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) +
                     (uint32_t)(a > 5.0f);
  return m | (signbit(v) ? 8u : 0u);
}

// Expand four e2m1 codes (one 16-bit group, code k in bits 4k..4k+3) into four e4m3 codes
// (byte k of the result). Every e2m1 value is an e4m3 value: the magnitudes map to the
// e4m3 codes 0x00 0x30 0x38 0x3C 0x40 0x44 0x48 0x4C (a byte permute looks them up) and
// the sign bit moves to bit 7 of its byte.
__device__ __forceinline__ uint32_t e2m1x4_to_e4m3x4(uint32_t x) {
  const uint32_t mag = __byte_perm(0x3C383000u, 0x4C484440u, x & 0x7777u);
  const uint32_t sg = ((x & 0x8u) << 4) | ((x & 0x80u) << 8) | ((x & 0x800u) << 12) |
                      ((x & 0x8000u) << 16);
  return mag | sg;
}

// Decode 4 codes (one 32-bit word, code k in byte k) to fp32. e4m3 -> f16 is exact.
__device__ __forceinline__ void e4m3x4_decode(uint32_t w, float (&f)[4]) {
  uint32_t h01, h23;
  asm("{ .reg .b16 lo, hi; mov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, hi; }"
      : "=r"(h01), "=r"(h23) : "r"(w));
  __half2 a = *reinterpret_cast<__half2*>(&h01);
  __half2 b = *reinterpret_cast<__half2*>(&h23);
  float2 fa = __half22float2(a), fb = __half22float2(b);
  f[0] = fa.x; f[1] = fa.y; f[2] = fb.x; f[3] = fb.y;
}

// Decode 2 codes (byte 0 -> low half, byte 1 -> high half) to a bf16x2 word. e4m3 -> bf16
// is exact: the code's sign and exponent/mantissa bits are placed in a bf16 whose
// exponent is 120 too small, then scaled by 2^120 with an exact bf16 multiply (subnormal
// codes land on bf16 subnormals first and become normal after the scaling).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two_codes_in_low16) {
  // byte k -> bits [16k+8, 16k+15]
  uint32_t t = __byte_perm(two_codes_in_low16, 0u, 0x1404);  // [c0<<8 | c1<<24]
  uint32_t mag = (t >> 4) & 0x07F007F0u;
  uint32_t sgn = t & 0x80008000u;
  uint32_t bits = mag | sgn;
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(bits), "r"(0x7B807B80u));
  return r;
}

// Four codes (byte k of w is code k) to two bf16x2 words (codes 0,1 -> lo; 2,3 -> hi),
// with the same exact placement-and-scale as e4m3x2_to_bf16x2.
__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t t0 = __byte_perm(w, 0u, 0x1404);   // c0 << 8 | c1 << 24
  const uint32_t t1 = __byte_perm(w, 0u, 0x3424);   // c2 << 8 | c3 << 24
  const uint32_t b0 = ((t0 >> 4) & 0x07F007F0u) | (t0 & 0x80008000u);
  const uint32_t b1 = ((t1 >> 4) & 0x07F007F0u) | (t1 & 0x80008000u);
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(lo) : "r"(b0), "r"(0x7B807B80u));
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(hi) : "r"(b1), "r"(0x7B807B80u));
}

// 16 codes -> 16 bf16 (two 16-byte chunks: codes 0-7 in lo, 8-15 in hi).
__device__ __forceinline__ void e4m3x16_to_bf16x16(const uint4& u, uint4& lo, uint4& hi) {
  e4m3x4_to_bf16x4(u.x, lo.x, lo.y);
  e4m3x4_to_bf16x4(u.y, lo.z, lo.w);
  e4m3x4_to_bf16x4(u.z, hi.x, hi.y);
  e4m3x4_to_bf16x4(u.w, hi.z, hi.w);
}

__device__ __forceinline__ int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Programmatic dependent launch. Every kernel of the library lets the next kernel of its
// stream start early (pdl_trigger, at its start) and, in each thread, waits for the kernels
// before it (pdl_wait: they have completed and their memory is visible) before it reads
// memory one of them may write or writes memory one of them may read. Work on the call's
// own inputs (queries, positions, block tables, weights) and on-chip setup may run before
// the wait, overlapping the previous kernel. Both are no-ops without the launch attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Floats between consecutive indexer score rows: rows start on 16-byte boundaries.
__host__ __device__ __forceinline__ int64_t score_row_stride(int64_t max_vis) {
  return (max_vis + 3) & ~(int64_t)3;
}

// Number of entries visible to a query at p: entry j qualifies iff its last covered
// position S*j + win_off + W - 1 is < p.
__host__ __device__ __forceinline__ int64_t visible_entries(int64_t p, int S, int W, int win_off) {
  int64_t num = p - win_off - W;
  if (num < 0) return 0;
  return num / S + 1;
}

}  // namespace v4a
