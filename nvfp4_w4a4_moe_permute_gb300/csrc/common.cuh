// Device-side building blocks shared by the minite kernels (sm_103a):
// NVFP4 scalar conversions, the warp-level row quantizer, the specified
// exponential, and thin inline-PTX wrappers for mbarrier, TMA and tcgen05.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/minite.h"

namespace minite {

constexpr int kWarp = 32;
constexpr float kE2M1Max = 6.0f;
constexpr float kGlobalNumerator = 2688.0f;  // 448 (E4M3 max) * 6 (E2M1 max)
constexpr float kFltMax = 3.402823466e+38f;

__device__ __forceinline__ void set_status(int32_t* status, int code) {
  if (status) atomicOr(status, 1 << code);
}

// Programmatic dependent launch: pdl_wait blocks the calling thread until the
// kernel launched before this one on the stream has completed and its writes
// are visible (it returns at once when this kernel was launched without the
// programmatic attribute). A kernel calls it before its first global memory
// access, so only prologue work that touches no global memory (barrier
// setup, TMEM allocation, tables in shared memory) overlaps the previous
// kernel's last CTAs. No kernel triggers its dependents early: measured on
// the CUDA-graph step, an early trigger slowed the step down.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ----------------------------------------------------------------------------
// BF16 / scalar format conversions
// ----------------------------------------------------------------------------

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
// v rounded to the nearest BF16 (ties to even), as a float. Rounding is
// monotone and odd, so the |x| maximum of a row rounded to BF16 is the
// rounded |x| maximum of the row.
__device__ __forceinline__ float bf16_round(float v) {
  return __uint_as_float(static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v))) << 16);
}

// Round to nearest even onto the E2M1 grid, saturating at +-6, sign kept.
// Returns one byte holding `lo` in bits 0..3 and `hi` in bits 4..7.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t out;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %2, %1;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(out) : "f"(lo), "f"(hi));
  return out & 0xFFu;
}

// Non-negative finite float -> unsigned E4M3 code (nearest even, saturate 448).
__device__ __forceinline__ uint32_t cvt_e4m3(float s) {
  uint16_t out;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(out) : "f"(s), "f"(0.0f));
  return out & 0xFFu;
}

// Unsigned E4M3 code (never 0x7F) -> float, exact.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
  uint32_t e = (c >> 3) & 0xF, m = c & 7;
  if (e == 0) return __fmul_rn(static_cast<float>(m), 0.001953125f);  // m * 2^-9
  return __uint_as_float(((e + 120u) << 23) | (m << 20));              // (1+m/8) * 2^(e-7)
}

// g = min(2688 / amax, FLT_MAX) for amax > 0, else 1.
__device__ __forceinline__ float global_scale(float amax) {
  if (!(amax > 0.0f)) return 1.0f;
  return fminf(__fdiv_rn(kGlobalNumerator, amax), kFltMax);
}

// x / 6 rounded to nearest for finite x >= 0, by Markstein's FMA-corrected
// division by a constant (q0 = x * RN(1/6); r = x - 6 q0 exactly; q = q0 + r
// RN(1/6)), with IEEE division kept for tiny x where the remainder could be
// inexact. Equality with IEEE division over every non-negative finite float
// is checked on the device by minite_test_div6_exhaustive.
__device__ __forceinline__ float div6_rn(float x) {
  constexpr float kSixth = 0.16666667163372039794921875f;  // RN(1/6)
  if (x < 1.0e-30f) return __fdiv_rn(x, kE2M1Max);
  const float q0 = __fmul_rn(x, kSixth);
  const float r = __fmaf_rn(-kE2M1Max, q0, x);
  return __fmaf_rn(r, kSixth, q0);
}

// Per-row table of encode factors: lane l holds RN(g / (1 + (l & 7) / 8)), g
// divided by each of the 8 E4M3 significands. A block's factor RN(g / sf) is
// the entry of sf's significand scaled by a power of two, which is exact
// whenever the result is a normal float (checked; IEEE division otherwise).
__device__ __forceinline__ float enc_table_entry(float g) {
  return __fdiv_rn(g, 1.0f + 0.125f * static_cast<float>(threadIdx.x & 7));
}

// One 16-element block: scale code from its amax and the row's global scale,
// and the factor that maps elements onto the E2M1 grid (0 when sf == 0).
// s = (amax_b / 6) * g; sf = E4M3(s); enc = min(g / sf, FLT_MAX).
// Warp-collective (one shuffle): every lane of the warp must call it. `tk` is
// the caller's table entry enc_table_entry(g); the table of this lane's row
// sits in lanes tbase .. tbase + 7.
struct BlockScale {
  uint32_t sf;
  float enc;
};
__device__ __forceinline__ BlockScale block_scale(float amax_b, float g, float tk,
                                                  int tbase = 0) {
  BlockScale r;
  const float s = __fmul_rn(div6_rn(amax_b), g);
  r.sf = cvt_e4m3(s);
  const uint32_t e = (r.sf >> 3) & 15, m = r.sf & 7;
  uint32_t idx;
  int k;
  if (e) {            // (1 + m/8) * 2^(e-7)
    idx = m;
    k = 7 - static_cast<int>(e);
  } else {            // m * 2^-9 = (1 + idx/8) * 2^(j-9)
    const int j = 31 - __clz(m | 1u);
    idx = (m << (3 - j)) & 7u;
    k = 9 - j;
  }
  const float t = __shfl_sync(0xffffffffu, tk, tbase + static_cast<int>(idx));
  float enc = __fmul_rn(t, __uint_as_float(static_cast<uint32_t>(127 + k) << 23));
  if (enc < 2.3509887016445750e-38f) enc = __fdiv_rn(g, e4m3_value(r.sf));  // below 2^-125
  r.enc = r.sf ? fminf(enc, kFltMax) : 0.0f;
  return r;
}

// 8 consecutive elements -> 4 bytes of packed codes (element 0 in the low nibble).
__device__ __forceinline__ uint32_t encode8(const float (&v)[8], float enc, bool zero) {
  if (zero) return 0u;
  uint32_t b0 = cvt_e2m1x2(__fmul_rn(v[0], enc), __fmul_rn(v[1], enc));
  uint32_t b1 = cvt_e2m1x2(__fmul_rn(v[2], enc), __fmul_rn(v[3], enc));
  uint32_t b2 = cvt_e2m1x2(__fmul_rn(v[4], enc), __fmul_rn(v[5], enc));
  uint32_t b3 = cvt_e2m1x2(__fmul_rn(v[6], enc), __fmul_rn(v[7], enc));
  return b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
}

__device__ __forceinline__ float amax8(const float (&v)[8]) {
  float m = fabsf(v[0]);
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
  return m;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& u, float (&v)[8]) {
  v[0] = bf16lo(u.x); v[1] = bf16hi(u.x); v[2] = bf16lo(u.y); v[3] = bf16hi(u.y);
  v[4] = bf16lo(u.z); v[5] = bf16hi(u.z); v[6] = bf16lo(u.w); v[7] = bf16hi(u.w);
}

// a / b for a >= 0, b > 0: the 32-bit division when both fit in 32 bits (the
// usual case; a 64-bit division is a long instruction sequence).
__device__ __forceinline__ int64_t div_nonneg(int64_t a, int64_t b) {
  if (((a | b) >> 32) == 0)
    return static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
  return a / b;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Offsets produced by the permutation must start at 0, be non-decreasing,
// end at most at `rows`, and the padded offsets must match the counts. A
// kernel that finds a violation skips all work and reports INVALID_ARG.
// Block-wide: every thread of the block must call it.
__device__ inline bool offsets_consistent(const int32_t* s_off, const int32_t* s_sfoff, int E,
                                   int64_t rows) {
  bool bad = false;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int cnt = s_off[e + 1] - s_off[e];
    if (cnt < 0 || s_sfoff[e + 1] - s_sfoff[e] != ((cnt + 127) & ~127)) bad = true;
  }
  if (threadIdx.x == 0 && (s_off[0] != 0 || s_sfoff[0] != 0 || s_off[E] > rows)) bad = true;
  return !__syncthreads_or(bad);
}

// Byte offset of the scale of (row r, SF column c) in a region with kc SF
// columns: 128-row x 4-column atoms of 512 bytes.
__device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t c, int64_t kc) {
  return ((r >> 7) * (kc >> 2) + (c >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (c & 3);
}

// ----------------------------------------------------------------------------
// Warp-level row quantizer. A row of C elements is split in chunks of 256;
// in chunk j lane l holds elements [256j + 8l, 256j + 8l + 8). Lanes 2b, 2b+1
// share one 16-element block; lanes 8a..8a+7 share one 4-column SF atom word.
// ----------------------------------------------------------------------------

// ----------------------------------------------------------------------------
// Lane-per-block quantizer core: one lane owns one whole 16-element block, so
// the block amax needs no shuffle and the block scale is computed once per
// block. A warp's 32 lanes cover 32 consecutive blocks (1 KB of BF16 input,
// 256 bytes of codes).
// ----------------------------------------------------------------------------

// 16 BF16 values from a 32-byte aligned address, streaming (read once).
__device__ __forceinline__ void ld_bf16x16(const uint16_t* p, uint32_t (&w)[8]) {
  asm("ld.global.cs.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                 "=r"(w[6]), "=r"(w[7])
               : "l"(p));
}

// Same values from a 16-byte aligned address (two 16-byte loads).
__device__ __forceinline__ void ld_bf16x16_a16(const uint16_t* p, uint32_t (&w)[8]) {
  const uint4 a = __ldcs(reinterpret_cast<const uint4*>(p));
  const uint4 b = __ldcs(reinterpret_cast<const uint4*>(p) + 1);
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

// max(|a|, |b|) per BF16 half, sign = sign(a) xor sign(b).
__device__ __forceinline__ uint32_t max_abs_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// min(|a|, |b|) per BF16 half, sign = sign(a) xor sign(b).
__device__ __forceinline__ uint32_t min_abs_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// max |x| over 16 BF16 values (exact: the result is one of the inputs).
__device__ __forceinline__ float amax_bf16x16(const uint32_t (&w)[8]) {
  const uint32_t m = max_abs_bf16x2(max_abs_bf16x2(max_abs_bf16x2(w[0], w[1]),
                                                   max_abs_bf16x2(w[2], w[3])),
                                    max_abs_bf16x2(max_abs_bf16x2(w[4], w[5]),
                                                   max_abs_bf16x2(w[6], w[7])));
  return fmaxf(__uint_as_float((m & 0x7FFFu) << 16), __uint_as_float(m & 0x7FFF0000u));
}

__device__ __forceinline__ void unpack_bf16x16(const uint32_t (&w)[8], float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16lo(w[i]);
    v[2 * i + 1] = bf16hi(w[i]);
  }
}

__device__ __forceinline__ float amax_f32x16(const float (&v)[16]) {
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1]));
  return fmaxf(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])),
               fmaxf(fmaxf(m[4], m[5]), fmaxf(m[6], m[7])));
}

// Two floats rounded to BF16 (nearest, ties to even) in one instruction: lo
// in bits 0..15, hi in bits 16..31 (each the same as __float2bfloat16_rn).
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(r) : "f"(lo), "f"(hi));
  return r;
}

// Elementwise a * b (IEEE float products) on pairs of floats.
__device__ __forceinline__ void mul_f32x2(float& a0, float& a1, float b0, float b1) {
  uint64_t p, q;
  asm("mov.b64 %0, {%1, %2};" : "=l"(p) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(q) : "f"(b0), "f"(b1));
  asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(p) : "l"(q));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a0), "=f"(a1) : "l"(p));
}

// 8 values -> 4 code bytes: E2M1(v_i * enc) with each product an IEEE float
// product (two per packed multiply); element 0 lands in the low nibble.
__device__ __forceinline__ uint32_t encode8_packed(float v0, float v1, float v2, float v3,
                                                   float v4, float v5, float v6, float v7,
                                                   float enc) {
  uint32_t out;
  asm("{\n\t"
      ".reg .b64 e2, p0, p1, p2, p3;\n\t"
      ".reg .f32 b0, b1, b2, b3, b4, b5, b6, b7;\n\t"
      ".reg .b8 c0, c1, c2, c3;\n\t"
      "mov.b64 e2, {%9, %9};\n\t"
      "mov.b64 p0, {%1, %2};\n\t"
      "mov.b64 p1, {%3, %4};\n\t"
      "mov.b64 p2, {%5, %6};\n\t"
      "mov.b64 p3, {%7, %8};\n\t"
      "mul.rn.f32x2 p0, p0, e2;\n\t"
      "mul.rn.f32x2 p1, p1, e2;\n\t"
      "mul.rn.f32x2 p2, p2, e2;\n\t"
      "mul.rn.f32x2 p3, p3, e2;\n\t"
      "mov.b64 {b0, b1}, p0;\n\t"
      "mov.b64 {b2, b3}, p1;\n\t"
      "mov.b64 {b4, b5}, p2;\n\t"
      "mov.b64 {b6, b7}, p3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c0, b1, b0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c1, b3, b2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c2, b5, b4;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c3, b7, b6;\n\t"
      "mov.b32 %0, {c0, c1, c2, c3};\n\t"
      "}"
      : "=r"(out)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7), "f"(enc));
  return out;
}

// One block of 16 values -> 8 code bytes (all zero when `zero`).
__device__ __forceinline__ uint2 encode16(const float (&v)[16], float enc, bool zero) {
  const uint32_t lo = encode8_packed(v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7], enc);
  const uint32_t hi = encode8_packed(v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15], enc);
  return zero ? make_uint2(0u, 0u) : make_uint2(lo, hi);
}

__device__ __forceinline__ void st_u64(uint8_t* p, uint2 v) {
  *reinterpret_cast<uint2*>(p) = v;
}

// One block: its scale code and 8 code bytes. Warp-collective (block_scale).
struct QBlock {
  uint2 codes;
  uint32_t sf;
};
__device__ __forceinline__ QBlock quant_block(const float (&v)[16], float am, float g, float tk,
                                              bool valid, int tbase = 0) {
  const BlockScale bs = block_scale(am, g, tk, tbase);
  QBlock r;
  r.sf = valid ? bs.sf : 0u;
  r.codes = encode16(v, bs.enc, r.sf == 0);
  return r;
}

// A row of nb <= 32*NCH blocks held by one warp, lane l owning blocks 32j + l
// as raw BF16 words. Loads return this lane's amax over its blocks.
template <int NCH, bool A32>
__device__ __forceinline__ float load_row_blocks(const uint16_t* row, int nb,
                                                 uint32_t (&w)[NCH][8], float (&am)[NCH]) {
  const int lane = threadIdx.x & 31;
  float m = 0.0f;
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int c = 32 * j + lane;
    if (c < nb) {
      if (A32) ld_bf16x16(row + 16 * c, w[j]);
      else ld_bf16x16_a16(row + 16 * c, w[j]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) w[j][i] = 0u;
    }
  }
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    am[j] = amax_bf16x16(w[j]);
    m = fmaxf(m, am[j]);
  }
  return m;
}

template <int NCH>
__device__ __forceinline__ void quant_row_blocks(const uint32_t (&w)[NCH][8],
                                                 const float (&am)[NCH], int nb, float g,
                                                 QBlock (&q)[NCH]) {
  const int lane = threadIdx.x & 31;
  const float tk = enc_table_entry(g);
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    if (32 * j < nb) {  // warp-uniform
      float v[16];
      unpack_bf16x16(w[j], v);
      q[j] = quant_block(v, am[j], g, tk, 32 * j + lane < nb);
    } else {
      q[j].codes = make_uint2(0u, 0u);
      q[j].sf = 0u;
    }
  }
}

// Codes of the row at codes_row (8 bytes per block); one scale byte per SF
// column (0 for the padding columns [nb, kc)) into the swizzled region sf_base
// at local row r.
template <int NCH>
__device__ __forceinline__ void store_row_blocks(const QBlock (&q)[NCH], int nb,
                                                 uint8_t* codes_row, uint8_t* sf_base,
                                                 int64_t r, int kc) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int c = 32 * j + lane;
    if (c < nb) st_u64(codes_row + 8 * c, q[j].codes);
    if (c < kc) sf_base[sf_offset(r, c, kc)] = static_cast<uint8_t>(q[j].sf);
  }
}

// ----------------------------------------------------------------------------
// The specified exponential: Cody-Waite reduction with a two-part ln 2 and a
// degree-7 Taylor polynomial, every step one IEEE float operation rounded to
// nearest (no contraction), inputs clamped to [-87, 88].
// ----------------------------------------------------------------------------

__device__ __forceinline__ float exp_spec(float x) {
  constexpr float kLog2e = 1.44269502162933349609375f;   // float32(log2 e)
  constexpr float kLn2Hi = 0.693145751953125f;           // ln 2 cut to 15 significant bits
  constexpr float kLn2Lo = 1.428606765330187045e-06f;    // float32(ln 2 - kLn2Hi)
  x = fminf(fmaxf(x, -87.0f), 88.0f);
  const float n = rintf(__fmul_rn(x, kLog2e));
  const float r = __fsub_rn(__fsub_rn(x, __fmul_rn(n, kLn2Hi)), __fmul_rn(n, kLn2Lo));
  float p = 1.0f / 5040.0f;
  p = __fadd_rn(__fmul_rn(p, r), 1.0f / 720.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f / 120.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f / 24.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f / 6.0f);
  p = __fadd_rn(__fmul_rn(p, r), 0.5f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  p = __fadd_rn(__fmul_rn(p, r), 1.0f);
  const int ni = static_cast<int>(n);
  return __fmul_rn(p, __uint_as_float(static_cast<uint32_t>(ni + 127) << 23));
}

// silu(g) = g / (1 + exp_spec(-g)), every step an IEEE float operation.
__device__ __forceinline__ float silu_spec(float g) {
  return __fdiv_rn(g, __fadd_rn(1.0f, exp_spec(-g)));
}

// The gates are BF16, so silu takes at most 2^16 distinct inputs: each CTA
// tabulates silu_spec in shared memory for |g| in [2^-24, 2^8) (32 binades,
// both signs, 32 KB) and evaluates the formula only for gates outside it.
// Entry index: 2 * (|g| bits - bits of 2^-24) + sign.
constexpr uint32_t kLutLo = (127u - 24u) << 7;  // BF16 bits of 2^-24
constexpr uint32_t kLutSpan = 32u << 7;          // 4096 magnitudes per sign
constexpr int kLutEntries = 2 * static_cast<int>(kLutSpan);

__device__ __forceinline__ uint32_t lut_gate_bits(int i) {
  return (static_cast<uint32_t>(i & 1) << 15) | (kLutLo + static_cast<uint32_t>(i >> 1));
}

__device__ inline void build_silu_lut_part(float* lut, int t, int nthreads) {
  for (int i = t; i < kLutEntries; i += nthreads)
    lut[i] = silu_spec(__uint_as_float(lut_gate_bits(i) << 16));
}

// A narrower table for kernels short of shared memory: |g| in [2^-16, 2^8)
// (24 binades, 24 KB), same entry order.
constexpr uint32_t kLut24Lo = (127u - 16u) << 7;
constexpr uint32_t kLut24Span = 24u << 7;
constexpr int kLut24Entries = 2 * static_cast<int>(kLut24Span);

__device__ inline void build_silu_lut24_part(float* lut, int t, int nthreads) {
  for (int i = t; i < kLut24Entries; i += nthreads)
    lut[i] = silu_spec(__uint_as_float(
        ((static_cast<uint32_t>(i & 1) << 15) | (kLut24Lo + static_cast<uint32_t>(i >> 1))) << 16));
}

// silu_spec of a gate that is a BF16 value (held as a float): the entry of the
// 24-binade table where |g| lies in [2^-16, 2^8), the formula elsewhere.
__device__ __forceinline__ float silu_bf16_lut24(const float* lut, float g) {
  const uint32_t bits = __float_as_uint(g) >> 16;
  const uint32_t off = (bits & 0x7FFFu) - kLut24Lo;
  return off < kLut24Span ? lut[2 * off + (bits >> 15)] : silu_spec(g);
}

// ----------------------------------------------------------------------------
// mbarrier / TMA / tcgen05 wrappers (inline PTX)
// ----------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}


__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
               :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// One wait attempt. The thread sleeps in the hardware until the phase
// completes or about `hint_ns` nanoseconds pass (suspend-time hint), so
// waiting warps do not spin on the barrier word that the copy engine and the
// tensor pipe update.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity,
                                              uint32_t hint_ns = 20000u) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns) : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: true when the phase with `parity` completed; false when
// `budget_ns` passed since the wait began, or *abort became non-zero first.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t budget_ns,
                                          volatile int* abort) {
  // no suspend-time hint: each attempt returns at once if the phase is not
  // complete (the grouped GEMMs measured 2-3% faster than with attempts that
  // may sleep 1 or 20 us), so a short budget also runs out on time
  if (mbar_try_wait(bar, parity, 0u)) return true;
  // the abort flag and the clock are checked after every failed attempt
  const uint64_t start = globaltimer();
  while (!mbar_try_wait(bar, parity, 0u)) {
    if (*abort) return false;
    if (globaltimer() - start > budget_ns) return false;
  }
  return true;
}

__device__ __forceinline__ void tma_prefetch_desc(const void* desc) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(desc)) : "memory");
}

// 2-D tiled TMA load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* desc, uint64_t* bar, int x,
                                            int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];"
      :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(desc)), "r"(smem_u32(bar)),
         "r"(x), "r"(y)
      : "memory");
}

// 3-D TMA load global -> shared, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* desc, uint64_t* bar, int x,
                                            int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];"
      :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(desc)), "r"(smem_u32(bar)),
         "r"(x), "r"(y), "r"(z)
      : "memory");
}

// 2-D tiled TMA store shared -> global of the box at (x, y), tracked in this
// thread's bulk async-group (commit with bulk_commit_group). x * element size
// must be a multiple of 16 bytes and x, y non-negative.
__device__ __forceinline__ void tma_store_2d(const void* desc, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
               :: "l"(reinterpret_cast<uint64_t>(desc)), "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// This thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// This thread's committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_group0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Untiled bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes),
         "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Whole warp: allocate `ncols` TMEM columns, address written to *dst (smem).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(smem_u32(dst)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
               :: "r"(taddr), "r"(ncols) : "memory");
}

// Make `bar` track completion of all prior tcgen05 async ops of this thread.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
      :: "r"(smem_u32(bar)) : "memory");
}

// D(tmem) (+)= A(smem) * B(smem)^T with NVFP4 block scales from TMEM.
__device__ __forceinline__ void tc_mma_nvfp4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                             uint32_t idesc, uint32_t sfa_tmem,
                                             uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
         "r"(accumulate)
      : "memory");
}

// Warp: load 32 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
      " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31},"
      " [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16-byte global store (address 16-byte aligned).
__device__ __forceinline__ void st_global_v4(void* ptr, uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};"
               :: "l"(ptr), "r"(a0), "r"(a1), "r"(a2), "r"(a3) : "memory");
}

// 32-byte global store (address 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void* ptr, uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t a4, uint32_t a5, uint32_t a6,
                                             uint32_t a7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               :: "l"(ptr), "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(a4), "r"(a5), "r"(a6),
                  "r"(a7)
               : "memory");
}

// Warp: store 16 / 32 consecutive 32-bit TMEM columns of this warp's 32 lanes.
__device__ __forceinline__ void tmem_st_16cols(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0],"
      " {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
         "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
         "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ----------------------------------------------------------------------------
// CTA-pair (cluster of 2) helpers
// ----------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// All threads of both CTAs of the cluster.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared::cluster address of the same shared variable in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Arrive on an mbarrier of the peer CTA with the default (release, CTA scope)
// semantics. Used after tcgen05.wait::st / wait::ld and
// tcgen05.fence::before_thread_sync to hand TMEM to the peer's MMA thread; a
// cluster-scope release costs ~1.4k cycles here (it waits for this SM's
// outstanding memory traffic), this form ~0.1k.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" :: "r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void st_shared_cluster(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" :: "r"(cluster_addr), "r"(v) : "memory");
}
// 2-D TMA load into this CTA's shared memory whose completion is counted on
// an mbarrier that may live in the peer CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const void* desc, uint32_t mbar_cluster,
                                                 int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile"
      ".mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
      :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(desc)), "r"(mbar_cluster), "r"(x),
         "r"(y)
      : "memory");
}
// One warp in each CTA of the pair, collectively.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(smem_u32(dst)), "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;"
               :: "r"(taddr), "r"(ncols) : "memory");
}
// Track the pair MMAs issued so far; arrive once on `bar` in every CTA of `mask`.
__device__ __forceinline__ void tc_commit_pair_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;"
      :: "r"(smem_u32(bar)), "h"(mask) : "memory");
}
// Pair MMA: M = 256 (128 rows from each CTA's A), N from both CTAs' B halves.
__device__ __forceinline__ void tc_mma_nvfp4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                  uint32_t idesc, uint32_t sfa_tmem,
                                                  uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      :: "r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
         "r"(accumulate)
      : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start, leading and stride
// byte offsets in 16-byte units, version 1 at bit 46, layout in bits 61..63.
enum : uint64_t { kLayoutNone = 0, kLayoutSwizzle128B = 2 };
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint64_t layout) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (layout << 61);
}

// Warp: load 8 consecutive fp32 columns at each of two TMEM addresses of this
// warp's 32 lanes, then wait; one statement, so that no use of the registers
// can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_8cols_x2(uint32_t ta, uint32_t tb, uint32_t (&a)[8],
                                                 uint32_t (&b)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%16];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8, %9, %10, %11, %12, %13, %14, %15}, [%17];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]),
        "=r"(a[7]), "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]),
        "=r"(b[6]), "=r"(b[7])
      : "r"(ta), "r"(tb)
      : "memory");
}

// One lane of the (converged) warp gets true.
__device__ __forceinline__ bool elect_one() {
  uint32_t r;
  asm volatile("{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(r));
  return r != 0;
}

// Named barrier `id` over `count` threads (whole warps).
__device__ __forceinline__ void bar_sync_named(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(count) : "memory");
}

// Device-scope stores and loads of global words (served by L2, not L1).
__device__ __forceinline__ void st_relaxed_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint4 ld_relaxed_gpu_v4(const uint32_t* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
  return v;
}
// block_scale for a thread that holds its own row: the encode factor is the
// IEEE quotient RN(g / sf) (clamped to FLT_MAX), which is what the table
// entry scaled by a power of two gives wherever that product is a normal
// float, and what block_scale computes below it.
__device__ __forceinline__ BlockScale block_scale_div(float amax_b, float g) {
  BlockScale r;
  r.sf = cvt_e4m3(__fmul_rn(div6_rn(amax_b), g));
  r.enc = r.sf ? fminf(__fdiv_rn(g, e4m3_value(r.sf)), kFltMax) : 0.0f;
  return r;
}

}  // namespace minite
