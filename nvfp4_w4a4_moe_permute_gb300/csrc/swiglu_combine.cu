// minite_swiglu_weighted_quant and minite_moe_combine.
//
// The weighted SwiGLU computes the activation amax inside the same pass and
// writes NVFP4 codes plus swizzled scales directly (miniTE report summary,
// section "Two complementary interventions"); the combine sums each token's
// k expert rows back into token order.
#include <mutex>

#include "common.cuh"
#include "host_util.h"

namespace minite {

// Byte offsets into a table of the two gates of a packed BF16 pair whose
// magnitudes both lie in [2^-24, 2^8): per 16-bit half h, t = h - bits of
// 2^-24 leaves the sign in bit 15 and the magnitude offset in bits 0..11
// (bits 12..14 clear); the offset moves to bits 3..14 and the sign to bit 2,
// i.e. 4 * (2 * offset + sign). No borrow crosses the halves since both are
// at least the subtrahend.
__device__ __forceinline__ void lut_offsets(uint32_t w, uint32_t& lo, uint32_t& hi) {
  constexpr uint32_t kMask = 0x7FF87FF8u;
  const uint32_t t = w - (kLutLo | (kLutLo << 16));
  const uint32_t r = ((t << 3) & kMask) | ((t >> 13) & ~kMask);
  lo = r & 0xFFFFu;
  hi = r >> 16;
}

__device__ __forceinline__ float lut_at(const float* lut, uint32_t byte_off) {
  return *reinterpret_cast<const float*>(reinterpret_cast<const char*>(lut) + byte_off);
}

// h = (silu(g) * u) * w for the 16 gates and ups of one block. Blocks whose
// gates all lie inside the table take one lookup per gate; any other block
// evaluates the formula for the gates outside it.
__device__ __forceinline__ void swiglu_block(const float* lut, const uint32_t (&wg)[8],
                                             const uint32_t (&wu)[8], float w, float (&h)[16]) {
  const uint32_t mx = max_abs_bf16x2(max_abs_bf16x2(max_abs_bf16x2(wg[0], wg[1]),
                                                    max_abs_bf16x2(wg[2], wg[3])),
                                     max_abs_bf16x2(max_abs_bf16x2(wg[4], wg[5]),
                                                    max_abs_bf16x2(wg[6], wg[7])));
  const uint32_t mn = min_abs_bf16x2(min_abs_bf16x2(min_abs_bf16x2(wg[0], wg[1]),
                                                    min_abs_bf16x2(wg[2], wg[3])),
                                     min_abs_bf16x2(min_abs_bf16x2(wg[4], wg[5]),
                                                    min_abs_bf16x2(wg[6], wg[7])));
  // magnitudes as BF16 bit patterns compare like unsigned integers
  const uint32_t hi_mag = max(mx & 0x7FFFu, (mx >> 16) & 0x7FFFu);
  const uint32_t lo_mag = min(mn & 0x7FFFu, (mn >> 16) & 0x7FFFu);
  if (lo_mag >= kLutLo && hi_mag < kLutLo + kLutSpan) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t a, b;
      lut_offsets(wg[i], a, b);
      h[2 * i] = lut_at(lut, a);
      h[2 * i + 1] = lut_at(lut, b);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t bits = (i & 1) ? (wg[i >> 1] >> 16) : (wg[i >> 1] & 0xFFFFu);
      const uint32_t off = (bits & 0x7FFFu) - kLutLo;
      h[i] = off < kLutSpan ? lut[2 * off + (bits >> 15)]
                            : silu_spec(__uint_as_float(bits << 16));
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    mul_f32x2(h[2 * i], h[2 * i + 1], bf16lo(wu[i]), bf16hi(wu[i]));
    mul_f32x2(h[2 * i], h[2 * i + 1], w, w);
  }
}

// Max over the LPR lanes of one row group (LPR = 32 or 16).
template <int LPR>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
  for (int o = LPR / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One warp holds 32 / LPR permuted rows at a time, LPR lanes per row; lane l
// of a row owns blocks l + LPR*j (j < NCH) of the row's intermediate, with
// the gates at [0, I) and the ups at [I, 2I) of the gate_up row. Every row's
// 4I input bytes are requested before any of them is used.
// KEEP_H: h is also stored as BF16 (round to nearest even) in h_out [M, I],
// and, when h_amax is given, each stored row's |h| maximum in h_amax [M].
constexpr int kSwThreads = 512;

__device__ __forceinline__ void st_bf16x16(uint16_t* p, const float (&v)[16]) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&b);
  }
  st_global_v8(p, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
}

template <int LPR, int NCH, bool KEEP_H>
__global__ void __launch_bounds__(kSwThreads, 1) swiglu_quant_kernel(
    const uint16_t* __restrict__ gu, const float* __restrict__ perm_w, int64_t M, int I, int E,
    const int32_t* __restrict__ expert_offsets, const int32_t* __restrict__ sf_row_offsets,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ sf, float* __restrict__ row_g,
    uint16_t* __restrict__ h_out, float* __restrict__ h_amax, int32_t* status) {
  extern __shared__ __align__(16) float smf[];
  float* lut = smf;
  int32_t* s_off = reinterpret_cast<int32_t*>(smf + kLutEntries);
  int32_t* s_sfoff = s_off + (E + 1);
  build_silu_lut_part(lut, threadIdx.x, blockDim.x);  // no global memory: overlaps the producer
  pdl_wait();
  for (int i = threadIdx.x; i <= E; i += blockDim.x) {
    s_off[i] = expert_offsets[i];
    s_sfoff[i] = sf_row_offsets[i];
  }
  __syncthreads();
  if (!offsets_consistent(s_off, s_sfoff, E, M)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, MINITE_ERR_INVALID_ARG);
    return;
  }

  constexpr int RPW = 32 / LPR;  // rows per warp
  const int lane = threadIdx.x & 31;
  const int l = lane % LPR;
  const int tbase = lane - l;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int nb = I / 16;
  const int kc = (nb + 3) & ~3;
  const int64_t used = s_off[E];
  for (int64_t base = warp * RPW; base < used; base += nwarps * RPW) {
    const int64_t m = base + lane / LPR;
    const bool live = m < used;
    const uint16_t* gr = gu + m * (2 * static_cast<int64_t>(I));
    uint32_t wg[NCH][8], wu[NCH][8];
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int c = l + LPR * j;
      if (live && c < nb) {
        ld_bf16x16(gr + 16 * c, wg[j]);
        ld_bf16x16(gr + I + 16 * c, wu[j]);
      }
    }
    const float w = live && perm_w ? perm_w[m] : 1.0f;
    float h[NCH][16], am[NCH];
    float rm = 0.0f;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      if (live && l + LPR * j < nb) {
        swiglu_block(lut, wg[j], wu[j], w, h[j]);
        if (KEEP_H) st_bf16x16(h_out + m * static_cast<int64_t>(I) + 16 * (l + LPR * j), h[j]);
      } else {
#pragma unroll
        for (int t = 0; t < 16; ++t) h[j][t] = 0.0f;
      }
      am[j] = amax_f32x16(h[j]);
      rm = fmaxf(rm, am[j]);
    }
    const float rmax = group_max<LPR>(rm);
    const float g = global_scale(rmax);
    const float tk = enc_table_entry(g);
    QBlock qb[NCH];
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      if (LPR * j < nb) {  // warp-uniform
        qb[j] = quant_block(h[j], am[j], g, tk, live && l + LPR * j < nb, tbase);
      } else {
        qb[j].codes = make_uint2(0u, 0u);
        qb[j].sf = 0u;
      }
    }
    if (live) {
      // expert of row m: the last e with s_off[e] <= m
      int lo = 0, hi = E;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_off[mid] <= m) lo = mid; else hi = mid;
      }
      const int64_t r = static_cast<int64_t>(s_sfoff[lo]) + (m - s_off[lo]);
      uint8_t* crow = codes + m * (I / 2);
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const int c = l + LPR * j;
        if (c < nb) st_u64(crow + 8 * c, qb[j].codes);
        if (c < kc) sf[sf_offset(r, c, kc)] = static_cast<uint8_t>(qb[j].sf);
      }
      if (l == 0) row_g[m] = g;
      if (KEEP_H && h_amax && l == 0) h_amax[m] = bf16_round(rmax);
    }
  }

  // zero the scale bytes of each expert's padding rows
  const int words = kc / 4;
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    const int cnt = s_off[e + 1] - s_off[e];
    const int pad = ((cnt + 127) & ~127) - cnt;
    for (int i = threadIdx.x; i < pad * words; i += blockDim.x) {
      const int64_t r = static_cast<int64_t>(s_sfoff[e]) + cnt + i / words;
      *reinterpret_cast<uint32_t*>(sf + sf_offset(r, 4 * (i % words), kc)) = 0u;
    }
  }
}

template <int LPR, int NCH>
static int launch_swiglu(const uint16_t* g, const float* perm_w, int64_t M, int I, int E,
                         const int32_t* off, const int32_t* sfoff, uint8_t* codes, uint8_t* sf,
                         float* row_g, uint16_t* h_out, float* h_amax, int32_t* status,
                         cudaStream_t s) {
  const size_t smem = kLutEntries * sizeof(float) + 2 * (E + 1) * sizeof(int32_t);
  // table (32 KB) + offsets stay under the default 48 KB of dynamic shared memory
  constexpr int rows_per_cta = kSwThreads / 32 * (32 / LPR);
  int64_t blocks = (M + rows_per_cta - 1) / rows_per_cta;
  const int64_t cap = static_cast<int64_t>(num_sms());
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 grid(static_cast<unsigned>(blocks)), block(kSwThreads);
  const cudaError_t e =
      h_out ? launch_pdl(swiglu_quant_kernel<LPR, NCH, true>, grid, block, smem, s, g, perm_w, M, I,
                         E, off, sfoff, codes, sf, row_g, h_out, h_amax, status)
            : launch_pdl(swiglu_quant_kernel<LPR, NCH, false>, grid, block, smem, s, g, perm_w, M,
                         I, E, off, sfoff, codes, sf, row_g, static_cast<uint16_t*>(nullptr),
                         static_cast<float*>(nullptr), status);
  if (e != cudaSuccess) return MINITE_ERR_CUDA;
  return MINITE_OK;
}

// ---------------------------------------------------------------------------
// SwiGLU backward: [dg | du] = d h / d [g | u] times dh, per permuted row, with
// d = 1 + exp(-g), s = 1/d, silu = g/d, silu' = s (1 + g (1 - s)),
// dg = ((dh u) w) silu', du = (dh silu) w, then per-row NVFP4 over the 2I
// values. silu and silu' of a BF16 gate come from per-CTA tables over the
// same 32 binades as the forward's (gates outside them take the formulas).
// ---------------------------------------------------------------------------

__device__ __forceinline__ void silu_dsilu_spec(float g, float& silu, float& dsilu) {
  const float d = __fadd_rn(1.0f, exp_spec(-g));
  const float sig = __fdiv_rn(1.0f, d);
  silu = __fdiv_rn(g, d);
  dsilu = __fmul_rn(sig, __fadd_rn(1.0f, __fmul_rn(g, __fsub_rn(1.0f, sig))));
}

__device__ void build_silu_bwd_luts(float* lut_s, float* lut_d, int t, int nthreads) {
  for (int i = t; i < kLutEntries; i += nthreads)
    silu_dsilu_spec(__uint_as_float(lut_gate_bits(i) << 16), lut_s[i], lut_d[i]);
}

// dg and du of one 16-element block from its gates, ups and dh (raw BF16).
__device__ __forceinline__ void swiglu_bwd_block(const float* lut_s, const float* lut_d,
                                                 const uint32_t (&wg)[8], const uint32_t (&wu)[8],
                                                 const uint32_t (&wd)[8], float w,
                                                 float (&dg)[16], float (&du)[16]) {
  const uint32_t mx = max_abs_bf16x2(max_abs_bf16x2(max_abs_bf16x2(wg[0], wg[1]),
                                                    max_abs_bf16x2(wg[2], wg[3])),
                                     max_abs_bf16x2(max_abs_bf16x2(wg[4], wg[5]),
                                                    max_abs_bf16x2(wg[6], wg[7])));
  const uint32_t mn = min_abs_bf16x2(min_abs_bf16x2(min_abs_bf16x2(wg[0], wg[1]),
                                                    min_abs_bf16x2(wg[2], wg[3])),
                                     min_abs_bf16x2(min_abs_bf16x2(wg[4], wg[5]),
                                                    min_abs_bf16x2(wg[6], wg[7])));
  const uint32_t hi_mag = max(mx & 0x7FFFu, (mx >> 16) & 0x7FFFu);
  const uint32_t lo_mag = min(mn & 0x7FFFu, (mn >> 16) & 0x7FFFu);
  float sl[16], ds[16];
  if (lo_mag >= kLutLo && hi_mag < kLutLo + kLutSpan) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t a, b;
      lut_offsets(wg[i], a, b);
      sl[2 * i] = lut_at(lut_s, a);
      ds[2 * i] = lut_at(lut_d, a);
      sl[2 * i + 1] = lut_at(lut_s, b);
      ds[2 * i + 1] = lut_at(lut_d, b);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint32_t bits = (i & 1) ? (wg[i >> 1] >> 16) : (wg[i >> 1] & 0xFFFFu);
      const uint32_t off = (bits & 0x7FFFu) - kLutLo;
      if (off < kLutSpan) {
        const uint32_t idx = 2 * off + (bits >> 15);
        sl[i] = lut_s[idx];
        ds[i] = lut_d[idx];
      } else {
        silu_dsilu_spec(__uint_as_float(bits << 16), sl[i], ds[i]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float d0 = bf16lo(wd[i]), d1 = bf16hi(wd[i]);
    float a0 = d0, a1 = d1;
    mul_f32x2(a0, a1, bf16lo(wu[i]), bf16hi(wu[i]));   // dh * u
    mul_f32x2(a0, a1, w, w);                           // * w
    mul_f32x2(a0, a1, ds[2 * i], ds[2 * i + 1]);       // * silu'
    dg[2 * i] = a0;
    dg[2 * i + 1] = a1;
    mul_f32x2(d0, d1, sl[2 * i], sl[2 * i + 1]);       // dh * silu
    mul_f32x2(d0, d1, w, w);                           // * w
    du[2 * i] = d0;
    du[2 * i + 1] = d1;
  }
}

// One warp per permuted row; lane l owns input blocks 32j + l (gates, ups and
// dh), which give output blocks 32j + l (dg) and I/16 + 32j + l (du). Rows of
// more than 64 blocks keep 2 x 16 x NCH values per lane live, so those
// variants run half as many threads per CTA to get the registers.
template <int NCH>
constexpr int bwd_threads() { return NCH <= 2 ? 512 : 256; }

// KEEP: [dg | du] is also stored as BF16 in dgu_out [M, 2I], and, when
// dgu_amax is given, each stored row's |x| maximum in dgu_amax [M].
template <int NCH, bool KEEP>
__global__ void __launch_bounds__(bwd_threads<NCH>(), 1) swiglu_bwd_quant_kernel(
    const uint16_t* __restrict__ gu, const uint16_t* __restrict__ dh,
    const float* __restrict__ perm_w, int64_t M, int I, int E,
    const int32_t* __restrict__ expert_offsets, const int32_t* __restrict__ sf_row_offsets,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ sf, float* __restrict__ row_g,
    uint16_t* __restrict__ dgu_out, float* __restrict__ dgu_amax, int32_t* status) {
  extern __shared__ __align__(16) float smf[];
  float* lut_s = smf;
  float* lut_d = smf + kLutEntries;
  int32_t* s_off = reinterpret_cast<int32_t*>(smf + 2 * kLutEntries);
  int32_t* s_sfoff = s_off + (E + 1);
  for (int i = threadIdx.x; i <= E; i += blockDim.x) {
    s_off[i] = expert_offsets[i];
    s_sfoff[i] = sf_row_offsets[i];
  }
  build_silu_bwd_luts(lut_s, lut_d, threadIdx.x, blockDim.x);
  __syncthreads();
  if (!offsets_consistent(s_off, s_sfoff, E, M)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, MINITE_ERR_INVALID_ARG);
    return;
  }
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int nb = I / 16;              // input blocks per row
  const int kc = (2 * nb + 3) & ~3;   // SF columns of the 2I-wide output
  const int64_t used = s_off[E];
  for (int64_t m = warp; m < used; m += nwarps) {
    const uint16_t* gr = gu + m * (2 * static_cast<int64_t>(I));
    const uint16_t* dr = dh + m * static_cast<int64_t>(I);
    const float w = perm_w ? perm_w[m] : 1.0f;
    float dgv[NCH][16], duv[NCH][16], amg[NCH], amu[NCH];
    float rm = 0.0f;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int c = 32 * j + lane;
      if (c < nb) {
        uint32_t wg[8], wu[8], wd[8];
        ld_bf16x16(gr + 16 * c, wg);
        ld_bf16x16(gr + I + 16 * c, wu);
        ld_bf16x16(dr + 16 * c, wd);
        swiglu_bwd_block(lut_s, lut_d, wg, wu, wd, w, dgv[j], duv[j]);
        if (KEEP) {
          uint16_t* o = dgu_out + m * (2 * static_cast<int64_t>(I)) + 16 * c;
          st_bf16x16(o, dgv[j]);
          st_bf16x16(o + I, duv[j]);
        }
      } else {
#pragma unroll
        for (int t = 0; t < 16; ++t) dgv[j][t] = duv[j][t] = 0.0f;
      }
      amg[j] = amax_f32x16(dgv[j]);
      amu[j] = amax_f32x16(duv[j]);
      rm = fmaxf(rm, fmaxf(amg[j], amu[j]));
    }
    const float rmax = warp_max(rm);
    const float g = global_scale(rmax);
    const float tk = enc_table_entry(g);
    QBlock qg[NCH], qu[NCH];
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      if (32 * j < nb) {  // warp-uniform
        const bool valid = 32 * j + lane < nb;
        qg[j] = quant_block(dgv[j], amg[j], g, tk, valid);
        qu[j] = quant_block(duv[j], amu[j], g, tk, valid);
      } else {
        qg[j].codes = qu[j].codes = make_uint2(0u, 0u);
        qg[j].sf = qu[j].sf = 0u;
      }
    }
    // expert of row m: the last e with s_off[e] <= m
    int lo = 0, hi = E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid] <= m) lo = mid; else hi = mid;
    }
    const int64_t r = static_cast<int64_t>(s_sfoff[lo]) + (m - s_off[lo]);
    uint8_t* crow = codes + m * static_cast<int64_t>(I);  // 2I codes = I bytes
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int c = 32 * j + lane;
      if (c < nb) {
        st_u64(crow + 8 * c, qg[j].codes);
        st_u64(crow + 8 * (nb + c), qu[j].codes);
        sf[sf_offset(r, c, kc)] = static_cast<uint8_t>(qg[j].sf);
        sf[sf_offset(r, nb + c, kc)] = static_cast<uint8_t>(qu[j].sf);
      }
    }
    if (lane == 0) row_g[m] = g;
    if (KEEP && dgu_amax && lane == 0) dgu_amax[m] = bf16_round(rmax);
  }

  // zero the scale bytes of each expert's padding rows
  const int words = kc / 4;
  for (int e = blockIdx.x; e < E; e += gridDim.x) {
    const int cnt = s_off[e + 1] - s_off[e];
    const int pad = ((cnt + 127) & ~127) - cnt;
    for (int i = threadIdx.x; i < pad * words; i += blockDim.x) {
      const int64_t r = static_cast<int64_t>(s_sfoff[e]) + cnt + i / words;
      *reinterpret_cast<uint32_t*>(sf + sf_offset(r, 4 * (i % words), kc)) = 0u;
    }
  }
}

template <int NCH, bool KEEP>
static cudaError_t bwd_smem_attr() {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(swiglu_bwd_quant_kernel<NCH, KEEP>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(2 * kLutEntries * sizeof(float) + 2 * 1025 * 4));
  });
  return attr;
}

template <int NCH>
static int launch_swiglu_bwd(const uint16_t* g, const uint16_t* dh, const float* perm_w,
                             int64_t M, int I, int E, const int32_t* off, const int32_t* sfoff,
                             uint8_t* codes, uint8_t* sf, float* row_g, uint16_t* dgu_out,
                             float* dgu_amax, int32_t* status, cudaStream_t s) {
  const size_t smem = 2 * kLutEntries * sizeof(float) + 2 * (E + 1) * sizeof(int32_t);
  if ((dgu_out ? bwd_smem_attr<NCH, true>() : bwd_smem_attr<NCH, false>()) != cudaSuccess)
    return MINITE_ERR_CUDA;
  constexpr int threads = bwd_threads<NCH>();
  int64_t blocks = (M + threads / 32 - 1) / (threads / 32);
  const int64_t cap = static_cast<int64_t>(num_sms());
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (dgu_out)
    swiglu_bwd_quant_kernel<NCH, true><<<static_cast<unsigned>(blocks), threads, smem, s>>>(
        g, dh, perm_w, M, I, E, off, sfoff, codes, sf, row_g, dgu_out, dgu_amax, status);
  else
    swiglu_bwd_quant_kernel<NCH, false><<<static_cast<unsigned>(blocks), threads, smem, s>>>(
        g, dh, perm_w, M, I, E, off, sfoff, codes, sf, row_g, nullptr, nullptr, status);
  return MINITE_OK;
}

// Work unit: (token t, column chunk of 512); lane l owns columns
// [512 ch + 16 l, +16). For each slot j in order the lane adds the 16 BF16
// values of row dest_row[t, j] into FP32 accumulators; up to 8 rows are in
// flight at once, and each warp requests the next unit's routing before it
// reads the current unit's rows.
template <bool A32>
__global__ void __launch_bounds__(256, 2) combine_kernel(const uint16_t* __restrict__ D,
                                                         const int32_t* __restrict__ dest_row,
                                                         int64_t T, int64_t M, int N, int k,
                                                         uint16_t* __restrict__ y,
                                                         int32_t* status) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int upt = (N + 511) / 512;
  const int64_t units = T * upt;
  int64_t u = warp;
  int nxt = -1;
  if (u < units && lane < k) nxt = dest_row[div_nonneg(u, upt) * k + lane];
  for (; u < units; u += nwarps) {
    const int64_t t = div_nonneg(u, upt);
    const int ch = static_cast<int>(u - t * upt);
    int my = nxt;
    const int64_t un = u + nwarps;
    if (un < units && lane < k) nxt = dest_row[div_nonneg(un, upt) * k + lane];
    if (my >= M) {
      set_status(status, MINITE_ERR_BAD_ROUTING);
      my = -1;
    }
    const int col = 512 * ch + 16 * lane;
    const int nv = col < N ? min(16, N - col) : 0;  // 0, 8 or 16 valid columns
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
    for (int j0 = 0; j0 < k; j0 += 8) {
      uint32_t v[8][8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int d = __shfl_sync(0xffffffffu, my, (j0 + jj) & 31);
        const uint16_t* src = D + static_cast<int64_t>(d) * N + col;
        if (j0 + jj < k && d >= 0 && nv == 16) {
          if (A32) ld_bf16x16(src, v[jj]);
          else ld_bf16x16_a16(src, v[jj]);
        } else if (j0 + jj < k && d >= 0 && nv == 8) {
          const uint4 a = __ldcs(reinterpret_cast<const uint4*>(src));
          v[jj][0] = a.x; v[jj][1] = a.y; v[jj][2] = a.z; v[jj][3] = a.w;
          v[jj][4] = v[jj][5] = v[jj][6] = v[jj][7] = 0u;
        }
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int d = __shfl_sync(0xffffffffu, my, (j0 + jj) & 31);
        if (j0 + jj < k && d >= 0 && nv > 0) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            acc[2 * i] = __fadd_rn(acc[2 * i], bf16lo(v[jj][i]));
            acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], bf16hi(v[jj][i]));
          }
        }
      }
    }
    if (nv > 0) {
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i]));
        const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i + 1]));
        o[i] = lo | (hi << 16);
      }
      uint16_t* dst = y + t * N + col;
      *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
      if (nv == 16) *reinterpret_cast<uint4*>(dst + 8) = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
}

}  // namespace minite

using namespace minite;

static int swiglu_weighted_quant_impl(const void* gate_up, const float* perm_w, int64_t M,
                                      int64_t I, int32_t E, const int32_t* expert_offsets,
                                      const int32_t* sf_row_offsets, uint8_t* codes, uint8_t* sf,
                                      float* row_g, void* h_out, float* h_amax,
                                      int32_t* status, minite_stream_t stream) {
  if (!gate_up || !expert_offsets || !sf_row_offsets || !codes || !sf || !row_g)
    return MINITE_ERR_INVALID_ARG;
  if (M < 1 || I < 64 || I % 64 != 0 || I > 2048 || E < 1 || E > 1024)
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (M >= (int64_t(1) << 31)) return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(gate_up, 32) || !aligned(codes, 16) || !aligned(sf, 16) || !aligned(h_out, 32) ||
      !aligned(h_amax, 4))
    return MINITE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint16_t* g = static_cast<const uint16_t*>(gate_up);
  uint16_t* h = static_cast<uint16_t*>(h_out);
  const int i = static_cast<int>(I);
  const int nb = i / 16;
  int rc;
  // 16 lanes per row when that leaves no lane idle or the row is short
  if (nb <= 16) rc = launch_swiglu<16, 1>(g, perm_w, M, i, E, expert_offsets, sf_row_offsets,
                                           codes, sf, row_g, h, h_amax, status, s);
  else if (nb <= 32) rc = launch_swiglu<16, 2>(g, perm_w, M, i, E, expert_offsets,
                                                sf_row_offsets, codes, sf, row_g, h, h_amax, status, s);
  else if (nb <= 48) rc = launch_swiglu<16, 3>(g, perm_w, M, i, E, expert_offsets,
                                                sf_row_offsets, codes, sf, row_g, h, h_amax, status, s);
  else if (nb <= 64) rc = launch_swiglu<32, 2>(g, perm_w, M, i, E, expert_offsets,
                                                sf_row_offsets, codes, sf, row_g, h, h_amax, status, s);
  else if (nb <= 96) rc = launch_swiglu<32, 3>(g, perm_w, M, i, E, expert_offsets,
                                                sf_row_offsets, codes, sf, row_g, h, h_amax, status, s);
  else rc = launch_swiglu<32, 4>(g, perm_w, M, i, E, expert_offsets, sf_row_offsets, codes, sf,
                                 row_g, h, h_amax, status, s);
  if (rc != MINITE_OK) return rc;
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}

extern "C" int minite_swiglu_weighted_quant(const void* gate_up, const float* perm_w, int64_t M,
                                            int64_t I, int32_t E,
                                            const int32_t* expert_offsets,
                                            const int32_t* sf_row_offsets, uint8_t* codes,
                                            uint8_t* sf, float* row_g, int32_t* status,
                                            minite_stream_t stream) {
  return swiglu_weighted_quant_impl(gate_up, perm_w, M, I, E, expert_offsets, sf_row_offsets,
                                    codes, sf, row_g, nullptr, nullptr, status, stream);
}

extern "C" int minite_swiglu_weighted_quant_keep_h(
    const void* gate_up, const float* perm_w, int64_t M, int64_t I, int32_t E,
    const int32_t* expert_offsets, const int32_t* sf_row_offsets, uint8_t* codes, uint8_t* sf,
    float* row_g, void* h_out, float* h_amax, int32_t* status, minite_stream_t stream) {
  if (!h_out) return MINITE_ERR_INVALID_ARG;
  return swiglu_weighted_quant_impl(gate_up, perm_w, M, I, E, expert_offsets, sf_row_offsets,
                                    codes, sf, row_g, h_out, h_amax, status, stream);
}

static int swiglu_backward_quant_impl(const void* gate_up, const void* dh, const float* perm_w,
                                      int64_t M, int64_t I, int32_t E,
                                      const int32_t* expert_offsets,
                                      const int32_t* sf_row_offsets, uint8_t* codes, uint8_t* sf,
                                      float* row_g, void* dgu_out, float* dgu_amax,
                                      int32_t* status, minite_stream_t stream) {
  if (!gate_up || !dh || !expert_offsets || !sf_row_offsets || !codes || !sf || !row_g)
    return MINITE_ERR_INVALID_ARG;
  if (M < 1 || I < 64 || I % 64 != 0 || I > 2048 || E < 1 || E > 1024)
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (M >= (int64_t(1) << 31)) return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(gate_up, 32) || !aligned(dh, 32) || !aligned(codes, 16) || !aligned(sf, 16) ||
      !aligned(dgu_out, 32) || !aligned(dgu_amax, 4))
    return MINITE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint16_t* g = static_cast<const uint16_t*>(gate_up);
  const uint16_t* d = static_cast<const uint16_t*>(dh);
  uint16_t* k = static_cast<uint16_t*>(dgu_out);
  const int i = static_cast<int>(I);
  const int nb = i / 16;
  int rc;
  if (nb <= 32) rc = launch_swiglu_bwd<1>(g, d, perm_w, M, i, E, expert_offsets, sf_row_offsets,
                                          codes, sf, row_g, k, dgu_amax, status, s);
  else if (nb <= 64) rc = launch_swiglu_bwd<2>(g, d, perm_w, M, i, E, expert_offsets,
                                               sf_row_offsets, codes, sf, row_g, k, dgu_amax, status, s);
  else if (nb <= 96) rc = launch_swiglu_bwd<3>(g, d, perm_w, M, i, E, expert_offsets,
                                               sf_row_offsets, codes, sf, row_g, k, dgu_amax, status, s);
  else rc = launch_swiglu_bwd<4>(g, d, perm_w, M, i, E, expert_offsets, sf_row_offsets, codes,
                                 sf, row_g, k, dgu_amax, status, s);
  if (rc != MINITE_OK) return rc;
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}

extern "C" int minite_swiglu_backward_quant(const void* gate_up, const void* dh,
                                            const float* perm_w, int64_t M, int64_t I, int32_t E,
                                            const int32_t* expert_offsets,
                                            const int32_t* sf_row_offsets, uint8_t* codes,
                                            uint8_t* sf, float* row_g, int32_t* status,
                                            minite_stream_t stream) {
  return swiglu_backward_quant_impl(gate_up, dh, perm_w, M, I, E, expert_offsets, sf_row_offsets,
                                    codes, sf, row_g, nullptr, nullptr, status, stream);
}

extern "C" int minite_swiglu_backward_quant_keep(const void* gate_up, const void* dh,
                                                 const float* perm_w, int64_t M, int64_t I,
                                                 int32_t E, const int32_t* expert_offsets,
                                                 const int32_t* sf_row_offsets, uint8_t* codes,
                                                 uint8_t* sf, float* row_g, void* dgu_out,
                                                 float* dgu_amax, int32_t* status,
                                                 minite_stream_t stream) {
  if (!dgu_out) return MINITE_ERR_INVALID_ARG;
  return swiglu_backward_quant_impl(gate_up, dh, perm_w, M, I, E, expert_offsets, sf_row_offsets,
                                    codes, sf, row_g, dgu_out, dgu_amax, status, stream);
}

extern "C" int minite_moe_combine(const void* expert_out, const int32_t* dest_row, int64_t T,
                                  int64_t M, int64_t N, int32_t k, void* y, int32_t* status,
                                  minite_stream_t stream) {
  if (!expert_out || !dest_row || !y) return MINITE_ERR_INVALID_ARG;
  if (T < 1 || M < 1 || N < 8 || N % 8 != 0 || k < 1 || k > 32 || N >= (int64_t(1) << 30))
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(expert_out, 16) || !aligned(y, 16)) return MINITE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t units = T * ((N + 511) / 512);
  int64_t blocks = (units + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 2;
  if (blocks > cap) blocks = cap;
  const uint16_t* d = static_cast<const uint16_t*>(expert_out);
  uint16_t* yy = static_cast<uint16_t*>(y);
  const int n = static_cast<int>(N);
  const dim3 grid(static_cast<unsigned>(blocks)), block(256);
  if (N % 16 == 0 && aligned(expert_out, 32))
    launch_pdl(combine_kernel<true>, grid, block, 0, s, d, dest_row, T, M, n, static_cast<int>(k),
               yy, status);
  else
    launch_pdl(combine_kernel<false>, grid, block, 0, s, d, dest_row, T, M, n, static_cast<int>(k),
               yy, status);
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}
