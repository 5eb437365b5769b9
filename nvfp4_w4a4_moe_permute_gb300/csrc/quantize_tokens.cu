// minite_quantize_tokens_nvfp4: one operand of a weight-gradient GEMM,
// quantized along tokens.
//
// The weight gradient of an expert sums over the expert's tokens, so its
// operands are the expert's permuted rows transposed ([channels, tokens]) and
// quantized in blocks of 16 consecutive tokens, with one global scale per
// expert (the scale may not vary along the summed axis). The pages run the
// backward in BF16 (miniTE report summary, "Respect the timing boundaries");
// this NVFP4 operand is a reading that keeps their layout choices: contiguous
// expert buffers, device-side offsets and the MMA scale layout written by the
// quantizer ("Two complementary interventions").
//
// Layout: expert e's tokens occupy columns [kofs[e], kofs[e] + count_e) of a
// [C, K_cap] code matrix (row pitch K_cap / 2 bytes), kofs being the prefix
// of the counts rounded up to 256 tokens (one 128-byte chunk of codes);
// columns up to kofs[e + 1] past the count hold code 0 and scale 0.
//
// Kernels
//   tokens_amax_kernel   per-expert |x| maximum: each CTA reduces a contiguous
//                        range of permuted rows (rows are expert-contiguous,
//                        so a range spans few experts) and issues one atomic
//                        per expert it touched.
//   token_rowmax_kernel, tokens_amax_gathered_kernel
//                        the same maximum when rows are gathered: each source
//                        row's maximum once, then the experts' maxima over
//                        their rows' sources (a token routed to k experts is
//                        read once instead of k times). With caller-given
//                        row maxima (the SwiGLU entries that keep their BF16
//                        output write them) only the second kernel runs, and
//                        the operand is read once, by the encoding.
//   tokens_quant_kernel  64-token x 256-channel tiles of one expert, gathered
//                        row by row into shared memory with per-thread
//                        asynchronous copies (two buffers). Each tile's
//                        position is decoded once and its source rows are
//                        looked up one tile ahead of its copies; thread c
//                        quantizes channel c's four 16-token blocks and
//                        writes 32 code bytes and 4 scale bytes, all
//                        contiguous.
#include <mutex>

#include "common.cuh"
#include "host_util.h"

namespace minite {

namespace {

constexpr int kTokT = 64;                   // tokens per tile
constexpr int kTokC = 256;                  // channels per tile (one per thread)
constexpr int kTokPitch = kTokC + 8;        // BF16 per staged row, 16-byte aligned rows
constexpr int kTokThreads = 256;
constexpr int kTokCtasPerSm = 3;           // resident CTAs per SM (shared memory)
constexpr int kTokAlign = 256;              // tokens: K alignment of each expert
constexpr int kAmaxRows = 64;               // permuted rows per CTA of the amax pass

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
               :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(valid ? 16 : 0)
               : "memory");
}

// Expert offsets must start at 0, not decrease and end at most at `rows`.
// Block-wide: every thread of the block must call it.
__device__ bool token_offsets_ok(const int32_t* s_off, int E, int64_t rows) {
  bool bad = false;
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    if (s_off[e + 1] < s_off[e]) bad = true;
  if (threadIdx.x == 0 && (s_off[0] != 0 || s_off[E] > rows)) bad = true;
  return !__syncthreads_or(bad);
}

// The expert of permuted row m: the last e with s_off[e] <= m.
__device__ __forceinline__ int expert_of(const int32_t* s_off, int E, int64_t m) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_off[mid] <= m) lo = mid; else hi = mid;
  }
  return lo;
}

// x: BF16 [x_rows, C]; permuted row m is x[row_src[m]] (or x[m] without
// row_src); at most m_cap permuted rows.
__global__ void __launch_bounds__(kTokThreads) tokens_amax_kernel(
    const uint16_t* __restrict__ x, int64_t x_rows, const int32_t* __restrict__ row_src,
    int64_t m_cap, int C, int E, const int32_t* __restrict__ expert_offsets,
    uint32_t* __restrict__ amax_bits, int32_t* status) {
  extern __shared__ int32_t s_off[];  // [E+1]
  for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = expert_offsets[i];
  __syncthreads();
  const int64_t src_rows = x_rows;
  if (!token_offsets_ok(s_off, E, m_cap)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, MINITE_ERR_INVALID_ARG);
    return;
  }
  const int64_t used = s_off[E];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = C / 8;
  for (int64_t r0 = static_cast<int64_t>(blockIdx.x) * kAmaxRows; r0 < used;
       r0 += static_cast<int64_t>(gridDim.x) * kAmaxRows) {
    const int64_t r1 = r0 + kAmaxRows < used ? r0 + kAmaxRows : used;
    // one warp per row; a warp keeps a running maximum while its rows stay in
    // one expert and flushes it with one atomic when the expert changes
    int cur = -1;
    float m = 0.0f;
    for (int64_t r = r0 + warp; r < r1; r += kTokThreads / 32) {
      const int e = expert_of(s_off, E, r);
      if (e != cur) {
        const float v = warp_max(m);
        if (cur >= 0 && lane == 0 && v > 0.0f) atomicMax(amax_bits + cur, __float_as_uint(v));
        cur = e;
        m = 0.0f;
      }
      int64_t src = r;
      if (row_src) {
        src = row_src[r];
        if (src < 0 || src >= src_rows) {  // warp-uniform
          if (lane == 0) set_status(status, MINITE_ERR_INVALID_ARG);
          continue;
        }
      }
      const uint4* row = reinterpret_cast<const uint4*>(x + src * C);
      for (int i = lane; i < nvec; i += 32) {
        float v[8];
        unpack_bf16x8(__ldg(row + i), v);
        m = fmaxf(m, amax8(v));
      }
    }
    const float v = warp_max(m);
    if (cur >= 0 && lane == 0 && v > 0.0f) atomicMax(amax_bits + cur, __float_as_uint(v));
  }
}

// |x| maximum of each source row, one warp per row.
__global__ void __launch_bounds__(kTokThreads) token_rowmax_kernel(
    const uint16_t* __restrict__ x, int64_t x_rows, int C, float* __restrict__ rowmax) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int nvec = C / 8;
  for (int64_t r = warp; r < x_rows; r += nwarps) {
    const uint4* row = reinterpret_cast<const uint4*>(x + r * C);
    uint32_t m = 0;  // packed |x| maximum of two BF16 halves
    for (int i = lane; i < nvec; i += 32) {
      const uint4 u = __ldg(row + i);
      m = max_abs_bf16x2(m, max_abs_bf16x2(max_abs_bf16x2(u.x, u.y), max_abs_bf16x2(u.z, u.w)));
    }
    float v = fmaxf(bf16lo(m & 0x7FFF7FFFu), bf16hi(m & 0x7FFF7FFFu));
    v = warp_max(v);
    if (lane == 0) rowmax[r] = v;
  }
}

// Per-expert maxima over the permuted rows' source-row maxima (row m's
// source is row_src[m], or m itself without row_src). A warp takes 32
// consecutive permuted rows; when they share an expert (the usual case, rows
// being expert-contiguous) it issues one atomic.
__global__ void __launch_bounds__(kTokThreads) tokens_amax_gathered_kernel(
    const float* __restrict__ rowmax, int64_t x_rows, const int32_t* __restrict__ row_src,
    int64_t m_cap, int E, const int32_t* __restrict__ expert_offsets,
    uint32_t* __restrict__ amax_bits, int32_t* status) {
  extern __shared__ int32_t s_off[];  // [E+1]
  pdl_wait();
  for (int i = threadIdx.x; i <= E; i += blockDim.x) s_off[i] = expert_offsets[i];
  __syncthreads();
  if (!token_offsets_ok(s_off, E, m_cap)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, MINITE_ERR_INVALID_ARG);
    return;
  }
  const int64_t used = s_off[E];
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t base = warp * 32; base < used; base += nwarps * 32) {
    const int64_t m = base + lane;
    float v = 0.0f;
    int e = -1;
    if (m < used) {
      e = expert_of(s_off, E, m);
      const int64_t src = row_src ? row_src[m] : m;
      if (src >= 0 && src < x_rows) v = rowmax[src];
      else set_status(status, MINITE_ERR_INVALID_ARG);
    }
    const int e0 = __shfl_sync(0xffffffffu, e, 0);
    if (__all_sync(0xffffffffu, e == e0 || e < 0)) {
      v = warp_max(v);
      if (lane == 0 && e0 >= 0 && v > 0.0f) atomicMax(amax_bits + e0, __float_as_uint(v));
    } else if (e >= 0 && v > 0.0f) {
      atomicMax(amax_bits + e, __float_as_uint(v));
    }
  }
}

// Per CTA: kofs (prefix of counts rounded up to kTokAlign) and the unit
// prefix (token tiles x channel tiles per expert) in shared memory, by warp 0.
__device__ void token_layout(const int32_t* s_off, int E, int nct, int64_t* s_kofs,
                             int64_t* s_upre) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int64_t kc = 0;
    if (lane == 0) { s_kofs[0] = 0; s_upre[0] = 0; }
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int64_t kp = 0;
      if (e < E) {
        const int64_t cnt = s_off[e + 1] - s_off[e];
        kp = (cnt + kTokAlign - 1) / kTokAlign * kTokAlign;
      }
      int64_t incl = kp;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (e < E) {
        s_kofs[e + 1] = kc + incl;
        s_upre[e + 1] = (kc + incl) / kTokT * nct;  // units of experts 0..e
      }
      kc += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kTokThreads) tokens_quant_kernel(
    const uint16_t* __restrict__ x, int64_t x_rows, const int32_t* __restrict__ row_src,
    int64_t m_cap, int C, int E, const int32_t* __restrict__ expert_offsets,
    const uint32_t* __restrict__ amax_bits, int64_t k_cap, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ sf, float* __restrict__ g_out, int32_t* __restrict__ kofs_out,
    int32_t* status) {
  extern __shared__ __align__(16) unsigned char smem_tok[];
  uint16_t* tiles = reinterpret_cast<uint16_t*>(smem_tok);  // [2][kTokT * kTokPitch]
  int64_t* s_kofs = reinterpret_cast<int64_t*>(tiles + 2 * kTokT * kTokPitch);  // [E+1]
  int64_t* s_upre = s_kofs + (E + 1);                                          // [E+1]
  int32_t* s_off = reinterpret_cast<int32_t*>(s_upre + (E + 1));               // [E+1]
  const int t = threadIdx.x;
  for (int i = t; i <= E; i += blockDim.x) s_off[i] = expert_offsets[i];
  __syncthreads();
  if (!token_offsets_ok(s_off, E, m_cap)) {
    if (blockIdx.x == 0 && t == 0) set_status(status, MINITE_ERR_INVALID_ARG);
    return;
  }
  const int nct = (C + kTokC - 1) / kTokC;
  token_layout(s_off, E, nct, s_kofs, s_upre);
  if (s_kofs[E] > k_cap) {  // block-uniform
    if (blockIdx.x == 0 && t == 0) set_status(status, MINITE_ERR_INVALID_ARG);
    return;
  }
  if (blockIdx.x == 0) {
    for (int e = t; e < E; e += blockDim.x) {
      g_out[e] = global_scale(__uint_as_float(amax_bits[e]));
      kofs_out[e] = static_cast<int32_t>(s_kofs[e]);
    }
    if (t == 0) kofs_out[E] = static_cast<int32_t>(s_kofs[E]);
  }
  const int64_t kc = k_cap / 16;        // scale columns
  const int64_t pitch = k_cap / 2;      // code bytes per channel row
  const int64_t units = s_upre[E];

  // unit u -> (expert, token tile, channel tile); expert -1 past the last unit
  struct Unit {
    int e, tt, ct;
  };
  auto unit_pos = [&](int64_t u) {
    Unit d{-1, 0, 0};
    if (u < units) {
      int lo = 0, hi = E;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_upre[mid] <= u) lo = mid; else hi = mid;
      }
      const int64_t rem = u - s_upre[lo];
      d.e = lo;
      d.tt = static_cast<int>(div_nonneg(rem, nct));
      d.ct = static_cast<int>(rem - static_cast<int64_t>(d.tt) * nct);
    }
    return d;
  };
  // This thread's 8 rows of a unit (rows warp + 8 i, 16-byte piece lane):
  // their source rows, looked up one tile ahead of the copies.
  auto srcs_of = [&](const Unit& d, int32_t (&sr)[8], uint32_t& vmask) {
    vmask = 0;
    if (d.e >= 0) {
      const int cnt = s_off[d.e + 1] - s_off[d.e];
      const bool cval = d.ct * kTokC + 8 * (t & 31) < C;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int tok = d.tt * kTokT + (t >> 5) + 8 * i;
        sr[i] = s_off[d.e] + tok;
        if (cval && tok < cnt) {
          vmask |= 1u << i;
          if (row_src) sr[i] = row_src[sr[i]];
        }
      }
    }
  };
  auto issue = [&](const Unit& d, const int32_t (&sr)[8], uint32_t vmask, uint16_t* buf) {
    if (d.e >= 0) {
      const uint16_t* xs = x + d.ct * kTokC + 8 * (t & 31);
      uint16_t* bs = buf + (t >> 5) * kTokPitch + 8 * (t & 31);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        bool valid = (vmask >> i) & 1u;
        const int64_t src = sr[i];
        if (valid && (src < 0 || src >= x_rows)) {
          set_status(status, MINITE_ERR_INVALID_ARG);
          valid = false;
        }
        cp_async16(bs + 8 * i * kTokPitch, valid ? xs + src * C : x, valid);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  const int64_t G = gridDim.x;
  int64_t u = blockIdx.x;
  Unit d0 = unit_pos(u), d1 = unit_pos(u + G);
  int32_t sr[8];  // source rows of the next tile to copy (valid where vm has the bit)
  uint32_t vm;
  srcs_of(d0, sr, vm);
  issue(d0, sr, vm, tiles);
  srcs_of(d1, sr, vm);
  int cur = 0;
  int ecur = -1;
  float g = 1.0f, tk = 1.0f;
  for (; u < units; u += G, cur ^= 1) {
    issue(d1, sr, vm, tiles + (cur ^ 1) * kTokT * kTokPitch);
    const Unit d2 = unit_pos(u + 2 * G);
    srcs_of(d2, sr, vm);
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncthreads();
    const int e = d0.e, tt = d0.tt;
    if (e != ecur) {  // block-uniform
      ecur = e;
      g = global_scale(__uint_as_float(amax_bits[e]));
      tk = enc_table_entry(g);
    }
    const uint16_t* tile = tiles + cur * kTokT * kTokPitch;
    const int c = d0.ct * kTokC + t;
    const bool valid = c < C;
    uint2 code[4];
    uint32_t sfw = 0;
#pragma unroll
    for (int rb = 0; rb < 4; ++rb) {
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        v[j] = __uint_as_float(static_cast<uint32_t>(tile[(16 * rb + j) * kTokPitch + t]) << 16);
      const QBlock q = quant_block(v, amax_f32x16(v), g, tk, valid);
      code[rb] = q.codes;
      sfw |= q.sf << (8 * rb);
    }
    if (valid) {
      const int64_t k0 = s_kofs[e] + static_cast<int64_t>(tt) * kTokT;  // first token column
      uint8_t* dst = codes + c * pitch + k0 / 2;
      st_global_v8(dst, code[0].x, code[0].y, code[1].x, code[1].y, code[2].x, code[2].y,
                   code[3].x, code[3].y);
      *reinterpret_cast<uint32_t*>(sf + sf_offset(c, k0 / 16, kc)) = sfw;
    }
    __syncthreads();  // the next iteration refills this buffer
    d0 = d1;
    d1 = d2;
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");

  // scale bytes of the padding channel rows [C, roundup(C, 128)), up to kofs[E]
  const int64_t pad_rows = ((C + 127) & ~127) - C;
  const int64_t words = s_kofs[E] / 64;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + t; i < pad_rows * words;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    *reinterpret_cast<uint32_t*>(sf + sf_offset(C + i / words, 4 * (i % words), kc)) = 0u;
}

}  // namespace
}  // namespace minite

using namespace minite;

namespace minite {
// Per-expert maxima, then (for gathered rows) one maximum per source row.
size_t tokens_workspace_bytes(int32_t E, int64_t x_rows) {
  const size_t a = (static_cast<size_t>(E) * sizeof(uint32_t) + 255) & ~size_t(255);
  return a + (x_rows > 0 ? static_cast<size_t>(x_rows) * sizeof(float) : 0);
}
}  // namespace minite

extern "C" int minite_quantize_tokens_nvfp4(const void* x, int64_t x_rows, const int32_t* row_src,
                                            const float* row_amax, int64_t m_cap, int64_t C, int32_t E,
                                            const int32_t* expert_offsets, int64_t k_cap,
                                            uint8_t* codes, uint8_t* sf, float* g_out,
                                            int32_t* kofs_out, void* workspace, size_t ws_bytes,
                                            int32_t* status, minite_stream_t stream) {
  if (!x || !expert_offsets || !codes || !sf || !g_out || !kofs_out || !workspace)
    return MINITE_ERR_INVALID_ARG;
  if (x_rows < 1 || m_cap < 1 || C < 16 || C % 16 != 0 || C > 65536 || E < 1 || E > 1024)
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (!row_src && m_cap > x_rows) return MINITE_ERR_INVALID_ARG;
  if (k_cap < kTokAlign || k_cap % kTokAlign != 0 || x_rows >= (int64_t(1) << 31) ||
      m_cap >= (int64_t(1) << 31) || C * (k_cap / 2) >= (int64_t(1) << 40))
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 16) || !aligned(codes, 32) || !aligned(sf, 4) || !aligned(workspace, 4) ||
      !aligned(row_amax, 4))
    return MINITE_ERR_INVALID_ARG;
  if (ws_bytes < tokens_workspace_bytes(E, row_src && !row_amax ? x_rows : 0))
    return MINITE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  uint32_t* amax = static_cast<uint32_t*>(workspace);
  if (cudaMemsetAsync(amax, 0, E * sizeof(uint32_t), s) != cudaSuccess) return MINITE_ERR_CUDA;
  const int c = static_cast<int>(C);
  int64_t ablocks = (m_cap + kAmaxRows - 1) / kAmaxRows;
  const int64_t acap = static_cast<int64_t>(num_sms()) * 8;
  if (ablocks > acap) ablocks = acap;
  if (row_src || row_amax) {
    const float* rowmax = row_amax;
    if (!rowmax) {  // each source row's maximum once
      float* rm = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                           tokens_workspace_bytes(E, 0));
      int64_t rblocks = (x_rows + kTokThreads / 32 - 1) / (kTokThreads / 32);
      if (rblocks > acap) rblocks = acap;
      token_rowmax_kernel<<<static_cast<unsigned>(rblocks), kTokThreads, 0, s>>>(xb, x_rows, c,
                                                                                rm);
      rowmax = rm;
    }
    int64_t gblocks = (m_cap + kTokThreads - 1) / kTokThreads;
    if (gblocks > acap) gblocks = acap;
    tokens_amax_gathered_kernel<<<static_cast<unsigned>(gblocks), kTokThreads,
                                  (E + 1) * sizeof(int32_t), s>>>(
        rowmax, x_rows, row_src, m_cap, E, expert_offsets, amax, status);
  } else {
    tokens_amax_kernel<<<static_cast<unsigned>(ablocks), kTokThreads, (E + 1) * sizeof(int32_t),
                         s>>>(xb, x_rows, row_src, m_cap, c, E, expert_offsets, amax, status);
  }
  const size_t smem = 2 * kTokT * kTokPitch * sizeof(uint16_t) +
                      2 * (E + 1) * sizeof(int64_t) + (E + 1) * sizeof(int32_t);
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(tokens_quant_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(2 * kTokT * kTokPitch * sizeof(uint16_t) +
                                                 2 * 1025 * sizeof(int64_t) + 1025 * 4));
  });
  if (attr != cudaSuccess) return MINITE_ERR_CUDA;
  const int64_t qblocks = static_cast<int64_t>(num_sms()) * kTokCtasPerSm;
  tokens_quant_kernel<<<static_cast<unsigned>(qblocks), kTokThreads, smem, s>>>(
      xb, x_rows, row_src, m_cap, c, E, expert_offsets, amax, k_cap, codes, sf, g_out, kofs_out,
      status);
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}
