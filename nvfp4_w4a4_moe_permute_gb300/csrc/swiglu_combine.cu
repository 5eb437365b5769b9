// minite_swiglu_weighted_quant and minite_moe_combine.
//
// The weighted SwiGLU computes the activation amax inside the same pass and
// writes NVFP4 codes plus swizzled scales directly (miniTE report summary,
// section "Two complementary interventions"); the combine sums each token's
// k expert rows back into token order.
#include "common.cuh"
#include "host_util.h"

namespace minite {

// Offsets produced by the permutation must start at 0, be non-decreasing,
// end at most at `rows`, and the padded offsets must match the counts. Any
// violation makes the kernels below skip all work and report INVALID_ARG.
// Block-wide: every thread of the block must call it.
__device__ bool offsets_consistent(const int32_t* s_off, const int32_t* s_sfoff, int E,
                                   int64_t rows) {
  bool bad = false;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int cnt = s_off[e + 1] - s_off[e];
    if (cnt < 0 || s_sfoff[e + 1] - s_sfoff[e] != ((cnt + 127) & ~127)) bad = true;
  }
  if (threadIdx.x == 0 && (s_off[0] != 0 || s_sfoff[0] != 0 || s_off[E] > rows)) bad = true;
  return !__syncthreads_or(bad);
}

template <int NCH>
__global__ void __launch_bounds__(256) swiglu_quant_kernel(
    const uint16_t* __restrict__ gu, const float* __restrict__ perm_w, int64_t M, int I, int E,
    const int32_t* __restrict__ expert_offsets, const int32_t* __restrict__ sf_row_offsets,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ sf, float* __restrict__ row_g,
    int32_t* status) {
  extern __shared__ int32_t sm[];
  int32_t* s_off = sm;
  int32_t* s_sfoff = sm + (E + 1);
  for (int i = threadIdx.x; i <= E; i += blockDim.x) {
    s_off[i] = expert_offsets[i];
    s_sfoff[i] = sf_row_offsets[i];
  }
  __syncthreads();
  if (!offsets_consistent(s_off, s_sfoff, E, M)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, MINITE_ERR_INVALID_ARG);
    return;
  }

  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int kc = ((I / 16) + 3) & ~3;
  const int64_t used = s_off[E];
  for (int64_t m = warp; m < used; m += nwarps) {
    // expert of row m: the last e with s_off[e] <= m
    int lo = 0, hi = E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid] <= m) lo = mid; else hi = mid;
    }
    const int e = lo;
    const uint16_t* gr = gu + m * (2 * static_cast<int64_t>(I));
    const float w = perm_w ? perm_w[m] : 1.0f;
    float h[NCH][8];
    float am = 0.0f;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int e0 = 256 * j + 8 * lane;
      if (e0 < I) {
        const uint4 ug = __ldcs(reinterpret_cast<const uint4*>(gr + e0));
        const uint4 uu = __ldcs(reinterpret_cast<const uint4*>(gr + I + e0));
        float gv[8], uv[8];
        unpack_bf16x8(ug, gv);
        unpack_bf16x8(uu, uv);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float silu = __fdiv_rn(gv[i], __fadd_rn(1.0f, exp_spec(-gv[i])));
          float v = __fmul_rn(silu, uv[i]);
          if (perm_w) v = __fmul_rn(v, w);
          h[j][i] = v;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) h[j][i] = 0.0f;
      }
      am = fmaxf(am, amax8(h[j]));
    }
    const float g = global_scale(warp_max(am));
    RowQuant<NCH> q;
    quantize_row_warp<NCH>(h, I, g, q);
    const int64_t r = static_cast<int64_t>(s_sfoff[e]) + (m - s_off[e]);
    store_row_warp<NCH>(q, I, codes + m * (I / 2), sf, r, kc);
    if (lane == 0) row_g[m] = g;
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

// One warp per token; lane l owns columns [256c + 8l, 256c + 8l + 8) of chunk c.
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ D,
                                                      const int32_t* __restrict__ dest_row,
                                                      int64_t T, int64_t M, int N, int k,
                                                      uint16_t* __restrict__ y, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t t = warp; t < T; t += nwarps) {
    int my = lane < k ? dest_row[t * k + lane] : -1;
    if (my >= M) {
      set_status(status, MINITE_ERR_BAD_ROUTING);
      my = -1;
    }
    for (int c0 = 0; c0 < N; c0 += 256) {
      const int col = c0 + 8 * lane;
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
      for (int j0 = 0; j0 < k; j0 += 8) {
        uint4 u[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int d = __shfl_sync(0xffffffffu, my, (j0 + jj) & 31);
          u[jj] = make_uint4(0, 0, 0, 0);
          if (j0 + jj < k && d >= 0 && col < N)
            u[jj] = __ldcs(reinterpret_cast<const uint4*>(D + static_cast<int64_t>(d) * N + col));
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int d = __shfl_sync(0xffffffffu, my, (j0 + jj) & 31);
          if (j0 + jj < k && d >= 0) {
            float v[8];
            unpack_bf16x8(u[jj], v);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], v[i]);
          }
        }
      }
      if (col < N) {
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i]));
          const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * i + 1]));
          o[i] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(y + t * N + col) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
}

}  // namespace minite

using namespace minite;

extern "C" int minite_swiglu_weighted_quant(const void* gate_up, const float* perm_w, int64_t M,
                                            int64_t I, int32_t E,
                                            const int32_t* expert_offsets,
                                            const int32_t* sf_row_offsets, uint8_t* codes,
                                            uint8_t* sf, float* row_g, int32_t* status,
                                            minite_stream_t stream) {
  if (!gate_up || !expert_offsets || !sf_row_offsets || !codes || !sf || !row_g)
    return MINITE_ERR_INVALID_ARG;
  if (M < 1 || I < 64 || I % 64 != 0 || I > 2048 || E < 1 || E > 1024)
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (M >= (int64_t(1) << 31)) return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(gate_up, 16) || !aligned(codes, 16) || !aligned(sf, 16))
    return MINITE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int64_t blocks = (M + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const size_t smem = 2 * (E + 1) * sizeof(int32_t);
  const uint16_t* g = static_cast<const uint16_t*>(gate_up);
  const int i = static_cast<int>(I);
  switch ((I + 255) / 256) {
#define MINITE_CASE(N)                                                                         \
  case N:                                                                                      \
    swiglu_quant_kernel<N><<<static_cast<unsigned>(blocks), 256, smem, s>>>(                   \
        g, perm_w, M, i, E, expert_offsets, sf_row_offsets, codes, sf, row_g, status);         \
    break;
    MINITE_CASE(1) MINITE_CASE(2) MINITE_CASE(3) MINITE_CASE(4) MINITE_CASE(5) MINITE_CASE(6)
    MINITE_CASE(7) MINITE_CASE(8)
#undef MINITE_CASE
    default: return MINITE_ERR_UNSUPPORTED_SHAPE;
  }
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}

extern "C" int minite_moe_combine(const void* expert_out, const int32_t* dest_row, int64_t T,
                                  int64_t M, int64_t N, int32_t k, void* y, int32_t* status,
                                  minite_stream_t stream) {
  if (!expert_out || !dest_row || !y) return MINITE_ERR_INVALID_ARG;
  if (T < 1 || M < 1 || N < 8 || N % 8 != 0 || k < 1 || k > 32 || N >= (int64_t(1) << 30))
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(expert_out, 16) || !aligned(y, 16)) return MINITE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int64_t blocks = (T + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  combine_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      static_cast<const uint16_t*>(expert_out), dest_row, T, M, static_cast<int>(N), k,
      static_cast<uint16_t*>(y), status);
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}
