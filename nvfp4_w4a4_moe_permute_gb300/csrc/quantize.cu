// minite_quantize_nvfp4: NVFP4 quantization of BF16 matrices with the MMA
// scale layout written directly by the quantizer.
//
// Per-token activation scaling follows the miniTE report summary, section
// "Follow the numerical execution path"; writing the swizzled scale layout
// from the quantizer itself follows its section "Two complementary
// interventions".
//
// Kernels
//   group_amax_kernel      per-group |x| maximum (weights), atomicMax on the
//                          float bits (all values are >= 0, so integer order
//                          equals float order).
//   quantize_rows_kernel   one warp per row, blocks of 16 along the row, the
//                          row held in registers (coalesced 16-byte loads).
//   quantize_cols_kernel   blocks of 16 along the rows of a group (the
//                          transposed, dgrad-layout copy of a weight): a
//                          64 x 128 tile is staged through shared memory.
#include "common.cuh"
#include "host_util.h"

namespace minite {

__global__ void group_amax_kernel(const uint16_t* __restrict__ x, int64_t elems_per_group,
                                  uint32_t* __restrict__ amax_bits) {
  const int64_t grp = blockIdx.y;
  const uint4* base = reinterpret_cast<const uint4*>(x + grp * elems_per_group);
  const int64_t nvec = elems_per_group / 8;
  float m = 0.0f;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nvec;
       i += (int64_t)gridDim.x * blockDim.x) {
    uint4 u = __ldcs(base + i);
    float v[8];
    unpack_bf16x8(u, v);
    m = fmaxf(m, amax8(v));
  }
  m = warp_max(m);
  __shared__ float red[32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
    v = warp_max(v);
    if (threadIdx.x == 0 && v > 0.0f) atomicMax(amax_bits + grp, __float_as_uint(v));
  }
}

template <int NCH>
__global__ void __launch_bounds__(256) quantize_rows_kernel(
    const uint16_t* __restrict__ x, int64_t groups, int64_t rows, int cols, int per_group,
    const float* __restrict__ g_in, const uint32_t* __restrict__ amax_bits,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ sf, float* __restrict__ g_out) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int kc = ((cols / 16) + 3) & ~3;
  const int64_t rows_pad = (rows + 127) & ~int64_t(127);
  const int64_t sf_group_bytes = rows_pad * kc;
  const int64_t total = groups * rows;

  for (int64_t row = warp; row < total; row += nwarps) {
    const int64_t grp = row / rows;
    const int64_t r = row - grp * rows;
    const uint16_t* xr = x + row * cols;
    float v[NCH][8];
    float am = 0.0f;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int e0 = 256 * j + 8 * lane;
      if (e0 < cols) {
        uint4 u = __ldcs(reinterpret_cast<const uint4*>(xr + e0));
        unpack_bf16x8(u, v[j]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) v[j][i] = 0.0f;
      }
      am = fmaxf(am, amax8(v[j]));
    }
    float g;
    if (per_group) {
      g = g_in ? g_in[grp] : global_scale(__uint_as_float(amax_bits[grp]));
    } else {
      g = global_scale(warp_max(am));
    }
    RowQuant<NCH> q;
    quantize_row_warp<NCH>(v, cols, g, q);
    store_row_warp<NCH>(q, cols, codes + row * (cols / 2), sf + grp * sf_group_bytes, r, kc);
    if (!per_group && lane == 0) g_out[row] = g;
  }

  // zero the scale bytes of the padding rows [rows, rows_pad) of every group
  const int64_t pad_rows = rows_pad - rows;
  for (int64_t p = warp; p < groups * pad_rows; p += nwarps) {
    const int64_t grp = p / pad_rows;
    const int64_t r = rows + (p - grp * pad_rows);
    for (int a = lane; a < kc / 4; a += 32)
      *reinterpret_cast<uint32_t*>(sf + grp * sf_group_bytes + sf_offset(r, 4 * a, kc)) = 0u;
  }

  if (per_group) {
    const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (t < groups) g_out[t] = g_in ? g_in[t] : global_scale(__uint_as_float(amax_bits[t]));
  }
}

// Transposed quantization of group matrices [rows, cols]: quantized row q is
// column q of the group, blocks of 16 run along the original rows.
// Tile: 64 original rows x 128 original columns; thread t handles quantized
// row q = tile_c0 + t/2 and the 32 original rows tile_r0 + 32*(t%2) + [0,32).
constexpr int kTR = 64, kTC = 128;
__global__ void __launch_bounds__(256) quantize_cols_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t cols, const float* __restrict__ g_in,
    const uint32_t* __restrict__ amax_bits, uint8_t* __restrict__ codes, uint8_t* __restrict__ sf,
    float* __restrict__ g_out) {
  __shared__ uint16_t tile[kTR][kTC + 1];
  const int64_t grp = blockIdx.z;
  const int64_t r0 = (int64_t)blockIdx.x * kTR;
  const int64_t c0 = (int64_t)blockIdx.y * kTC;
  const uint16_t* xg = x + grp * rows * cols;
  const int t = threadIdx.x;

  // load: 16 threads per row segment of 128 columns, 16 rows per pass
#pragma unroll
  for (int pass = 0; pass < kTR / 16; ++pass) {
    const int lr = pass * 16 + t / 16;
    const int lc = (t % 16) * 8;
    const int64_t gr = r0 + lr, gc = c0 + lc;
    uint4 u = make_uint4(0, 0, 0, 0);
    if (gr < rows && gc < cols) u = __ldcs(reinterpret_cast<const uint4*>(xg + gr * cols + gc));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      tile[lr][lc + 2 * i] = static_cast<uint16_t>(w[i] & 0xFFFF);
      tile[lr][lc + 2 * i + 1] = static_cast<uint16_t>(w[i] >> 16);
    }
  }
  __syncthreads();

  const float g = g_in ? g_in[grp] : global_scale(__uint_as_float(amax_bits[grp]));
  const float tk = enc_table_entry(g);
  const int lq = t / 2, half = t % 2;
  const int64_t q = c0 + lq;               // quantized row
  const int64_t e0 = r0 + 32 * half;       // first quantized column of this thread
  const int kc = static_cast<int>(((rows / 16) + 3) & ~int64_t(3));
  const int64_t rows_pad_q = (cols + 127) & ~int64_t(127);
  uint32_t packed[4];
  uint32_t sfpair = 0;
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    float v[16];
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      v[i] = __uint_as_float(static_cast<uint32_t>(tile[32 * half + 16 * b + i][lq]) << 16);
      am = fmaxf(am, fabsf(v[i]));
    }
    const bool valid = (e0 + 16 * b) < rows;
    BlockScale bs = block_scale(am, g, tk);
    const uint32_t s = valid ? bs.sf : 0u;
    const bool zero = !valid || s == 0;
    float lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) { lo[i] = v[i]; hi[i] = v[8 + i]; }
    packed[2 * b] = encode8(lo, bs.enc, zero);
    packed[2 * b + 1] = encode8(hi, bs.enc, zero);
    sfpair |= s << (8 * b);
  }
  const uint32_t other = __shfl_down_sync(0xffffffffu, sfpair, 1);
  const size_t sf_group_bytes = static_cast<size_t>(rows_pad_q) * kc;
  if (q < cols) {
    uint8_t* crow = codes + (grp * cols + q) * (rows / 2);
    if (e0 < rows) *reinterpret_cast<uint2*>(crow + e0 / 2) = make_uint2(packed[0], packed[1]);
    if (e0 + 16 < rows)
      *reinterpret_cast<uint2*>(crow + e0 / 2 + 8) = make_uint2(packed[2], packed[3]);
  }
  const int64_t col = r0 / 16;  // SF column of this tile's first block (multiple of 4)
  if (half == 0 && q < rows_pad_q && col < kc) {
    const uint32_t word = (q < cols) ? (sfpair | (other << 16)) : 0u;
    *reinterpret_cast<uint32_t*>(sf + grp * sf_group_bytes + sf_offset(q, col, kc)) = word;
  }
  if (blockIdx.x == 0 && blockIdx.y == 0 && t == 0) g_out[grp] = g;
}

template <int NCH>
static void launch_rows(const uint16_t* x, int64_t groups, int64_t rows, int cols, int per_group,
                        const float* g_in, const uint32_t* amax, uint8_t* codes, uint8_t* sf,
                        float* g_out, cudaStream_t s) {
  const int64_t total = groups * ((rows + 127) & ~int64_t(127));
  int64_t blocks = (total + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  if (per_group && blocks * 256 < groups) blocks = (groups + 255) / 256;
  quantize_rows_kernel<NCH><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
      x, groups, rows, cols, per_group, g_in, amax, codes, sf, g_out);
}

}  // namespace minite

using namespace minite;

extern "C" int minite_quantize_nvfp4(const void* x, int64_t groups, int64_t rows, int64_t cols,
                                     int scale_mode, int orientation, const float* gscale_in,
                                     uint8_t* codes, uint8_t* sf, float* gscale_out,
                                     void* workspace, size_t ws_bytes, int32_t* status,
                                     minite_stream_t stream) {
  (void)status;
  if (!x || !codes || !sf || !gscale_out) return MINITE_ERR_INVALID_ARG;
  if (scale_mode != MINITE_SCALE_PER_ROW && scale_mode != MINITE_SCALE_PER_GROUP)
    return MINITE_ERR_INVALID_ARG;
  if (orientation != MINITE_ALONG_COLS && orientation != MINITE_ALONG_ROWS)
    return MINITE_ERR_INVALID_ARG;
  if (groups <= 0 || rows <= 0 || cols <= 0) return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 16) || !aligned(codes, 4) || !aligned(sf, 4)) return MINITE_ERR_INVALID_ARG;
  const bool per_group = scale_mode == MINITE_SCALE_PER_GROUP;
  if (gscale_in && !per_group) return MINITE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  const int64_t Cq = orientation == MINITE_ALONG_COLS ? cols : rows;
  if (Cq % 16 != 0 || cols % 8 != 0) return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (orientation == MINITE_ALONG_ROWS && !per_group) return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (orientation == MINITE_ALONG_COLS && cols > 4096) return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (groups * rows * cols >= (int64_t(1) << 40)) return MINITE_ERR_UNSUPPORTED_SHAPE;

  uint32_t* amax = nullptr;
  if (per_group && !gscale_in) {
    if (!workspace || ws_bytes < minite_workspace_bytes(MINITE_OP_QUANTIZE, groups, 0, 0, 0))
      return MINITE_ERR_INVALID_ARG;
    amax = static_cast<uint32_t*>(workspace);
    if (cudaMemsetAsync(amax, 0, groups * sizeof(uint32_t), s) != cudaSuccess)
      return MINITE_ERR_CUDA;
    const int64_t per = rows * cols;
    int64_t bx = (per / 8 + 255) / 256;
    const int64_t want = (num_sms() * 8 + groups - 1) / groups;
    if (bx > want) bx = want;
    if (bx < 1) bx = 1;
    dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(groups));
    group_amax_kernel<<<grid, 256, 0, s>>>(xb, per, amax);
  }

  if (orientation == MINITE_ALONG_COLS) {
    const int nch = static_cast<int>((cols + 255) / 256);
    const int c = static_cast<int>(cols);
    const int pg = per_group ? 1 : 0;
    switch (nch) {
#define MINITE_CASE(N) \
  case N: launch_rows<N>(xb, groups, rows, c, pg, gscale_in, amax, codes, sf, gscale_out, s); break;
      MINITE_CASE(1) MINITE_CASE(2) MINITE_CASE(3) MINITE_CASE(4) MINITE_CASE(5) MINITE_CASE(6)
      MINITE_CASE(7) MINITE_CASE(8) MINITE_CASE(9) MINITE_CASE(10) MINITE_CASE(11)
      MINITE_CASE(12) MINITE_CASE(13) MINITE_CASE(14) MINITE_CASE(15) MINITE_CASE(16)
#undef MINITE_CASE
      default: return MINITE_ERR_UNSUPPORTED_SHAPE;
    }
  } else {
    dim3 grid(static_cast<unsigned>((rows + kTR - 1) / kTR),
              static_cast<unsigned>((cols + kTC - 1) / kTC), static_cast<unsigned>(groups));
    quantize_cols_kernel<<<grid, 256, 0, s>>>(xb, rows, cols, gscale_in, amax, codes, sf,
                                              gscale_out);
  }
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}
