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
//   quantize_token_rows_kernel
//                          one warp per row, blocks of 16 along the row, the
//                          row held in registers between its maximum and its
//                          encoding: per-row scales (activations) or the
//                          group's scale (weights along K).
//   quantize_group_blocks_kernel
//                          the group-scaled form for rows longer than 2048: a
//                          flat stream of 32-block chunks per warp.
//   quantize_tiles_kernel  blocks of 16 along the rows of a group (the
//                          transposed, dgrad-layout copy of a weight), and
//                          optionally the forward copy from the same read:
//                          128 x 128 tiles staged through shared memory with
//                          per-thread asynchronous copies (two buffers).
#include <mutex>

#include "common.cuh"
#include "host_util.h"

namespace minite {

// Each thread keeps kAmaxU 32-byte loads in flight and takes maxima on packed
// BF16 pairs (|x| compares like the unsigned magnitude bits).
constexpr int kAmaxU = 4;
__global__ void __launch_bounds__(256) group_amax_kernel(const uint16_t* __restrict__ x,
                                                         int64_t elems_per_group,
                                                         uint32_t* __restrict__ amax_bits) {
  pdl_wait();
  const int64_t grp = blockIdx.y;
  const uint16_t* base = x + grp * elems_per_group;
  const int64_t nvec = elems_per_group / 16;                    // 32-byte vectors
  const bool a32 = (reinterpret_cast<uintptr_t>(base) & 31) == 0;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  float m = 0.0f;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < nvec;
       i += kAmaxU * stride) {
    uint32_t w[kAmaxU][8];
#pragma unroll
    for (int u = 0; u < kAmaxU; ++u) {
      const int64_t v = i + u * stride;
      if (v < nvec) {
        if (a32) ld_bf16x16(base + 16 * v, w[u]);
        else ld_bf16x16_a16(base + 16 * v, w[u]);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) w[u][j] = 0u;
      }
    }
#pragma unroll
    for (int u = 0; u < kAmaxU; ++u) m = fmaxf(m, amax_bf16x16(w[u]));
  }
  // the tail of a group whose size is not a multiple of 16 elements
  for (int64_t e = nvec * 16 + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
       e < elems_per_group; e += stride)
    m = fmaxf(m, fabsf(bf16lo(base[e])));
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

// Per-group quantization along columns as one flat stream of blocks: the
// blocks of group grp are numbered row-major, b = r * nb + c, and cut into
// chunks of 32 (one per lane). Warp w owns a contiguous range of chunks and
// keeps kU of them in flight; the group's g and encode table are refreshed
// only when the group changes.
constexpr int kU = 2;
template <bool A32>
__global__ void __launch_bounds__(256, 4) quantize_group_blocks_kernel(
    const uint16_t* __restrict__ x, int64_t groups, int64_t rows, int nb, uint32_t nb_magic,
    const float* __restrict__ g_in, const uint32_t* __restrict__ amax_bits,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ sf, float* __restrict__ g_out) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int kc = (nb + 3) & ~3;
  const int64_t rows_pad = (rows + 127) & ~int64_t(127);
  const int64_t sf_group_bytes = rows_pad * kc;
  const uint32_t bpg = static_cast<uint32_t>(rows * nb);  // blocks per group (< 2^32)
  const int64_t cpg = (bpg + 31) / 32;
  const int64_t total = groups * cpg;
  const int64_t per = (total + nwarps - 1) / nwarps;
  int64_t q = warp * per;
  const int64_t q_end = q + per < total ? q + per : total;
  int64_t grp = q / cpg;
  int64_t qin = q - grp * cpg;
  int64_t cur = -1;
  float g = 1.0f, tk = 1.0f;
  while (q < q_end) {
    uint32_t w[kU][8];
    int64_t gq[kU];
    uint32_t bq[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      gq[u] = grp;
      bq[u] = static_cast<uint32_t>(qin) * 32u + lane;
      if (q + u < q_end && bq[u] < bpg) {
        const uint16_t* src = x + (grp * bpg + bq[u]) * 16;
        if (A32) ld_bf16x16(src, w[u]);
        else ld_bf16x16_a16(src, w[u]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[u][i] = 0u;
      }
      if (++qin == cpg) { qin = 0; ++grp; }
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (q + u >= q_end) break;  // warp-uniform
      if (gq[u] != cur) {         // warp-uniform
        cur = gq[u];
        g = g_in ? g_in[cur] : global_scale(__uint_as_float(amax_bits[cur]));
        tk = enc_table_entry(g);
      }
      const bool valid = bq[u] < bpg;
      float v[16];
      unpack_bf16x16(w[u], v);
      const QBlock qb = quant_block(v, amax_bf16x16(w[u]), g, tk, valid);
      if (valid) {
        // r = bq / nb: nb_magic = floor(2^32 / nb) undershoots by at most one
        uint32_t r = __umulhi(bq[u], nb_magic);
        uint32_t c = bq[u] - r * static_cast<uint32_t>(nb);
        if (c >= static_cast<uint32_t>(nb)) { c -= nb; ++r; }
        st_u64(codes + (gq[u] * bpg + bq[u]) * 8, qb.codes);
        sf[gq[u] * sf_group_bytes + sf_offset(r, c, kc)] = static_cast<uint8_t>(qb.sf);
        if (c + 1 == static_cast<uint32_t>(nb)) {  // last block of the row: pad columns
          for (int cc = nb; cc < kc; ++cc) sf[gq[u] * sf_group_bytes + sf_offset(r, cc, kc)] = 0;
        }
      }
    }
    q += kU;
  }

  // zero the scale bytes of the padding rows [rows, rows_pad) of every group
  const int64_t pad_rows = rows_pad - rows;
  for (int64_t p = warp; p < groups * pad_rows; p += nwarps) {
    const int64_t gp = p / pad_rows;
    const int64_t r = rows + (p - gp * pad_rows);
    for (int a = lane; a < kc / 4; a += 32)
      *reinterpret_cast<uint32_t*>(sf + gp * sf_group_bytes + sf_offset(r, 4 * a, kc)) = 0u;
  }
  const int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (t < groups) g_out[t] = g_in ? g_in[t] : global_scale(__uint_as_float(amax_bits[t]));
}

// Quantization along columns, one warp per row, lane l owning blocks 32j + l,
// the row held in registers between its amax and its encoding. Per-row
// (activation) scales, or with PG the group's scale (g_in[grp], else from
// the group maximum in amax_bits).
template <int NCH, bool A32, bool PG>
__global__ void __launch_bounds__(256) quantize_token_rows_kernel(
    const uint16_t* __restrict__ x, int64_t groups, int64_t rows, int cols,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ sf, float* __restrict__ g_out,
    const float* __restrict__ g_in, const uint32_t* __restrict__ amax_bits) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int nb = cols / 16;
  const int kc = (nb + 3) & ~3;
  const int64_t rows_pad = (rows + 127) & ~int64_t(127);
  const int64_t sf_group_bytes = rows_pad * kc;
  const int64_t total = groups * rows;
  for (int64_t i = warp; i < total; i += nwarps) {
    // per-group scales follow the group-maxima pass, which reads the groups in
    // order: taking the rows last to first starts where that pass ended, on
    // bytes still in L2
    const int64_t row = PG ? total - 1 - i : i;
    const int64_t grp = div_nonneg(row, rows);
    const int64_t r = row - grp * rows;
    uint32_t w[NCH][8];
    float am[NCH];
    const float m = load_row_blocks<NCH, A32>(x + row * cols, nb, w, am);
    float g;
    if (PG) g = g_in ? g_in[grp] : global_scale(__uint_as_float(amax_bits[grp]));
    else g = global_scale(warp_max(m));
    QBlock qb[NCH];
    quant_row_blocks<NCH>(w, am, nb, g, qb);
    store_row_blocks<NCH>(qb, nb, codes + row * (cols / 2), sf + grp * sf_group_bytes, r, kc);
    if (lane == 0 && (!PG || r == 0)) g_out[PG ? grp : row] = g;
  }
  const int64_t pad_rows = rows_pad - rows;
  for (int64_t p = warp; p < groups * pad_rows; p += nwarps) {
    const int64_t gp = p / pad_rows;
    const int64_t r = rows + (p - gp * pad_rows);
    for (int a = lane; a < kc / 4; a += 32)
      *reinterpret_cast<uint32_t*>(sf + gp * sf_group_bytes + sf_offset(r, 4 * a, kc)) = 0u;
  }
}

// Per-group quantization of weights [rows, cols] in the transposed (dgrad)
// orientation, and with FWD also in the forward one, from one read of each
// weight: 128 x 128 tiles of x[grp] are staged in shared memory (two buffers,
// the next tile's per-thread asynchronous copies in flight while the current
// one is quantized). Every thread takes four blocks of each copy it writes:
// of the transposed copy, column t % 128 of the tile and its rows
// 64 (t / 128) .. + 64; of the forward copy, row t / 2 and its columns
// 64 (t % 2) .. + 64; each gives 32 contiguous code bytes and one 4-byte
// scale word. Both copies use the group's global scale (g_in, else from the
// group maxima in amax_bits; after that maxima pass the tiles are taken last
// to first, starting on the bytes it left in L2).
constexpr int kDR = 128, kDC = 128, kDPitch = kDC + 8;  // pitch in BF16, rows 16-byte aligned
constexpr int kDTile = kDR * kDPitch;
constexpr size_t kDualSmem = 2 * kDTile * sizeof(uint16_t);

__device__ __forceinline__ void cp_async16_zfill(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
               :: "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(valid ? 16 : 0)
               : "memory");
}

// Shape constants of the quantization of one weight shape.
struct DualGeom {
  int rows, cols, tr, tc;        // tiles per group: tr x tc
  int nbk, nbn, kck, kcn;        // blocks per quantized row, SF columns (forward, transposed)
  int64_t sfk_group, sfn_group;  // SF bytes per group
  bool v8k, v8n;                 // 32-byte code stores allowed
};

__device__ __forceinline__ DualGeom dual_geom(int rows, int cols, const uint8_t* codes_k,
                                              const uint8_t* codes_n) {
  DualGeom G;
  G.rows = rows; G.cols = cols;
  G.tr = (rows + kDR - 1) / kDR; G.tc = (cols + kDC - 1) / kDC;
  G.nbk = cols / 16; G.nbn = rows / 16;
  G.kck = (G.nbk + 3) & ~3; G.kcn = (G.nbn + 3) & ~3;
  G.sfk_group = static_cast<int64_t>((rows + 127) & ~127) * G.kck;
  G.sfn_group = static_cast<int64_t>((cols + 127) & ~127) * G.kcn;
  // 32-byte code stores where every destination row starts 32-byte aligned
  G.v8k = (cols / 2) % 32 == 0 && (reinterpret_cast<uintptr_t>(codes_k) & 31) == 0;
  G.v8n = (rows / 2) % 32 == 0 && (reinterpret_cast<uintptr_t>(codes_n) & 31) == 0;
  return G;
}

// Every thread of the block: per-thread asynchronous copies of the 128 x 128
// tile (r0, c0) of group xg into buf (zero-filled outside the matrix), as
// one commit group.
__device__ __forceinline__ void dual_fetch(const uint16_t* xg, const DualGeom& G, int r0, int c0,
                                           uint16_t* buf, const uint16_t* any_valid) {
  const int t = threadIdx.x;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int q = t + 256 * i;  // 16-byte piece q of the tile: row q / 16, piece q % 16
    const int lr = q >> 4, seg = q & 15;
    const bool valid = r0 + lr < G.rows && c0 + 8 * seg < G.cols;
    const uint16_t* src =
        valid ? xg + static_cast<int64_t>(r0 + lr) * G.cols + c0 + 8 * seg : any_valid;
    cp_async16_zfill(buf + lr * kDPitch + 8 * seg, src, valid);
  }
}

// Four 8-byte code blocks at dst (blocks g0 .. g0 + 3 of a row of nb): one
// 32-byte store where allowed, else the blocks below nb one by one.
__device__ __forceinline__ void store_code4(uint8_t* dst, const uint2 (&code)[4], int g0, int nb,
                                            bool v8) {
  if (v8 && g0 + 4 <= nb) {
    st_global_v8(dst, code[0].x, code[0].y, code[1].x, code[1].y, code[2].x, code[2].y,
                 code[3].x, code[3].y);
  } else {
#pragma unroll
    for (int b = 0; b < 4; ++b)
      if (g0 + b < nb) st_u64(dst + 8 * b, code[b]);
  }
}

// Every thread of the block (256): quantize the staged tile (r0, c0) of
// group grp in the transposed orientation and, with FWD, the forward one,
// with the group's global scale g.
template <bool FWD>
__device__ __forceinline__ void dual_tile_quant(const uint16_t* tile, const DualGeom& G,
                                                int64_t grp, int r0, int c0, float g, float tk,
                                                uint8_t* __restrict__ codes_k,
                                                uint8_t* __restrict__ sf_k,
                                                uint8_t* __restrict__ codes_n,
                                                uint8_t* __restrict__ sf_n) {
  const int t = threadIdx.x;
  {
    // ---- one tile column, 4 blocks along the rows (transposed copy)
    const int lc = t & (kDC - 1), rb0 = 4 * (t >> 7);
    const int c = c0 + lc;
    const int gr = r0 / 16 + rb0;  // multiple of 4
    uint2 code[4];
    uint32_t sfw = 0;
#pragma unroll
    for (int rb = 0; rb < 4; ++rb) {
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        v[j] = __uint_as_float(static_cast<uint32_t>(tile[(16 * (rb0 + rb) + j) * kDPitch + lc])
                               << 16);
      const bool valid = c < G.cols && gr + rb < G.nbn;
      const QBlock q = quant_block(v, amax_f32x16(v), g, tk, valid);
      code[rb] = q.codes;
      sfw |= q.sf << (8 * rb);
    }
    if (c < G.cols && gr < G.kcn) {
      if (gr < G.nbn)
        store_code4(codes_n + (grp * G.cols + c) * static_cast<int64_t>(G.rows / 2) + 8 * gr, code,
                    gr, G.nbn, G.v8n);
      *reinterpret_cast<uint32_t*>(sf_n + grp * G.sfn_group + sf_offset(c, gr, G.kcn)) = sfw;
    }
  }
  if (FWD) {
    // ---- half a tile row, 4 blocks along the columns (forward copy)
    const int lr = t >> 1, half = t & 1;
    const int r = r0 + lr;
    uint2 code[4];
    uint32_t sfw = 0;
#pragma unroll
    for (int cb = 0; cb < 4; ++cb) {
      const uint4* src =
          reinterpret_cast<const uint4*>(tile + lr * kDPitch + 64 * half + 16 * cb);
      const uint4 a0 = src[0], a1 = src[1];
      const uint32_t w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      float v[16];
      unpack_bf16x16(w, v);
      const bool valid = r < G.rows && c0 / 16 + 4 * half + cb < G.nbk;
      const QBlock q = quant_block(v, amax_bf16x16(w), g, tk, valid);
      code[cb] = q.codes;
      sfw |= q.sf << (8 * cb);
    }
    const int gc = c0 / 16 + 4 * half;  // multiple of 4
    if (r < G.rows && gc < G.nbk) {
      store_code4(codes_k + (grp * G.rows + r) * static_cast<int64_t>(G.cols / 2) + 8 * gc, code,
                  gc, G.nbk, G.v8k);
      *reinterpret_cast<uint32_t*>(sf_k + grp * G.sfk_group + sf_offset(r, gc, G.kck)) = sfw;
    }
  }
}

// Scale bytes of the padding rows of the copies written (the forward one with
// FWD), groups [g0, g1), split over `nthreads` threads numbered from `gt`.
template <bool FWD>
__device__ __forceinline__ void dual_zero_padding(const DualGeom& G, int64_t g0, int64_t g1,
                                                  int64_t gt, int64_t nthreads,
                                                  uint8_t* __restrict__ sf_k,
                                                  uint8_t* __restrict__ sf_n) {
  const int64_t pk = ((G.rows + 127) & ~127) - G.rows, pn = ((G.cols + 127) & ~127) - G.cols;
  const int wk = G.kck / 4, wn = G.kcn / 4;
  if (FWD) {
    for (int64_t i = gt; i < (g1 - g0) * pk * wk; i += nthreads) {
      const int64_t grp = g0 + i / (pk * wk);
      const int64_t rem = i % (pk * wk);
      *reinterpret_cast<uint32_t*>(sf_k + grp * G.sfk_group +
                                   sf_offset(G.rows + rem / wk, 4 * (rem % wk), G.kck)) = 0u;
    }
  }
  for (int64_t i = gt; i < (g1 - g0) * pn * wn; i += nthreads) {
    const int64_t grp = g0 + i / (pn * wn);
    const int64_t rem = i % (pn * wn);
    *reinterpret_cast<uint32_t*>(sf_n + grp * G.sfn_group +
                                 sf_offset(G.cols + rem / wn, 4 * (rem % wn), G.kcn)) = 0u;
  }
}

template <bool FWD>
__global__ void __launch_bounds__(256) quantize_tiles_kernel(
    const uint16_t* __restrict__ x, int64_t groups, int rows, int cols,
    const float* __restrict__ g_in, const uint32_t* __restrict__ amax_bits,
    uint8_t* __restrict__ codes_k, uint8_t* __restrict__ sf_k, uint8_t* __restrict__ codes_n,
    uint8_t* __restrict__ sf_n, float* __restrict__ g_out) {
  extern __shared__ __align__(16) uint16_t dtiles[];  // [2][kDTile]
  pdl_wait();
  const int t = threadIdx.x;
  const DualGeom G = dual_geom(rows, cols, codes_k, codes_n);
  const int64_t per_group = static_cast<int64_t>(G.tr) * G.tc;
  const int64_t ntiles = groups * per_group;
  // tile ti -> (group, first row, first column), decoded once per tile and
  // carried from its copies to its quantization
  struct TilePos {
    int64_t grp;
    int r0, c0;
  };
  auto pos = [&](int64_t ti) {
    TilePos p{-1, 0, 0};
    if (ti < ntiles) {
      const int64_t k = g_in ? ti : ntiles - 1 - ti;
      p.grp = div_nonneg(k, per_group);
      const int rem = static_cast<int>(k - p.grp * per_group);
      const int a = rem / G.tc;
      p.r0 = a * kDR;
      p.c0 = (rem - a * G.tc) * kDC;
    }
    return p;
  };
  auto fetch = [&](const TilePos& p, uint16_t* buf) {
    if (p.grp >= 0)
      dual_fetch(x + p.grp * static_cast<int64_t>(rows) * cols, G, p.r0, p.c0, buf, x);
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  int64_t ti = blockIdx.x;
  TilePos p0 = pos(ti), p1 = pos(ti + gridDim.x);
  fetch(p0, dtiles);
  int cur = 0;
  int64_t gcur = -1;
  float g = 1.0f, tk = 1.0f;
  for (; ti < ntiles; ti += gridDim.x, cur ^= 1) {
    fetch(p1, dtiles + (cur ^ 1) * kDTile);
    const TilePos p2 = pos(ti + 2 * static_cast<int64_t>(gridDim.x));
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncthreads();
    if (p0.grp != gcur) {  // block-uniform
      gcur = p0.grp;
      g = g_in ? g_in[gcur] : global_scale(__uint_as_float(amax_bits[gcur]));
      tk = enc_table_entry(g);
    }
    dual_tile_quant<FWD>(dtiles + cur * kDTile, G, p0.grp, p0.r0, p0.c0, g, tk, codes_k, sf_k,
                         codes_n, sf_n);
    __syncthreads();  // the next iteration refills this buffer
    p0 = p1;
    p1 = p2;
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");

  // zero the scale bytes of the padding rows, and publish g
  const int64_t gt = blockIdx.x * static_cast<int64_t>(blockDim.x) + t;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  dual_zero_padding<FWD>(G, 0, groups, gt, nthreads, sf_k, sf_n);
  for (int64_t grp = gt; grp < groups; grp += nthreads)
    g_out[grp] = g_in ? g_in[grp] : global_scale(__uint_as_float(amax_bits[grp]));
}

// One launch of quantize_tiles_kernel<FWD> (three CTAs per SM: two 34 KB tile
// buffers each).
template <bool FWD>
static int launch_tiles(const uint16_t* x, int64_t groups, int64_t rows, int64_t cols,
                        const float* g_in, const uint32_t* amax, uint8_t* codes_k, uint8_t* sf_k,
                        uint8_t* codes_n, uint8_t* sf_n, float* g_out, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(quantize_tiles_kernel<FWD>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kDualSmem));
  });
  if (attr != cudaSuccess) return MINITE_ERR_CUDA;
  const int64_t tiles = groups * ((rows + kDR - 1) / kDR) * ((cols + kDC - 1) / kDC);
  int64_t blocks = static_cast<int64_t>(num_sms()) * 3;
  if (blocks > tiles) blocks = tiles;
  if (blocks * 256 < groups) blocks = (groups + 255) / 256;  // g_out: thread t < groups
  if (launch_pdl(quantize_tiles_kernel<FWD>, dim3(static_cast<unsigned>(blocks)), dim3(256),
                 kDualSmem, s, x, groups, static_cast<int>(rows), static_cast<int>(cols), g_in,
                 amax, codes_k, sf_k, codes_n, sf_n, g_out) != cudaSuccess)
    return MINITE_ERR_CUDA;
  return MINITE_OK;
}

template <int NCH, bool PG>
static void launch_token_rows(const uint16_t* x, int64_t groups, int64_t rows, int cols, bool a32,
                              uint8_t* codes, uint8_t* sf, float* g_out, const float* g_in,
                              const uint32_t* amax, cudaStream_t s) {
  const int64_t total = groups * ((rows + 127) & ~int64_t(127));
  int64_t blocks = (total + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
  if (blocks > cap) blocks = cap;
  const dim3 grid(static_cast<unsigned>(blocks)), block(256);
  if (a32)
    launch_pdl(quantize_token_rows_kernel<NCH, true, PG>, grid, block, 0, s, x, groups, rows, cols,
               codes, sf, g_out, g_in, amax);
  else
    launch_pdl(quantize_token_rows_kernel<NCH, false, PG>, grid, block, 0, s, x, groups, rows, cols,
               codes, sf, g_out, g_in, amax);
}

static void launch_group_blocks(const uint16_t* x, int64_t groups, int64_t rows, int cols,
                                bool a32, const float* g_in, const uint32_t* amax,
                                uint8_t* codes, uint8_t* sf, float* g_out, cudaStream_t s) {
  const int nb = cols / 16;
  const uint32_t magic = nb == 1 ? 0xFFFFFFFFu
                                 : static_cast<uint32_t>((uint64_t(1) << 32) / uint64_t(nb));
  const int64_t chunks = groups * ((rows * nb + 31) / 32);
  int64_t blocks = static_cast<int64_t>(num_sms()) * 4;
  const int64_t need = (chunks + 8 * kU - 1) / (8 * kU);
  if (blocks > need) blocks = need;
  const int64_t min_blocks = (groups + 255) / 256;  // g_out is written by thread t < groups
  if (blocks < min_blocks) blocks = min_blocks;
  if (blocks < 1) blocks = 1;
  if (a32)
    launch_pdl(quantize_group_blocks_kernel<true>, dim3(static_cast<unsigned>(blocks)), dim3(256),
               0, s, x, groups, rows, nb, magic, g_in, amax, codes, sf, g_out);
  else
    launch_pdl(quantize_group_blocks_kernel<false>, dim3(static_cast<unsigned>(blocks)), dim3(256),
               0, s, x, groups, rows, nb, magic, g_in, amax, codes, sf, g_out);
}

// Per-group |x| maxima into amax (zeroed first), one grid over all groups.
static int launch_group_amax(const uint16_t* x, int64_t groups, int64_t per_group,
                             uint32_t* amax, cudaStream_t s) {
  if (cudaMemsetAsync(amax, 0, groups * sizeof(uint32_t), s) != cudaSuccess)
    return MINITE_ERR_CUDA;
  int64_t bx = (per_group / 16 + 256 * kAmaxU - 1) / (256 * kAmaxU);
  const int64_t want = (num_sms() * 8 + groups - 1) / groups;
  if (bx > want) bx = want;
  if (bx < 1) bx = 1;
  dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(groups));
  if (launch_pdl(group_amax_kernel, grid, dim3(256), 0, s, x, per_group, amax) != cudaSuccess)
    return MINITE_ERR_CUDA;
  return MINITE_OK;
}

}  // namespace minite

using namespace minite;

extern "C" int minite_quantize_nvfp4_dual(const void* x, int64_t groups, int64_t rows,
                                          int64_t cols, uint8_t* codes_k, uint8_t* sf_k,
                                          uint8_t* codes_n, uint8_t* sf_n, float* gscale_out,
                                          void* workspace, size_t ws_bytes, int32_t* status,
                                          minite_stream_t stream) {
  (void)status;
  if (!x || !codes_k || !sf_k || !codes_n || !sf_n || !gscale_out || !workspace)
    return MINITE_ERR_INVALID_ARG;
  if (groups <= 0 || rows <= 0 || cols <= 0 || rows % 16 != 0 || cols % 16 != 0)
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (rows >= (int64_t(1) << 30) || cols >= (int64_t(1) << 30) ||
      groups * rows * cols >= (int64_t(1) << 40))
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 16) || !aligned(codes_k, 8) || !aligned(codes_n, 8) || !aligned(sf_k, 4) ||
      !aligned(sf_n, 4))
    return MINITE_ERR_INVALID_ARG;
  if (ws_bytes < minite_workspace_bytes(MINITE_OP_QUANTIZE, groups, 0, 0, 0))
    return MINITE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  uint32_t* amax = static_cast<uint32_t*>(workspace);
  const int rc = launch_group_amax(xb, groups, rows * cols, amax, s);
  if (rc != MINITE_OK) return rc;
  return launch_tiles<true>(xb, groups, rows, cols, nullptr, amax, codes_k, sf_k, codes_n, sf_n,
                            gscale_out, s);
}

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
  if (!aligned(x, 16) || !aligned(codes, 8) || !aligned(sf, 4)) return MINITE_ERR_INVALID_ARG;
  const bool per_group = scale_mode == MINITE_SCALE_PER_GROUP;
  if (gscale_in && !per_group) return MINITE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  const int64_t Cq = orientation == MINITE_ALONG_COLS ? cols : rows;
  if (Cq % 16 != 0 || cols % 8 != 0) return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (orientation == MINITE_ALONG_ROWS &&
      (!per_group || rows >= (int64_t(1) << 30) || cols >= (int64_t(1) << 30)))
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (orientation == MINITE_ALONG_COLS && cols > 4096) return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (groups * rows * cols >= (int64_t(1) << 40)) return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (per_group && rows * (cols / 16) >= (int64_t(1) << 32)) return MINITE_ERR_UNSUPPORTED_SHAPE;

  uint32_t* amax = nullptr;
  if (per_group && !gscale_in) {
    if (!workspace || ws_bytes < minite_workspace_bytes(MINITE_OP_QUANTIZE, groups, 0, 0, 0))
      return MINITE_ERR_INVALID_ARG;
    amax = static_cast<uint32_t*>(workspace);
    const int rc = launch_group_amax(xb, groups, rows * cols, amax, s);
    if (rc != MINITE_OK) return rc;
  }

  if (orientation == MINITE_ALONG_COLS) {
    const int c = static_cast<int>(cols);
    const bool a32 = aligned(x, 32);
    if (per_group) {
      // one warp per row when the row fits in registers, else the flat block stream
      switch ((cols / 16 + 31) / 32) {
#define MINITE_CASE(N)                                                                   \
  case N:                                                                                \
    launch_token_rows<N, true>(xb, groups, rows, c, a32, codes, sf, gscale_out, gscale_in, \
                               amax, s);                                                 \
    break;
        MINITE_CASE(1) MINITE_CASE(2) MINITE_CASE(3) MINITE_CASE(4)
#undef MINITE_CASE
        default:
          launch_group_blocks(xb, groups, rows, c, a32, gscale_in, amax, codes, sf, gscale_out, s);
      }
    } else {
      switch ((cols / 16 + 31) / 32) {
#define MINITE_CASE(N) \
  case N:                                                                                \
    launch_token_rows<N, false>(xb, groups, rows, c, a32, codes, sf, gscale_out, nullptr,  \
                                nullptr, s);                                             \
    break;
        MINITE_CASE(1) MINITE_CASE(2) MINITE_CASE(3) MINITE_CASE(4) MINITE_CASE(5)
        MINITE_CASE(6) MINITE_CASE(7) MINITE_CASE(8)
#undef MINITE_CASE
        default: return MINITE_ERR_UNSUPPORTED_SHAPE;
      }
    }
  } else {
    const int rc = launch_tiles<false>(xb, groups, rows, cols, gscale_in, amax, nullptr, nullptr,
                                       codes, sf, gscale_out, s);
    if (rc != MINITE_OK) return rc;
  }
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}
