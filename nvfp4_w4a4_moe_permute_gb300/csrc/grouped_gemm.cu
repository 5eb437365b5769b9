// minite_grouped_gemm_nvfp4: block-scaled FP4 x FP4 grouped GEMM over the
// experts of a MoE layer, one persistent launch for all experts.
//
// Grouped GEMMs over experts are where the W4A4 speed-up is won or lost
// ("miniTE accélère le RL en NVFP4 sur B300", section "Diagnostic, alignement
// et noyaux rapides"); the operands are contiguous expert buffers described by
// device-side offsets, with no host-side splitting or repacking (miniTE
// report summary, section "Two complementary interventions").
//
// Design (sm_103a):
//  * Output tile 128 x 256; K consumed 256 elements (128 bytes of packed
//    E2M1) per pipeline stage; one tcgen05.mma of kind mxf4nvf4 with 4X block
//    scaling covers K = 64 (M = 128, N = 256), so a stage is 4 MMAs.
//  * Warp 0 (producer): TMA (128-byte swizzle) loads the A and B code tiles;
//    plain bulk copies load the scale atoms, which the permutation and the
//    quantizers already wrote in the MMA layout.
//  * Warp 1 (MMA issuer): one thread issues only MMAs and commits, with
//    descriptors advanced by constant offsets, so the tensor pipe never waits
//    on the issuing thread.
//  * Warps 2..5 (scale warps): read each stage's scale atoms from shared
//    memory and write them to a TMEM ring with tcgen05.st, replicated into
//    the four 32-lane quarters (the layout a 32x128b.warpx4 copy produces).
//    This keeps scale movement off the tensor pipe, where copies and MMAs
//    would otherwise share issue bandwidth.
//  * Warps 6..21 (epilogue): four warps per TMEM lane quarter, each draining
//    64 of the 256 accumulator columns (two 32-column loads) and releasing
//    the accumulator right after the second; the next tile's MMAs then overlap
//    the rest of the scaling by 1/(g_a[row] * g_w[e]), conversion and stores
//    (rows of the tile's expert only).
//  * TMEM: 256 accumulator columns + a 4-deep ring of 48 scale columns.
//  * Static round-robin tile schedule over one CTA per SM; the tile list is
//    derived on the device from expert_offsets.
//  * Fixed K order, no split-K, one tile shape: a row's result depends only
//    on its own codes and its expert's weights (batch invariance).
//  * Every mbarrier wait is bounded by a %globaltimer budget; on expiry the
//    CTA records MINITE_ERR_TIMEOUT, drains its in-flight copies and MMAs,
//    frees TMEM and exits.
//
// Kernels (all bit-identical; the automatic choice is the third where it
// applies): grouped_gemm_kernel (above, one-chunk stages; any K % 64 == 0),
// grouped_gemm_dc_kernel (128 x 256 tiles, two-chunk stages loaded with one
// 3-D box per operand and scale atoms from a separate producer warp) and
// grouped_gemm_pair_deep_kernel (256 x 256 tiles with tcgen05.mma.cta_group::2
// on the two SMs of a cluster, five one-chunk stages that carry their scale
// atoms). Measured on the pair kernel, neither the operand loads (copies
// stopped after the first stages: within 3% of the real time) nor the
// tensor pipe (128 cycles per MMA when fed) sets the pace: each K chunk's
// MMAs wait for its scale atoms, which are copied only once the stage's
// previous MMAs complete and then pass through the scale warps into TMEM.
// The output stores were the other limit: with a lane owning a row, every
// store instruction touched 32 different 128-byte lines and the epilogue
// warps fell behind the single-buffered accumulator (with the stores left
// out, gate_up took 0.32 instead of 0.44 ms and down 0.22 instead of 0.39 ms
// on the skewed layer). The BF16 epilogue therefore transposes chunks among
// groups of four lanes so that each instruction writes whole row segments,
// and the pair kernel hands full 32-row boxes to TMA stores from a 2 KB
// staging buffer per warp.
//
// minite_gate_up_swiglu_quant_nvfp4 runs the pair kernel's second instance
// (SWIGLU): the even CTA loads gate rows and the odd CTA the matching up
// rows, so each accumulator holds gate and up columns of the same 128
// intermediate columns; the epilogue applies the weighted SwiGLU and, once
// the I/128 tiles of a 256-row block have published their rows' partial |h|
// maxima (flagged per-row slots in a workspace), quantizes h to NVFP4.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "host_util.h"

namespace minite {

namespace gemm {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK_BYTES = 128;                 // 256 E2M1 values per row per stage
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK_BYTES;        // 16 KB
constexpr int B_BYTES = BN * BK_BYTES;        // 32 KB
constexpr int SF_ATOM = 512;                  // 128 rows x 4 scales (one K = 64 step)
constexpr int SFA_BYTES = 4 * SF_ATOM;        // 4 K-steps
constexpr int SFB_BYTES = 4 * SF_ATOM * (BN / 128);
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr int NUM_EPI_WARPS = 16;                 // four per TMEM lane quarter, 64 columns each
constexpr int EPI_WARP0 = 6;
constexpr int NUM_WARPS = EPI_WARP0 + NUM_EPI_WARPS;
constexpr int NUM_THREADS = NUM_WARPS * 32;
constexpr int EPI_COLS = BN / (NUM_EPI_WARPS / 4);  // accumulator columns per epilogue warp
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = BN;
constexpr int NSF = 4;                                   // scale ring depth
constexpr uint32_t SF_COLS = 16 + 16 * (BN / 128);       // A: 4 x 4 cols, B: 4 x 4 x (BN/128)
constexpr uint32_t SF_COL0 = ACC_COLS;
static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte swizzle alignment");
static_assert(SF_COL0 + NSF * SF_COLS <= TMEM_COLS, "TMEM budget");

// Instruction descriptor of tcgen05.mma kind::mxf4nvf4: A and B E2M1 (format
// code 1 in this kind), both K-major, UE4M3 scales (bit 23 clear), scale
// factor ids 0, N >> 3 at bit 17, M >> 4 at bit 24, dense K = 64.
constexpr uint32_t make_idesc() {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
         (static_cast<uint32_t>(BM >> 4) << 24);
}

struct Smem {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t sf_full[NSF];
  uint64_t sf_empty[NSF];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int total_tiles;
  int pad_;
};

// Fields of the fused gate_up + weighted SwiGLU + NVFP4 epilogue (unused by
// the plain GEMMs).
struct SwigluParams {
  const float* perm_w;   // [M] routing weights, or null (weight 1)
  uint8_t* h_codes;      // [M, I/2]
  uint8_t* h_sf;         // per-expert padded regions, kc = I/16 scale columns
  float* h_g;            // [M]
  uint32_t* amax;        // [M, roundup(I/128, 4)] zeroed: per row, each tile's partial |h|
                         // maximum (float bits) with bit 31 set once written
  int I;
};

struct Params {
  const float* a_g;
  const float* b_g;
  const uint8_t* a_sf;
  const uint8_t* b_sf;
  const int32_t* offsets;
  const int32_t* sf_offsets;
  void* out;
  int32_t* status;
  int64_t M;          // rows of A / out (weight gradient: rows of A, i.e. channels)
  int N, K, E;        // weight gradient: K = token columns allocated per operand row
  int out_fp32;
  int c_tma;          // CTA-pair kernel: BF16 output staged per warp, written by TMA stores
  uint64_t budget_ns;
  SwigluParams sw;
};

struct Tile {
  int e, nt;
  int row0;           // first permuted row of the tile (weight gradient: first A row)
  int rows;           // valid rows (<= 128)
  int sf_rb;          // 128-row block of A's scales
  int kz0;            // first 128-byte K chunk (0 for the forward GEMMs)
  int kt;             // K chunks of the tile
};

// tile index -> (expert, m block, n block). tiles_prefix[e] = 128-row m blocks
// before expert e; s_off = expert_offsets (both in shared memory). With
// validated offsets the A scale block of m block `mt` is mt itself, since
// sf_row_offsets[e] / 128 = sum of ceil(count / 128) = tiles_prefix[e].
__device__ __forceinline__ Tile decode_tile(int t, int n_tiles, const int32_t* tiles_prefix,
                                            const int32_t* s_off, const Params& p) {
  Tile r;
  const int mt = t / n_tiles;
  r.nt = t - mt * n_tiles;
  int lo = 0, hi = p.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tiles_prefix[mid] <= mt) lo = mid; else hi = mid;
  }
  r.e = lo;
  const int ml = mt - tiles_prefix[lo];
  r.row0 = s_off[lo] + ml * BM;
  r.rows = min(BM, s_off[lo + 1] - r.row0);
  r.sf_rb = mt;
  r.kz0 = 0;
  r.kt = (p.K + 255) / 256;
  return r;
}

// Weight-gradient tile index -> (expert, A row block, B column block):
// tiles_prefix[e] = A row blocks of the experts before e that have tokens;
// s_kofs = the operands' token offsets (multiples of 256). Expert e's K range
// is [s_kofs[e], s_kofs[e + 1]).
__device__ __forceinline__ Tile decode_tile_wg(int t, int n_tiles, const int32_t* tiles_prefix,
                                               const int32_t* s_kofs, const Params& p) {
  Tile r;
  const int mt = t / n_tiles;
  r.nt = t - mt * n_tiles;
  int lo = 0, hi = p.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tiles_prefix[mid] <= mt) lo = mid; else hi = mid;
  }
  r.e = lo;
  const int ml = mt - tiles_prefix[lo];
  r.row0 = ml * BM;
  r.rows = min(BM, static_cast<int>(p.M) - r.row0);
  r.sf_rb = ml;
  r.kz0 = s_kofs[lo] / 256;
  r.kt = (s_kofs[lo + 1] - s_kofs[lo]) / 256;
  return r;
}

template <bool WG>
__device__ __forceinline__ Tile decode_any(int t, int n_tiles, const int32_t* tiles_prefix,
                                           const int32_t* s_off, const Params& p) {
  if constexpr (WG) return decode_tile_wg(t, n_tiles, tiles_prefix, s_off, p);
  else return decode_tile(t, n_tiles, tiles_prefix, s_off, p);
}

__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// One epilogue warp's drain of EPI_COLS (= 64) accumulator columns of its 32
// TMEM lanes into 32 packed BF16 pairs per lane (the row's columns scaled by
// `scale`), as two 32-column loads; `release` runs on lane 0 once the second
// has landed (the MMA may then overwrite the accumulator). The first half is
// packed (paired products, one two-value conversion) before the second load.
template <typename Release>
__device__ __forceinline__ void drain_bf16x64(uint32_t tbase, float scale, Release release,
                                              uint32_t (&pk)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t r[32];
    tmem_ld_32cols(tbase + 32 * c, r);
    if (c == 1) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) release();
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float lo = __uint_as_float(r[2 * j]), hi = __uint_as_float(r[2 * j + 1]);
      mul_f32x2(lo, hi, scale, scale);
      pk[16 * c + j] = pack_bf16x2_rn(lo, hi);
    }
  }
}

// Stores 128 bytes of each of a warp's 32 consecutive rows: the columns
// [n0, n0 + 128 / sizeof(T)) below N of a row-major [*, ld] array of T (64
// BF16 or 32 FP32 columns); lane L holds row row0 + L as 32 words (four
// 32-byte chunks). A lane owning a whole row would make every store
// instruction touch 32 different 128-byte lines; instead the four lanes of
// each group g exchange chunks (a 4 x 4 transpose by three shuffles and two
// rotations on each side) so that lane (g, t) stores chunk t of rows
// 4g..4g+3, one row per instruction: each instruction writes 8 whole
// 128-byte row segments. `vmask` has bit L set when row row0 + L exists.
// Call on all 32 lanes.
template <typename T>
__device__ __forceinline__ void store_rows_x4(T* out, int64_t ld, int64_t row0, int n0, int N,
                                              uint32_t vmask, uint32_t (&pk)[32]) {
  static_assert(sizeof(T) == 2 || sizeof(T) == 4, "BF16 or FP32 rows");
  const int lane = threadIdx.x & 31;
  const int t = lane & 3;
  const int gbase = lane & ~3;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    // sender side: y[s] = chunk (t - s) & 3, the chunk lane gbase + ((t - s) & 3) needs
    const uint32_t c0 = pk[w], c1 = pk[8 + w], c2 = pk[16 + w], c3 = pk[24 + w];
    const uint32_t a0 = (t & 1) ? c1 : c0, a1 = (t & 1) ? c0 : c3, a2 = (t & 1) ? c3 : c2,
                   a3 = (t & 1) ? c2 : c1;
    const uint32_t y1 = (t & 2) ? a3 : a1, y2 = (t & 2) ? a0 : a2, y3 = (t & 2) ? a1 : a3;
    // r[s] = chunk t of group row (t + s) & 3
    const uint32_t r0 = (t & 2) ? a2 : a0;
    const uint32_t r1 = __shfl_sync(0xffffffffu, y1, gbase | ((t + 1) & 3));
    const uint32_t r2 = __shfl_sync(0xffffffffu, y2, gbase | ((t + 2) & 3));
    const uint32_t r3 = __shfl_sync(0xffffffffu, y3, gbase | ((t + 3) & 3));
    // receiver side: chunk t of group row u is r[(u - t) & 3]
    const uint32_t b0 = (t & 1) ? r3 : r0, b1 = (t & 1) ? r0 : r1, b2 = (t & 1) ? r1 : r2,
                   b3 = (t & 1) ? r2 : r3;
    pk[w] = (t & 2) ? b2 : b0;
    pk[8 + w] = (t & 2) ? b3 : b1;
    pk[16 + w] = (t & 2) ? b0 : b2;
    pk[24 + w] = (t & 2) ? b1 : b3;
  }
  const int col = n0 + (32 / static_cast<int>(sizeof(T))) * t;
  T* o = out + (row0 + gbase) * ld + col;
#pragma unroll
  for (int u = 0; u < 4; ++u)
    if (((vmask >> (gbase + u)) & 1u) && col < N)
      st_global_v8(o + static_cast<int64_t>(u) * ld, pk[8 * u], pk[8 * u + 1], pk[8 * u + 2],
                   pk[8 * u + 3], pk[8 * u + 4], pk[8 * u + 5], pk[8 * u + 6], pk[8 * u + 7]);
}

// One epilogue warp: drain EPI_COLS (= 64) accumulator columns of its 32 TMEM
// lanes (row `row` on each lane, consecutive over the lanes) as two 32-column
// loads, call `release` on lane 0 as soon as the second has landed (the MMA
// may then overwrite the accumulator), scale by `scale`, round to BF16 (or
// keep FP32) and store the row's columns [n0, n0 + 64) below N. Call on all
// 32 lanes.
template <typename Release>
__device__ __forceinline__ void epilogue_slice(const Params& p, uint32_t tbase, bool valid,
                                               int64_t row, int n0, float scale, Release release) {
  static_assert(EPI_COLS == 64, "two 32-column TMEM loads per epilogue warp");
  const int lane = threadIdx.x & 31;
  if (!p.out_fp32) {
    uint32_t pk[32];
    drain_bf16x64(tbase, scale, release, pk);
    store_rows_x4(static_cast<uint16_t*>(p.out), p.N, row - lane, n0, p.N,
                  __ballot_sync(0xffffffffu, valid), pk);
  } else {
    const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
      uint32_t r[32];
      tmem_ld_32cols(tbase + 32 * c, r);
      if (c == 1) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release();
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__fmul_rn(__uint_as_float(r[j]), scale));
      store_rows_x4(static_cast<float*>(p.out), p.N, row - lane, n0 + 32 * c, p.N, vmask, r);
    }
  }
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Smem& S = *reinterpret_cast<Smem*>(stages + STAGES * STAGE_BYTES);
  int32_t* tiles_prefix = reinterpret_cast<int32_t*>(&S + 1);   // [E+1]
  int32_t* s_off = tiles_prefix + (p.E + 1);                    // [E+1] expert_offsets

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KT = (p.K + 255) / 256;       // pipeline stages per tile
  const int KSTEPS = p.K / 64;            // MMAs per tile
  const int atoms_per_rb = p.K / 64;      // scale atoms per 128-row block
  const int n_tiles = (p.N + BN - 1) / BN;
  const int rb_per_expert = (p.N + 127) / 128;   // 128-row scale blocks of one weight

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int b = 0; b < NSF; ++b) {
      mbar_init(&S.sf_full[b], 4);
      mbar_init(&S.sf_empty[b], 1);
    }
    mbar_init(&S.acc_full, 1);
    mbar_init(&S.acc_empty, NUM_EPI_WARPS);
    mbar_init(&S.drain, 1);
    S.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&S.tmem_base, TMEM_COLS);
  if (warp == 2) {
    // m-block prefix over experts, validating the device offsets on the way
    int carry = 0;
    bool bad = false;
    if (lane == 0) tiles_prefix[0] = 0;
    for (int base = 0; base < p.E; base += 32) {
      const int e = base + lane;
      int cnt = 0;
      if (e < p.E) {
        const int o0 = __ldg(p.offsets + e), o1 = __ldg(p.offsets + e + 1);
        const int s0 = __ldg(p.sf_offsets + e), s1 = __ldg(p.sf_offsets + e + 1);
        s_off[e + 1] = o1;
        if (e == 0) s_off[0] = o0;
        cnt = o1 - o0;
        if (cnt < 0 || s1 - s0 != ((cnt + 127) & ~127) || (e == 0 && (o0 != 0 || s0 != 0)) ||
            (e == p.E - 1 && o1 > p.M))
          bad = true;
        cnt = cnt > 0 ? (cnt + BM - 1) / BM : 0;
      }
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (e < p.E) tiles_prefix[e + 1] = carry + incl;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      S.total_tiles = bad ? 0 : carry * n_tiles;
      if (bad && blockIdx.x == 0) set_status(p.status, MINITE_ERR_INVALID_ARG);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem = S.tmem_base;
  const int total = S.total_tiles;
  volatile int* abort_flag = &S.abort_flag;
  const uint64_t budget = p.budget_ns;
  constexpr uint64_t kDrainBudget = 200000000ull;  // 200 ms for in-flight work at exit

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t armed_mask = 0, armed_parity = 0;   // per stage: armed at least once, last parity
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const size_t sfb_expert = static_cast<size_t>(rb_per_expert) * atoms_per_rb * SF_ATOM;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile tl = decode_tile(t, n_tiles, tiles_prefix, s_off, p);
        // the second 128-row scale block of B exists only inside the padded weight
        const int nrb = min(BN / 128, rb_per_expert - tl.nt * (BN / 128));
        for (int kt = 0; kt < KT; ++kt) {
          if (!mbar_wait(&S.empty[stage], phase ^ 1u, budget, abort_flag)) { ok = false; break; }
          const int ks = min(4, KSTEPS - 4 * kt);
          uint8_t* sA = stages + stage * STAGE_BYTES;
          uint8_t* sB = sA + A_BYTES;
          uint8_t* sSFA = sB + B_BYTES;
          uint8_t* sSFB = sSFA + SFA_BYTES;
          mbar_arrive_expect_tx(&S.full[stage], A_BYTES + B_BYTES +
                                                    static_cast<uint32_t>(ks * (1 + nrb)) * SF_ATOM);
          tma_load_2d(sA, &tmap_a, &S.full[stage], kt * BK_BYTES, tl.row0);
          tma_load_2d(sB, &tmap_b, &S.full[stage], kt * BK_BYTES, tl.e * p.N + tl.nt * BN);
          bulk_load(sSFA,
                    p.a_sf + (static_cast<size_t>(tl.sf_rb) * atoms_per_rb + 4 * kt) * SF_ATOM,
                    ks * SF_ATOM, &S.full[stage]);
          for (int rb = 0; rb < nrb; ++rb)
            bulk_load(sSFB + rb * 4 * SF_ATOM,
                      p.b_sf + tl.e * sfb_expert +
                          (static_cast<size_t>(tl.nt * (BN / 128) + rb) * atoms_per_rb + 4 * kt) *
                              SF_ATOM,
                      ks * SF_ATOM, &S.full[stage]);
          armed_mask |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        *abort_flag = 1;
        set_status(p.status, MINITE_ERR_TIMEOUT);
      }
      // drain: every armed stage's copies must have landed before exit
      volatile int no_abort = 0;
      for (int s = 0; s < STAGES; ++s)
        if (armed_mask & (1u << s))
          mbar_wait(&S.full[s], (armed_parity >> s) & 1u, kDrainBudget, &no_abort);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc();
      const uint64_t adesc0 = smem_desc(smem_u32(stages), 16, 1024, kLayoutSwizzle128B);
      const uint64_t bdesc0 = smem_desc(smem_u32(stages + A_BYTES), 16, 1024, kLayoutSwizzle128B);
      int stage = 0, sfb = 0;
      uint32_t phase = 0, sf_phase = 0, acc_phase = 0;
      bool ok = true;
      bool issued = false;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        if (!mbar_wait(&S.acc_empty, acc_phase ^ 1u, budget, abort_flag)) { ok = false; break; }
        tc_fence_after();
        for (int kt = 0; kt < KT; ++kt) {
          if (!mbar_wait(&S.full[stage], phase, budget, abort_flag) ||
              !mbar_wait(&S.sf_full[sfb], sf_phase, budget, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const int ks = min(4, KSTEPS - 4 * kt);
          const uint64_t soff = static_cast<uint64_t>(stage * STAGE_BYTES) >> 4;
          const uint32_t sf_t = tmem + SF_COL0 + sfb * SF_COLS;
          for (int s = 0; s < ks; ++s)
            tc_mma_nvfp4(tmem, adesc0 + soff + 2 * s, bdesc0 + soff + 2 * s, idesc, sf_t + 4 * s,
                         sf_t + 16 + 4 * (BN / 128) * s, (kt | s) != 0);
          issued = true;
          tc_commit(&S.empty[stage]);
          tc_commit(&S.sf_empty[sfb]);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          if (++sfb == NSF) { sfb = 0; sf_phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(&S.acc_full);
        acc_phase ^= 1u;
      }
      if (!ok) {
        *abort_flag = 1;
        set_status(p.status, MINITE_ERR_TIMEOUT);
      }
      if (issued) {
        // drain: all MMAs of this thread complete before TMEM is freed
        tc_commit(&S.drain);
        volatile int no_abort = 0;
        mbar_wait(&S.drain, 0, kDrainBudget, &no_abort);
      }
    }
  } else if (warp < EPI_WARP0) {
    // ------------------------------------------------------------ scale warps
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int stage = 0, sfb = 0;
    uint32_t phase = 0, sf_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const Tile tl = decode_tile(t, n_tiles, tiles_prefix, s_off, p);
      const int nrb = min(BN / 128, rb_per_expert - tl.nt * (BN / 128));
      for (int kt = 0; kt < KT; ++kt) {
        if (!mbar_wait(&S.sf_empty[sfb], sf_phase ^ 1u, budget, abort_flag) ||
            !mbar_wait(&S.full[stage], phase, budget, abort_flag))
          ok = false;
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        const int ks = min(4, KSTEPS - 4 * kt);
        const uint8_t* sSFA = stages + stage * STAGE_BYTES + A_BYTES + B_BYTES;
        const uint8_t* sSFB = sSFA + SFA_BYTES;
        // lane i of every quarter holds atom row i: the scales of rows i, i+32, i+64, i+96
        uint32_t ra[16];
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (s < ks) v = lds128(sSFA + s * SF_ATOM + lane * 16);
          ra[4 * s] = v.x; ra[4 * s + 1] = v.y; ra[4 * s + 2] = v.z; ra[4 * s + 3] = v.w;
        }
        const uint32_t col = tmem + lane_base + SF_COL0 + sfb * SF_COLS;
        tmem_st_16cols(col, ra);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // k-steps 2h, 2h+1: columns 8s + 4rb of the B region
          uint32_t rbv[16];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int s = 2 * h + j;
#pragma unroll
            for (int rb = 0; rb < 2; ++rb) {
              uint4 v = make_uint4(0, 0, 0, 0);
              if (s < ks && rb < nrb) v = lds128(sSFB + (rb * 4 + s) * SF_ATOM + lane * 16);
              const int c = 8 * j + 4 * rb;
              rbv[c] = v.x; rbv[c + 1] = v.y; rbv[c + 2] = v.z; rbv[c + 3] = v.w;
            }
          }
          tmem_st_16cols(col + 16 + 16 * h, rbv);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.sf_full[sfb]);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        if (++sfb == NSF) { sfb = 0; sf_phase ^= 1u; }
      }
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      set_status(p.status, MINITE_ERR_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;                 // TMEM lanes this warp may access
    const int cb = (warp - EPI_WARP0) >> 2;       // accumulator columns [64 cb, 64 cb + 64)
    const int r_in_tile = quarter * 32 + lane;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = decode_tile(t, n_tiles, tiles_prefix, s_off, p);
      const bool valid = r_in_tile < tl.rows;
      const int64_t row = static_cast<int64_t>(tl.row0) + r_in_tile;
      float scale = 0.0f;
      if (valid) scale = __frcp_rn(__fmul_rn(__ldg(p.a_g + row), __ldg(p.b_g + tl.e)));
      if (!mbar_wait(&S.acc_full, acc_phase, budget, abort_flag)) ok = false;
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      acc_phase ^= 1u;
      tc_fence_after();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + cb * EPI_COLS;
      epilogue_slice(p, tbase, valid, row, tl.nt * BN + cb * EPI_COLS, scale,
                     [&] { mbar_arrive(&S.acc_empty); });
    }
    if (!ok && lane == 0) {
      *abort_flag = 1;
      set_status(p.status, MINITE_ERR_TIMEOUT);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ============================================================================
// CTA-pair building blocks (cta_group::2): a cluster of two CTAs on the two
// SMs of a TPC computes a 256 x 256 output tile (M = 256: each CTA holds 128
// rows of A; N = 256: each CTA holds 128 rows of B). The MMA thread of the
// even CTA issues for the pair; both CTAs' A/B loads count on its barriers.
// Each CTA's TMEM needs its own 128 rows' A scales and all 256 rows' B scales.
// ============================================================================

constexpr int P_A_BYTES = 128 * BK_BYTES;             // this CTA's 128 rows of A
constexpr int P_B_BYTES = 128 * BK_BYTES;             // this CTA's 128 rows of B
constexpr int P_STAGE_BYTES = P_A_BYTES + P_B_BYTES;  // 32 KB, counted on the even CTA's barrier
constexpr int P_SFA_BYTES = 4 * SF_ATOM;              // this CTA's A scales, 4 K-steps
constexpr int P_SFB_BYTES = 8 * SF_ATOM;              // both 128-row blocks of B scales
constexpr int P_SLOT_BYTES = P_SFA_BYTES + P_SFB_BYTES;  // 6 KB of scale atoms per chunk
constexpr uint32_t P_SF_COLS = 16 + 32;               // A: 4 x 4, B: 4 x 8 (256 rows)
static_assert(P_STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte swizzle alignment");
constexpr uint16_t kPairMask = 0x3;

constexpr uint32_t make_idesc_pair() {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(BN >> 3) << 17) |
         (static_cast<uint32_t>(256 >> 4) << 24);
}

struct PTile {
  int e, nt;
  int row0;      // first permuted row of the pair tile (the even CTA's first row)
  int rows;      // valid rows from row0 (<= 256)
  int sf_rb0;    // first 128-row scale block of the pair tile
  int sf_rbs;    // scale blocks of the expert from sf_rb0 on
};

// s_off = expert_offsets, s_sfb = sf_row_offsets / 128 (shared memory);
// tiles_prefix[e] = 256-row m blocks before expert e.
__device__ __forceinline__ PTile decode_pair_tile(int t, int n_tiles, const int32_t* tiles_prefix,
                                                  const int32_t* s_off, const int32_t* s_sfb,
                                                  const Params& p) {
  PTile r;
  const int mt = t / n_tiles;
  r.nt = t - mt * n_tiles;
  int lo = 0, hi = p.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tiles_prefix[mid] <= mt) lo = mid; else hi = mid;
  }
  r.e = lo;
  const int ml = mt - tiles_prefix[lo];
  r.row0 = s_off[lo] + ml * 256;
  r.rows = min(256, s_off[lo + 1] - r.row0);
  r.sf_rb0 = s_sfb[lo] + 2 * ml;
  r.sf_rbs = s_sfb[lo + 1] - r.sf_rb0;
  return r;
}

// Walks this cluster's k-tiles in order: tiles t = cid, cid + ncl, ...,
// k-tiles 0..KT-1 of each.
struct KIter {
  int t, kt, ncl, total, KT, n_tiles;
  PTile tl;
  __device__ __forceinline__ bool valid() const { return t < total; }
  const int32_t *prefix, *s_off, *s_sfb;
  __device__ __forceinline__ void start(int cid, int ncl_, int total_, int KT_, int n_tiles_,
                                        const int32_t* prefix_, const int32_t* s_off_,
                                        const int32_t* s_sfb_, const Params& p) {
    t = cid; kt = 0; ncl = ncl_; total = total_; KT = KT_; n_tiles = n_tiles_;
    prefix = prefix_; s_off = s_off_; s_sfb = s_sfb_;
    if (t < total) tl = decode_pair_tile(t, n_tiles, prefix, s_off, s_sfb, p);
  }
  __device__ __forceinline__ void advance(const Params& p) {
    if (++kt == KT) {
      kt = 0;
      t += ncl;
      if (t < total) tl = decode_pair_tile(t, n_tiles, prefix, s_off, s_sfb, p);
    }
  }
};

constexpr int Q_CH = 2;                                  // 128-byte K chunks per stage
constexpr int Q_SFA_BYTES = 4 * Q_CH * SF_ATOM;          // 4 KB: 8 k-steps of A scales
constexpr int Q_SFB_BYTES = 2 * 4 * Q_CH * SF_ATOM;      // 8 KB: 8 k-steps of both B blocks
constexpr int Q_SLOT_BYTES = Q_SFA_BYTES + Q_SFB_BYTES;  // 12 KB
constexpr int Q_SF_WARP = NUM_WARPS;                     // the scale-slot producer warp
constexpr int Q_THREADS = (NUM_WARPS + 1) * 32;

// ============================================================================
// Single-CTA kernel with two-chunk stages: the 128 x 256 tile of the
// single-CTA kernel, with each stage covering two 128-byte K chunks (eight
// MMAs, 1024 tensor cycles) loaded by one 3-D box per operand, so that the
// producer spends two copy instructions per 1024 tensor cycles instead of
// five per 512. Scale atoms come from a separate scale-producer warp, three
// copies per stage (A: 8 atoms; B: 8 atoms of each 128-row block) into two
// 12 KB slots, which the scale warps walk chunk by chunk into the TMEM ring.
// ============================================================================

constexpr int D_STAGES = 2;
constexpr int D_A_BYTES = Q_CH * A_BYTES;                 // 32 KB
constexpr int D_B_BYTES = Q_CH * B_BYTES;                 // 64 KB
constexpr int D_STAGE_BYTES = D_A_BYTES + D_B_BYTES;      // 96 KB
constexpr int D_SLOTS = 2;
static_assert(D_STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte swizzle alignment");

struct DSmem {
  uint64_t full[D_STAGES];
  uint64_t empty[D_STAGES];
  uint64_t sfdata[D_SLOTS];
  uint64_t sfread[D_SLOTS];
  uint64_t sf_full[NSF];
  uint64_t sf_empty[NSF];
  uint64_t acc_full;
  uint64_t acc_empty;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int total_tiles;
  int pad_;
};

// Walks this CTA's (tile, stage) pairs in order; a tile has
// ceil(tl.kt / Q_CH) stages.
template <bool WG>
struct DIter {
  int t, kd, ncl, total, n_tiles;
  Tile tl;
  const int32_t *prefix, *s_off;
  __device__ __forceinline__ bool valid() const { return t < total; }
  __device__ __forceinline__ int stages() const { return (tl.kt + Q_CH - 1) / Q_CH; }
  __device__ __forceinline__ void start(int t0, int ncl_, int total_, int n_tiles_,
                                        const int32_t* prefix_, const int32_t* s_off_,
                                        const Params& p) {
    t = t0; kd = 0; ncl = ncl_; total = total_; n_tiles = n_tiles_;
    prefix = prefix_; s_off = s_off_;
    if (t < total) tl = decode_any<WG>(t, n_tiles, prefix, s_off, p);
  }
  __device__ __forceinline__ void advance(const Params& p) {
    if (++kd == stages()) {
      kd = 0;
      t += ncl;
      if (t < total) tl = decode_any<WG>(t, n_tiles, prefix, s_off, p);
    }
  }
};

// WG: weight-gradient mode. A [M channels, K tokens] and B [N channels, K
// tokens] are token-axis operands whose expert e occupies token columns
// [kofs[e], kofs[e + 1]) (p.offsets = kofs); the tile (e, A rows, B columns)
// sums over that range and is written to out[e]; the scale is
// 1 / (a_g[e] * b_g[e]).
template <bool WG>
__global__ void __maxnreg__(80)
grouped_gemm_dc_kernel(const __grid_constant__ CUtensorMap tmap_a,
                       const __grid_constant__ CUtensorMap tmap_b, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* slots = stages + D_STAGES * D_STAGE_BYTES;
  DSmem& S = *reinterpret_cast<DSmem*>(slots + D_SLOTS * Q_SLOT_BYTES);
  int32_t* tiles_prefix = reinterpret_cast<int32_t*>(&S + 1);   // [E+1]
  int32_t* s_off = tiles_prefix + (p.E + 1);                    // [E+1] expert_offsets (WG: kofs)

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int atoms_per_rb = p.K / 64;       // scale atoms per 128-row block of A or B
  const int n_tiles = (p.N + BN - 1) / BN;
  const int rb_per_expert = (p.N + 127) / 128;
  const size_t sfb_expert = static_cast<size_t>(rb_per_expert) * atoms_per_rb * SF_ATOM;

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    for (int s = 0; s < D_STAGES; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int s = 0; s < D_SLOTS; ++s) {
      mbar_init(&S.sfdata[s], 1);
      mbar_init(&S.sfread[s], 4);
    }
    for (int b = 0; b < NSF; ++b) {
      mbar_init(&S.sf_full[b], 4);
      mbar_init(&S.sf_empty[b], 1);
    }
    mbar_init(&S.acc_full, 1);
    mbar_init(&S.acc_empty, NUM_EPI_WARPS);
    mbar_init(&S.drain, 1);
    S.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(&S.tmem_base, TMEM_COLS);
  // everything above touches only this CTA's shared memory and TMEM
  pdl_wait();
  if (warp == 2) {
    // m-block prefix over experts, validating the device offsets on the way
    int carry = 0;
    bool bad = false;
    if (lane == 0) tiles_prefix[0] = 0;
    for (int base = 0; base < p.E; base += 32) {
      const int e = base + lane;
      int cnt = 0;
      if (e < p.E) {
        const int o0 = __ldg(p.offsets + e), o1 = __ldg(p.offsets + e + 1);
        s_off[e + 1] = o1;
        if (e == 0) s_off[0] = o0;
        cnt = o1 - o0;
        if constexpr (WG) {
          // token ranges: from 0, multiples of 256, within the K columns
          if (cnt < 0 || cnt % 256 != 0 || (e == 0 && o0 != 0) || (e == p.E - 1 && o1 > p.K))
            bad = true;
          cnt = cnt > 0 ? static_cast<int>((p.M + BM - 1) / BM) : 0;
        } else {
          const int s0 = __ldg(p.sf_offsets + e), s1 = __ldg(p.sf_offsets + e + 1);
          if (cnt < 0 || s1 - s0 != ((cnt + 127) & ~127) || (e == 0 && (o0 != 0 || s0 != 0)) ||
              (e == p.E - 1 && o1 > p.M))
            bad = true;
          cnt = cnt > 0 ? (cnt + BM - 1) / BM : 0;
        }
      }
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (e < p.E) tiles_prefix[e + 1] = carry + incl;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      S.total_tiles = bad ? 0 : carry * n_tiles;
      if (bad && blockIdx.x == 0) set_status(p.status, MINITE_ERR_INVALID_ARG);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem = S.tmem_base;
  const int total = S.total_tiles;
  volatile int* abort_flag = &S.abort_flag;
  const uint64_t budget = p.budget_ns;
  constexpr uint64_t kDrainBudget = 200000000ull;
  auto fail = [&](int code) {
    *abort_flag = 1;
    set_status(p.status, code);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ A/B producer
    if (lane == 0) {
      uint32_t armed_mask = 0, armed_parity = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      DIter<WG> it;
      it.start(blockIdx.x, gridDim.x, total, n_tiles, tiles_prefix, s_off, p);
      while (it.valid()) {
        if (!mbar_wait(&S.empty[stage], phase ^ 1u, budget, abort_flag)) { ok = false; break; }
        uint8_t* sA = stages + stage * D_STAGE_BYTES;
        uint8_t* sB = sA + D_A_BYTES;
        const int z = it.tl.kz0 + Q_CH * it.kd;
        // a tile's last stage may hold one chunk: its second box lies in the
        // next expert's range (or past the columns, zero-filled) and is unused
        mbar_arrive_expect_tx(&S.full[stage], D_STAGE_BYTES);
        tma_load_3d(sA, &tmap_a, &S.full[stage], 0, it.tl.row0, z);
        tma_load_3d(sB, &tmap_b, &S.full[stage], 0,
                    (WG ? 0 : it.tl.e * p.N) + it.tl.nt * BN, z);
        armed_mask |= 1u << stage;
        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == D_STAGES) { stage = 0; phase ^= 1u; }
        it.advance(p);
      }
      if (!ok) fail(MINITE_ERR_TIMEOUT);
      volatile int no_abort = 0;
      for (int s = 0; s < D_STAGES; ++s)
        if (armed_mask & (1u << s))
          mbar_wait(&S.full[s], (armed_parity >> s) & 1u, kDrainBudget, &no_abort);
    }
  } else if (warp == Q_SF_WARP) {
    // ------------------------------------------------------------ scale-slot producer
    if (lane == 0) {
      uint32_t slot_mask = 0, slot_parity = 0;
      int slot = 0;
      uint32_t slot_phase = 0;
      bool ok = true;
      DIter<WG> it;
      it.start(blockIdx.x, gridDim.x, total, n_tiles, tiles_prefix, s_off, p);
      while (it.valid()) {
        if (!mbar_wait(&S.sfread[slot], slot_phase ^ 1u, budget, abort_flag)) { ok = false; break; }
        const Tile& tl = it.tl;
        const int na = min(4 * Q_CH, 4 * tl.kt - 4 * Q_CH * it.kd);  // atoms (k-steps) in this stage
        const int a0 = 4 * tl.kz0 + 4 * Q_CH * it.kd;               // first atom of the stage
        const int nrb = min(BN / 128, rb_per_expert - tl.nt * (BN / 128));
        uint8_t* sSFA = slots + slot * Q_SLOT_BYTES;
        uint8_t* sSFB = sSFA + Q_SFA_BYTES;
        mbar_arrive_expect_tx(&S.sfdata[slot], static_cast<uint32_t>(na * (1 + nrb)) * SF_ATOM);
        bulk_load(sSFA, p.a_sf + (static_cast<size_t>(tl.sf_rb) * atoms_per_rb + a0) * SF_ATOM,
                  na * SF_ATOM, &S.sfdata[slot]);
        for (int rb = 0; rb < nrb; ++rb)
          bulk_load(sSFB + rb * 4 * Q_CH * SF_ATOM,
                    p.b_sf + (WG ? 0 : tl.e * sfb_expert) +
                        (static_cast<size_t>(tl.nt * (BN / 128) + rb) * atoms_per_rb + a0) *
                            SF_ATOM,
                    na * SF_ATOM, &S.sfdata[slot]);
        slot_mask |= 1u << slot;
        slot_parity = (slot_parity & ~(1u << slot)) | (slot_phase << slot);
        if (++slot == D_SLOTS) { slot = 0; slot_phase ^= 1u; }
        it.advance(p);
      }
      if (!ok) fail(MINITE_ERR_TIMEOUT);
      volatile int no_abort = 0;
      for (int s = 0; s < D_SLOTS; ++s)
        if (slot_mask & (1u << s))
          mbar_wait(&S.sfdata[s], (slot_parity >> s) & 1u, kDrainBudget, &no_abort);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc();
      const uint64_t adesc0 = smem_desc(smem_u32(stages), 16, 1024, kLayoutSwizzle128B);
      const uint64_t bdesc0 = smem_desc(smem_u32(stages + D_A_BYTES), 16, 1024, kLayoutSwizzle128B);
      int stage = 0, sfb = 0;
      uint32_t phase = 0, sf_phase = 0, acc_phase = 0;
      bool ok = true;
      bool issued = false;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile tl = decode_any<WG>(t, n_tiles, tiles_prefix, s_off, p);
        const int KT = tl.kt, KD = (tl.kt + Q_CH - 1) / Q_CH, KSTEPS = 4 * tl.kt;
        if (!mbar_wait(&S.acc_empty, acc_phase ^ 1u, budget, abort_flag)) { ok = false; break; }
        tc_fence_after();
        for (int kd = 0; kd < KD && ok; ++kd) {
          if (!mbar_wait(&S.full[stage], phase, budget, abort_flag)) { ok = false; break; }
          const int nch = min(Q_CH, KT - Q_CH * kd);
          for (int c = 0; c < nch; ++c) {
            if (!mbar_wait(&S.sf_full[sfb], sf_phase, budget, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const int kt = Q_CH * kd + c;
            const int ks = min(4, KSTEPS - 4 * kt);
            const uint64_t aoff = static_cast<uint64_t>(stage * D_STAGE_BYTES + c * A_BYTES) >> 4;
            const uint64_t boff = static_cast<uint64_t>(stage * D_STAGE_BYTES + c * B_BYTES) >> 4;
            const uint32_t sf_t = tmem + SF_COL0 + sfb * SF_COLS;
            for (int s = 0; s < ks; ++s)
              tc_mma_nvfp4(tmem, adesc0 + aoff + 2 * s, bdesc0 + boff + 2 * s, idesc, sf_t + 4 * s,
                           sf_t + 16 + 4 * (BN / 128) * s, (kt | s) != 0);
            issued = true;
            tc_commit(&S.sf_empty[sfb]);
            if (++sfb == NSF) { sfb = 0; sf_phase ^= 1u; }
          }
          if (!ok) break;
          tc_commit(&S.empty[stage]);
          if (++stage == D_STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(&S.acc_full);
        acc_phase ^= 1u;
      }
      if (!ok) fail(MINITE_ERR_TIMEOUT);
      if (issued) {
        // drain: all MMAs of this thread complete before TMEM is freed
        tc_commit(&S.drain);
        volatile int no_abort = 0;
        mbar_wait(&S.drain, 0, kDrainBudget, &no_abort);
      }
    }
  } else if (warp < EPI_WARP0) {
    // ------------------------------------------------------------ scale warps
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int slot = 0, sfb = 0;
    uint32_t slot_phase = 0, sf_phase = 0;
    bool ok = true;
    DIter<WG> it;
    it.start(blockIdx.x, gridDim.x, total, n_tiles, tiles_prefix, s_off, p);
    while (it.valid() && ok) {
      const int nrb = min(BN / 128, rb_per_expert - it.tl.nt * (BN / 128));
      const int nch = min(Q_CH, it.tl.kt - Q_CH * it.kd);
      const int KSTEPS = 4 * it.tl.kt;
      if (!mbar_wait(&S.sfdata[slot], slot_phase, budget, abort_flag)) ok = false;
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      const uint8_t* sSFA = slots + slot * Q_SLOT_BYTES;
      const uint8_t* sSFB = sSFA + Q_SFA_BYTES;
      for (int c = 0; c < nch; ++c) {
        const int ks = min(4, KSTEPS - 4 * (Q_CH * it.kd + c));
        // lane i of every quarter holds atom row i: the scales of rows i, i+32, i+64, i+96
        uint32_t ra[16];
#pragma unroll
        for (int st = 0; st < 4; ++st) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (st < ks) v = lds128(sSFA + (4 * c + st) * SF_ATOM + lane * 16);
          ra[4 * st] = v.x; ra[4 * st + 1] = v.y; ra[4 * st + 2] = v.z; ra[4 * st + 3] = v.w;
        }
        uint32_t rbv[2][16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          // k-steps 2h, 2h+1: columns 8s + 4rb of the B region
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int st = 2 * h + j;
#pragma unroll
            for (int rb = 0; rb < 2; ++rb) {
              uint4 v = make_uint4(0, 0, 0, 0);
              if (st < ks && rb < nrb)
                v = lds128(sSFB + (rb * 4 * Q_CH + 4 * c + st) * SF_ATOM + lane * 16);
              const int cc = 8 * j + 4 * rb;
              rbv[h][cc] = v.x; rbv[h][cc + 1] = v.y; rbv[h][cc + 2] = v.z; rbv[h][cc + 3] = v.w;
            }
          }
        }
        if (c == nch - 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.sfread[slot]);
        }
        if (!mbar_wait(&S.sf_empty[sfb], sf_phase ^ 1u, budget, abort_flag)) ok = false;
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        const uint32_t col = tmem + lane_base + SF_COL0 + sfb * SF_COLS;
        tmem_st_16cols(col, ra);
        tmem_st_16cols(col + 16, rbv[0]);
        tmem_st_16cols(col + 32, rbv[1]);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.sf_full[sfb]);
        if (++sfb == NSF) { sfb = 0; sf_phase ^= 1u; }
      }
      if (++slot == D_SLOTS) { slot = 0; slot_phase ^= 1u; }
      it.advance(p);
    }
    if (!ok && lane == 0) fail(MINITE_ERR_TIMEOUT);
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;                 // TMEM lanes this warp may access
    const int cb = (warp - EPI_WARP0) >> 2;       // accumulator columns [64 cb, 64 cb + 64)
    const int r_in_tile = quarter * 32 + lane;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const Tile tl = decode_any<WG>(t, n_tiles, tiles_prefix, s_off, p);
      const bool valid = r_in_tile < tl.rows;
      const int64_t row = static_cast<int64_t>(tl.row0) + r_in_tile +
                          (WG ? static_cast<int64_t>(tl.e) * p.M : 0);  // output row
      float scale = 0.0f;
      if (valid)
        scale = __frcp_rn(__fmul_rn(__ldg(p.a_g + (WG ? tl.e : row)), __ldg(p.b_g + tl.e)));
      if (!mbar_wait(&S.acc_full, acc_phase, budget, abort_flag)) ok = false;
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      acc_phase ^= 1u;
      tc_fence_after();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + cb * EPI_COLS;
      epilogue_slice(p, tbase, valid, row, tl.nt * BN + cb * EPI_COLS, scale,
                     [&] { mbar_arrive(&S.acc_empty); });
    }
    if (!ok && lane == 0) fail(MINITE_ERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ============================================================================
// CTA-pair kernel with a deep operand pipeline (default for the forward and
// dgrad GEMMs). The pair's two SMs compute a 256 x 256 tile with
// tcgen05.mma.cta_group::2: each CTA holds 128 rows of A and 128 of the 256
// B rows, so an SM streams 32 KB of operands per 128-byte K chunk instead of
// the 48 KB of a single-CTA 128 x 256 tile (64 instead of 96 bytes per
// tensor cycle). A chunk's scale atoms travel in the same pipeline stage as
// its A/B tiles and are written to the TMEM slot of that stage, so the stage
// count (five) is also the scale look-ahead, and a stage's MMA commit frees
// its shared memory and its TMEM scale slot at once. Copy instructions are
// split between two producer threads (A/B tiles; scale atoms) so that
// neither issues more than three per chunk.
//
// Per chunk and stage s:
//   warp 0 (each CTA): waits empty[s]; two TMA boxes (A rows, B rows) whose
//     bytes count on the leader's full[s] (the leader arms it for both CTAs).
//   warp 22 (each CTA): waits empty[s]; bulk copies of this CTA's A atoms and
//     both 128-row blocks of B atoms, counted on its own sfdata[s].
//   warps 2..5 (each CTA): wait sfdata[s]; write the atoms into TMEM slot s
//     (tcgen05.st, replicated into the four lane quarters); arrive on the
//     leader's sf_full[s] (eight arrivals: four warps per CTA).
//   warp 1 of the leader (the whole warp, one elected lane issuing): waits
//     full[s] and sf_full[s]; four pair MMAs; commits empty[s] to both CTAs.
//   warps 6..21 (each CTA): after the tile's last commit (acc_full), drain
//     the 128 x 256 accumulator of this CTA's rows, arrive on the leader's
//     acc_empty (32 arrivals), then scale, convert and store: with c_tma
//     (BF16 output, staging fits) each warp writes its 32 rows x 64 columns
//     as two 32 x 32 TMA boxes through its 2 KB of staging, rows past the
//     expert's end by transposed plain stores.
// ============================================================================

constexpr int R_STAGES = 5;
constexpr int R_AB_BYTES = P_STAGE_BYTES;   // 32 KB: this CTA's A and B rows of one chunk
constexpr int R_SF_BYTES = P_SLOT_BYTES;    // 6 KB: this CTA's A atoms, both B blocks' atoms
constexpr int R_SF_WARP = NUM_WARPS;        // warp 22: scale-copy producer
constexpr int R_THREADS = (NUM_WARPS + 1) * 32;
constexpr int R_C_WARP_BYTES = 2048;                  // 32 rows x 32 BF16 columns
constexpr int R_C_BYTES = NUM_EPI_WARPS * R_C_WARP_BYTES;
static_assert(SF_COL0 + R_STAGES * P_SF_COLS <= TMEM_COLS, "TMEM budget");
static_assert(R_SF_BYTES % 16 == 0, "bulk copy alignment");

struct RSmem {
  uint64_t full[R_STAGES];     // leader: both CTAs' A/B bytes of the stage
  uint64_t empty[R_STAGES];    // both CTAs: the stage's MMAs completed
  uint64_t sfdata[R_STAGES];   // both CTAs: this CTA's scale bytes of the stage
  uint64_t sf_full[R_STAGES];  // leader: both CTAs' scale warps filled TMEM slot s
  uint64_t acc_full;           // both CTAs: the tile's MMAs completed
  uint64_t acc_empty;          // leader: every epilogue warp of both CTAs drained
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int total_tiles;
  int pad_;
};

// 80 registers: the 23 warps spread over the SM's four sub-partitions put six
// on one of them, and 6 x 32 x 80 = 15360 of its 16384 registers is the most
// that fits (88 would not).
template <bool SWIGLU>
__global__ void __maxnreg__(80)
grouped_gemm_pair_deep_kernel(const __grid_constant__ CUtensorMap tmap_a,
                              const __grid_constant__ CUtensorMap tmap_b,
                              const __grid_constant__ CUtensorMap tmap_c, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sf_area = stages + R_STAGES * R_AB_BYTES;
  uint8_t* c_area = sf_area + R_STAGES * R_SF_BYTES;   // c_tma: R_C_WARP_BYTES per epilogue warp
  RSmem& S = *reinterpret_cast<RSmem*>(c_area + (!SWIGLU && p.c_tma ? R_C_BYTES : 0));
  int32_t* tiles_prefix = reinterpret_cast<int32_t*>(&S + 1);   // [E+1]
  int32_t* s_off = tiles_prefix + (p.E + 1);                    // [E+1] expert_offsets
  int32_t* s_sfb = s_off + (p.E + 1);                           // [E+1] sf_row_offsets / 128
  float* lut = reinterpret_cast<float*>(
      (reinterpret_cast<uintptr_t>(s_sfb + (p.E + 1)) + 15) & ~uintptr_t(15));  // SWIGLU: silu table
  float* epi_part = lut + kLut24Entries;   // SWIGLU: [2][4 quarters][4 warps][32] row partial maxima

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(num_clusters_x());
  const int KT = (p.K + 255) / 256;
  const int KSTEPS = p.K / 64;
  const int atoms_per_rb = p.K / 64;
  const int n_tiles = (p.N + BN - 1) / BN;
  const int rb_per_expert = (p.N + 127) / 128;
  const size_t sfb_expert = static_cast<size_t>(rb_per_expert) * atoms_per_rb * SF_ATOM;

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    for (int s = 0; s < R_STAGES; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
      mbar_init(&S.sfdata[s], 1);
      mbar_init(&S.sf_full[s], 8);
    }
    mbar_init(&S.acc_full, 1);
    mbar_init(&S.acc_empty, 2 * NUM_EPI_WARPS);
    mbar_init(&S.drain, 1);
    S.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc_pair(&S.tmem_base, TMEM_COLS);
  if constexpr (SWIGLU) build_silu_lut24_part(lut, threadIdx.x, R_THREADS);
  // everything above touches only this CTA's shared memory and TMEM
  pdl_wait();
  if (warp == 2) {
    // 256-row m-block prefix over experts, validating the device offsets
    int carry = 0;
    bool bad = false;
    if (lane == 0) tiles_prefix[0] = 0;
    for (int base = 0; base < p.E; base += 32) {
      const int e = base + lane;
      int cnt = 0;
      if (e < p.E) {
        const int o0 = __ldg(p.offsets + e), o1 = __ldg(p.offsets + e + 1);
        const int s0 = __ldg(p.sf_offsets + e), s1 = __ldg(p.sf_offsets + e + 1);
        s_off[e + 1] = o1;
        s_sfb[e + 1] = s1 / 128;
        if (e == 0) { s_off[0] = o0; s_sfb[0] = s0 / 128; }
        cnt = o1 - o0;
        if (cnt < 0 || s1 - s0 != ((cnt + 127) & ~127) || (e == 0 && (o0 != 0 || s0 != 0)) ||
            (e == p.E - 1 && o1 > p.M))
          bad = true;
        cnt = cnt > 0 ? (cnt + 255) / 256 : 0;
      }
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      if (e < p.E) tiles_prefix[e + 1] = carry + incl;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      S.total_tiles = bad ? 0 : carry * n_tiles;
      if (bad && blockIdx.x == 0) set_status(p.status, MINITE_ERR_INVALID_ARG);
    }
  }
  // both CTAs' barriers exist and TMEM is allocated before any cross-CTA traffic
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();

  const uint32_t tmem = S.tmem_base;
  const int total = S.total_tiles;
  volatile int* abort_flag = &S.abort_flag;
  const uint32_t peer_abort = mapa_shared(smem_u32(&S.abort_flag), rank ^ 1u);
  const uint32_t leader_full0 = mapa_shared(smem_u32(&S.full[0]), 0);
  const uint32_t leader_sf_full0 = mapa_shared(smem_u32(&S.sf_full[0]), 0);
  const uint32_t leader_acc_empty = mapa_shared(smem_u32(&S.acc_empty), 0);
  const uint64_t budget = p.budget_ns;
  constexpr uint64_t kDrainBudget = 200000000ull;
  auto fail = [&](int code) {
    *abort_flag = 1;
    st_shared_cluster(peer_abort, 1u);
    set_status(p.status, code);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ A/B producer
    if (lane == 0) {
      uint32_t armed_mask = 0, armed_parity = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      KIter it;
      it.start(cid, ncl, total, KT, n_tiles, tiles_prefix, s_off, s_sfb, p);
      while (it.valid()) {
        if (!mbar_wait(&S.empty[stage], phase ^ 1u, budget, abort_flag)) { ok = false; break; }
        uint8_t* sA = stages + stage * R_AB_BYTES;
        uint8_t* sB = sA + P_A_BYTES;
        if (rank == 0) mbar_arrive_expect_tx(&S.full[stage], 2 * R_AB_BYTES);
        const uint32_t fb = leader_full0 + 8u * stage;
        tma_load_2d_pair(sA, &tmap_a, fb, it.kt * BK_BYTES,
                         it.tl.row0 + 128 * static_cast<int>(rank));
        // SWIGLU: the even CTA loads gate rows [128 nt, +128), the odd CTA the
        // up rows [I + 128 nt, +128) of the expert's [2I, K] weight
        const int b_row = SWIGLU ? it.tl.e * p.N + static_cast<int>(rank) * (p.N / 2) + it.tl.nt * 128
                                 : it.tl.e * p.N + it.tl.nt * BN + 128 * static_cast<int>(rank);
        tma_load_2d_pair(sB, &tmap_b, fb, it.kt * BK_BYTES, b_row);
        armed_mask |= 1u << stage;
        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == R_STAGES) { stage = 0; phase ^= 1u; }
        it.advance(p);
      }
      if (!ok) fail(MINITE_ERR_TIMEOUT);
      volatile int no_abort = 0;
      if (rank == 0) {
        // both CTAs' A/B copies count on these barriers: all armed stages landed
        for (int s = 0; s < R_STAGES; ++s)
          if (armed_mask & (1u << s))
            mbar_wait(&S.full[s], (armed_parity >> s) & 1u, kDrainBudget, &no_abort);
      } else if (!ok) {
        // this CTA's copies count on the other CTA's barriers: give any copy
        // still in flight time to land before the CTA can exit
        const uint64_t t0 = globaltimer();
        while (globaltimer() - t0 < 100000ull) {}
      }
    }
  } else if (warp == R_SF_WARP) {
    // ------------------------------------------------------------ scale-copy producer
    if (lane == 0) {
      uint32_t armed_mask = 0, armed_parity = 0;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      KIter it;
      it.start(cid, ncl, total, KT, n_tiles, tiles_prefix, s_off, s_sfb, p);
      while (it.valid()) {
        if (!mbar_wait(&S.empty[stage], phase ^ 1u, budget, abort_flag)) { ok = false; break; }
        const PTile& tl = it.tl;
        const int ks = min(4, KSTEPS - 4 * it.kt);
        const bool a_ok = static_cast<int>(rank) < tl.sf_rbs;   // this CTA's A block exists
        const int nrb = SWIGLU ? 2 : min(2, rb_per_expert - tl.nt * 2);  // B blocks inside the weight
        uint8_t* sSFA = sf_area + stage * R_SF_BYTES;
        uint8_t* sSFB = sSFA + P_SFA_BYTES;
        mbar_arrive_expect_tx(&S.sfdata[stage],
                              static_cast<uint32_t>(ks * ((a_ok ? 1 : 0) + nrb)) * SF_ATOM);
        if (a_ok)
          bulk_load(sSFA,
                    p.a_sf + (static_cast<size_t>(tl.sf_rb0 + static_cast<int>(rank)) * atoms_per_rb +
                              4 * it.kt) * SF_ATOM,
                    ks * SF_ATOM, &S.sfdata[stage]);
        for (int rb = 0; rb < nrb; ++rb) {
          // SWIGLU: the gate block nt, then the up block I / 128 + nt
          const int brb = SWIGLU ? (rb == 0 ? tl.nt : p.N / 256 + tl.nt) : tl.nt * 2 + rb;
          bulk_load(sSFB + rb * 4 * SF_ATOM,
                    p.b_sf + tl.e * sfb_expert +
                        (static_cast<size_t>(brb) * atoms_per_rb + 4 * it.kt) * SF_ATOM,
                    ks * SF_ATOM, &S.sfdata[stage]);
        }
        armed_mask |= 1u << stage;
        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == R_STAGES) { stage = 0; phase ^= 1u; }
        it.advance(p);
      }
      if (!ok) fail(MINITE_ERR_TIMEOUT);
      // this CTA's scale copies count on its own barriers
      volatile int no_abort = 0;
      for (int s = 0; s < R_STAGES; ++s)
        if (armed_mask & (1u << s))
          mbar_wait(&S.sfdata[s], (armed_parity >> s) & 1u, kDrainBudget, &no_abort);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    // The whole warp runs the loop, so the stage, the phases and every
    // descriptor are warp-uniform values; every lane takes the barrier waits
    // (one instruction for the warp) and one elected lane issues the MMAs and
    // commits. Issued from a one-lane branch instead, the per-chunk loop took
    // ~165 cycles per MMA, above the tensor pipe's 128.
    if (rank == 0) {
      constexpr uint32_t idesc = make_idesc_pair();
      const uint64_t adesc0 = smem_desc(smem_u32(stages), 16, 1024, kLayoutSwizzle128B);
      const uint64_t bdesc0 = smem_desc(smem_u32(stages + P_A_BYTES), 16, 1024, kLayoutSwizzle128B);
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      bool issued = false;
      for (int t = cid; t < total && ok; t += ncl) {
        if (!__all_sync(0xffffffffu, mbar_wait(&S.acc_empty, acc_phase ^ 1u, budget, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kt = 0; kt < KT; ++kt) {
          const bool w_ok = mbar_wait(&S.full[stage], phase, budget, abort_flag) &&
                            mbar_wait(&S.sf_full[stage], phase, budget, abort_flag);
          if (!__all_sync(0xffffffffu, w_ok)) { ok = false; break; }
          tc_fence_after();
          const int ks = min(4, KSTEPS - 4 * kt);
          const uint64_t soff = static_cast<uint64_t>(stage * R_AB_BYTES) >> 4;
          const uint32_t sf_t = tmem + SF_COL0 + stage * P_SF_COLS;
          if (elect_one()) {
#pragma unroll
            for (int s = 0; s < 4; ++s)
              if (s < ks)
                tc_mma_nvfp4_pair(tmem, adesc0 + soff + 2 * s, bdesc0 + soff + 2 * s, idesc,
                                  sf_t + 4 * s, sf_t + 16 + 8 * s, (kt | s) != 0);
            tc_commit_pair_mc(&S.empty[stage], kPairMask);
          }
          __syncwarp();
          issued = true;
          if (++stage == R_STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (elect_one()) tc_commit_pair_mc(&S.acc_full, kPairMask);
        __syncwarp();
        acc_phase ^= 1u;
      }
      if (!ok && lane == 0) fail(MINITE_ERR_TIMEOUT);
      if (issued) {
        // all MMAs complete before TMEM is freed
        if (elect_one()) tc_commit_pair_mc(&S.drain, 0x1);
        __syncwarp();
        volatile int no_abort = 0;
        mbar_wait(&S.drain, 0, kDrainBudget, &no_abort);
      }
    }
  } else if (warp < EPI_WARP0) {
    // ------------------------------------------------------------ scale warps
    const int quarter = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    KIter it;
    it.start(cid, ncl, total, KT, n_tiles, tiles_prefix, s_off, s_sfb, p);
    while (it.valid()) {
      const bool a_ok = static_cast<int>(rank) < it.tl.sf_rbs;
      const int nrb = SWIGLU ? 2 : min(2, rb_per_expert - it.tl.nt * 2);
      const int ks = min(4, KSTEPS - 4 * it.kt);
      if (!mbar_wait(&S.sfdata[stage], phase, budget, abort_flag)) ok = false;
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      const uint8_t* sSFA = sf_area + stage * R_SF_BYTES;
      const uint8_t* sSFB = sSFA + P_SFA_BYTES;
      // lane i of every quarter holds atom row i: the scales of rows i, i+32, i+64, i+96
      uint32_t ra[16], rbv[32];
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (a_ok && s < ks) v = lds128(sSFA + s * SF_ATOM + lane * 16);
        ra[4 * s] = v.x; ra[4 * s + 1] = v.y; ra[4 * s + 2] = v.z; ra[4 * s + 3] = v.w;
#pragma unroll
        for (int rb = 0; rb < 2; ++rb) {
          uint4 w = make_uint4(0, 0, 0, 0);
          if (rb < nrb && s < ks) w = lds128(sSFB + (rb * 4 + s) * SF_ATOM + lane * 16);
          const int c = 8 * s + 4 * rb;
          rbv[c] = w.x; rbv[c + 1] = w.y; rbv[c + 2] = w.z; rbv[c + 3] = w.w;
        }
      }
      // TMEM slot `stage` is free: its previous chunk's MMAs completed before
      // the scale producer could refill this stage (both wait on empty[stage])
      const uint32_t col = tmem + lane_base + SF_COL0 + stage * P_SF_COLS;
      tmem_st_16cols(col, ra);
      tmem_st_16cols(col + 16, *reinterpret_cast<const uint32_t(*)[16]>(&rbv[0]));
      tmem_st_16cols(col + 32, *reinterpret_cast<const uint32_t(*)[16]>(&rbv[16]));
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(&S.sf_full[stage]);
        else mbar_arrive_remote(leader_sf_full0 + 8u * stage);
      }
      if (++stage == R_STAGES) { stage = 0; phase ^= 1u; }
      it.advance(p);
    }
    if (!ok && lane == 0) fail(MINITE_ERR_TIMEOUT);
  } else if (SWIGLU && warp < EPI_WARP0 + NUM_EPI_WARPS) {
    // ------------------------------------------------------------ fused SwiGLU epilogue
    // Warp (quarter, cb) holds TMEM lanes 32 quarter.. of this CTA: gate
    // columns [32 cb, +32) and the matching up columns [128 + 32 cb, +32),
    // i.e. intermediate columns 128 nt + 32 cb + [0, 32) of its row, two
    // NVFP4 blocks. A row's global scale needs the |h| maximum over all I
    // columns, spread over the n_tiles CTA tiles of its m-block, which
    // n_tiles clusters run at the same time: the four warps of a quarter
    // combine their partial maxima in shared memory, one of them publishes the
    // CTA's value in the row's slot nt (bit 31 set marks it written; the
    // maxima are non-negative floats), and every warp polls its rows' n_tiles
    // slots before quantizing. A warp that hits a timeout stops working but
    // keeps the quarter's barrier cadence, so no barrier is left waiting.
    const int quarter = warp & 3;
    const int cb = (warp - EPI_WARP0) >> 2;
    const int r_in_tile = static_cast<int>(rank) * 128 + quarter * 32 + lane;
    const uint32_t qbar = 2 + static_cast<uint32_t>(quarter);   // named barrier of the quarter
    const SwigluParams& sw = p.sw;
    const int I = sw.I;
    const int kc = I / 16;
    const int stride = (n_tiles + 3) & ~3;                        // slot words per row
    uint32_t acc_phase = 0;
    int it = 0;
    bool failed = false;
    for (int t = cid; t < total; t += ncl, ++it) {
      const PTile tl = decode_pair_tile(t, n_tiles, tiles_prefix, s_off, s_sfb, p);
      const bool valid = r_in_tile < tl.rows;
      const int64_t row = static_cast<int64_t>(tl.row0) + r_in_tile;
      float scale = 0.0f, w = 1.0f;
      if (valid) {
        scale = __frcp_rn(__fmul_rn(__ldg(p.a_g + row), __ldg(p.b_g + tl.e)));
        if (sw.perm_w) w = __ldg(sw.perm_w + row);
      }
      bool ok = !failed &&
                __all_sync(0xffffffffu, mbar_wait(&S.acc_full, acc_phase, budget, abort_flag));
      if (!ok && !failed) {
        failed = true;
        if (lane == 0) fail(MINITE_ERR_TIMEOUT);
      }
      float h[2][16];
      float part = 0.0f;
      if (ok) {
        acc_phase ^= 1u;
        tc_fence_after();
        const uint32_t tb = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + 32 * cb;
        // 8 gate and 8 up columns at a time: the BF16 values the plain GEMM
        // would store (kept in gate_up when asked), then h; nothing else stays
        // live between steps, so the 80 registers hold without spilling
        uint16_t* o = static_cast<uint16_t*>(p.out) + row * p.N + tl.nt * 128 + 32 * cb;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          uint32_t rg[8], ru[8];
          tmem_ld_8cols_x2(tb + 8 * b, tb + 128 + 8 * b, rg, ru);
          if (b == 3) {
            // every accumulator column this warp reads is in registers
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              if (rank == 0) mbar_arrive(&S.acc_empty);
              else mbar_arrive_remote(leader_acc_empty);
            }
          }
          uint32_t gw[4], uw[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float g0 = __uint_as_float(rg[2 * j]), g1 = __uint_as_float(rg[2 * j + 1]);
            float u0 = __uint_as_float(ru[2 * j]), u1 = __uint_as_float(ru[2 * j + 1]);
            mul_f32x2(g0, g1, scale, scale);
            mul_f32x2(u0, u1, scale, scale);
            gw[j] = pack_bf16x2_rn(g0, g1);
            uw[j] = pack_bf16x2_rn(u0, u1);
          }
          if (p.out && valid) {
            st_global_v4(o + 8 * b, gw[0], gw[1], gw[2], gw[3]);
            st_global_v4(o + I + 8 * b, uw[0], uw[1], uw[2], uw[3]);
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float h0 = silu_bf16_lut24(lut, bf16lo(gw[j]));
            float h1 = silu_bf16_lut24(lut, bf16hi(gw[j]));
            mul_f32x2(h0, h1, bf16lo(uw[j]), bf16hi(uw[j]));
            mul_f32x2(h0, h1, w, w);
            h[b >> 1][8 * (b & 1) + 2 * j] = h0;
            h[b >> 1][8 * (b & 1) + 2 * j + 1] = h1;
          }
        }
        part = fmaxf(fmaxf(part, amax_f32x16(h[0])), amax_f32x16(h[1]));
      }
      // the quarter's four partial maxima of each row meet in shared memory
      // (two buffers: a warp is at most one tile ahead of the others here)
      float* pm = epi_part + (it & 1) * 512 + quarter * 128;
      pm[cb * 32 + lane] = part;
      __syncwarp();
      bar_sync_named(qbar, 128);
      uint32_t* slots = sw.amax + row * stride;
      if (ok && cb == 0 && valid) {
        const float m = fmaxf(fmaxf(pm[lane], pm[32 + lane]), fmaxf(pm[64 + lane], pm[96 + lane]));
        st_relaxed_gpu(slots + tl.nt, 0x80000000u | __float_as_uint(m));
      }
      if (!ok) continue;
      // wait for the row's n_tiles slots (all lanes of the warp together)
      float rmax = 0.0f;
      bool have = !valid;
      const uint64_t t0 = globaltimer();
      while (true) {
        if (!have) {
          uint32_t m = 0u, all = 0x80000000u;
          for (int q = 0; q < n_tiles; q += 4) {
            const uint4 v = ld_relaxed_gpu_v4(slots + q);
            const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (q + i < n_tiles) { all &= x[i]; m = max(m, x[i] & 0x7FFFFFFFu); }
          }
          if (all) { have = true; rmax = __uint_as_float(m); }
        }
        if (__all_sync(0xffffffffu, have)) break;
        // one decision for the whole warp: every lane must leave together
        const bool stop = *abort_flag != 0 || globaltimer() - t0 > budget;
        if (__any_sync(0xffffffffu, stop)) {
          failed = true;
          if (lane == 0) fail(MINITE_ERR_TIMEOUT);
          break;
        }
        __nanosleep(32);
      }
      if (failed) continue;
      const float g = global_scale(rmax);
      const int64_t sfr = static_cast<int64_t>(tl.sf_rb0) * 128 + r_in_tile;
      const int c0 = 8 * tl.nt + 2 * cb;   // first of this thread's two block columns
      if (valid) {
        const BlockScale s0 = block_scale_div(amax_f32x16(h[0]), g);
        const BlockScale s1 = block_scale_div(amax_f32x16(h[1]), g);
        const uint2 q0 = encode16(h[0], s0.enc, s0.sf == 0);
        const uint2 q1 = encode16(h[1], s1.enc, s1.sf == 0);
        *reinterpret_cast<uint4*>(sw.h_codes + row * (I / 2) + 64 * tl.nt + 16 * cb) =
            make_uint4(q0.x, q0.y, q1.x, q1.y);
        *reinterpret_cast<uint16_t*>(sw.h_sf + sf_offset(sfr, c0, kc)) =
            static_cast<uint16_t>(s0.sf | (s1.sf << 8));
        if (tl.nt == 0 && cb == 0) sw.h_g[row] = g;
      } else if (r_in_tile < 128 * tl.sf_rbs) {
        // a padding row of the expert's last 128-row scale block
        *reinterpret_cast<uint16_t*>(sw.h_sf + sf_offset(sfr, c0, kc)) = 0;
      }
    }
  } else if (warp < EPI_WARP0 + NUM_EPI_WARPS) {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int cb = (warp - EPI_WARP0) >> 2;
    const int r_in_tile = static_cast<int>(rank) * 128 + quarter * 32 + lane;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int t = cid; t < total; t += ncl) {
      const PTile tl = decode_pair_tile(t, n_tiles, tiles_prefix, s_off, s_sfb, p);
      const bool valid = r_in_tile < tl.rows;
      const int64_t row = static_cast<int64_t>(tl.row0) + r_in_tile;
      float scale = 0.0f;
      if (valid) scale = __frcp_rn(__fmul_rn(__ldg(p.a_g + row), __ldg(p.b_g + tl.e)));
      if (!mbar_wait(&S.acc_full, acc_phase, budget, abort_flag)) ok = false;
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      acc_phase ^= 1u;
      tc_fence_after();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + cb * EPI_COLS;
      auto release = [&] {
        if (rank == 0) mbar_arrive(&S.acc_empty);
        else mbar_arrive_remote(leader_acc_empty);
      };
      const int n0 = tl.nt * BN + cb * EPI_COLS;
      if (!p.c_tma) {
        epilogue_slice(p, tbase, valid, row, n0, scale, release);
        continue;
      }
      uint32_t pk[32];
      drain_bf16x64(tbase, scale, release, pk);
      const uint32_t vmask = __ballot_sync(0xffffffffu, valid);
      if (vmask != 0xffffffffu || n0 + EPI_COLS > p.N) {
        // the expert's last rows (a box would cross into the next expert's)
        store_rows_x4(static_cast<uint16_t*>(p.out), p.N, row - lane, n0, p.N, vmask, pk);
        continue;
      }
      // two 32 x 32 boxes through this warp's 2 KB of staging: lane = row,
      // its 64 bytes as four 16-byte chunks, chunk c at c ^ ((lane >> 1) & 3)
      // (the output tensor map's 64-byte swizzle, conflict-free shared stores)
      uint8_t* cst = c_area + (warp - EPI_WARP0) * R_C_WARP_BYTES;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (lane == 0) bulk_wait_group_read0();   // the previous box has left the buffer
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 4; ++c)
          *reinterpret_cast<uint4*>(cst + lane * 64 + 16 * (c ^ ((lane >> 1) & 3))) =
              make_uint4(pk[16 * h + 4 * c], pk[16 * h + 4 * c + 1], pk[16 * h + 4 * c + 2],
                         pk[16 * h + 4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmap_c, cst, n0 + 32 * h, static_cast<int>(row));
          bulk_commit_group();
        }
      }
    }
    if (lane == 0) bulk_wait_group0();   // every box written before the CTA exits
    if (!ok && lane == 0) fail(MINITE_ERR_TIMEOUT);
  }

  // no cross-CTA traffic may target a CTA that has left: both wait here, then
  // free the pair's TMEM together
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, TMEM_COLS);
}

// Zero `n` words (the fused epilogue's row maxima and counters) once the
// previous kernel on the stream has finished with them.
__global__ void zero_words_kernel(uint32_t* __restrict__ w, int64_t n) {
  pdl_wait();
  const int64_t i0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = 4 * i0; i < n; i += 4 * step) {
    if (i + 4 <= n) *reinterpret_cast<uint4*>(w + i) = make_uint4(0u, 0u, 0u, 0u);
    else for (int64_t j = i; j < n; ++j) w[j] = 0u;
  }
}

}  // namespace gemm

// Workspace of minite_gate_up_swiglu_quant_nvfp4: per row, one slot word for
// each of the I / 128 tiles of its m-block (the tile's partial |h| maximum
// with bit 31 set once written), rows padded to 4 words.
size_t swiglu_fused_workspace_words(int64_t M, int64_t I) {
  const int64_t stride = (I / 128 + 3) / 4 * 4;
  return static_cast<size_t>(M * stride);
}

// ---------------------------------------------------------------- host side

namespace {

std::atomic<uint64_t> g_budget_ns{0};
std::atomic<int> g_gemm_variant{0};  // 0 auto, 1 single-CTA, 2 CTA-pair, 4 pair two-chunk, 5 single two-chunk

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, uint64_t inner_bytes, uint64_t rows,
              uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner_bytes, rows};
  cuuint64_t strides[1] = {inner_bytes};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(gemm::BK_BYTES), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// BF16 output [rows, N] for TMA stores: boxes of 32 rows x 32 columns (64
// bytes, 64-byte swizzle).
bool make_map_out(CUtensorMap* m, const void* base, uint64_t N, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {N, rows};
  cuuint64_t strides[1] = {N * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same operand as 3-D: {128 bytes of a K chunk, rows, K / 128 chunks} with
// strides {row pitch, 128 bytes}; a box of 2 chunks lands as two consecutive
// 128-byte-swizzled chunk tiles. Only for K a multiple of 256, so that no
// chunk runs past the end of a row.
bool make_map3(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows,
               uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(gemm::BK_BYTES), rows, row_bytes / gemm::BK_BYTES};
  cuuint64_t strides[2] = {row_bytes, static_cast<cuuint64_t>(gemm::BK_BYTES)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(gemm::BK_BYTES), box_rows,
                       static_cast<cuuint32_t>(gemm::Q_CH)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace {

// Clusters of two CTAs of `kernel` that can be resident at once on the
// current device (queried once per device and kernel).
template <int Tag, typename Kernel>
int resident_pairs(Kernel kernel, int threads, size_t smem) {
  static std::atomic<int> cache[64];   // one per Tag: kernels of one type share a type
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int v = cache[dev].load();
  if (v > 0) return v;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * static_cast<unsigned>(num_sms() / 2));
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n <= 0) return 0;
  if (n > num_sms() / 2) n = num_sms() / 2;
  cache[dev].store(n);
  return n;
}

// Launch `pairs` clusters of two CTAs with programmatic stream serialization.
template <typename... KArgs, typename... Args>
cudaError_t launch_pair_pdl(void (*kernel)(KArgs...), int pairs, int threads, size_t smem,
                            cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace

uint64_t wait_budget_ns() {
  const uint64_t v = g_budget_ns.load();
  return v ? v : 2000000000ull;
}

}  // namespace minite

using namespace minite;

extern "C" void minite_set_wait_budget_ns(uint64_t ns) { g_budget_ns.store(ns); }

extern "C" void minite_set_gemm_variant(int variant) {
  g_gemm_variant.store(variant == 1 || variant == 5 || variant == 6 ? variant : 0);
}

extern "C" int minite_grouped_gemm_nvfp4(const uint8_t* a_codes, const uint8_t* a_sf,
                                         const float* a_g, const uint8_t* b_codes,
                                         const uint8_t* b_sf, const float* b_g,
                                         const int32_t* expert_offsets,
                                         const int32_t* sf_row_offsets, int64_t M_total,
                                         int64_t N, int64_t K, int32_t E, void* out,
                                         int out_dtype, int32_t* status,
                                         minite_stream_t stream) {
  using namespace gemm;
  if (!a_codes || !a_sf || !a_g || !b_codes || !b_sf || !b_g || !expert_offsets ||
      !sf_row_offsets || !out)
    return MINITE_ERR_INVALID_ARG;
  if (out_dtype != MINITE_OUT_BF16 && out_dtype != MINITE_OUT_FP32) return MINITE_ERR_INVALID_ARG;
  if (M_total < 1 || M_total >= (int64_t(1) << 31) || N < 32 || N % 32 != 0 || K < 64 ||
      K % 64 != 0 || E < 1 || E > 1024 || N * E >= (int64_t(1) << 31) || K > (1 << 20))
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(a_codes, 128) || !aligned(b_codes, 128) || !aligned(a_sf, 16) ||
      !aligned(b_sf, 16) || !aligned(out, 32))
    return MINITE_ERR_INVALID_ARG;
  // automatic choice: the CTA-pair kernel (measured fastest on the MoE
  // shapes: gate_up 0.445 against 0.457 ms, dgrad 0.232 against 0.234 ms, down
  // even), else the single-CTA kernels
  int variant = g_gemm_variant.load();
  if (variant == 0) variant = 6;
  const size_t d_smem = 1024 + D_STAGES * D_STAGE_BYTES + D_SLOTS * Q_SLOT_BYTES + sizeof(DSmem) +
                        2 * (E + 1) * sizeof(int32_t);
  // the two-chunk kernel reads whole 128-byte chunks of every row
  if (variant == 5 && (K % 256 != 0 || d_smem > 232448)) variant = 1;
  const size_t r_smem = 1024 + R_STAGES * (R_AB_BYTES + R_SF_BYTES) + sizeof(RSmem) +
                        3 * (E + 1) * sizeof(int32_t);
  if (variant == 6 && r_smem > 232448) variant = 1;
  // BF16 output of the CTA-pair kernel through TMA stores when the staging fits
  const bool c_tma = variant == 6 && out_dtype == MINITE_OUT_BF16 && r_smem + R_C_BYTES <= 232448;
  CUtensorMap tc;
  if (c_tma && !make_map_out(&tc, out, N, M_total)) return MINITE_ERR_CUDA;
  CUtensorMap ta, tb;
  if (variant == 5) {
    if (!make_map3(&ta, a_codes, K / 2, M_total, BM) || !make_map3(&tb, b_codes, K / 2, N * E, BN))
      return MINITE_ERR_CUDA;
  } else {
    const uint32_t b_box = variant == 6 ? 128u : static_cast<uint32_t>(BN);
    if (!make_map(&ta, a_codes, K / 2, M_total, BM) || !make_map(&tb, b_codes, K / 2, N * E, b_box))
      return MINITE_ERR_CUDA;
  }
  Params p = {};
  p.a_g = a_g;
  p.b_g = b_g;
  p.a_sf = a_sf;
  p.b_sf = b_sf;
  p.offsets = expert_offsets;
  p.sf_offsets = sf_row_offsets;
  p.out = out;
  p.status = status;
  p.M = M_total;
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.E = E;
  p.out_fp32 = out_dtype == MINITE_OUT_FP32;
  p.c_tma = c_tma ? 1 : 0;
  p.budget_ns = wait_budget_ns();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t n_tiles = (N + BN - 1) / BN;
  if (variant == 1) {
    const size_t smem = 1024 + STAGES * STAGE_BYTES + sizeof(Smem) + 2 * (E + 1) * sizeof(int32_t);
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
      attr_err = cudaFuncSetAttribute(grouped_gemm_kernel,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    });
    if (attr_err != cudaSuccess || smem > 232448) return MINITE_ERR_CUDA;
    // one CTA per SM, never more CTAs than the largest possible tile count
    const int64_t max_tiles = (M_total / BM + E) * n_tiles;
    int grid = num_sms();
    if (max_tiles < grid) grid = static_cast<int>(max_tiles);
    grouped_gemm_kernel<<<grid, NUM_THREADS, smem, s>>>(ta, tb, p);
  } else if (variant == 5) {
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
      attr_err = cudaFuncSetAttribute(grouped_gemm_dc_kernel<false>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    });
    if (attr_err != cudaSuccess) return MINITE_ERR_CUDA;
    const int64_t max_tiles = (M_total / BM + E) * n_tiles;
    int grid = num_sms();
    if (max_tiles < grid) grid = static_cast<int>(max_tiles);
    if (launch_pdl(grouped_gemm_dc_kernel<false>, dim3(grid), dim3(Q_THREADS), d_smem, s, ta, tb,
                   p) != cudaSuccess)
      return MINITE_ERR_CUDA;
  } else if (variant == 6) {
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
      attr_err = cudaFuncSetAttribute(grouped_gemm_pair_deep_kernel<false>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    });
    if (attr_err != cudaSuccess) return MINITE_ERR_CUDA;
    // one CTA per SM in clusters of two: as many pairs as can be resident at
    // once (a GPC with an odd SM count leaves one SM out), never more pairs
    // than pair tiles
    const int64_t max_pairs = (M_total / 256 + E) * n_tiles;
    const size_t smem = r_smem + (c_tma ? R_C_BYTES : 0);
    int pairs = c_tma ? resident_pairs<2>(grouped_gemm_pair_deep_kernel<false>, R_THREADS, smem)
                      : resident_pairs<0>(grouped_gemm_pair_deep_kernel<false>, R_THREADS, smem);
    if (pairs <= 0) return MINITE_ERR_CUDA;
    if (max_pairs < pairs) pairs = static_cast<int>(max_pairs);
    // without c_tma the kernel does not read its third tensor map
    if (launch_pair_pdl(grouped_gemm_pair_deep_kernel<false>, pairs, R_THREADS, smem, s, ta, tb,
                        c_tma ? tc : tb, p) != cudaSuccess)
      return MINITE_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}

extern "C" int minite_gate_up_swiglu_quant_nvfp4(
    const uint8_t* a_codes, const uint8_t* a_sf, const float* a_g, const uint8_t* b_codes,
    const uint8_t* b_sf, const float* b_g, const int32_t* expert_offsets,
    const int32_t* sf_row_offsets, int64_t M_total, int64_t I, int64_t K, int32_t E,
    const float* perm_w, void* gate_up, uint8_t* h_codes, uint8_t* h_sf, float* h_g,
    void* workspace, size_t ws_bytes, int32_t* status, minite_stream_t stream) {
  using namespace gemm;
  if (!a_codes || !a_sf || !a_g || !b_codes || !b_sf || !b_g || !expert_offsets ||
      !sf_row_offsets || !h_codes || !h_sf || !h_g || !workspace)
    return MINITE_ERR_INVALID_ARG;
  if (M_total < 1 || M_total >= (int64_t(1) << 31) || I < 128 || I % 128 != 0 || I > 8192 ||
      K < 64 || K % 64 != 0 || K > (1 << 20) || E < 1 || E > 1024 ||
      2 * I * E >= (int64_t(1) << 31))
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(a_codes, 128) || !aligned(b_codes, 128) || !aligned(a_sf, 16) ||
      !aligned(b_sf, 16) || !aligned(h_codes, 16) || !aligned(h_sf, 16) || !aligned(workspace, 16) ||
      (gate_up && !aligned(gate_up, 32)))
    return MINITE_ERR_INVALID_ARG;
  const size_t words = swiglu_fused_workspace_words(M_total, I);
  if (ws_bytes < words * sizeof(uint32_t)) return MINITE_ERR_INVALID_ARG;
  // stages, scale slots, barriers, the three offset tables and the silu table
  const size_t smem = 1024 + R_STAGES * (R_AB_BYTES + R_SF_BYTES) + sizeof(RSmem) +
                      3 * (E + 1) * sizeof(int32_t) + 16 + kLut24Entries * sizeof(float) +
                      2 * 512 * sizeof(float);
  if (smem > 232448) return MINITE_ERR_UNSUPPORTED_SHAPE;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(grouped_gemm_pair_deep_kernel<true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
  });
  if (attr_err != cudaSuccess) return MINITE_ERR_CUDA;
  // every m-block's I/128 tiles run at once on I/128 clusters (consecutive
  // cluster ids): launch a multiple of I/128 clusters, all resident together
  const int n_tiles = static_cast<int>(I / 128);
  int pairs = resident_pairs<1>(grouped_gemm_pair_deep_kernel<true>, R_THREADS, smem);
  if (pairs <= 0) return MINITE_ERR_CUDA;
  pairs = pairs / n_tiles * n_tiles;
  if (pairs == 0) return MINITE_ERR_UNSUPPORTED_SHAPE;
  const int64_t max_pairs = (M_total / 256 + E) * n_tiles;
  if (max_pairs < pairs) pairs = static_cast<int>(max_pairs);
  CUtensorMap ta, tb;
  if (!make_map(&ta, a_codes, K / 2, M_total, BM) || !make_map(&tb, b_codes, K / 2, 2 * I * E, 128))
    return MINITE_ERR_CUDA;
  Params p = {};
  p.a_g = a_g;
  p.b_g = b_g;
  p.a_sf = a_sf;
  p.b_sf = b_sf;
  p.offsets = expert_offsets;
  p.sf_offsets = sf_row_offsets;
  p.out = gate_up;
  p.status = status;
  p.M = M_total;
  p.N = static_cast<int>(2 * I);
  p.K = static_cast<int>(K);
  p.E = E;
  p.out_fp32 = 0;
  p.budget_ns = wait_budget_ns();
  uint32_t* ws = static_cast<uint32_t*>(workspace);
  p.sw.perm_w = perm_w;
  p.sw.h_codes = h_codes;
  p.sw.h_sf = h_sf;
  p.sw.h_g = h_g;
  p.sw.amax = ws;
  p.sw.I = static_cast<int>(I);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t zero_blocks = std::min<int64_t>(num_sms(), (static_cast<int64_t>(words) + 1023) / 1024);
  if (launch_pdl(zero_words_kernel, dim3(static_cast<unsigned>(zero_blocks)), dim3(256), 0, s, ws,
                 static_cast<int64_t>(words)) != cudaSuccess)
    return MINITE_ERR_CUDA;
  if (launch_pair_pdl(grouped_gemm_pair_deep_kernel<true>, pairs, R_THREADS, smem, s, ta, tb, tb, p) !=
      cudaSuccess)
    return MINITE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}

extern "C" int minite_grouped_gemm_wgrad_nvfp4(const uint8_t* a_codes, const uint8_t* a_sf,
                                               const float* a_g, const uint8_t* b_codes,
                                               const uint8_t* b_sf, const float* b_g,
                                               const int32_t* kofs, int32_t E, int64_t M,
                                               int64_t N, int64_t k_cap, void* out,
                                               int out_dtype, int32_t* status,
                                               minite_stream_t stream) {
  using namespace gemm;
  if (!a_codes || !a_sf || !a_g || !b_codes || !b_sf || !b_g || !kofs || !out)
    return MINITE_ERR_INVALID_ARG;
  if (out_dtype != MINITE_OUT_BF16 && out_dtype != MINITE_OUT_FP32) return MINITE_ERR_INVALID_ARG;
  if (M < 1 || M > 65536 || N < 32 || N % 32 != 0 || N > 65536 || E < 1 || E > 1024 ||
      k_cap < 256 || k_cap % 256 != 0 || k_cap >= (int64_t(1) << 31) ||
      int64_t(E) * M * N >= (int64_t(1) << 40))
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(a_codes, 128) || !aligned(b_codes, 128) || !aligned(a_sf, 16) ||
      !aligned(b_sf, 16) || !aligned(out, 32))
    return MINITE_ERR_INVALID_ARG;
  const size_t d_smem = 1024 + D_STAGES * D_STAGE_BYTES + D_SLOTS * Q_SLOT_BYTES + sizeof(DSmem) +
                        2 * (E + 1) * sizeof(int32_t);
  if (d_smem > 232448) return MINITE_ERR_UNSUPPORTED_SHAPE;
  CUtensorMap ta, tb;
  if (!make_map3(&ta, a_codes, k_cap / 2, M, BM) || !make_map3(&tb, b_codes, k_cap / 2, N, BN))
    return MINITE_ERR_CUDA;
  Params p = {};
  p.a_g = a_g;
  p.b_g = b_g;
  p.a_sf = a_sf;
  p.b_sf = b_sf;
  p.offsets = kofs;
  p.sf_offsets = kofs;
  p.out = out;
  p.status = status;
  p.M = M;
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(k_cap);
  p.E = E;
  p.out_fp32 = out_dtype == MINITE_OUT_FP32;
  p.budget_ns = wait_budget_ns();
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(grouped_gemm_dc_kernel<true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
  });
  if (attr_err != cudaSuccess) return MINITE_ERR_CUDA;
  const int64_t max_tiles = int64_t(E) * ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  int grid = num_sms();
  if (max_tiles < grid) grid = static_cast<int>(max_tiles);
  if (launch_pdl(grouped_gemm_dc_kernel<true>, dim3(grid), dim3(Q_THREADS), d_smem,
                 reinterpret_cast<cudaStream_t>(stream), ta, tb, p) != cudaSuccess)
    return MINITE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}
