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
//  * Tile 128 x BN (BN = 128) of the output, K consumed 256 elements (128
//    bytes of packed E2M1) per pipeline stage; one tcgen05.mma of kind
//    mxf4nvf4 with 4X block scaling covers K = 64, so a stage is 4 MMAs.
//  * Warp 0: producer. TMA (128-byte swizzle) loads the A and B code tiles;
//    plain bulk copies load the scale atoms, which the permutation and the
//    quantizers already wrote in the MMA layout, so they need no reshuffle.
//  * Warp 1: MMA issuer. Copies the scale atoms shared -> TMEM with
//    tcgen05.cp (32x128b, replicated to the four lane quarters) and issues
//    the MMAs into a TMEM accumulator; tcgen05.commit frees smem stages and
//    publishes finished accumulators.
//  * Warps 2..5: epilogue. tcgen05.ld the accumulator, multiply by
//    1/(g_a[row] * g_w[e]), convert, and store rows of this expert only.
//  * Two TMEM accumulators so the epilogue of one tile overlaps the main
//    loop of the next; a static round-robin tile schedule over a grid of one
//    CTA per SM. The tile list is derived on the device from expert_offsets.
//  * Fixed K order, no split-K, one tile shape: a row's result depends only
//    on its own codes and its expert's weights (batch invariance).
//  * Every mbarrier wait is bounded by a %globaltimer budget; on expiry the
//    CTA records MINITE_ERR_TIMEOUT, drains its in-flight copies and MMAs,
//    frees TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "host_util.h"

namespace minite {

namespace gemm {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK_BYTES = 128;                 // 256 E2M1 values per row per stage
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK_BYTES;        // 16 KB
constexpr int B_BYTES = BN * BK_BYTES;        // 16 KB
constexpr int SF_ATOM = 512;                  // 128 rows x 4 scales
constexpr int SFA_BYTES = 4 * SF_ATOM;        // 4 K-steps of 64
constexpr int SFB_BYTES = 4 * SF_ATOM * (BN / 128);
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COLS = BN;             // fp32 accumulator: one column per n
constexpr uint32_t SFA_COL = 2 * ACC_COLS;    // 2 x 16 columns
constexpr uint32_t SFB_COL = SFA_COL + 32;    // 2 x 16 columns (BN = 128)
static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte swizzle alignment");
static_assert(SFB_COL + 32 <= TMEM_COLS, "TMEM budget");

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
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int total_tiles;
  int pad_;
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
  int64_t M;          // rows of A / out
  int N, K, E;
  int out_fp32;
  uint64_t budget_ns;
};

struct Tile {
  int e, nt;
  int row0;           // first permuted row of the tile
  int rows;           // valid rows (<= 128)
  int sf_rb;          // 128-row block of A's scales
};

// tile index -> (expert, m block, n block); tiles_prefix[e] = m blocks before e.
__device__ __forceinline__ Tile decode_tile(int t, int n_tiles, const int32_t* tiles_prefix,
                                            const Params& p) {
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
  const int off0 = __ldg(p.offsets + lo), off1 = __ldg(p.offsets + lo + 1);
  r.row0 = off0 + ml * BM;
  r.rows = min(BM, off1 - r.row0);
  r.sf_rb = __ldg(p.sf_offsets + lo) / 128 + ml;
  return r;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b, const Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Smem& S = *reinterpret_cast<Smem*>(stages + STAGES * STAGE_BYTES);
  int32_t* tiles_prefix = reinterpret_cast<int32_t*>(&S + 1);   // [E+1]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int KT = (p.K + 255) / 256;       // pipeline stages per tile
  const int KSTEPS = p.K / 64;            // MMAs per tile
  const int atoms_per_rb = p.K / 64;      // scale atoms per 128-row block
  const int n_tiles = (p.N + BN - 1) / BN;

  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.acc_full[b], 1);
      mbar_init(&S.acc_empty[b], 4);
    }
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
    uint32_t armed[STAGES];
#pragma unroll
    for (int s = 0; s < STAGES; ++s) armed[s] = 0;
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      const size_t sfb_expert = static_cast<size_t>((p.N + 127) / 128) * atoms_per_rb * SF_ATOM;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const Tile tl = decode_tile(t, n_tiles, tiles_prefix, p);
        for (int kt = 0; kt < KT; ++kt) {
          if (!mbar_wait(&S.empty[stage], phase ^ 1u, budget, abort_flag)) { ok = false; break; }
          const int ks = min(4, KSTEPS - 4 * kt);
          uint8_t* sA = stages + stage * STAGE_BYTES;
          uint8_t* sB = sA + A_BYTES;
          uint8_t* sSFA = sB + B_BYTES;
          uint8_t* sSFB = sSFA + SFA_BYTES;
          mbar_arrive_expect_tx(&S.full[stage],
                                A_BYTES + B_BYTES + 2 * static_cast<uint32_t>(ks) * SF_ATOM);
          tma_load_2d(sA, &tmap_a, &S.full[stage], kt * BK_BYTES, tl.row0);
          tma_load_2d(sB, &tmap_b, &S.full[stage], kt * BK_BYTES, tl.e * p.N + tl.nt * BN);
          bulk_load(sSFA,
                    p.a_sf + (static_cast<size_t>(tl.sf_rb) * atoms_per_rb + 4 * kt) * SF_ATOM,
                    ks * SF_ATOM, &S.full[stage]);
          bulk_load(sSFB,
                    p.b_sf + tl.e * sfb_expert +
                        (static_cast<size_t>(tl.nt) * atoms_per_rb + 4 * kt) * SF_ATOM,
                    ks * SF_ATOM, &S.full[stage]);
          ++armed[stage];
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
        if (armed[s]) mbar_wait(&S.full[s], (armed[s] - 1) & 1u, kDrainBudget, &no_abort);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc();
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      bool issued = false;
      int local = 0;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++local) {
        const int buf = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!mbar_wait(&S.acc_empty[buf], acc_phase ^ 1u, budget, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * ACC_COLS;
        for (int kt = 0; kt < KT; ++kt) {
          if (!mbar_wait(&S.full[stage], phase, budget, abort_flag)) { ok = false; break; }
          tc_fence_after();
          const int ks = min(4, KSTEPS - 4 * kt);
          uint8_t* sA = stages + stage * STAGE_BYTES;
          uint8_t* sB = sA + A_BYTES;
          uint8_t* sSFA = sB + B_BYTES;
          uint8_t* sSFB = sSFA + SFA_BYTES;
          const uint32_t sfa_t = tmem + SFA_COL + (kt & 1) * 16;
          const uint32_t sfb_t = tmem + SFB_COL + (kt & 1) * 16;
          for (int s = 0; s < ks; ++s) {
            tc_cp_sf(sfa_t + 4 * s, smem_desc(smem_u32(sSFA + s * SF_ATOM), 0, 128, kLayoutNone));
            tc_cp_sf(sfb_t + 4 * s, smem_desc(smem_u32(sSFB + s * SF_ATOM), 0, 128, kLayoutNone));
          }
          for (int s = 0; s < ks; ++s) {
            const uint64_t ad = smem_desc(smem_u32(sA + 32 * s), 16, 1024, kLayoutSwizzle128B);
            const uint64_t bd = smem_desc(smem_u32(sB + 32 * s), 16, 1024, kLayoutSwizzle128B);
            tc_mma_nvfp4(d_tmem, ad, bd, idesc, sfa_t + 4 * s, sfb_t + 4 * s, (kt | s) != 0);
          }
          issued = true;
          tc_commit(&S.empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(&S.acc_full[buf]);
      }
      if (!ok) {
        *abort_flag = 1;
        set_status(p.status, MINITE_ERR_TIMEOUT);
      }
      if (issued) {
        // drain: all MMAs and scale copies of this thread complete before TMEM is freed
        tc_commit(&S.drain);
        volatile int no_abort = 0;
        mbar_wait(&S.drain, 0, kDrainBudget, &no_abort);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;            // TMEM lanes this warp may access
    const int r_in_tile = quarter * 32 + lane;
    int local = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++local) {
      const int buf = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if (!mbar_wait(&S.acc_full[buf], acc_phase, budget, abort_flag)) ok = false;
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      const Tile tl = decode_tile(t, n_tiles, tiles_prefix, p);
      const bool valid = r_in_tile < tl.rows;
      const int64_t row = static_cast<int64_t>(tl.row0) + r_in_tile;
      float scale = 0.0f;
      if (valid) scale = __frcp_rn(__fmul_rn(__ldg(p.a_g + row), __ldg(p.b_g + tl.e)));
      const uint32_t tbase = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + buf * ACC_COLS;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32cols(tbase + c * 32, r);
        const int n = tl.nt * BN + c * 32;
        if (valid && n < p.N) {
          if (p.out_fp32) {
            float4* o = reinterpret_cast<float4*>(static_cast<float*>(p.out) + row * p.N + n);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              o[i] = make_float4(__fmul_rn(__uint_as_float(r[4 * i]), scale),
                                 __fmul_rn(__uint_as_float(r[4 * i + 1]), scale),
                                 __fmul_rn(__uint_as_float(r[4 * i + 2]), scale),
                                 __fmul_rn(__uint_as_float(r[4 * i + 3]), scale));
          } else {
            uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + row * p.N + n);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t w[4];
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float lo = __fmul_rn(__uint_as_float(r[8 * i + 2 * j]), scale);
                const float hi = __fmul_rn(__uint_as_float(r[8 * i + 2 * j + 1]), scale);
                w[j] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
                       (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
              }
              o[i] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.acc_empty[buf]);
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

}  // namespace gemm

// ---------------------------------------------------------------- host side

namespace {

std::atomic<uint64_t> g_budget_ns{0};

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

}  // namespace

uint64_t wait_budget_ns() {
  const uint64_t v = g_budget_ns.load();
  return v ? v : 2000000000ull;
}

}  // namespace minite

using namespace minite;

extern "C" void minite_set_wait_budget_ns(uint64_t ns) { g_budget_ns.store(ns); }

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
      !aligned(b_sf, 16) || !aligned(out, 16))
    return MINITE_ERR_INVALID_ARG;
  CUtensorMap ta, tb;
  if (!make_map(&ta, a_codes, K / 2, M_total, BM) || !make_map(&tb, b_codes, K / 2, N * E, BN))
    return MINITE_ERR_CUDA;
  Params p;
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
  p.budget_ns = wait_budget_ns();
  const size_t smem = 1024 + STAGES * STAGE_BYTES + sizeof(Smem) + (E + 1) * sizeof(int32_t);
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(grouped_gemm_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
  });
  if (attr_err != cudaSuccess || smem > 232448) return MINITE_ERR_CUDA;
  // one CTA per SM, never more CTAs than the largest possible tile count
  const int64_t max_tiles = (M_total / BM + E) * ((N + BN - 1) / BN);
  int grid = num_sms();
  if (max_tiles < grid) grid = static_cast<int>(max_tiles);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  grouped_gemm_kernel<<<grid, NUM_THREADS, smem, s>>>(ta, tb, p);
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}
