// minite_moe_permute_quant: MoE token permutation fused with the per-token
// amax, NVFP4 quantization and the scale-layout swizzle.
//
// The miniTE report summary, section "Two complementary interventions",
// computes the amax during the permutation (so no separate scan of the
// activations), writes experts into contiguous buffers described by
// device-side metadata, and fuses the scale-layout conversion into
// quantization. Per-token scales follow its section "Follow the numerical
// execution path".
//
// Four launches, no host synchronization:
//   permute_rank_kernel      one warp per token chunk: stable in-chunk rank of
//                            every (token, slot) pair (kept in dest_row) and
//                            the chunk's expert histogram -> table[e][chunk];
//                            also resets the scan's completion counter.
//   permute_scan_kernel      one block per expert: exclusive prefix of its
//                            chunk counts; the last block to finish turns the
//                            expert totals into expert_offsets / sf_row_offsets.
//   permute_quant_kernel     one warp per token: completes its pairs' permuted
//                            rows (offset + chunk base + local rank) with
//                            perm_src and perm_w, reads the token once,
//                            quantizes it once in registers and writes its
//                            codes to its k destination rows, its scales and
//                            global scale in token order.
//   permute_sf_gather_kernel the swizzled scale layout, one 128-row block of
//                            whole 512-byte atoms at a time, from the
//                            token-order scales through perm_src.
// Without room for the token-order staging (the allocation-free entry point
// on large problems) the quant kernel writes each row's scales itself, one
// 4-byte word per lane and row, and there is no gather.
#include <mutex>

#include "common.cuh"
#include "host_util.h"

namespace minite {

constexpr int kPermThreads = 256;

struct PermWs {
  uint32_t* counter;  // scan completion counter
  int32_t* totals;    // [E]
  int32_t* table;     // [E][nchunks]
  uint8_t* sfc;       // [T][kc] each token's scale bytes, token order (or null)
  float* gtok;        // [T] each token's global scale (or null)
};

static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Scratch of the ranking and scan (the histogram table).
static size_t perm_ws_base_bytes(int64_t T, int E, int k) {
  const int64_t ct = permute_chunk_tokens(k);
  const int64_t nchunks = (T + ct - 1) / ct;
  return 256 + align256(static_cast<size_t>(E) * 4) + align256(static_cast<size_t>(E) * nchunks * 4);
}

// Plus the token-order scale bytes and global scales that the scale gather
// turns into the swizzled layout.
static size_t perm_ws_bytes(int64_t T, int64_t H, int E, int k) {
  const size_t kc = static_cast<size_t>(((H / 16) + 3) & ~int64_t(3));
  return perm_ws_base_bytes(T, E, k) + align256(static_cast<size_t>(T) * kc) +
         align256(static_cast<size_t>(T) * 4);
}

static PermWs perm_ws(void* ws, int64_t T, int64_t H, int E, int k, bool compact) {
  PermWs w;
  char* p = static_cast<char*>(ws);
  w.counter = reinterpret_cast<uint32_t*>(p);
  w.totals = reinterpret_cast<int32_t*>(p + 256);
  w.table = reinterpret_cast<int32_t*>(p + 256 + align256(static_cast<size_t>(E) * 4));
  w.sfc = nullptr;
  w.gtok = nullptr;
  if (compact) {
    const size_t kc = static_cast<size_t>(((H / 16) + 3) & ~int64_t(3));
    char* q = p + perm_ws_base_bytes(T, E, k);
    w.sfc = reinterpret_cast<uint8_t*>(q);
    w.gtok = reinterpret_cast<float*>(q + align256(static_cast<size_t>(T) * kc));
  }
  return w;
}

// One warp per chunk of ct tokens (ct * k <= 512 pairs): the stable rank of
// every pair among the chunk's pairs with the same expert, in pair order, 32
// pairs at a time. Lanes carrying the same expert find each other with a
// match, take their order among themselves from the match mask and continue
// a per-expert running count kept in shared memory; the final counts are the
// chunk's histogram. The local rank goes to dest_row (completed later).
constexpr int kRankWarps = 4;  // chunks per block
__global__ void __launch_bounds__(32 * kRankWarps) permute_rank_kernel(
    const int32_t* __restrict__ ids, int64_t T, int k, int E, int ct, int nchunks,
    int32_t* __restrict__ table, int32_t* __restrict__ dest_row, uint32_t* __restrict__ counter,
    int32_t* status) {
  pdl_wait();
  extern __shared__ int32_t cnt_all[];  // [kRankWarps][E]
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int c = blockIdx.x * kRankWarps + wid;
  int32_t* cnt = cnt_all + wid * E;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  if (blockIdx.x == 0 && threadIdx.x == 0) *counter = 0u;
  __syncwarp();
  if (c >= nchunks) return;
  const int64_t p0 = static_cast<int64_t>(c) * ct * k;
  const int npairs = static_cast<int>(min(static_cast<int64_t>(c + 1) * ct, T) * k - p0);
  bool bad = false;
  // all of the chunk's ids requested at once (at most 16 per lane)
  int ids_r[16];
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const int p = 32 * r + lane;
    ids_r[r] = p < npairs ? ids[p0 + p] : -1;
  }
#pragma unroll
  for (int r = 0; r < 16; ++r) {
    const int b = 32 * r;
    if (b >= npairs) break;  // warp-uniform
    const int p = b + lane;
    const int e = ids_r[r];
    const bool valid = e >= 0 && e < E;
    if (p < npairs && !valid) bad = true;
    const uint32_t mask = __match_any_sync(0xffffffffu, valid ? e : E + lane);
    const int before = __popc(mask & ((1u << lane) - 1u));
    const int run = valid ? cnt[e] : 0;
    __syncwarp();
    if (valid && before == 0) cnt[e] = run + __popc(mask);
    __syncwarp();
    if (p < npairs) dest_row[p0 + p] = valid ? run + before : -1;
  }
  if (bad) set_status(status, MINITE_ERR_BAD_ROUTING);
  __syncwarp();
  for (int e = lane; e < E; e += 32) table[static_cast<int64_t>(e) * nchunks + c] = cnt[e];
}

// Exclusive scan of one value per thread over a 256-thread block; returns the
// block total through *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_sums[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int s = lane < (kPermThreads / 32) ? warp_sums[lane] : 0;
    int si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += t;
    }
    if (lane < (kPermThreads / 32)) warp_sums[lane] = si - s;
    if (lane == 31) warp_sums[32] = si;
  }
  __syncthreads();
  const int res = warp_sums[wid] + incl - v;
  *total = warp_sums[32];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(kPermThreads) permute_scan_kernel(
    int32_t* __restrict__ table, int nchunks, int E, uint32_t* __restrict__ counter,
    int32_t* __restrict__ totals, int32_t* __restrict__ expert_offsets,
    int32_t* __restrict__ sf_row_offsets) {
  pdl_wait();
  __shared__ int warp_sums[33];
  __shared__ int is_last;
  const int e = blockIdx.x;
  int32_t* row = table + static_cast<int64_t>(e) * nchunks;
  int carry = 0;
  for (int base = 0; base < nchunks; base += kPermThreads) {
    const int i = base + threadIdx.x;
    const int v = i < nchunks ? row[i] : 0;
    int tot;
    const int ex = block_exclusive_scan(v, warp_sums, &tot);
    if (i < nchunks) row[i] = carry + ex;
    carry += tot;
  }
  if (threadIdx.x == 0) {
    totals[e] = carry;
    __threadfence();
    is_last = (atomicAdd(counter, 1u) == static_cast<uint32_t>(E - 1));
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  int off = 0, sfoff = 0;
  for (int base = 0; base < E; base += kPermThreads) {
    const int i = base + threadIdx.x;
    const int cnt = i < E ? __ldcg(totals + i) : 0;
    int tot, tot_pad;
    const int ex = block_exclusive_scan(cnt, warp_sums, &tot);
    const int ex_pad = block_exclusive_scan((cnt + 127) & ~127, warp_sums, &tot_pad);
    if (i < E) {
      expert_offsets[i] = off + ex;
      sf_row_offsets[i] = sfoff + ex_pad;
    }
    off += tot;
    sfoff += tot_pad;
  }
  if (threadIdx.x == 0) {
    expert_offsets[E] = off;
    sf_row_offsets[E] = sfoff;
  }
}

// Quantize and scatter, one warp per token over a grid of resident blocks:
// the warp reads the token once (lane l owns blocks 32i + l), quantizes it
// once in registers and writes its codes, scales and g to each of its k
// permuted rows. Each warp requests its next token (row and routing) before
// it writes the current one.
// ids == nullptr: the routing comes from the caller (dest_row and offsets of
// an earlier permutation), which is then checked on the device; only the
// token-order scale mode (sfc != nullptr) is used this way.
// With ids, the warp also completes its token's routing (what a separate
// pass would do): each pair's permuted row is the expert's offset plus the
// chunk's base for the expert (the scan's table) plus the pair's rank within
// the chunk (left in dest_row by the ranking), written back to dest_row with
// perm_src and perm_w of that row.
template <int NCH>
__global__ void __launch_bounds__(kPermThreads, NCH <= 5 ? 3 : 2) permute_quant_kernel(
    const uint16_t* __restrict__ x, const int32_t* __restrict__ ids, int64_t T, int H, int E,
    int k, const int32_t* __restrict__ expert_offsets,
    const int32_t* __restrict__ sf_row_offsets, int32_t* __restrict__ dest_row,
    const int32_t* __restrict__ table, int ct, int nchunks, const float* __restrict__ topk_w,
    int32_t* __restrict__ perm_src, float* __restrict__ perm_w,
    uint8_t* __restrict__ codes, uint8_t* __restrict__ sf, float* __restrict__ row_g,
    uint8_t* __restrict__ sfc, float* __restrict__ gtok, int32_t* status) {
  pdl_wait();
  extern __shared__ int32_t sm[];
  int32_t* s_off = sm;                 // [E+1]
  int32_t* s_sfoff = s_off + (E + 1);  // [E+1]
  for (int i = threadIdx.x; i <= E; i += blockDim.x) {
    s_off[i] = expert_offsets[i];
    s_sfoff[i] = sf_row_offsets[i];
  }
  __syncthreads();
  if (ids == nullptr && !offsets_consistent(s_off, s_sfoff, E, T * k)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, MINITE_ERR_INVALID_ARG);
    return;
  }
  const int used = s_off[E];
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int nb = H / 16;
  const int kc = (nb + 3) & ~3;
  // Direct scale stores: lane l writes the 4-byte word of atoms l, l + 32
  // (scale columns 4a .. 4a + 3) of each destination row. Column c is block
  // c of the row, held by lane c % 32 in chunk c / 32, so the word of atom
  // l + 32 m gathers byte (l / 8 + 4 m) of the packed chunk scales of lanes
  // (4 l + i) % 32, i = 0..3.
  const int natoms = kc >> 2;
  const int src0 = (4 * lane) & 31;
  const uint32_t bsel = static_cast<uint32_t>(lane >> 3);   // byte within a packed word
  const bool a32 = (reinterpret_cast<uintptr_t>(x) & 31) == 0;
  uint32_t w[NCH][8];
  float am[NCH];
  float m = 0.0f;
  int dest = -1, e = -1;  // pair (t, lane)
  auto fetch = [&](int64_t t) {
    if (lane < k) {
      dest = dest_row[t * k + lane];
      if (ids) {
        e = ids[t * k + lane];
        if (dest >= 0)   // a valid id: dest is the pair's rank within its chunk
          dest += s_off[e] + table[static_cast<int64_t>(e) * nchunks + t / ct];
      } else {
        e = 0;
      }
    }
    const uint16_t* xr = x + t * H;
    m = a32 ? load_row_blocks<NCH, true>(xr, nb, w, am)
            : load_row_blocks<NCH, false>(xr, nb, w, am);
  };
  int64_t t = warp;
  if (t < T) fetch(t);
  while (t < T) {
    const float g = global_scale(warp_max(m));
    QBlock qb[NCH];
    quant_row_blocks<NCH>(w, am, nb, g, qb);
    const int dcur = dest, ecur = e;
    const int64_t tcur = t;
    if (ids && lane < k) {
      dest_row[tcur * k + lane] = dcur;
      if (dcur >= 0) {
        perm_src[dcur] = static_cast<int32_t>(tcur);
        if (perm_w) perm_w[dcur] = topk_w[tcur * k + lane];
      }
    }
    t += nwarps;
    if (t < T) fetch(t);
    if (sfc) {
      // scales once per token, in token order; the scale gather places them
#pragma unroll
      for (int jj = 0; jj < NCH; ++jj) {
        const int cc = 32 * jj + lane;
        if (cc < kc) sfc[tcur * kc + cc] = static_cast<uint8_t>(qb[jj].sf);
      }
      if (lane == 0) gtok[tcur] = g;
    }
    // this lane's scale words: atom lane + 32 m for m < (natoms + 31) / 32
    uint32_t sw[(NCH + 3) / 4];
    if (!sfc) {
#pragma unroll
      for (int m = 0; m < (NCH + 3) / 4; ++m) {
        // packed scales of chunks 4m .. 4m + 3 of this lane (zero past the row)
        uint32_t pk = 0u;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (4 * m + q < NCH) pk |= (qb[4 * m + q].sf & 0xFFu) << (8 * q);
        uint32_t word = 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t v = __shfl_sync(0xffffffffu, pk, src0 + i);
          word |= ((v >> (8 * bsel)) & 0xFFu) << (8 * i);
        }
        sw[m] = word;
      }
    }
    for (int j = 0; j < k; ++j) {
      const int d = __shfl_sync(0xffffffffu, dcur, j);
      if (d < 0) continue;  // warp-uniform
      if (d >= used) {      // only a caller-given routing can point past the used rows
        if (lane == 0) set_status(status, MINITE_ERR_INVALID_ARG);
        continue;
      }
      const int ej = __shfl_sync(0xffffffffu, ecur, j);
      uint8_t* crow = codes + static_cast<int64_t>(d) * (H / 2);
#pragma unroll
      for (int jj = 0; jj < NCH; ++jj) {
        const int cc = 32 * jj + lane;
        if (cc < nb) st_u64(crow + 8 * cc, qb[jj].codes);
      }
      if (!sfc) {
        const int64_t r = static_cast<int64_t>(s_sfoff[ej]) + (d - s_off[ej]);
        uint8_t* srow = sf + ((r >> 7) * natoms) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4;
#pragma unroll
        for (int m = 0; m < (NCH + 3) / 4; ++m) {
          const int a = lane + 32 * m;
          if (a < natoms) *reinterpret_cast<uint32_t*>(srow + a * 512) = sw[m];
        }
        if (lane == 0) row_g[d] = g;
      }
    }
  }
  if (sfc) return;  // the scale gather writes every scale row, padding included

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

// Scale gather: writes the swizzled scale layout one 128-row block (one row of
// atoms, 128 x kc bytes) at a time, in order, from the token-order scales:
// row r of an expert's region holds the scales of token perm_src[p] for its
// permuted row p, or zeros past the expert's rows. Thread unit (line i of 32,
// group of 4 atoms): reads 16 bytes of each of the rows i, i+32, i+64, i+96
// and writes the 16-byte line i of each of the 4 atoms, so a warp writes
// whole 512-byte atoms. Also row_g[p] = the token's g.
__global__ void __launch_bounds__(kPermThreads) permute_sf_gather_kernel(
    const uint8_t* __restrict__ sfc, const float* __restrict__ gtok,
    const int32_t* __restrict__ perm_src, const int32_t* __restrict__ expert_offsets,
    const int32_t* __restrict__ sf_row_offsets, int64_t T, int k, int E, int kc,
    uint8_t* __restrict__ sf, float* __restrict__ row_g, int32_t* status) {
  pdl_wait();
  extern __shared__ int32_t sm[];
  int32_t* s_off = sm;                 // [E+1]
  int32_t* s_sfoff = s_off + (E + 1);  // [E+1]
  for (int i = threadIdx.x; i <= E; i += blockDim.x) {
    s_off[i] = expert_offsets[i];
    s_sfoff[i] = sf_row_offsets[i];
  }
  __syncthreads();
  if (!offsets_consistent(s_off, s_sfoff, E, T * k)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, MINITE_ERR_INVALID_ARG);
    return;
  }
  // a permuted row's source token, or -1 (with the error bit) if out of range
  auto source = [&](int p) {
    const int tk = perm_src[p];
    if (tk < 0 || tk >= T) {
      set_status(status, MINITE_ERR_INVALID_ARG);
      return -1;
    }
    return tk;
  };
  const int t = threadIdx.x;
  const int natoms = kc / 4;
  const int ngroups = (natoms + 3) / 4;
  const int nblocks = s_sfoff[E] / 128;
  for (int blk = blockIdx.x; blk < nblocks; blk += gridDim.x) {
    // expert of the block: the last e with s_sfoff[e] <= 128 blk
    int lo = 0, hi = E;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_sfoff[mid] <= 128 * blk) lo = mid; else hi = mid;
    }
    const int row0 = 128 * blk - s_sfoff[lo];  // local row of the block's first row
    const int cnt = s_off[lo + 1] - s_off[lo];
    const int p0 = s_off[lo] + row0;
    if (t < 128 && row0 + t < cnt) {
      const int tk = source(p0 + t);
      row_g[p0 + t] = tk >= 0 ? gtok[tk] : 0.0f;
    }
    for (int u = t; u < 32 * ngroups; u += blockDim.x) {
      const int i = u & 31, ag = u >> 5;
      int tok[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) tok[q] = row0 + 32 * q + i < cnt ? source(p0 + 32 * q + i) : -1;
      uint32_t wv[4][4];  // [q][atom j]: 4 scale bytes of row 32q+i, columns 4(4ag+j) ..
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint8_t* src = sfc + static_cast<int64_t>(tok[q]) * kc + 16 * ag;
        if (tok[q] >= 0 && 4 * ag + 4 <= natoms && kc % 16 == 0) {
          const uint4 v = *reinterpret_cast<const uint4*>(src);
          wv[q][0] = v.x; wv[q][1] = v.y; wv[q][2] = v.z; wv[q][3] = v.w;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            wv[q][j] = (tok[q] >= 0 && 4 * ag + j < natoms)
                           ? *reinterpret_cast<const uint32_t*>(src + 4 * j) : 0u;
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int a = 4 * ag + j;
        if (a < natoms)
          *reinterpret_cast<uint4*>(sf + (static_cast<int64_t>(blk) * natoms + a) * 512 + 16 * i) =
              make_uint4(wv[0][j], wv[1][j], wv[2][j], wv[3][j]);
      }
    }
  }
}

}  // namespace minite

using namespace minite;

namespace minite {
size_t permute_workspace_bytes(int64_t T, int64_t H, int32_t E, int32_t k) {
  return perm_ws_bytes(T, H, E, k);
}
// The combine backward keeps only the token-order scales and global scales.
size_t combine_backward_workspace_bytes(int64_t T, int64_t H) {
  const size_t kc = static_cast<size_t>(((H / 16) + 3) & ~int64_t(3));
  return align256(static_cast<size_t>(T) * kc) + align256(static_cast<size_t>(T) * 4);
}
}  // namespace minite

// The per-token quantization (codes to every destination row; scales to the
// token-order scratch when compact, else straight to the rows) and, when
// compact, the scale gather. ids == nullptr: caller-given routing.
static int launch_quant_gather(const void* x, const int32_t* topk_ids, int64_t T, int64_t H,
                               int32_t E, int32_t k, const int32_t* expert_offsets,
                               const int32_t* sf_row_offsets, int32_t* perm_src,
                               int32_t* dest_row, const int32_t* table, int ct, int nchunks,
                               const float* topk_w, float* perm_w, uint8_t* codes, uint8_t* sf,
                               float* row_g, const PermWs& w, bool compact, int32_t* status,
                               cudaStream_t s) {
  const size_t smem = 2 * (E + 1) * sizeof(int32_t);
  const int nch = static_cast<int>((H / 16 + 31) / 32);
  const uint16_t* xb = static_cast<const uint16_t*>(x);
  const int h = static_cast<int>(H);
  const int per_sm = nch <= 5 ? 3 : 2;
  int64_t qblocks = (T + kPermThreads / 32 - 1) / (kPermThreads / 32);
  if (qblocks > static_cast<int64_t>(num_sms()) * per_sm) qblocks = num_sms() * per_sm;
  if (qblocks < 1) qblocks = 1;
  switch (nch) {
#define MINITE_CASE(N)                                                                     \
  case N:                                                                                  \
    launch_pdl(permute_quant_kernel<N>, dim3(static_cast<unsigned>(qblocks)),              \
               dim3(kPermThreads), smem, s, xb, topk_ids, T, h, E, k, expert_offsets,      \
               sf_row_offsets, dest_row, table, ct, nchunks, topk_w, perm_src, perm_w,     \
               codes, sf, row_g, w.sfc, w.gtok, status);                                   \
    break;
    MINITE_CASE(1) MINITE_CASE(2) MINITE_CASE(3) MINITE_CASE(4) MINITE_CASE(5) MINITE_CASE(6)
    MINITE_CASE(7) MINITE_CASE(8)
#undef MINITE_CASE
    default: return MINITE_ERR_UNSUPPORTED_SHAPE;
  }
  if (compact) {
    const int kc = static_cast<int>(((H / 16) + 3) & ~int64_t(3));
    int64_t gblocks = (T * k) / 128 + E;   // upper bound of the 128-row scale blocks
    const int64_t cap = static_cast<int64_t>(num_sms()) * 8;
    if (gblocks > cap) gblocks = cap;
    launch_pdl(permute_sf_gather_kernel, dim3(static_cast<unsigned>(gblocks)), dim3(kPermThreads),
               smem, s, static_cast<const uint8_t*>(w.sfc), static_cast<const float*>(w.gtok),
               perm_src, expert_offsets, sf_row_offsets, T, static_cast<int>(k),
               static_cast<int>(E), kc, sf, row_g, status);
  }
  return MINITE_OK;
}

// compact = true: scales go to a token-order scratch and the scale gather
// writes the swizzled layout with whole-atom stores (needs the full
// workspace); false: each token's scales are scattered to its k rows.
static int permute_quant_impl(const void* x, const int32_t* topk_ids, const float* topk_w,
                              int64_t T, int64_t H, int32_t E, int32_t k, uint8_t* codes,
                              uint8_t* sf, float* row_g, int32_t* expert_offsets,
                              int32_t* sf_row_offsets, int32_t* perm_src, int32_t* dest_row,
                              float* perm_w, void* workspace, size_t ws_bytes, bool compact,
                              int32_t* status, minite_stream_t stream) {
  if (!x || !topk_ids || !codes || !sf || !row_g || !expert_offsets || !sf_row_offsets ||
      !perm_src || !dest_row || !workspace)
    return MINITE_ERR_INVALID_ARG;
  if ((topk_w == nullptr) != (perm_w == nullptr)) return MINITE_ERR_INVALID_ARG;
  if (T < 1 || H < 64 || H % 64 != 0 || H > 4096 || E < 1 || E > 1024 || k < 1 || k > 32)
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (T * k >= (int64_t(1) << 31) || (T * k + 128 * int64_t(E)) * ((H / 16 + 3) & ~3) >= (int64_t(1) << 40))
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(sf, 16) || !aligned(workspace, 256))
    return MINITE_ERR_INVALID_ARG;
  if (ws_bytes < (compact ? perm_ws_bytes(T, H, E, k) : perm_ws_base_bytes(T, E, k)))
    return MINITE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int ct = permute_chunk_tokens(k);
  const int nchunks = static_cast<int>((T + ct - 1) / ct);
  PermWs w = perm_ws(workspace, T, H, E, k, compact);

  const int rank_blocks = (nchunks + kRankWarps - 1) / kRankWarps;
  launch_pdl(permute_rank_kernel, dim3(rank_blocks), dim3(32 * kRankWarps),
             kRankWarps * E * sizeof(int32_t), s, topk_ids, T, static_cast<int>(k),
             static_cast<int>(E), ct, nchunks, w.table, dest_row, w.counter, status);
  launch_pdl(permute_scan_kernel, dim3(E), dim3(kPermThreads), 0, s, w.table, nchunks,
             static_cast<int>(E), w.counter, w.totals, expert_offsets, sf_row_offsets);
  const int rc = launch_quant_gather(x, topk_ids, T, H, E, k, expert_offsets, sf_row_offsets,
                                     perm_src, dest_row, w.table, ct, nchunks, topk_w, perm_w,
                                     codes, sf, row_g, w, compact, status, s);
  if (rc != MINITE_OK) return rc;
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}

extern "C" int minite_moe_permute_quant(const void* x, const int32_t* topk_ids,
                                        const float* topk_w, int64_t T, int64_t H, int32_t E,
                                        int32_t k, uint8_t* codes, uint8_t* sf, float* row_g,
                                        int32_t* expert_offsets, int32_t* sf_row_offsets,
                                        int32_t* perm_src, int32_t* dest_row, float* perm_w,
                                        void* workspace, size_t ws_bytes, int32_t* status,
                                        minite_stream_t stream) {
  return permute_quant_impl(x, topk_ids, topk_w, T, H, E, k, codes, sf, row_g, expert_offsets,
                            sf_row_offsets, perm_src, dest_row, perm_w, workspace, ws_bytes,
                            true, status, stream);
}

// The backward of the combine: dD[dest_row[t, j]] = dY[t] for every routed
// pair, i.e. dY laid out like the forward's permuted activations. Each token
// of dY is quantized once (per-token NVFP4) and its codes written to its k
// rows, reusing the forward permutation's routing instead of ranking the
// routing ids again.
extern "C" int minite_moe_combine_backward_quant(
    const void* dy, int64_t T, int64_t H, int32_t E, int32_t k, const int32_t* dest_row,
    const int32_t* expert_offsets, const int32_t* sf_row_offsets, const int32_t* perm_src,
    uint8_t* codes, uint8_t* sf, float* row_g, void* workspace, size_t ws_bytes,
    int32_t* status, minite_stream_t stream) {
  if (!dy || !dest_row || !expert_offsets || !sf_row_offsets || !perm_src || !codes || !sf ||
      !row_g || !workspace)
    return MINITE_ERR_INVALID_ARG;
  if (T < 1 || H < 64 || H % 64 != 0 || H > 4096 || E < 1 || E > 1024 || k < 1 || k > 32)
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (T * k >= (int64_t(1) << 31) ||
      (T * k + 128 * int64_t(E)) * ((H / 16 + 3) & ~3) >= (int64_t(1) << 40))
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(dy, 16) || !aligned(codes, 16) || !aligned(sf, 16) || !aligned(workspace, 256))
    return MINITE_ERR_INVALID_ARG;
  if (ws_bytes < combine_backward_workspace_bytes(T, H)) return MINITE_ERR_INVALID_ARG;
  PermWs w = {};
  const size_t kc = static_cast<size_t>(((H / 16) + 3) & ~int64_t(3));
  w.sfc = static_cast<uint8_t*>(workspace);
  w.gtok = reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(T * kc));
  // the forward's routing, read only (no ids: dest_row, perm_src untouched)
  const int rc = launch_quant_gather(dy, nullptr, T, H, E, k, expert_offsets, sf_row_offsets,
                                     const_cast<int32_t*>(perm_src), const_cast<int32_t*>(dest_row),
                                     nullptr, 1, 1, nullptr, nullptr, codes, sf, row_g, w, true,
                                     status, reinterpret_cast<cudaStream_t>(stream));
  if (rc != MINITE_OK) return rc;
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of minite_moe_permute_quant.
//
// Some callers cannot call cudaMalloc or hand out device memory at the point
// where they run the permutation: a host application whose memory plan is
// fixed before it starts, a plugin that receives only its input and output
// buffers from the framework that loads it, or a latency-critical loop that
// must not enter the allocator. For them this entry point takes the same
// inputs and outputs but keeps its scratch (the per-chunk expert histogram
// and the scan counter) in one fixed array in the library's own device
// memory, so the call performs no allocation of any kind.
//
// The array is file-scope device memory: every GPU that loads the library
// holds it until the process exits. Its device address is looked up once
// per device (cudaGetSymbolAddress, under a mutex) on the first call made
// while that device is current; make that first call before capturing a
// stream. The address is kept for the life of the process, so it does not
// survive cudaDeviceReset (which unloads the module holding the array); a
// process that resets its device must not call this entry point again. All
// calls on a device share the array, so two calls whose work
// overlaps on the GPU (different streams, no ordering between them) race
// and must not be issued. The kernels rewrite every scratch word they read
// on each call (histogram entries, the counter and, when they fit, the
// token-order scales), so nothing left by an earlier call needs clearing.
// When the token-order scales do not fit, each token's scales are scattered
// straight to its k rows instead (same results).
// ---------------------------------------------------------------------------

namespace {
constexpr size_t kStaticScratchBytes = size_t(2) << 20;  // 2 MiB
__device__ __align__(256) unsigned char g_permute_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[64] = {};
}  // namespace

extern "C" int minite_moe_permute_quant_noalloc(
    const void* x, const int32_t* topk_ids, const float* topk_w, int64_t T, int64_t H,
    int32_t E, int32_t k, uint8_t* codes, uint8_t* sf, float* row_g, int32_t* expert_offsets,
    int32_t* sf_row_offsets, int32_t* perm_src, int32_t* dest_row, float* perm_w,
    int32_t* status, minite_stream_t stream) {
  if (T < 1 || E < 1 || E > 1024 || k < 1 || k > 32 || H < 64 || H > 4096)
    return MINITE_ERR_UNSUPPORTED_SHAPE;
  if (perm_ws_base_bytes(T, E, k) > kStaticScratchBytes) return MINITE_ERR_SCRATCH_LIMIT;
  // token-order scale staging when it fits in the array as well
  const bool compact = perm_ws_bytes(T, H, E, k) <= kStaticScratchBytes;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MINITE_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_permute_scratch) != cudaSuccess || !addr)
        return MINITE_ERR_CUDA;
      g_scratch_addr[dev] = addr;
    }
    scratch = g_scratch_addr[dev];
  }
  return permute_quant_impl(x, topk_ids, topk_w, T, H, E, k, codes, sf, row_g, expert_offsets,
                            sf_row_offsets, perm_src, dest_row, perm_w, scratch,
                            kStaticScratchBytes, compact, status, stream);
}
