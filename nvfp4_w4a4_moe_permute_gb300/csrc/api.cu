// Small entry points of the minite C ABI: status strings, version,
// workspace sizing, and the converter test hook.
#include <atomic>

#include "common.cuh"
#include "host_util.h"

namespace minite {

size_t permute_workspace_bytes(int64_t T, int64_t H, int32_t E, int32_t k);
size_t combine_backward_workspace_bytes(int64_t T, int64_t H);
size_t tokens_workspace_bytes(int32_t E, int64_t x_rows);
size_t swiglu_fused_workspace_words(int64_t M, int64_t I);

int num_sms() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int v = cache[dev].load();
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
    v = 148;
  cache[dev].store(v);
  return v;
}

__global__ void convert_test_kernel(const float* __restrict__ in, int64_t n,
                                    uint8_t* __restrict__ out_e2m1, uint8_t* __restrict__ out_e4m3,
                                    float* __restrict__ out_exp) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float v = in[i];
    if (out_e2m1) out_e2m1[i] = static_cast<uint8_t>(cvt_e2m1x2(v, 0.0f) & 0xF);
    if (out_e4m3) out_e4m3[i] = static_cast<uint8_t>(cvt_e4m3(v));
    if (out_exp) out_exp[i] = exp_spec(v);
  }
}

// SplitMix64 finaliser (Steele, Lea and Flood, 2014), for the converter digests.
__device__ __forceinline__ unsigned long long splitmix64(unsigned long long z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Digests of the converters over chunks of 2^20 consecutive float32 bit
// patterns: per chunk and converter, the sum modulo 2^64 of
// splitmix64(((pattern << 32) | result) ^ salt) over the finite inputs (E4M3:
// +0 and the positive ones). 16 blocks of 256 threads per chunk.
constexpr int kDigestChunkBits = 20;
constexpr int kDigestBlocksPerChunk = 16;
__global__ void __launch_bounds__(256) convert_digest_kernel(unsigned long long first_chunk,
                                                             unsigned long long* __restrict__ digests) {
  const unsigned long long chunk = first_chunk + blockIdx.x / kDigestBlocksPerChunk;
  const uint32_t per_block = (1u << kDigestChunkBits) / kDigestBlocksPerChunk;
  const uint32_t base = static_cast<uint32_t>(chunk << kDigestChunkBits) +
                        (blockIdx.x % kDigestBlocksPerChunk) * per_block;
  unsigned long long d0 = 0, d1 = 0, d2 = 0;
  for (uint32_t i = threadIdx.x; i < per_block; i += blockDim.x) {
    const uint32_t b = base + i;
    if ((b & 0x7F800000u) == 0x7F800000u) continue;  // inf / NaN
    const float v = __uint_as_float(b);
    const unsigned long long key = static_cast<unsigned long long>(b) << 32;
    d0 += splitmix64((key | (cvt_e2m1x2(v, 0.0f) & 0xFu)) ^ 0x243F6A8885A308D3ull);
    if (v > 0.0f || b == 0u) d1 += splitmix64((key | cvt_e4m3(v)) ^ 0x13198A2E03707344ull);
    d2 += splitmix64((key | __float_as_uint(exp_spec(v))) ^ 0xA4093822299F31D0ull);
  }
  d0 = warp_sum_u64(d0);
  d1 = warp_sum_u64(d1);
  d2 = warp_sum_u64(d2);
  if ((threadIdx.x & 31) == 0) {
    unsigned long long* out = digests + 3 * (blockIdx.x / kDigestBlocksPerChunk);
    atomicAdd(out, d0);
    atomicAdd(out + 1, d1);
    atomicAdd(out + 2, d2);
  }
}

// Every non-negative finite float x: count x with div6_rn(x) != IEEE x / 6.
__global__ void div6_exhaustive_kernel(unsigned long long* mismatches) {
  unsigned long long bad = 0;
  for (uint32_t b = blockIdx.x * blockDim.x + threadIdx.x; b < 0x7F800000u;
       b += gridDim.x * blockDim.x) {
    const float x = __uint_as_float(b);
    if (__float_as_uint(div6_rn(x)) != __float_as_uint(__fdiv_rn(x, 6.0f))) ++bad;
  }
  if (bad) atomicAdd(mismatches, bad);
}

}  // namespace minite

using namespace minite;

extern "C" size_t minite_workspace_bytes(int op, int64_t a, int64_t b, int32_t E, int32_t k) {
  (void)b;
  switch (op) {
    case MINITE_OP_QUANTIZE:
      return a > 0 ? static_cast<size_t>(a) * sizeof(uint32_t) : 0;
    case MINITE_OP_PERMUTE_QUANT:
      return (a > 0 && b > 0 && E > 0 && k > 0) ? permute_workspace_bytes(a, b, E, k) : 0;
    case MINITE_OP_COMBINE_BACKWARD_QUANT:
      return (a > 0 && b > 0) ? combine_backward_workspace_bytes(a, b) : 0;
    case MINITE_OP_QUANTIZE_TOKENS:
      return (a > 0 && a <= 1024 && b >= 0) ? tokens_workspace_bytes(static_cast<int32_t>(a), b) : 0;
    case MINITE_OP_GATE_UP_SWIGLU:
      return (a > 0 && b >= 128) ? swiglu_fused_workspace_words(a, b) * sizeof(uint32_t) : 0;
    default:
      return 0;
  }
}

extern "C" const char* minite_status_string(int status) {
  switch (status) {
    case MINITE_OK: return "ok";
    case MINITE_ERR_INVALID_ARG: return "invalid argument";
    case MINITE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MINITE_ERR_CUDA: return "CUDA error";
    case MINITE_ERR_TIMEOUT: return "device pipeline wait timed out";
    case MINITE_ERR_BAD_ROUTING: return "routing id out of range";
    case MINITE_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the built-in array holds";
    default: return "unknown status";
  }
}

extern "C" const char* minite_version(void) { return "0.1.0"; }

extern "C" int minite_test_convert(const float* in, int64_t n, uint8_t* out_e2m1,
                                   uint8_t* out_e4m3, float* out_exp, minite_stream_t stream) {
  if (!in || n < 0) return MINITE_ERR_INVALID_ARG;
  if (n == 0) return MINITE_OK;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 65536) blocks = 65536;
  convert_test_kernel<<<static_cast<unsigned>(blocks), 256, 0,
                        reinterpret_cast<cudaStream_t>(stream)>>>(in, n, out_e2m1, out_e4m3,
                                                                  out_exp);
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}

extern "C" int minite_test_convert_digest(unsigned long long first_chunk,
                                          unsigned long long n_chunks,
                                          unsigned long long* digests, minite_stream_t stream) {
  if (!digests || first_chunk + n_chunks > (1ull << (32 - kDigestChunkBits)) ||
      n_chunks > (1ull << 16))
    return MINITE_ERR_INVALID_ARG;
  if (n_chunks == 0) return MINITE_OK;
  convert_digest_kernel<<<static_cast<unsigned>(n_chunks * kDigestBlocksPerChunk), 256, 0,
                          reinterpret_cast<cudaStream_t>(stream)>>>(first_chunk, digests);
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}

extern "C" int minite_test_div6_exhaustive(unsigned long long* mismatches, minite_stream_t stream) {
  if (!mismatches) return MINITE_ERR_INVALID_ARG;
  div6_exhaustive_kernel<<<4 * num_sms(), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      mismatches);
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}
