// Small entry points of the minite C ABI: status strings, version,
// workspace sizing, and the converter test hook.
#include <atomic>

#include "common.cuh"
#include "host_util.h"

namespace minite {

size_t permute_workspace_bytes(int64_t T, int64_t H, int32_t E, int32_t k);
size_t combine_backward_workspace_bytes(int64_t T, int64_t H);
size_t tokens_workspace_bytes(int32_t E, int64_t x_rows);

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

extern "C" int minite_test_div6_exhaustive(unsigned long long* mismatches, minite_stream_t stream) {
  if (!mismatches) return MINITE_ERR_INVALID_ARG;
  div6_exhaustive_kernel<<<4 * num_sms(), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      mismatches);
  return cudaGetLastError() == cudaSuccess ? MINITE_OK : MINITE_ERR_CUDA;
}
