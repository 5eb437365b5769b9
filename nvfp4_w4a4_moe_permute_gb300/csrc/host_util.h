// Host-side helpers shared by the entry points of the minite library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace minite {

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Streaming multiprocessors of the current device (queried once per device).
int num_sms();

// Budget of the GEMM's bounded pipeline waits, in nanoseconds.
uint64_t wait_budget_ns();

// Token-chunk size of the permutation for top-k = k (pairs per chunk <= 512).
inline int permute_chunk_tokens(int k) {
  int ct = 512 / (k > 0 ? k : 1);
  return ct < 1 ? 1 : ct;
}

// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel on the stream finishes; it must call pdl_wait() before
// touching global memory (every kernel launched this way does).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace minite
