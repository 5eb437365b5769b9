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

}  // namespace minite
