// Helpers shared by the CUDA translation units of the library.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace tree {

constexpr int kSMs = 152;  // GB300: 2 dies x 76 SMs

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

inline int launch_status(const char *what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(TREE_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
  return TREE_OK;
}

inline cudaStream_t as_stream(tree_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

// Number of SMs of the current device (cached per process; GB300 has 152).
int sm_count();

}  // namespace tree
