// Host-side helpers shared by the C-ABI files (api.cu, api_bf16.cu,
// api_fp8.cu): carving caller-owned buffers into aligned sub-buffers,
// alignment checks and CUDA-error propagation.
#pragma once
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdint>

#include "mxg.h"

namespace mxg {
namespace api {

constexpr int64_t kAlign = 256;   // every sub-buffer of saved / workspace starts on 256 bytes

inline int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

// Device pointers must be 32-byte aligned (the GEMM epilogues move whole
// 32-byte sectors); a null pointer passes (nullable arguments).
inline bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// Consecutive sub-buffers of one caller-owned buffer, each kAlign-aligned.
struct Carver {
  int64_t off = 0;
  int64_t take(int64_t bytes) {
    const int64_t o = off;
    off = align_up(off + bytes, kAlign);
    return o;
  }
};

template <typename T>
inline T* at(void* base, int64_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(base) + off);
}
template <typename T>
inline const T* at(const void* base, int64_t off) {
  return reinterpret_cast<const T*>(static_cast<const uint8_t*>(base) + off);
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? MXG_OK : MXG_ERR_CUDA; }

// An NVTX range around the host code that enqueues one stage's launches, so a
// profiler's timeline names every kernel by its stage ("mxg.fwd.gate_up", ...).
// NVTX v3 is header-only: without a profiler attached a range costs a few
// nanoseconds and loads nothing.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace api
}  // namespace mxg

#define MXG_TRY(expr)                                 \
  do {                                                \
    if ((expr) != cudaSuccess) return MXG_ERR_CUDA;   \
  } while (0)
