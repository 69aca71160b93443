// mxg_route_permute_noalloc: the permute with its scratch held in a static
// device array instead of a caller-provided workspace.
//
// For callers that cannot allocate device memory at the point where they route
// tokens — e.g. code running inside a framework's memory pool, or a host
// runtime that owns all allocations and hands out only the input and output
// buffers.  The call still
// takes the caller's inputs and outputs; only the per-call scratch (per-chunk
// expert counts and bases, the row offsets) lives in a fixed-size array that
// every GPU loading this library keeps until the process exits.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace mxg {
namespace {

// The scratch: 256 KB per device, shared by every call of the entry point.
static __device__ __align__(256) int32_t g_permute_scratch[MXG_NOALLOC_SCRATCH_BYTES / 4];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch for the current device, looked up once per
// device (a host-side runtime query; no allocation).
cudaError_t scratch_for_current_device(int32_t** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace mxg

using namespace mxg;

extern "C" size_t mxg_route_permute_noalloc_max_entries(int E) {
  if (E <= 0) return 0;
  // scratch ints used: counts + bases (one per chunk and expert) + E+1 offsets
  const int64_t room = MXG_NOALLOC_SCRATCH_BYTES / 4 - (E + 1);
  const int64_t chunks = room / (2 * static_cast<int64_t>(E));
  return chunks > 0 ? static_cast<size_t>(chunks) * 4096u : 0u;
}

extern "C" int mxg_route_permute_noalloc(const int32_t* ids, int T, int k, int E, int32_t* split_sizes,
                                         int32_t* src_of_row, int32_t* row_of_src, int32_t* padded_offsets,
                                         int32_t* dev_status, void* stream) {
  if (!ids || !split_sizes || !src_of_row || !row_of_src || !padded_offsets || !dev_status) return MXG_ERR_ARG;
  if (T <= 0 || k <= 0 || E <= 0) return MXG_ERR_ARG;
  if (k > E || E > 256) return MXG_ERR_SHAPE;
  const int64_t R = static_cast<int64_t>(T) * k;
  if (R > static_cast<int64_t>(mxg_route_permute_noalloc_max_entries(E))) return MXG_ERR_WORKSPACE;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(ids) | reinterpret_cast<uintptr_t>(split_sizes) |
                        reinterpret_cast<uintptr_t>(src_of_row) | reinterpret_cast<uintptr_t>(row_of_src) |
                        reinterpret_cast<uintptr_t>(padded_offsets);
  if (mis & 31u) return MXG_ERR_ALIGN;
  int32_t* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return MXG_ERR_CUDA;
  const int nblk = permute_num_blocks(static_cast<int>(R));
  // Every scratch entry is written (counts, then bases and offsets) before it is
  // read within the call, so nothing has to be cleared between calls.
  PermuteParams p{};
  p.ids = ids;
  p.R = static_cast<int32_t>(R);
  p.E = E;
  p.counts = scratch;
  p.bases = scratch + static_cast<int64_t>(nblk) * E;
  p.offsets = scratch + 2 * static_cast<int64_t>(nblk) * E;
  p.padded_offsets = padded_offsets;
  p.pad = 128;
  p.split_sizes = split_sizes;
  p.src_of_row = src_of_row;
  p.row_of_src = row_of_src;
  p.status = dev_status;
  return launch_permute(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MXG_OK : MXG_ERR_CUDA;
}
