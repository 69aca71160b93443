// Row movement for tokens that travel between the grouped layout and token
// order outside the fused MLP call: a row gather (dispatch of tokens to their
// experts' order, the return of expert rows, the per-row probabilities) and
// the expansion of split_sizes into the group id of every row (a caller whose
// tokens arrive already grouped: "BioNeMo Uses Grouped Kernels and MXFP8",
// "Grouping fragmented expert workloads", the GroupedLinear call with one
// token count per expert).  HBM-bound: every byte is read once and written
// once, in 16-byte vectors where the row size allows.
#include "common.cuh"
#include "kernels.h"

namespace mxg {
namespace {

// One thread per 16-byte (VEC = 4 words) or 4-byte (VEC = 1) piece of a row.
template <int VEC>
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint32_t* __restrict__ src, int64_t src_rows,
                                                          int64_t row_words, const int32_t* __restrict__ index,
                                                          int div, int64_t rows, uint32_t* __restrict__ dst,
                                                          int32_t* status) {
  const int64_t pieces = row_words / VEC;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= rows * pieces) return;
  const int64_t r = i / pieces, c = i % pieces;
  const int32_t f = index[r];
  const int64_t sr = f < 0 ? -1 : f / div;
  uint32_t* d = dst + r * row_words + c * VEC;
  if (sr < 0 || sr >= src_rows) {
    if (c == 0) report(status, MXG_ERR_INDEX);
    if constexpr (VEC == 4) *reinterpret_cast<uint4*>(d) = make_uint4(0u, 0u, 0u, 0u);
    else *d = 0u;
    return;
  }
  const uint32_t* p = src + sr * row_words + c * VEC;
  if constexpr (VEC == 4) *reinterpret_cast<uint4*>(d) = __ldg(reinterpret_cast<const uint4*>(p));
  else *d = __ldg(p);
}

// Group id of every row from the split sizes (E <= 1024): one block scans the
// sizes into offsets in shared memory; then every thread labels rows with a
// binary search of the offsets.
__global__ void __launch_bounds__(1024) expand_splits_kernel(const int32_t* __restrict__ split, int E, int64_t R,
                                                             int32_t* __restrict__ ids, int32_t* status) {
  __shared__ int64_t s_off[1025];
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  const int64_t v = tid < E ? split[tid] : 0;
  if (v < 0) s_bad = 1;
  s_off[tid + 1] = v;
  if (tid == 0) s_off[0] = 0;
  __syncthreads();
  for (int d = 1; d < 1024; d <<= 1) {                  // inclusive scan of s_off[1..1024]
    const int64_t a = tid >= d ? s_off[tid + 1 - d] : 0;
    __syncthreads();
    s_off[tid + 1] += a;
    __syncthreads();
  }
  if (s_bad || s_off[E] != R) {
    if (blockIdx.x == 0 && tid == 0) report(status, MXG_ERR_OFFSETS);
  }
  const bool ok = !s_bad;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + tid; r < R;
       r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int id = -1;
    if (ok && r < s_off[E]) {
      int lo = 0, hi = E - 1;                          // the last e with s_off[e] <= r
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_off[mid] <= r) lo = mid;
        else hi = mid - 1;
      }
      id = lo;
    }
    ids[r] = id;
  }
}

// One CTA per padded row: 16-byte code chunks by the threads, then the
// row's scale bytes, each to its tensor-core-layout position.
__global__ void __launch_bounds__(128) place_rows_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s,
                                                         int64_t src_rows, const int32_t* __restrict__ src,
                                                         const int32_t* rows_valid, int cols,
                                                         uint8_t* __restrict__ q_out, uint8_t* __restrict__ s_out,
                                                         int64_t sf_rows, const float* __restrict__ probs,
                                                         float* __restrict__ probs_perm, int32_t* status) {
  const int64_t p = blockIdx.x;
  if (rows_valid != nullptr && p >= *rows_valid) return;
  int f = src[p];
  if (f >= src_rows) {
    if (threadIdx.x == 0) report(status, MXG_ERR_INDEX);
    f = -1;
  }
  const int chunks = cols / 16;
  uint4* dq = reinterpret_cast<uint4*>(q_out + p * cols);
  const uint4* sq = f >= 0 ? reinterpret_cast<const uint4*>(q + static_cast<int64_t>(f) * cols) : nullptr;
  for (int c = threadIdx.x; c < chunks; c += blockDim.x) dq[c] = f >= 0 ? __ldg(sq + c) : make_uint4(0u, 0u, 0u, 0u);
  const int nb = cols / 32;
  for (int b = threadIdx.x; b < nb; b += blockDim.x)
    s_out[sf_mma_offset(p, b, sf_rows)] = f >= 0 ? s[static_cast<int64_t>(f) * nb + b] : uint8_t{0};
  if (probs_perm != nullptr && threadIdx.x == 0) probs_perm[p] = f >= 0 ? probs[f] : 0.f;
}

}  // namespace

cudaError_t launch_place_rows(const uint8_t* q, const uint8_t* s, int64_t src_rows, const int32_t* src, int64_t rows,
                              const int32_t* rows_valid, int cols, uint8_t* q_out, uint8_t* s_out, int64_t sf_rows,
                              const float* probs, float* probs_perm, int32_t* status, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  place_rows_kernel<<<static_cast<unsigned>(rows), 128, 0, st>>>(q, s, src_rows, src, rows_valid, cols, q_out, s_out,
                                                                 sf_rows, probs, probs_perm, status);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void* src, int64_t src_rows, int64_t row_bytes, const int32_t* index, int div,
                               int64_t rows, void* dst, int32_t* status, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const bool v16 = row_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
  const int64_t words = row_bytes / 4;
  const int64_t n = rows * (v16 ? words / 4 : words);
  const int64_t grid = (n + 255) / 256;
  if (v16)
    gather_rows_kernel<4><<<static_cast<unsigned>(grid), 256, 0, s>>>(
        static_cast<const uint32_t*>(src), src_rows, words, index, div, rows, static_cast<uint32_t*>(dst), status);
  else
    gather_rows_kernel<1><<<static_cast<unsigned>(grid), 256, 0, s>>>(
        static_cast<const uint32_t*>(src), src_rows, words, index, div, rows, static_cast<uint32_t*>(dst), status);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_expand_splits(const int32_t* split_sizes, int E, int64_t R, int32_t* ids, int32_t* status,
                                 cudaStream_t s) {
  if (R <= 0) return cudaSuccess;
  const int64_t want = (R + 1023) / 1024;
  const unsigned grid = static_cast<unsigned>(want < 1216 ? want : 1216);   // 8 blocks per SM at most
  expand_splits_kernel<<<grid, 1024, 0, s>>>(split_sizes, E, R, ids, status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mxg
