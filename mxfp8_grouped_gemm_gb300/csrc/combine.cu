// Unpermute/combine and the routing-probability gradient reduction.
//
// BioNeMo Uses Grouped Kernels and MXFP8, Fig. 1: expert outputs are combined
// per token as a weighted sum.  The weight (routing probability) is already
// applied inside ScaledSwiGLU ("Fusing precision conversion and expert
// computation"), so the combine sums the token's k expert rows:
//   y[t] = sum_j Y[row(t, j)]   (fp32 accumulation in j order, bf16 store).
#include "common.cuh"
#include "kernels.h"

namespace mxg {

namespace {

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4& q) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] += __uint_as_float(w[i] << 16);
    acc[2 * i + 1] += __uint_as_float(w[i] & 0xffff0000u);
  }
}

// One thread per 8 consecutive columns (16-byte vectors) of one token.  Up to
// eight slots, the thread requests all its row indices and then all its rows
// before it adds any (the adds still run in slot order), so k loads are in
// flight per thread instead of one dependent pair at a time.
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ src,
                                                      const int32_t* __restrict__ prow_of_src, int T, int k,
                                                      int H, uint16_t* __restrict__ out, int64_t src_rows,
                                                      int32_t* status) {
  const int vecs = H >> 3;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(T) * vecs) return;
  const int t = static_cast<int>(idx / vecs);
  const int v = static_cast<int>(idx % vecs);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  if (k <= 8) {
    int pr[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) pr[j] = j < k ? prow_of_src[static_cast<int64_t>(t) * k + j] : -1;
    uint4 q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (pr[j] >= src_rows) {
        if (v == 0) report(status, MXG_ERR_INDEX);
        pr[j] = -1;
      }
      q[j] = pr[j] >= 0 ? *reinterpret_cast<const uint4*>(src + static_cast<int64_t>(pr[j]) * H + v * 8)
                        : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (pr[j] >= 0) add_bf16x8(acc, q[j]);
  } else {
    for (int j = 0; j < k; ++j) {
      const int pr = prow_of_src[static_cast<int64_t>(t) * k + j];
      if (pr < 0) continue;
      if (pr >= src_rows) {
        if (v == 0) report(status, MXG_ERR_INDEX);
        continue;
      }
      add_bf16x8(acc, *reinterpret_cast<const uint4*>(src + static_cast<int64_t>(pr) * H + v * 8));
    }
  }
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  *reinterpret_cast<uint4*>(out + static_cast<int64_t>(t) * H + v * 8) = o;
}

// dprobs[f] = sum over column tiles of the per-row partials of its padded row.
__global__ void __launch_bounds__(256) dprob_kernel(const float* __restrict__ part, int ld,
                                                    const int32_t* __restrict__ prow_of_src, int R,
                                                    float* __restrict__ dprobs) {
  const int f = blockIdx.x * blockDim.x + threadIdx.x;
  if (f >= R) return;
  const int pr = prow_of_src[f];
  float s = 0.f;
  if (pr >= 0)
    for (int i = 0; i < ld; ++i) s += part[static_cast<int64_t>(pr) * ld + i];
  dprobs[f] = s;
}

}  // namespace

cudaError_t launch_combine(const uint16_t* src, const int32_t* prow_of_src, int T, int k, int H, uint16_t* out,
                           cudaStream_t s, int64_t src_rows, int32_t* status) {
  const int64_t n = static_cast<int64_t>(T) * (H / 8);
  const int64_t grid = (n + 255) / 256;
  if (grid == 0) return cudaSuccess;
  combine_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(src, prow_of_src, T, k, H, out, src_rows, status);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_dprob(const float* part, int ld, const int32_t* prow_of_src, int R, float* dprobs,
                         cudaStream_t s) {
  const int grid = (R + 255) / 256;
  if (grid == 0) return cudaSuccess;
  dprob_kernel<<<grid, 256, 0, s>>>(part, ld, prow_of_src, R, dprobs);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mxg
