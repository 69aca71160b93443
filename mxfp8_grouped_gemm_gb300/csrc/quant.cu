// MXFP8 quantiser: bf16 -> E4M3 codes + E8M0 scales, row-wise (blocks of 32
// along a row) and/or column-wise (blocks of 32 consecutive rows, stored
// transposed), with an optional row gather.  One pass over the source serves
// the activations (gathered into the per-expert padded layout, both
// orientations), the weights (both orientations, batched over experts) and the
// standalone call.
//
// Format: BioNeMo Uses Grouped Kernels and MXFP8, "Reducing memory pressure
// with MXFP8", Fig. 3 (E4M3 values, one E8M0 scale per 32 consecutive values).
// Scale rule: OCP MX v1.0 (floor(log2 amax) - 8, clamp, RNE, saturate).
#include "common.cuh"
#include "kernels.h"

namespace mxg {

namespace {

constexpr int kRows = 32;    // rows per CTA tile (one column-wise block)
constexpr int kCols = 128;   // columns per CTA tile (four row-wise blocks)
constexpr int kPad = 8;      // smem row padding (bf16 elements)

__global__ void __launch_bounds__(128) quant_kernel(const QuantParams P) {
  __shared__ __align__(16) uint16_t tile[kRows][kCols + kPad];
  const int p0 = blockIdx.x * kRows;
  const int c0 = blockIdx.y * kCols;
  const int b = blockIdx.z;
  const int tid = threadIdx.x;
  if (P.rows_valid != nullptr && p0 >= *P.rows_valid) return;

  const uint16_t* xb = P.x + static_cast<int64_t>(b) * P.x_batch_stride;
  // 32 rows x 128 bf16 = 512 vectors of 16 bytes
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int i = tid + it * 128;
    const int r = i >> 4, v = i & 15;
    const int p = p0 + r;
    int64_t srow = p;
    bool zero = false;
    if (P.src_rows != nullptr) {
      const int f = P.src_rows[p];
      if (f < 0) zero = true;
      else srow = f / P.src_div;
    }
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (!zero) val = *reinterpret_cast<const uint4*>(xb + srow * P.ld_x + c0 + v * 8);
    *reinterpret_cast<uint4*>(&tile[r][v * 8]) = val;
  }
  if (P.probs_perm != nullptr && blockIdx.y == 0 && b == 0 && tid < kRows) {
    const int p = p0 + tid;
    const int f = P.src_rows != nullptr ? P.src_rows[p] : p;
    P.probs_perm[p] = f < 0 ? 0.f : P.probs[f];
  }
  __syncthreads();

  if (P.q_row != nullptr) {
    // thread -> (row r, 32-column block j)
    const int r = tid >> 2, j = tid & 3;
    float v[32];
    uint32_t amax = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      v[i] = bf16_bits_to_float(tile[r][j * 32 + i]);
      amax = max(amax, __float_as_uint(v[i]) & 0x7fffffffu);
    }
    const uint32_t sb = mx_scale_byte(amax);
    const float inv = mx_inv_scale(sb);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] *= inv;
    uint32_t w[8];
    encode32(v, w);
    const int64_t grow = static_cast<int64_t>(b) * P.rows + p0 + r;
    uint4* dst = reinterpret_cast<uint4*>(P.q_row + grow * P.cols + c0 + j * 32);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    int64_t srow = grow;
    if (P.sf_row_interleave > 0) {
      const int half = P.sf_row_interleave;
      const int lr = p0 + r;
      const int jj = lr % half;
      srow = static_cast<int64_t>(b) * P.rows + (jj / 64) * 128 + (lr / half) * 64 + (jj % 64);
    }
    P.s_row[sf_offset(P.layout, srow, (c0 >> 5) + j, P.sf_row_rows, P.cols >> 5)] = static_cast<uint8_t>(sb);
  }

  if (P.q_col != nullptr) {
    // thread -> column c0 + tid, the 32 rows of this tile form one block
    float v[32];
    uint32_t amax = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      v[i] = bf16_bits_to_float(tile[i][tid]);
      amax = max(amax, __float_as_uint(v[i]) & 0x7fffffffu);
    }
    const uint32_t sb = mx_scale_byte(amax);
    const float inv = mx_inv_scale(sb);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] *= inv;
    uint32_t w[8];
    encode32(v, w);
    const int64_t gcol = static_cast<int64_t>(b) * P.cols + c0 + tid;
    uint4* dst = reinterpret_cast<uint4*>(P.q_col + gcol * P.ld_col + p0);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    P.s_col[sf_offset(P.layout, gcol, p0 >> 5, P.sf_col_rows, P.ld_col >> 5)] = static_cast<uint8_t>(sb);
  }
}

}  // namespace

cudaError_t launch_quant(const QuantParams& p, cudaStream_t s) {
  dim3 grid(p.rows / kRows, p.cols / kCols, p.batch);
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
  quant_kernel<<<grid, 128, 0, s>>>(p);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mxg
