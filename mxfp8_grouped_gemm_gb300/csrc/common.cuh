// Shared device helpers: status reporting, bf16 packing, MXFP8 encoding and
// the tensor-core scale-factor layout.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <cstdint>

#include "mxg.h"

namespace mxg {

// A kernel wait that has not completed after this long gives up and reports
// MXG_ERR_TIMEOUT (all legitimate waits are microseconds).
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void report(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// ------------------------------------------------------------- bf16 helpers
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Two fp32 -> packed bf16x2 (round to nearest even); lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Packed fp32 pairs (the f32x2 forms of add, sub, mul and fma, sm_100 and
// later): one instruction for two lanes, each rounded exactly like the scalar
// instruction (round to nearest even, no flush to zero).
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{.reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n add.rn.f32x2 rd, ra, rb;\n"
      " mov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  float2 d;
  asm("{.reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n sub.rn.f32x2 rd, ra, rb;\n"
      " mov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{.reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mul.rn.f32x2 rd, ra, rb;\n"
      " mov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{.reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
      " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
// ------------------------------------------------------------ MXFP8 encode
// Scale byte from the bit pattern of a block's max magnitude (a finite fp32
// >= 0): shared exponent floor(log2 amax) - 8, clamped at -127, plus bias 127.
// For a normal amax with exponent field Ef that is Ef - 8; below 2^-119 (and
// for zero) it clamps to byte 0.
__device__ __forceinline__ uint32_t mx_scale_byte(uint32_t amax_bits) {
  const int ef = static_cast<int>(amax_bits >> 23);
  return static_cast<uint32_t>(ef > 8 ? ef - 8 : 0);
}

// 2^(127 - byte) as fp32: the factor that brings the block into E4M3 range.
__device__ __forceinline__ float mx_inv_scale(uint32_t byte) {
  return __uint_as_float((254u - byte) << 23);
}

// Per-tensor FP8 (current scaling): the MX scale rule with a whole tensor as
// the block, from the tensor's largest magnitude amax: codes are E4M3(v *
// fp8_scale(amax)), fp8_scale = 2^-(floor(log2 amax) - 8) (clamped like the
// E8M0 byte); a GEMM on two such operands multiplies its fp32 accumulator by
// fp8_dequant(amax_a) * fp8_dequant(amax_b), both exact powers of two.
__device__ __forceinline__ float fp8_scale(float amax) {
  return mx_inv_scale(mx_scale_byte(__float_as_uint(amax) & 0x7fffffffu));
}
__device__ __forceinline__ float fp8_dequant(float amax) {
  return __uint_as_float(mx_scale_byte(__float_as_uint(amax) & 0x7fffffffu) << 23);
}

// Two fp32 -> two E4M3 codes (round to nearest even, saturate to +-448);
// a in the low byte, b in the high byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// Four fp32 -> four E4M3 codes in one word (a in the lowest byte).
__device__ __forceinline__ uint32_t cvt_e4m3x4(float a, float b, float c, float d) {
  uint32_t r;
  asm("{.reg .b16 lo, hi;\n cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n"
      " mov.b32 %0, {lo, hi};}"
      : "=r"(r) : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}

// 32 values already multiplied by the inverse scale -> 32 codes in 8 words.
__device__ __forceinline__ void encode32(const float (&v)[32], uint32_t (&w)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t lo = cvt_e4m3x2(v[4 * i + 0], v[4 * i + 1]);
    const uint32_t hi = cvt_e4m3x2(v[4 * i + 2], v[4 * i + 3]);
    w[i] = lo | (hi << 16);
  }
}

// The same codes with each word packed by one move (the quantiser's form:
// measured faster there, a little slower inside the GEMM epilogues).
__device__ __forceinline__ void encode32_x4(const float (&v)[32], uint32_t (&w)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = cvt_e4m3x4(v[4 * i + 0], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

// ----------------------------------------------------------------- top-k
// One warp routes one token: lane l holds logits l, l+32, ... (E <= 256); k
// rounds of a warp argmax (ties to the lower id) pick the experts in
// descending order, then softmax over the chosen logits.  `row` may be global
// or shared memory.
// Returns, on lane j < k, the id it wrote to ids_out[j].
__device__ __forceinline__ int warp_topk_softmax(const float* row, int E, int k, int lane, int32_t* ids_out,
                                                 float* probs_out) {
  float v[8];
  uint32_t taken = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int e = lane + 32 * q;
    v[q] = e < E ? row[e] : -FLT_MAX;
    if (e >= E) taken |= 1u << q;
  }
  float my_val = 0.f;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -FLT_MAX;
    int bi = 0x7fffffff;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (!(taken >> q & 1u) && (bi == 0x7fffffff || v[q] > bv)) {   // first max within the lane = lowest id
        bv = v[q];
        bi = lane + 32 * q;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_val = bv;
      my_id = bi;
    }
  }
  const float vmax = __shfl_sync(0xffffffffu, my_val, 0);
  const float w = lane < k ? expf(my_val - vmax) : 0.f;
  float sum = w;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane < k) {
    ids_out[lane] = my_id;
    probs_out[lane] = w / sum;
  }
  return my_id;
}

// The same route by one thread (E <= 64, k <= 8): k passes over the row pick
// the largest untaken logit (ties to the lower id), and the softmax sums the
// chosen weights in the order of the warp version's butterfly
// ((w0 + w4) + (w2 + w6)) + ((w1 + w5) + (w3 + w7)) (missing terms are
// zeros), so ids and probabilities are bit-identical to warp_topk_softmax.
// Writes ids_out[0..k) and probs_out[0..k); sel[0..k) receives the ids.
__device__ __forceinline__ void thread_topk_softmax(const float* row, int E, int k, int32_t* ids_out,
                                                   float* probs_out, int (&sel)[8]) {
  float val[8];
  uint64_t taken = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    sel[j] = 0;
    val[j] = 0.f;
    if (j >= k) continue;
    float bv = -FLT_MAX;
    int bi = -1;
    for (int e = 0; e < E; ++e) {
      const float v = row[e];
      if (!((taken >> e) & 1ull) && (bi < 0 || v > bv)) {
        bv = v;
        bi = e;
      }
    }
    taken |= 1ull << bi;
    val[j] = bv;
    sel[j] = bi;
  }
  float w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = j < k ? expf(val[j] - val[0]) : 0.f;
  const float sum = ((w[0] + w[4]) + (w[2] + w[6])) + ((w[1] + w[5]) + (w[3] + w[7]));
#pragma unroll
  for (int j = 0; j < 8; ++j)
    if (j < k) {
      ids_out[j] = sel[j];
      probs_out[j] = w[j] / sum;
    }
}

// ------------------------------------------------------- scale-factor layout
// Byte offset of the scale of (row r, 32-block b) for a matrix with `rows`
// rows (multiple of 128): 512-byte atoms of 128 rows x 4 blocks, K-chunk-major.
// Inside an atom, 32 "lines" of 16 bytes: line (r%32) holds the 4 blocks of
// rows r%32, 32+r%32, 64+r%32, 96+r%32 — what the tensor core's 32x128b
// shared->TMEM copy expects.
__host__ __device__ __forceinline__ int64_t sf_mma_offset(int64_t r, int64_t b, int64_t rows) {
  return ((b >> 2) * (rows >> 7) + (r >> 7)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (b & 3);
}

__host__ __device__ __forceinline__ int64_t sf_offset(int layout, int64_t r, int64_t b, int64_t rows,
                                                       int64_t nblocks) {
  return layout == MXG_LAYOUT_MMA ? sf_mma_offset(r, b, rows) : r * nblocks + b;
}

}  // namespace mxg
