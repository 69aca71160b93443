// MXFP8 quantiser: bf16 -> E4M3 codes + E8M0 scales, row-wise (blocks of 32
// along a row) and/or column-wise (blocks of 32 consecutive rows, stored
// transposed), with an optional row gather.  One pass over the source serves
// the activations (gathered into the per-expert padded layout, both
// orientations), the weights (both orientations, batched over experts) and the
// standalone call.
//
// Format: BioNeMo Uses Grouped Kernels and MXFP8, "Reducing memory pressure
// with MXFP8", Fig. 3 (E4M3 values, one E8M0 scale per 32 consecutive values).
// The same pass also serves the BF16 path: gathered and transposed bf16
// copies (b_row / b_col) instead of codes.
// Scale rule: OCP MX v1.0 (floor(log2 amax) - 8, clamp, RNE, saturate).
#include "common.cuh"
#include "kernels.h"

namespace mxg {

namespace {

constexpr int kRows = 32;    // rows per CTA tile (one column-wise block)
constexpr int kCols = 128;   // columns per CTA tile (four row-wise blocks)
constexpr int kStride = kCols + 8;   // bf16 per smem row (272 bytes: 16-byte aligned, spreads banks)

// Shared-memory position of 16-byte chunk c of staged row r: chunks are
// permuted by XOR with 2*((r/8)%4), so that the eight rows of one transposed
// 8x8 load (rows 2m + {0,1,8,9,16,17,24,25}) fall in eight different bank
// groups.
__device__ __forceinline__ int chunk_pos(int r, int c) { return c ^ (((r >> 3) & 3) << 1); }

// Largest magnitude of packed bf16 pairs, as fp32 bits: max.xorsign.abs
// keeps the larger magnitude of each lane pair (its sign bit, the XOR of the
// operands' signs, is cleared at the end), one instruction per word.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t pair_max_bits(const uint32_t* w, int n) {
  uint32_t m = w[0];
#pragma unroll
  for (int i = 1; i < n; ++i) m = absmax_bf16x2(m, w[i]);
  m &= 0x7fff7fffu;
  return max(m << 16, m & 0xffff0000u);
}

__device__ __forceinline__ void quant_store32(float (&v)[32], uint8_t* dst, uint8_t* sdst, uint32_t amax) {
  const uint32_t sb = mx_scale_byte(amax);
  const float2 inv = make_float2(mx_inv_scale(sb), mx_inv_scale(sb));
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float2 t = mul2(make_float2(v[i], v[i + 1]), inv);
    v[i] = t.x;
    v[i + 1] = t.y;
  }
  uint32_t w[8];
  encode32_x4(v, w);
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(w[0], w[1], w[2], w[3]);
  d[1] = make_uint4(w[4], w[5], w[6], w[7]);
  *sdst = static_cast<uint8_t>(sb);
}

// Per-tensor FP8: the thread's 32 values times the tensor's scale, as codes.
__device__ __forceinline__ void quant_store32_pt(float (&v)[32], uint8_t* dst, float s) {
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] *= s;
  uint32_t w[8];
  encode32_x4(v, w);
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(w[0], w[1], w[2], w[3]);
  d[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
               "l"(gsrc)
               : "memory");
}

// Four 8x8 bf16 matrices from shared memory, transposed: thread t receives,
// for matrix m, the two elements (rows 2(t%4), 2(t%4)+1; column t/4) of that
// matrix as one packed word.  Threads 8m..8m+7 give the row addresses of m.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t saddr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(saddr));
}

// Column-wise MX of one warp's 32-row x 32-column block (columns col0..+31 of
// the staged tile): ldmatrix.trans hands each quad of lanes one column with
// lane j of the quad holding rows 8j..8j+7 in order (the row addresses are
// permuted so that matrix m's fragment rows 2j, 2j+1 are tile rows 8j+2m,
// 8j+2m+1); the quad reduces the block maximum with two shuffles and each lane
// writes its 8 codes as one 8-byte store.
template <bool PT>
__device__ __forceinline__ void quant_col_block(const QuantParams& P, const uint16_t* buf, int col0, int64_t gcol0,
                                                int p0, int lane, float pt_s) {
  const int m = lane >> 3, i = lane & 7;
  const int srow = 8 * (i >> 1) + 2 * m + (i & 1);
  const uint16_t* rowp = buf + srow * kStride;
  const int j = lane & 3;
  // this lane's output column for ct = 0 and the steps to the next 8 columns:
  // the codes' row (column of x) advances by 8, and so does the scale's row
  // (inside one 32-row group of the tensor-core layout: 8 rows = 128 bytes)
  const int64_t gc = gcol0 + (lane >> 2);
  uint8_t* qdst = P.q_col + gc * P.ld_col + p0 + 8 * j;
  const int64_t qstep = 8 * P.ld_col;
  const bool store_scale = j == 0 && !PT;
  int64_t soff = 0, sstep = 0;
  if (store_scale) {
    soff = sf_offset(P.layout, gc, p0 >> 5, P.sf_col_rows, P.ld_col >> 5);
    sstep = P.layout == MXG_LAYOUT_MMA ? 128 : 8 * (P.ld_col >> 5);
  }
#pragma unroll
  for (int ct = 0; ct < 4; ++ct) {
    uint32_t r[4];
    ldsm_x4_trans(static_cast<uint32_t>(__cvta_generic_to_shared(rowp + chunk_pos(srow, (col0 >> 3) + ct) * 8)), r);
    float v[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      v[2 * q] = __uint_as_float(r[q] << 16);
      v[2 * q + 1] = __uint_as_float(r[q] & 0xffff0000u);
    }
    uint32_t sb = 0;
    float inv = pt_s;                         // per-tensor FP8: the tensor's scale
    if constexpr (!PT) {                      // MX: the block's own scale
      uint32_t amax = pair_max_bits(r, 4);
      amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      sb = mx_scale_byte(amax);
      inv = mx_inv_scale(sb);
    }
    uint32_t w[2];
    const float2 inv2 = make_float2(inv, inv);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float2 lo = mul2(make_float2(v[4 * q], v[4 * q + 1]), inv2);
      const float2 hi = mul2(make_float2(v[4 * q + 2], v[4 * q + 3]), inv2);
      w[q] = cvt_e4m3x4(lo.x, lo.y, hi.x, hi.y);
    }
    *reinterpret_cast<uint2*>(qdst + ct * qstep) = make_uint2(w[0], w[1]);
    if (store_scale) P.s_col[soff + ct * sstep] = static_cast<uint8_t>(sb);
  }
}

// Transposed bf16 copy of one warp's 32-row x 32-column block: the same
// transposed loads as quant_col_block, each lane writing its column's 8
// consecutive rows as one 16-byte store.
__device__ __forceinline__ void copy_col_block(const QuantParams& P, const uint16_t* buf, int col0, int64_t gcol0,
                                               int p0, int lane) {
  const int m = lane >> 3, i = lane & 7;
  const int srow = 8 * (i >> 1) + 2 * m + (i & 1);
  const uint16_t* rowp = buf + srow * kStride;
  const int j = lane & 3;
#pragma unroll
  for (int ct = 0; ct < 4; ++ct) {
    uint32_t r[4];
    ldsm_x4_trans(static_cast<uint32_t>(__cvta_generic_to_shared(rowp + chunk_pos(srow, (col0 >> 3) + ct) * 8)), r);
    const int64_t gcol = gcol0 + ct * 8 + (lane >> 2);
    *reinterpret_cast<uint4*>(P.b_col + gcol * P.ld_col + p0 + 8 * j) = make_uint4(r[0], r[1], r[2], r[3]);
  }
}

constexpr int kTilesPerCta = 8;      // 32-row tiles walked by one CTA

// Stage one 32 x 128 tile into shared memory asynchronously.  Thread tid
// copies 16-byte chunk tid % 16 of rows tid / 16 + 8 i (i < 4).  Gathered
// rows: s_off holds each of the CTA's rows' element offset from x (-1: a zero
// padding row), so a copy is one shared load, one add and the copy.
template <bool GATHER>
__device__ __forceinline__ void stage_tile(const uint16_t* xc, int64_t ld_x, int p0, int rel0, uint16_t* buf, int tid,
                                           const int64_t* s_off) {
  const int vv = tid & 15;
#pragma unroll
  for (int it = 0; it < 4; ++it) {
    const int rr = (tid >> 4) + it * 8;
    uint16_t* dst = buf + rr * kStride + chunk_pos(rr, vv) * 8;
    if constexpr (GATHER) {
      const int64_t off = s_off[rel0 + rr];
      if (off < 0) *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      else cp_async16(dst, xc + off);
    } else {
      cp_async16(dst, xc + static_cast<int64_t>(p0 + rr) * ld_x);
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// One CTA walks up to kTilesPerCta tiles of 32 rows x 128 columns, loading
// tile t+1 (asynchronous 16-byte copies into the other shared buffer) while it
// quantises tile t.  Row-wise: thread t quantises the 32-value block (row t/4,
// columns 32*(t%4)..) read back with 16-byte loads.  Column-wise: warp w
// quantises columns 32w..32w+31 over the tile's 32 rows from transposed
// matrix loads (quant_col_block).  The mode (gathered rows, row-wise and
// column-wise outputs, per-tensor scale) is a template argument, so the tile
// loop carries no run-time mode tests; the bf16 pass-through outputs of the
// BF16 path stay run-time options.  Ten CTAs per SM (48 registers, no spills):
// the kernel waits mostly on shared-memory and shuffle results, and two more
// CTAs than eight gave the gathered passes 2 % (twelve spill and lose 2-6 %).
template <bool GATHER, bool ROW, bool COL, bool PT>
__device__ __forceinline__ void quant_tiles(const QuantParams& P, int bx, int by, int bz) {
  __shared__ __align__(16) uint16_t tile[2][kRows * kStride];
  __shared__ int64_t s_off[GATHER ? kTilesPerCta * kRows : 1];
  const int c0 = by * kCols;
  const int b = bz;
  const int tid = threadIdx.x;
  const int first = bx * kTilesPerCta * kRows;
  int limit = P.rows;
  if (P.rows_valid != nullptr) limit = min(limit, *P.rows_valid);
  const int ntiles = min(kTilesPerCta, (limit - first + kRows - 1) / kRows);
  if (ntiles <= 0) return;
  const uint16_t* xb = P.x + static_cast<int64_t>(b) * P.x_batch_stride;
  const uint16_t* xc = xb + c0 + (tid & 15) * 8;      // this thread's 16-byte column chunk
  if constexpr (GATHER) {
    // the CTA's source rows resolved once: a row map entry divided by the
    // number of rows per source row, or a search of the group offsets
    for (int i = tid; i < ntiles * kRows; i += 128) {
      const int p = first + i;
      int f = -1;
      if (P.src_rows != nullptr) {
        const int v = P.src_rows[p];
        f = v < 0 ? -1 : (P.src_div == 1 ? v : v / P.src_div);
      } else if (p < limit) {
        int lo = 0, hi = P.groups - 1;     // the last group g with grp_poff[g] <= p
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (P.grp_poff[mid] <= p) lo = mid;
          else hi = mid - 1;
        }
        const int src = P.grp_off[lo] + (p - P.grp_poff[lo]);
        f = src < P.grp_off[lo + 1] ? src : -1;
      }
      s_off[i] = f < 0 ? int64_t{-1} : static_cast<int64_t>(f) * P.ld_x;
    }
    __syncthreads();
    if (P.probs_perm != nullptr && blockIdx.y == 0 && b == 0) {
      for (int i = tid; i < ntiles * kRows; i += 128) {
        const int pp = first + i;
        const int f = P.src_rows != nullptr ? P.src_rows[pp] : pp;
        P.probs_perm[pp] = f < 0 ? 0.f : P.probs[f];
      }
    }
  }

  stage_tile<GATHER>(xc, P.ld_x, first, 0, tile[0], tid, s_off);
  for (int t = 0; t < ntiles; ++t) {
    const int p0 = first + t * kRows;
    if (t + 1 < ntiles) {
      stage_tile<GATHER>(xc, P.ld_x, p0 + kRows, (t + 1) * kRows, tile[(t + 1) & 1], tid, s_off);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const uint16_t* buf = tile[t & 1];
    float pt_s = 1.f;
    if constexpr (PT) {
      int g = b;
      if (P.pt_group_off != nullptr) {      // the row group holding this tile (groups are 32-row aligned)
        g = 0;
        while (g + 1 < P.pt_groups && P.pt_group_off[g + 1] <= p0) ++g;
      }
      pt_s = fp8_scale(P.pt_amax[g]);
    }
    if constexpr (ROW) {
      const int r = tid >> 2, j = tid & 3;
      const int p = p0 + r;
      float v[32];
      uint32_t wv[16];
      const uint4* s4 = reinterpret_cast<const uint4*>(buf + r * kStride);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 q = s4[chunk_pos(r, 4 * j + i)];
        wv[4 * i] = q.x;
        wv[4 * i + 1] = q.y;
        wv[4 * i + 2] = q.z;
        wv[4 * i + 3] = q.w;
      }
      const uint32_t blk_max = PT ? 0u : pair_max_bits(wv, 16);
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        v[2 * h] = __uint_as_float(wv[h] << 16);
        v[2 * h + 1] = __uint_as_float(wv[h] & 0xffff0000u);
      }
      const int64_t grow = static_cast<int64_t>(b) * P.rows + p;
      if constexpr (PT)
        quant_store32_pt(v, P.q_row + grow * P.cols + c0 + j * 32, pt_s);
      else
        quant_store32(v, P.q_row + grow * P.cols + c0 + j * 32,
                      P.s_row + sf_offset(P.layout, grow, (c0 >> 5) + j, P.sf_row_rows, P.cols >> 5),
                      blk_max);
    }
    if constexpr (COL) {
      const int warp = tid >> 5;
      quant_col_block<PT>(P, buf, warp * 32, static_cast<int64_t>(b) * P.cols + c0 + warp * 32, p0, tid & 31, pt_s);
    }
    if (P.b_row != nullptr) {
      const int r = tid >> 2, j = tid & 3;
      const uint4* s4 = reinterpret_cast<const uint4*>(buf + r * kStride);
      uint4* d = reinterpret_cast<uint4*>(P.b_row + (static_cast<int64_t>(b) * P.rows + p0 + r) * P.cols + c0 + j * 32);
#pragma unroll
      for (int i = 0; i < 4; ++i) d[i] = s4[chunk_pos(r, 4 * j + i)];
    }
    if (P.b_col != nullptr) {
      const int warp = tid >> 5;
      copy_col_block(P, buf, warp * 32, static_cast<int64_t>(b) * P.cols + c0 + warp * 32, p0, tid & 31);
    }
    __syncthreads();   // buffer t&1 is refilled two tiles later
  }
}

template <bool GATHER, bool ROW, bool COL, bool PT>
__global__ void __launch_bounds__(128, 10) quant_kernel(const QuantParams P) {
  quant_tiles<GATHER, ROW, COL, PT>(P, blockIdx.x, blockIdx.y, blockIdx.z);
}

// Two tensors of the same mode in one launch (the weights: W_gate_up, then
// W_down): blocks [0, n0) walk the first tensor's grid (gx0 x gy0 x batch,
// x fastest), the rest the second's.  As two launches, each ended with a
// partly filled last wave; here the second tensor's blocks fill the first's.
template <bool GATHER, bool ROW, bool COL, bool PT>
__global__ void __launch_bounds__(128, 10) quant_kernel2(const QuantParams P0, const QuantParams P1, int gx0, int gy0,
                                                          int n0, int gx1, int gy1) {
  const int id = static_cast<int>(blockIdx.x);
  if (id < n0) {
    quant_tiles<GATHER, ROW, COL, PT>(P0, id % gx0, (id / gx0) % gy0, id / (gx0 * gy0));
  } else {
    const int j = id - n0;
    quant_tiles<GATHER, ROW, COL, PT>(P1, j % gx1, (j / gx1) % gy1, j / (gx1 * gy1));
  }
}

// Largest magnitude per tensor: a CTA of 256 threads reads a 32-row x
// 256-column tile (thread t: row t/8, 32 columns, four 16-byte loads), reduces
// over the warp and adds one atomic maximum per warp (non-negative floats
// order like their bit patterns).
__global__ void __launch_bounds__(256) amax_kernel(const AmaxParams P) {
  const int b = blockIdx.z;
  const int p0 = blockIdx.x * 32;
  int limit = P.rows;
  if (P.rows_valid != nullptr) limit = min(limit, *P.rows_valid);
  if (p0 >= limit) return;
  const int p = p0 + (threadIdx.x >> 3);
  const int c = blockIdx.y * 256 + (threadIdx.x & 7) * 32;
  uint32_t m = 0;
  if (p < limit) {
    int64_t srow = p;
    if (P.src_rows != nullptr) {
      const int f = P.src_rows[p];
      srow = f < 0 ? -1 : f / P.src_div;
    }
    if (srow >= 0) {
      const uint4* src = reinterpret_cast<const uint4*>(P.x + static_cast<int64_t>(b) * P.x_batch_stride +
                                                        srow * P.ld_x + c);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 q = src[i];
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) m = max(m, max((w[h] << 16) & 0x7fffffffu, w[h] & 0x7fff0000u));
      }
    }
  }
  m = __reduce_max_sync(0xffffffffu, m);
  if ((threadIdx.x & 31) == 0 && m != 0) {
    int g = b;
    if (P.group_off != nullptr) {
      g = 0;
      while (g + 1 < P.groups && P.group_off[g + 1] <= p0) ++g;
    }
    atomicMax(reinterpret_cast<unsigned int*>(P.amax + g), m);
  }
}

// Padded offsets of grouped rows, one block: every thread takes a contiguous
// run of groups, checks them, sums their padded sizes; a block-wide scan of
// the run totals gives each run's start.
__global__ void __launch_bounds__(1024) group_pad_kernel(const int32_t* __restrict__ off, int groups, int rows,
                                                         int align, int64_t cap, int32_t* __restrict__ poff,
                                                         int32_t* status) {
  __shared__ int64_t s_tot[1024];
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  if (tid == 0) s_bad = (off[0] != 0 || off[groups] != rows) ? 1 : 0;
  const int per = (groups + blockDim.x - 1) / blockDim.x;
  const int g0 = min(groups, tid * per), g1 = min(groups, g0 + per);
  int64_t tot = 0;
  bool bad = false;
  for (int g = g0; g < g1; ++g) {
    const int a = off[g], b = off[g + 1];
    if (b < a) bad = true;
    tot += (static_cast<int64_t>(b - a) + align - 1) / align * align;
  }
  s_tot[tid] = tot;
  __syncthreads();
  if (bad) s_bad = 1;
  for (int d = 1; d < static_cast<int>(blockDim.x); d <<= 1) {      // inclusive scan of the run totals
    const int64_t v = tid >= d ? s_tot[tid - d] : 0;
    __syncthreads();
    s_tot[tid] += v;
    __syncthreads();
  }
  const bool fail = s_bad != 0 || s_tot[blockDim.x - 1] > cap;
  if (fail) {
    for (int g = tid; g <= groups; g += blockDim.x) poff[g] = 0;
    if (tid == 0) report(status, MXG_ERR_OFFSETS);
    return;
  }
  int64_t run = s_tot[tid] - tot;
  for (int g = g0; g < g1; ++g) {
    poff[g] = static_cast<int32_t>(run);
    run += (static_cast<int64_t>(off[g + 1] - off[g]) + align - 1) / align * align;
  }
  if (tid == blockDim.x - 1) poff[groups] = static_cast<int32_t>(s_tot[tid]);
}

}  // namespace

cudaError_t launch_group_pad(const int32_t* off, int groups, int rows, int align, int64_t cap, int32_t* poff,
                             int32_t* status, cudaStream_t s) {
  group_pad_kernel<<<1, 1024, 0, s>>>(off, groups, rows, align, cap, poff, status);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_amax(const AmaxParams& p, cudaStream_t s) {
  dim3 grid((p.rows + 31) / 32, p.cols / 256, p.batch);
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
  amax_kernel<<<grid, 256, 0, s>>>(p);
  count_launch();
  return cudaGetLastError();
}

template <bool G, bool R, bool C, bool PT>
void launch_mode(const QuantParams& p, dim3 grid, cudaStream_t s) {
  quant_kernel<G, R, C, PT><<<grid, 128, 0, s>>>(p);
}

static int quant_mode(const QuantParams& p) {
  return (p.src_rows != nullptr || p.grp_off != nullptr ? 1 : 0) | (p.q_row != nullptr ? 2 : 0) |
         (p.q_col != nullptr ? 4 : 0) | (p.pt_amax != nullptr ? 8 : 0);
}

static dim3 quant_grid(const QuantParams& p) {
  return dim3((p.rows / kRows + kTilesPerCta - 1) / kTilesPerCta, p.cols / kCols, p.batch);
}

cudaError_t launch_quant2(const QuantParams& a, const QuantParams& b, cudaStream_t s) {
  const dim3 ga = quant_grid(a), gb = quant_grid(b);
  const int64_t na = static_cast<int64_t>(ga.x) * ga.y * ga.z, nb = static_cast<int64_t>(gb.x) * gb.y * gb.z;
  // the same outputs as two launches; one launch needs one mode and a grid that fits
  if (quant_mode(a) != quant_mode(b) || na == 0 || nb == 0 || na + nb > INT32_MAX) {
    cudaError_t err = launch_quant(a, s);
    return err != cudaSuccess ? err : launch_quant(b, s);
  }
  const unsigned n = static_cast<unsigned>(na + nb);
  const int gx0 = static_cast<int>(ga.x), gy0 = static_cast<int>(ga.y), n0 = static_cast<int>(na);
  const int gx1 = static_cast<int>(gb.x), gy1 = static_cast<int>(gb.y);
  switch (quant_mode(a)) {
    case 6: quant_kernel2<false, true, true, false><<<n, 128, 0, s>>>(a, b, gx0, gy0, n0, gx1, gy1); break;
    case 2: quant_kernel2<false, true, false, false><<<n, 128, 0, s>>>(a, b, gx0, gy0, n0, gx1, gy1); break;
    default: {
      cudaError_t err = launch_quant(a, s);
      return err != cudaSuccess ? err : launch_quant(b, s);
    }
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_quant(const QuantParams& p, cudaStream_t s) {
  dim3 grid = quant_grid(p);
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
  const int mode = quant_mode(p);
  switch (mode) {
    case 0: launch_mode<false, false, false, false>(p, grid, s); break;
    case 1: launch_mode<true, false, false, false>(p, grid, s); break;
    case 2: launch_mode<false, true, false, false>(p, grid, s); break;
    case 3: launch_mode<true, true, false, false>(p, grid, s); break;
    case 4: launch_mode<false, false, true, false>(p, grid, s); break;
    case 5: launch_mode<true, false, true, false>(p, grid, s); break;
    case 6: launch_mode<false, true, true, false>(p, grid, s); break;
    case 7: launch_mode<true, true, true, false>(p, grid, s); break;
    case 10: launch_mode<false, true, false, true>(p, grid, s); break;
    case 11: launch_mode<true, true, false, true>(p, grid, s); break;
    case 12: launch_mode<false, false, true, true>(p, grid, s); break;
    case 13: launch_mode<true, false, true, true>(p, grid, s); break;
    case 14: launch_mode<false, true, true, true>(p, grid, s); break;
    case 15: launch_mode<true, true, true, true>(p, grid, s); break;
    default: return cudaErrorInvalidValue;   // a per-tensor scale without any code output
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace mxg
