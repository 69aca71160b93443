// Persistent grouped MXFP8 GEMM for sm_103a: TMA-fed, tcgen05 block-scaled
// MMA (kind::mxf8f6f4, E4M3 x E4M3, E8M0 scale per 32 along K), fp32
// accumulators in TMEM, warp-specialised.
//
// Grouping (BioNeMo Uses Grouped Kernels and MXFP8, "Grouping fragmented
// expert workloads"): every expert keeps its own weight matrix; one launch
// covers all experts.  Two shapes:
//   row-grouped   : rows [poff[e], poff[e+1]) of A use expert e's B
//                   (forward GEMMs and activation gradients);
//   token-grouped : the contraction runs over tokens [poff[e], poff[e+1]),
//                   one output matrix per expert (weight gradients).
// The tile scheduler reads the 128-aligned group offsets on the device; the
// host never sees the split sizes.
//
// Epilogues (TMEM -> registers, one thread per output row):
//   EPI_BF16    : store fp32 accumulators as bf16.
//   EPI_ACC_F32 : (weight gradients) add the fp32 accumulators into an fp32
//                 gradient buffer (main_grad accumulation across micro-batches).
//   EPI_SWIGLU  : gate-up tile = 128 gate + 128 up columns; h = p*SiLU(g)*u
//                 (ScaledSwiGLU, "Fusing precision conversion and expert
//                 computation"), re-quantised to MXFP8 row-wise (the down
//                 GEMM's A) and token-column-wise (the down wgrad's B); the
//                 pre-activation g|u is kept in bf16 for the backward (MXFP8:
//                 in 32 x 32 tiles, gu_tile_offset).
//   EPI_DSWIGLU : dH tile -> dg = dH p u s (1 + g (1-s)), du = dH p g s
//                 (s = sigmoid(g)), d(prob) partial sum_i dH g s u; dGU
//                 quantised row-wise (dgrad A) and token-column-wise (wgrad A).
//                 With BN = 256 the accumulator is single-buffered, so dH is
//                 first parked as bf16 pairs in spare TMEM columns and the
//                 accumulator released; the math then overlaps the next
//                 tile's MMAs, and the dGU codes leave through per-warp
//                 shared tiles by TMA stores.
//
// CTA = 12 warps: warp 0 issues TMA, warp 1 owns TMEM and issues the MMAs,
// warp 2 copies each stage's scale factors into TMEM, warps 4-11 run the
// epilogue (warp w reads TMEM lanes 32*(w%4)..+31, half of the tile's columns
// each).
// Tile 128 x BN x 128 (BN = 256 or 128) on one SM, or 256 x 256 x 128 on a
// CTA pair (cta_group::2: each SM holds its 128 rows of A and half of B, so
// the operand bytes per MMA flop drop by a third); 4-8-stage smem ring with a
// matching ring of scale-factor slots in TMEM; the accumulator is
// double-buffered in TMEM when it fits next to them (BN = 128).  Every wait is
// bounded; a wait that gives up records MXG_ERR_TIMEOUT, stops the CTA's
// pipeline and still frees TMEM.
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace mxg {

namespace {

constexpr int BM = 128;
constexpr int BK = 128;
// warp 0 TMA, warp 1 MMA, warp 2 scale-factor copies, warp 3 idle, warps 4-11
// epilogue (two per TMEM lane quadrant)
constexpr int kThreads = 384;

// Operand kinds: MXFP8 (E4M3 + E8M0 block scales in TMEM), bf16, and E4M3
// with one scale per expert tensor applied in the epilogue.
enum Opk { OPK_MX = 0, OPK_BF16 = 1, OPK_F8 = 2 };

template <int BN, int EPI, bool PAIR, int OPK = OPK_MX, bool KG = false>
struct Cfg {
  // contraction elements per stage: one 128-byte swizzle row of A and B
  static constexpr int kKElems = OPK == OPK_BF16 ? 64 : 128;
  static constexpr int CG = PAIR ? 2 : 1;
  static constexpr int kTileM = PAIR ? 2 * BM : BM;         // rows of one tile (both CTAs)
  static constexpr int kBRows = PAIR ? BN / 2 : BN;         // rows of B held by one CTA
  static constexpr int kAcc = BN == 128 ? 2 : 1;            // accumulator buffers in TMEM
  static constexpr int kABytes = BM * BK;
  static constexpr int kBBytes = kBRows * BK;
  static constexpr int kSfaBytes = OPK == OPK_MX ? BM * 4 : 0;   // 128 rows x 4 blocks of 32
  static constexpr int kSfbBytes = OPK == OPK_MX ? BN * 4 : 0;   // every CTA holds the tile's full SFB
  static constexpr uint32_t kTx = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kStageBytes = (kTx + 1023) / 1024 * 1024;
  // dSwiGLU at BN = 256 parks the tile's dH as packed bf16 in TMEM columns
  // [kDsCol, kDsCol + 128) so the accumulator is released before the epilogue
  // math.  MXFP8 gate-up and dSwiGLU at BN = 256: a 32 x 20-word scratch per
  // epilogue warp for the column-wise quantiser (20 KB, what a six-stage ring
  // leaves free); BN = 128 dSwiGLU keeps a 32 x 33 fp32 transpose tile per warp.
  static constexpr bool kDsTmem = EPI == 2 && BN == 256;
  static constexpr uint32_t kDsCol = 384;
  // MXFP8 dSwiGLU at BN = 256 stores its dGU codes by TMA through a 4 KB
  // shared tile per epilogue warp (epi_dswiglu_tma), beside the 2.5 KB
  // scratch: a five-stage ring.
  static constexpr bool kDsTma = EPI == 2 && BN == 256 && OPK == OPK_MX;
  static constexpr int kDsWarpBytes = 4096 + 32 * 20 * 4;
  // MXFP8 pair GEMMs with a bf16 epilogue (the weight gradients' dW, down,
  // dgrad-gate-up) or the fp32 main_grad epilogue write by TMA from a 2 KB
  // shared tile per epilogue warp (epi_tma_out; epi_bf16 when a combine is
  // fused, its stores completed before the combine counters): the ring keeps
  // six stages.
  static constexpr bool kTmaOut = PAIR && OPK == OPK_MX && (EPI == 0 || (KG && EPI == 3));
  // MXFP8 gate-up: the saved g|u leave as bulk copies through the column
  // quantiser's scratch
  static constexpr bool kSwTma = EPI == 1 && OPK == OPK_MX;
  static constexpr int kXposeBytes = kDsTma                                    ? 8 * kDsWarpBytes
                                     : kTmaOut                                 ? 8 * 2048
                                     : EPI == 2 && BN == 128                   ? 8 * 32 * 33 * 4
                                     : (EPI == 1 || EPI == 2) && OPK == OPK_MX ? 8 * 32 * 20 * 4
                                                                               : 0;
  static constexpr int kCtrlBytes = 2048;
  static constexpr int kStages = (232448 - 1024 - kCtrlBytes - kXposeBytes) / kStageBytes > 8
                                     ? 8
                                     : (232448 - 1024 - kCtrlBytes - kXposeBytes) / kStageBytes;
  // Scale factors in TMEM: one slot per smem stage (SFA 4 columns, then SFB
  // 4 per 128 rows), so the copy for the next K step never overwrites scales
  // that MMAs still in the tensor pipe are reading.
  static constexpr uint32_t kSfCol = kAcc * BN;             // first TMEM column of the slots
  static constexpr uint32_t kSfSlot = OPK == OPK_MX ? 4 + BN / 32 : 0;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kCtrlBytes + kXposeBytes;
  static_assert(kSfCol + kStages * kSfSlot <= (kDsTmem ? kDsCol : 512u), "TMEM budget");
  static_assert(kABytes == BM * 128, "stage rows are one 128-byte swizzle row");
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(!PAIR || BN == 256, "CTA-pair tiles are 256 x 256");
};

struct TileCoord {
  int e;      // expert
  int m0;     // first row of the tile (padded row, or row of D_e)
  int nt;     // column-tile index
  int kbeg;   // first contraction index
  int num_k;  // number of 128-wide contraction steps
};

__device__ __forceinline__ uint32_t f2u(float f) { return __float_as_uint(f); }
__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

// 32 bf16 of a read-only global row (64 bytes, 32-byte aligned) as fp32.
__device__ __forceinline__ void load_bf16_32(const uint16_t* src, float (&v)[32]) {
  uint32_t w[16];
  ld_global_nc_v8(src, w);
  ld_global_nc_v8(src + 16, w + 8);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    v[2 * j] = u2f(w[j] << 16);
    v[2 * j + 1] = u2f(w[j] & 0xffff0000u);
  }
}

// The MXFP8 path keeps the gate-up output g|u for the backward in 32 x 32
// tiles: the tile of rows 32·rb.. and columns 32·cb.. of the gate half (cb <
// I/32) starts at element (rb·I/32 + cb)·2048 and holds the gate block, then
// the up block of the same columns, each as two 16-column halves of 32 rows x
// 16 values (row r of half h at h·512 + r·16).  A warp owning the tile's 32
// rows reads each half as one contiguous kilobyte (lane r: its row's 32
// bytes), where rows of a [rows][2I] matrix are 4I bytes apart and every lane
// touched its own sector: those scattered loads slowed the concurrent MMAs of
// the dgrad-down GEMM (its tensor pipe by ~7 %).
__device__ __forceinline__ int64_t gu_tile_offset(int I, int tok0, int col) {
  return (static_cast<int64_t>(tok0 >> 5) * (I >> 5) + (col >> 5)) * 2048;
}

// Lane `lane`'s 32 values of one block (gate or up) of a g|u tile, as fp32.
__device__ __forceinline__ void load_gu_block32(const uint16_t* blk, int lane, float (&v)[32]) {
  uint32_t w[16];
  ld_global_nc_v8(blk + lane * 16, w);
  ld_global_nc_v8(blk + 512 + lane * 16, w + 8);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    v[2 * j] = u2f(w[j] << 16);
    v[2 * j + 1] = u2f(w[j] & 0xffff0000u);
  }
}

// Row-wise MX of one thread's 32 consecutive values: codes to dst (32 bytes),
// scale byte returned.
__device__ __forceinline__ uint32_t row_quant32(const float (&h)[32], uint8_t* dst) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(h[i]));
  const uint32_t sb = mx_scale_byte(f2u(amax));
  const float2 inv = make_float2(mx_inv_scale(sb), mx_inv_scale(sb));
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float2 t = mul2(make_float2(h[i], h[i + 1]), inv);
    v[i] = t.x;
    v[i + 1] = t.y;
  }
  uint32_t w[8];
  encode32(v, w);
  st_global_v8(dst, w);
  return sb;
}

// Row-wise MX of one thread's 32 values into a 32-row x 32-byte shared tile
// for a TMA store: row `lane` at lane·32, its two 16-byte halves swapped when
// bit 2 of the row is set (the tensor map's 32-byte swizzle: conflict-free).
// Returns the scale byte.
__device__ __forceinline__ uint32_t row_quant32_staged(const float (&h)[32], uint8_t* tile, int lane) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(h[i]));
  const uint32_t sb = mx_scale_byte(f2u(amax));
  const float2 inv = make_float2(mx_inv_scale(sb), mx_inv_scale(sb));
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float2 t = mul2(make_float2(h[i], h[i + 1]), inv);
    v[i] = t.x;
    v[i + 1] = t.y;
  }
  uint32_t w[8];
  encode32(v, w);
  const int sw = (lane >> 2) & 1;
  uint8_t* row = tile + lane * 32;
  *reinterpret_cast<uint4*>(row + (sw << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(row + ((sw ^ 1) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
  return sb;
}

// Column-wise MX of the warp's 32 x 32 block (lane l holds row tok0 + l; for
// each column col0 + i the 32 rows form one block, tok0 32-aligned and inside
// one expert group; codes go to qc[(col0 + i) * ld + tok0 + row]) through a
// 32 x 33 fp32 shared tile: the warp writes
// its 32 rows, each lane then reads one column (its 32 tokens), quantises it in
// registers and writes the 32 codes as one contiguous run of the transposed
// output.  Bank-conflict free in both directions.
__device__ __forceinline__ void col_quant32_xpose(const float (&h)[32], float* xp, uint8_t* qc, uint8_t* sc,
                                                  int64_t ld, int64_t sc_rows, int64_t col0, int64_t tok0,
                                                  int lane) {
#pragma unroll
  for (int i = 0; i < 32; ++i) xp[lane * 33 + i] = h[i];
  __syncwarp();
  float v[32];
  uint32_t amax = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = xp[i * 33 + lane];
    amax = max(amax, f2u(v[i]) & 0x7fffffffu);
  }
  __syncwarp();
  const uint32_t sb = mx_scale_byte(amax);
  const float inv = mx_inv_scale(sb);
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] *= inv;
  uint32_t w[8];
  encode32(v, w);
  uint4* d = reinterpret_cast<uint4*>(qc + (col0 + lane) * ld + tok0);
  d[0] = make_uint4(w[0], w[1], w[2], w[3]);
  d[1] = make_uint4(w[4], w[5], w[6], w[7]);
  sc[sf_mma_offset(col0 + lane, tok0 >> 5, sc_rows)] = static_cast<uint8_t>(sb);
}

// The same column-wise MX through the warp's own 32 x 16 fp32 scratch: lane
// l's 64-byte slot is at slot + l * pitch words (16-byte aligned; pitch % 8 ==
// 4, so rows 12 or 20 apart start 16 banks apart, and eight consecutive rows'
// slots start in distinct groups of four banks).  Two passes of 16 columns:
// every lane writes its row's 16 values, then reads one column (cl = lane % 16)
// for half of the block's rows, lanes 0-15 rows 0-15 and lanes 16-31 rows
// 16-31 taken in the order 16 + (j ^ 4), so that at each read the two
// half-warps cover the 32 banks once.  The halves' maxima meet in one shuffle
// and each lane stores its 16 codes as one 16-byte run of the transposed
// output (lanes l and l + 16 fill one 32-byte sector).
//
// STAGED: the codes go to a 32-column x 32-byte shared tile for a TMA store
// instead (column c = 16·pass + cl at c·32, its two 16-byte halves swapped
// when bit 2 of c is set: the tensor map's 32-byte swizzle, so the eight lanes
// of each store phase cover the 32 banks once); qc and ld are then unused.
template <bool STAGED = false>
__device__ __forceinline__ void col_quant32_slots(const float (&h)[32], float* slot, int pitch, uint8_t* qc,
                                                  uint8_t* sc, int64_t ld, int64_t sc_rows, int64_t col0,
                                                  int64_t tok0, int lane) {
  const int g = lane >> 4, cl = lane & 15;
  float4* mine = reinterpret_cast<float4*>(slot + lane * pitch);
  // rows j ^ (4g) of this half: j with bit 2 clear sit 4g rows below j, the others 4g rows above
  const float* lo = slot + (16 * g + 4 * g) * pitch + cl;
  const float* hi = slot + (16 * g - 4 * g) * pitch + cl;
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    __syncwarp();  // the previous pass's readers are done with the slots
#pragma unroll
    for (int k = 0; k < 4; ++k)
      mine[k] = make_float4(h[16 * pass + 4 * k], h[16 * pass + 4 * k + 1], h[16 * pass + 4 * k + 2],
                            h[16 * pass + 4 * k + 3]);
    __syncwarp();
    float v[16];
    float m = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      v[j] = (j & 4) ? hi[j * pitch] : lo[j * pitch];
      m = fmaxf(m, fabsf(v[j]));
    }
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
    const uint32_t sb = mx_scale_byte(f2u(m));
    const float2 inv = make_float2(mx_inv_scale(sb), mx_inv_scale(sb));
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 lo = mul2(make_float2(v[4 * i], v[4 * i + 1]), inv);
      const float2 hi = mul2(make_float2(v[4 * i + 2], v[4 * i + 3]), inv);
      w[i] = cvt_e4m3x2(lo.x, lo.y) | (cvt_e4m3x2(hi.x, hi.y) << 16);
    }
    // v[j] holds row j ^ (4g): for g = 1 the words of rows 0-3 / 4-7 (and 8-11 / 12-15) trade places
    const uint4 out = g ? make_uint4(w[1], w[0], w[3], w[2]) : make_uint4(w[0], w[1], w[2], w[3]);
    const int64_t col = col0 + 16 * pass + cl;
    if constexpr (STAGED) {
      const int c = 16 * pass + cl;
      *reinterpret_cast<uint4*>(qc + c * 32 + ((g ^ ((c >> 2) & 1)) << 4)) = out;
    } else {
      *reinterpret_cast<uint4*>(qc + col * ld + tok0 + 16 * g) = out;
    }
    if (g == 0) sc[sf_mma_offset(col, tok0 >> 5, sc_rows)] = static_cast<uint8_t>(sb);
  }
}

// bf16 outputs of the fused epilogues (BF16 and FP8 paths): the transposed
// copy (column col0+i, row tok0+lane: for each column the warp writes 32
// consecutive bf16) and, below, the thread's 32 values as one 64-byte run of
// its row.
// The row store returns the largest magnitude written (as bf16 bits:
// non-negative bf16 values order like their bit patterns; the FP8 path's amax).
__device__ __forceinline__ uint32_t row_store_bf16_amax(const float (&h)[32], uint16_t* dst) {
  uint32_t w[16];
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    w[i] = pack_bf16x2(h[2 * i], h[2 * i + 1]);
    m = max(m, max(w[i] & 0x7fffu, (w[i] >> 16) & 0x7fffu));
  }
  st_global_v8(dst, w);
  st_global_v8(dst + 16, w + 8);
  return m;
}

// Per-tensor FP8: fold this warp's largest magnitude (bf16 bits) into the
// expert tensor's amax (fp32 bits; non-negative floats order like integers).
__device__ __forceinline__ void warp_amax_to(float* amax, uint32_t m_bf16, int lane) {
  const uint32_t m = __reduce_max_sync(0xffffffffu, m_bf16);
  if (lane == 0 && m != 0) atomicMax(reinterpret_cast<unsigned int*>(amax), m << 16);
}

__device__ __forceinline__ void col_store_bf16(const float (&h)[32], uint16_t* yc, int64_t ld, int64_t col0,
                                               int64_t tok0, int lane) {
  uint16_t* dst = yc + col0 * ld + tok0 + lane;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const __nv_bfloat16 v = __float2bfloat16_rn(h[i]);
    *dst = *reinterpret_cast<const uint16_t*>(&v);
    dst += ld;
  }
}

// Hand the accumulator buffer back to the MMA warp (all of this warp's TMEM
// loads have completed).  A single CTA, or rank 0 of a pair, arrives on its own
// barrier.  Rank 1 of a pair signals rank 0 with a 4-byte asynchronous store
// into rank 0's shared memory that completes transaction bytes on rank 0's
// barrier: measured on GB300, an mbarrier arrive through the cluster window
// became visible to the waiting MMA thread only 2-4k cycles later, against a
// few hundred for these two paths.
struct AccRelease {
  uint32_t bar;   // rank 0 / single CTA: own barrier (shared window); rank 1: rank 0's barrier (cluster window)
  uint32_t land;  // rank 1: this warp's 4-byte slot in rank 0's shared memory (cluster window)
  bool peer;      // rank 1 of a CTA pair
};

__device__ __forceinline__ void release_acc(const AccRelease& rl, int lane) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) {
    if (rl.peer) st_async_complete_tx(rl.land, 1u, rl.bar);
    else mbar_arrive_u32(rl.bar);
  }
}

// bf16 store.  The thread owns half of its row's BN columns; it drains them
// from TMEM into packed bf16 registers, releases the accumulator, then stores,
// so the next tile's MMAs overlap the global stores.
// The factor that turns a per-tensor FP8 tile's accumulators into values:
// the dequantisation factors of the expert's A and B tensors (1 otherwise).
template <int OPK>
__device__ __forceinline__ float tile_scale(const GemmArgs& P, const TileCoord& tc) {
  if constexpr (OPK == OPK_F8) return fp8_dequant(P.amax_a[tc.e]) * fp8_dequant(P.amax_b[tc.e]);
  return 1.f;
}

// Combine fused into a row-grouped bf16 epilogue.  The thread has just
// stored its half row (COLS columns) of padded row m0 + row, which is slot j of
// token t.  It counts its segment in for (t, column tile, half); the thread
// that brings the count to k sums the token's k segments in slot order (fp32,
// from bf16: the same arithmetic as the combine kernel), writes y[t]'s segment
// and resets the counter.  Each writer fences its stores before its atomic,
// and the summing thread fences after it and reads through L2, so it sees the
// other CTAs' segments.  No thread waits on another.
template <int BN, int COLS>
__device__ __forceinline__ void fused_combine(const GemmArgs& P, const TileCoord& tc, int row, int hf,
                                              const uint32_t (&packed)[COLS / 2]) {
  const int prow = tc.m0 + row;
  const int f = P.cmb_prow_src[prow];
  if (f < 0) return;                              // padding row
  const int k = P.cmb_k;
  const int t = f / k;
  int32_t* cnt = P.cmb_count + (static_cast<int64_t>(t) * (P.N / BN) + tc.nt) * 2 + hf;
  __threadfence();
  if (atomicAdd(cnt, 1) != k - 1) return;
  __threadfence();
  *cnt = 0;
  const int64_t c0 = static_cast<int64_t>(tc.nt) * BN + hf * COLS;
  const int32_t* slots = P.cmb_prow_of_src + static_cast<int64_t>(t) * k;
#pragma unroll
  for (int jc = 0; jc < COLS / 16; ++jc) {
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
    for (int j = 0; j < k; ++j) {
      const int pr = slots[j];
      uint32_t w[8];
      if (pr == prow) {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = packed[8 * jc + i];
      } else {
        ld_global_cg_v8(P.d + static_cast<int64_t>(pr) * P.ldd + c0 + 16 * jc, w);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        acc[2 * i] += u2f(w[i] << 16);
        acc[2 * i + 1] += u2f(w[i] & 0xffff0000u);
      }
    }
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
    st_global_v8(P.cmb_out + static_cast<int64_t>(t) * P.N + c0 + 16 * jc, o);
  }
}

// stg / tmO (MXFP8 pair tiles with a fused combine): the warp's 2 KB shared
// tile and the output's tensor map; the rows then leave by TMA and complete
// before the combine's counters see them (otherwise stg is null).
template <int BN, bool KG, int OPK>
__device__ __forceinline__ void epi_bf16(const GemmArgs& P, const TileCoord& tc, uint32_t tb, int row, int hf,
                                         const AccRelease& tempty, int lane, uint8_t* stg = nullptr,
                                         const CUtensorMap* tmO = nullptr) {
  constexpr int COLS = BN / 2;
  const float f = tile_scale<OPK>(P, tc);
  uint32_t packed[COLS / 2];
#pragma unroll
  for (int c = 0; c < COLS / 32; c += 2) {
    uint32_t r0[32], r1[32];
    tmem_ld_32x32b_x32(tb + hf * COLS + c * 32, r0);
    tmem_ld_32x32b_x32(tb + hf * COLS + (c + 1) * 32, r1);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if constexpr (OPK == OPK_F8) {
        packed[c * 16 + i] = pack_bf16x2(u2f(r0[2 * i]) * f, u2f(r0[2 * i + 1]) * f);
        packed[(c + 1) * 16 + i] = pack_bf16x2(u2f(r1[2 * i]) * f, u2f(r1[2 * i + 1]) * f);
      } else {
        packed[c * 16 + i] = pack_bf16x2(u2f(r0[2 * i]), u2f(r0[2 * i + 1]));
        packed[(c + 1) * 16 + i] = pack_bf16x2(u2f(r1[2 * i]), u2f(r1[2 * i + 1]));
      }
    }
  }
  release_acc(tempty, lane);
  if (stg != nullptr) {
    // 32-row x 64-byte boxes through the warp's tile (64-byte swizzle), as in
    // epi_tma_out; then every box has been written to global memory and made
    // visible to generic loads (the combine's readers) before any lane of the
    // warp signals its row through the combine counter
    const int y = tc.m0 + (row & ~31);
    const int x0 = tc.nt * BN + hf * COLS;
    const int sw = (lane >> 1) & 3;
    uint8_t* srow = stg + lane * 64;
#pragma unroll
    for (int bx = 0; bx < COLS / 32; ++bx) {
      if (lane == 0) bulk_wait_group_read<0>();
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(srow + ((j ^ sw) << 4)) =
            make_uint4(packed[16 * bx + 4 * j], packed[16 * bx + 4 * j + 1], packed[16 * bx + 4 * j + 2],
                       packed[16 * bx + 4 * j + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(tmO, stg, x0 + 32 * bx, y);
        bulk_commit_group();
      }
    }
    if (lane == 0) {
      bulk_wait_group<0>();
      fence_proxy_async_global();
    }
    __syncwarp();
  } else {
    uint16_t* drow = KG ? P.d + static_cast<int64_t>(tc.e) * P.M * P.N + static_cast<int64_t>(tc.m0 + row) * P.N +
                              tc.nt * BN + hf * COLS
                        : P.d + static_cast<int64_t>(tc.m0 + row) * P.ldd + tc.nt * BN + hf * COLS;
#pragma unroll
    for (int j = 0; j < COLS / 16; ++j) st_global_v8(drow + 16 * j, packed + 8 * j);
  }
  if constexpr (!KG)
    if (P.cmb_out != nullptr) fused_combine<BN, COLS>(P, tc, row, hf, packed);
}

// Weight-gradient tile added into an fp32 gradient buffer (main_grad): the
// thread drains its half row of fp32 accumulators, releases the accumulator,
// then reads, adds and writes back 32 bytes at a time.  Each element of the
// buffer belongs to exactly one tile, so the update is a plain
// read-modify-write.
template <int BN>
__device__ __forceinline__ void epi_acc_f32(const GemmArgs& P, const TileCoord& tc, uint32_t tb, int row, int hf,
                                            const AccRelease& tempty, int lane) {
  constexpr int COLS = BN / 2;
  uint32_t v[COLS / 32][32];
#pragma unroll
  for (int c = 0; c < COLS / 32; ++c) tmem_ld_32x32b_x32(tb + hf * COLS + c * 32, v[c]);
  tmem_ld_wait();
  release_acc(tempty, lane);
  float* drow = P.dacc + static_cast<int64_t>(tc.e) * P.M * P.N + static_cast<int64_t>(tc.m0 + row) * P.N +
                tc.nt * BN + hf * COLS;
#pragma unroll
  for (int j = 0; j < COLS / 8; ++j) {
    uint32_t w[8];
    ld_global_v8(drow + 8 * j, w);
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = f2u(u2f(w[i]) + u2f(v[j / 4][8 * (j % 4) + i]));
    st_global_v8(drow + 8 * j, w);
  }
}

// MXFP8 pair tiles with a plain output (weight gradients; down and
// dgrad-gate-up without a fused combine): the thread's 128
// accumulator columns leave through the warp's 2 KB shared tile, a 32-row x
// 64-byte box (64-byte swizzle: 16-byte chunk j of row r at
// (j ^ ((r / 2) % 4)) · 16, conflict-free), by TMA: stored as bf16 dW (four
// boxes of 32 columns), or added into the fp32 main_grad by the memory system
// (eight boxes of 16 columns; a tensor-map reduce-add, the same single fp32
// addition per element as a read-modify-write).  One lane per output row made
// the per-lane global stores touch 32 rows per instruction.
template <int BN, bool KG, bool ACC>
__device__ __forceinline__ void epi_tma_out(const GemmArgs& P, const TileCoord& tc, uint32_t tb, int q, int hf,
                                           const AccRelease& tempty, int lane, uint8_t* stg, const CUtensorMap* tmO) {
  constexpr int COLS = BN / 2;
  uint32_t v[COLS / 32][32];
#pragma unroll
  for (int c = 0; c < COLS / 32; ++c) tmem_ld_32x32b_x32(tb + hf * COLS + c * 32, v[c]);
  tmem_ld_wait();
  release_acc(tempty, lane);
  // this warp's 32 rows: of the [E·M][N] weight gradient, or of the padded rows
  const int y = (KG ? tc.e * P.M : 0) + tc.m0 + q * 32;
  const int x0 = tc.nt * BN + hf * COLS;
  const int sw = (lane >> 1) & 3;
  uint8_t* row = stg + lane * 64;
  constexpr int BOXES = ACC ? COLS / 16 : COLS / 32;    // 64-byte rows: 16 fp32 or 32 bf16
#pragma unroll
  for (int bx = 0; bx < BOXES; ++bx) {
    uint32_t w[16];
    if constexpr (ACC) {
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = v[bx / 2][16 * (bx % 2) + i];
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(u2f(v[bx][2 * i]), u2f(v[bx][2 * i + 1]));
    }
    if (lane == 0) bulk_wait_group_read<0>();   // the previous box has been read out of the tile
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint4*>(row + ((j ^ sw) << 4)) = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if constexpr (ACC) tma_reduce_add_2d(tmO, stg, x0 + 16 * bx, y);
      else tma_store_2d(tmO, stg, x0 + 32 * bx, y);
      bulk_commit_group();
    }
  }
}

// Gate-up tile: accumulator columns [0, BN/2) = gate j0.., [BN/2, BN) = up j0..
// (j0 = nt * BN/2).  The thread owns BN/4 h columns (half hf).  It drains its
// accumulator columns into registers, releases the accumulator, then computes
// h in fp32 and quantises and stores while the next tile's MMAs run.
// MXFP8 (stage_gu): the saved g|u leave as 2 KB bulk copies (one gate or up
// block of a g|u tile, gu_tile_offset) through the warp's column-quantiser
// scratch, one block at a time, before the column quantiser takes it back.
template <int BN, int OPK>
__device__ __forceinline__ void epi_swiglu(const GemmArgs& P, const TileCoord& tc, uint32_t tb, int q, int lane,
                                           int hf, const AccRelease& tempty, float* slots, bool stage_gu = false) {
  constexpr int HC = BN / 2;          // h columns per tile
  constexpr int CH = HC / 64;         // 32-column chunks per thread
  const int64_t tok0 = tc.m0 + q * 32;
  const int64_t r = tok0 + lane;
  const float p = P.probs_perm[r];
  const int64_t I = P.I;
  const int j0 = tc.nt * HC + hf * (HC / 2);
  const bool save = P.gu_save != nullptr;
  uint32_t g[CH][32], u[CH][32];
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    tmem_ld_32x32b_x32(tb + hf * (HC / 2) + c * 32, g[c]);
    tmem_ld_32x32b_x32(tb + HC + hf * (HC / 2) + c * 32, u[c]);
  }
  tmem_ld_wait();
  release_acc(tempty, lane);
  if constexpr (OPK == OPK_F8) {        // per-tensor FP8: accumulators -> values
    const float f = tile_scale<OPK>(P, tc);
#pragma unroll
    for (int c = 0; c < CH; ++c)
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        g[c][i] = f2u(u2f(g[c][i]) * f);
        u[c][i] = f2u(u2f(u[c][i]) * f);
      }
  }
  uint32_t hmax = 0;
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int64_t col = j0 + c * 32;
    float h[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float gf = u2f(g[c][i]);
      h[i] = p * __fdividef(gf, 1.f + __expf(-gf)) * u2f(u[c][i]);
    }
    if (save) {
      uint32_t gp[16], up[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        gp[i] = pack_bf16x2(u2f(g[c][2 * i]), u2f(g[c][2 * i + 1]));
        up[i] = pack_bf16x2(u2f(u[c][2 * i]), u2f(u[c][2 * i + 1]));
      }
      if (OPK == OPK_MX && stage_gu) {
        // the gate block, then the up block, of g|u tile (tok0/32, col/32),
        // each staged in its global order: lane's 32 bytes of half h at
        // (32·h + lane)·32, written as two 16-byte pieces of which lanes with
        // bit 2 set write the second first (eight consecutive lanes then
        // cover the 32 banks once)
        uint8_t* stg = reinterpret_cast<uint8_t*>(slots);
        const int sw = (lane >> 2) & 1;
        uint16_t* dst = P.gu_save + gu_tile_offset(static_cast<int>(I), static_cast<int>(tok0), static_cast<int>(col));
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t* w = half ? up : gp;
          if (lane == 0) bulk_wait_group_read<0>();    // the previous block has left the scratch
          __syncwarp();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint8_t* srow = stg + (32 * h + lane) * 32;
            const uint4 a = make_uint4(w[8 * h], w[8 * h + 1], w[8 * h + 2], w[8 * h + 3]);
            const uint4 b = make_uint4(w[8 * h + 4], w[8 * h + 5], w[8 * h + 6], w[8 * h + 7]);
            *reinterpret_cast<uint4*>(srow + (sw << 4)) = sw ? b : a;
            *reinterpret_cast<uint4*>(srow + ((sw ^ 1) << 4)) = sw ? a : b;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            bulk_store_s2g(dst + 1024 * half, stg, 2048);
            bulk_commit_group();
          }
        }
        if (lane == 0) bulk_wait_group_read<0>();      // the scratch is the column quantiser's again
        __syncwarp();
      } else {
        uint16_t* gs = P.gu_save + r * (2 * I) + col;
        st_global_v8(gs, gp);
        st_global_v8(gs + 16, gp + 8);
        st_global_v8(gs + I, up);
        st_global_v8(gs + I + 16, up + 8);
      }
    }
    if constexpr (OPK != OPK_MX) {
      hmax = max(hmax, row_store_bf16_amax(h, P.y_row + r * P.y_row_ld + col));
      if (P.y_col != nullptr) col_store_bf16(h, P.y_col, P.y_col_ld, col, tok0, lane);
    } else {
      const uint32_t sb = row_quant32(h, P.q_out + r * P.q_out_ld + col);
      P.s_out[sf_mma_offset(r, col >> 5, P.s_out_rows)] = static_cast<uint8_t>(sb);
      if (P.qc_out != nullptr) col_quant32_slots(h, slots, 20, P.qc_out, P.sc_out, P.qc_ld, P.sc_rows, col, tok0, lane);
    }
  }
  if constexpr (OPK == OPK_F8) warp_amax_to(P.amax_out + tc.e, hmax, lane);
}

// dgrad-down tile: accumulator = dH columns nt*BN.., the thread owns half hf.
// Partial d(prob) sums go to dp_part[r][2*nt + hf].
template <int BN>
__device__ __forceinline__ void epi_dswiglu(const GemmArgs& P, const TileCoord& tc, uint32_t tb, int q, int lane,
                                            int hf, const AccRelease& tempty, float* xp) {
  constexpr int COLS = BN / 2;
  const int64_t tok0 = tc.m0 + q * 32;
  const int64_t r = tok0 + lane;
  const float p = P.probs_perm[r];
  const int64_t I = P.I;
  const int j0 = tc.nt * BN + hf * COLS;
  float dp = 0.f;
#pragma unroll 1
  for (int c = 0; c < COLS / 32; ++c) {
    uint32_t dh[32];
    tmem_ld_32x32b_x32(tb + hf * COLS + c * 32, dh);
    const int64_t col = j0 + c * 32;
    float g[32], u[32], dg[32];
    const uint16_t* blk = P.gu_save + gu_tile_offset(static_cast<int>(I), static_cast<int>(tok0), static_cast<int>(col));
    load_gu_block32(blk, lane, g);
    load_gu_block32(blk + 1024, lane, u);
    tmem_ld_wait();
    if (c == COLS / 32 - 1) release_acc(tempty, lane);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float gf = g[i], uf = u[i];
      const float s = __fdividef(1.f, 1.f + __expf(-gf));
      const float sl = gf * s;
      const float a = u2f(dh[i]) * p;
      dg[i] = a * uf * s * (1.f + gf * (1.f - s));
      u[i] = a * sl;                       // du
      dp += u2f(dh[i]) * sl * uf;
    }
    uint32_t sb = row_quant32(dg, P.q_out + r * P.q_out_ld + col);
    P.s_out[sf_mma_offset(r, col >> 5, P.s_out_rows)] = static_cast<uint8_t>(sb);
    col_quant32_xpose(dg, xp, P.qc_out, P.sc_out, P.qc_ld, P.sc_rows, col, tok0, lane);
    sb = row_quant32(u, P.q_out + r * P.q_out_ld + I + col);
    P.s_out[sf_mma_offset(r, (I + col) >> 5, P.s_out_rows)] = static_cast<uint8_t>(sb);
    col_quant32_xpose(u, xp, P.qc_out, P.sc_out, P.qc_ld, P.sc_rows, I + col, tok0, lane);
  }
  P.dp_part[r * P.dp_ld + 2 * tc.nt + hf] = dp;
}


// BN = 256: drain the thread's 128 dH columns and park them as 64 packed
// bf16 pairs in the warp's own TMEM columns (tstage: this warp's lanes,
// columns kDsCol + 64·hf ..), then release the accumulator, so the dSwiGLU
// math runs from there while the next tile's MMAs fill the accumulator.
template <int OPK>
__device__ __forceinline__ void park_dh(const GemmArgs& P, const TileCoord& tc, uint32_t tb, int hf, int lane,
                                        const AccRelease& tempty, uint32_t tstage) {
  constexpr int COLS = 128;
  const float f = tile_scale<OPK>(P, tc);         // per-tensor FP8: accumulators -> dH
#pragma unroll
  for (int c = 0; c < COLS / 32; c += 2) {
    uint32_t a0[32], a1[32];
    tmem_ld_32x32b_x32(tb + hf * COLS + c * 32, a0);
    tmem_ld_32x32b_x32(tb + hf * COLS + (c + 1) * 32, a1);
    tmem_ld_wait();
    if constexpr (OPK == OPK_F8) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        a0[i] = f2u(u2f(a0[i]) * f);
        a1[i] = f2u(u2f(a1[i]) * f);
      }
    }
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      w[i] = pack_bf16x2(u2f(a0[2 * i]), u2f(a0[2 * i + 1]));
      w[16 + i] = pack_bf16x2(u2f(a1[2 * i]), u2f(a1[2 * i + 1]));
    }
    tmem_st_32x32b_x32(tstage + 16 * c, w);
  }
  tmem_st_wait();
  release_acc(tempty, lane);
}

// The parked dH of 32-column chunk c as fp32.
__device__ __forceinline__ void unpark_dh(uint32_t tstage, int c, float (&dh)[32]) {
  uint32_t w[16];
  tmem_ld_32x32b_x16(tstage + 16 * c, w);
  tmem_ld_wait();
#pragma unroll
  for (int m = 0; m < 16; ++m) {
    dh[2 * m] = u2f(w[m] << 16);
    dh[2 * m + 1] = u2f(w[m] & 0xffff0000u);
  }
}

// dSwiGLU of 32 columns of one row: dg, du (into u) and the d(prob) partial
// sum_i dH g s u.  s = sigmoid(g), sl = silu(g) = g s,
// d silu(g)/dg = s (1 + g (1 - s)) = s + sl (1 - s); pairs of columns as
// packed fp32 pairs.
__device__ __forceinline__ void dswiglu32(const float (&dh)[32], const float (&g)[32], float (&u)[32], float p,
                                          float2& dp2, float (&dg)[32]) {
  const float2 one2 = make_float2(1.f, 1.f), p2 = make_float2(p, p);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float2 g2 = make_float2(g[i], g[i + 1]), u2 = make_float2(u[i], u[i + 1]);
    const float2 dh2 = make_float2(dh[i], dh[i + 1]);
    const float2 d2 = add2(one2, make_float2(__expf(-g2.x), __expf(-g2.y)));
    const float2 s2 = make_float2(__fdividef(1.f, d2.x), __fdividef(1.f, d2.y));
    const float2 sl2 = mul2(g2, s2);
    const float2 t2 = mul2(dh2, u2);
    dp2 = fma2(t2, sl2, dp2);
    const float2 dg2 = mul2(mul2(t2, p2), fma2(sl2, sub2(one2, s2), s2));
    const float2 du2 = mul2(mul2(dh2, p2), sl2);
    dg[i] = dg2.x;
    dg[i + 1] = dg2.y;
    u[i] = du2.x;
    u[i + 1] = du2.y;
  }
}

// BF16 and per-tensor FP8 dgrad-down at BN = 256: dH parked in TMEM, the
// saved g|u read with plain loads, dGU written in bf16 (row-major, and
// transposed for the weight gradient; FP8: with the expert's amax).
template <int OPK>
__device__ __forceinline__ void epi_dswiglu_staged(const GemmArgs& P, const TileCoord& tc, uint32_t tb, int q,
                                                   int lane, int hf, const AccRelease& tempty, uint32_t tstage) {
  constexpr int COLS = 128;
  const int64_t tok0 = tc.m0 + q * 32;
  const int64_t r = tok0 + lane;
  park_dh<OPK>(P, tc, tb, hf, lane, tempty, tstage);
  const float p = P.probs_perm[r];
  const int64_t I = P.I;
  const int j0 = tc.nt * 256 + hf * COLS;
  float2 dp2 = make_float2(0.f, 0.f);
  uint32_t gmax = 0;
#pragma unroll 1
  for (int c = 0; c < COLS / 32; ++c) {
    const int64_t col = j0 + c * 32;
    float dh[32], g[32], u[32], dg[32];
    unpark_dh(tstage, c, dh);
    load_bf16_32(P.gu_save + r * (2 * I) + col, g);
    load_bf16_32(P.gu_save + r * (2 * I) + I + col, u);
    dswiglu32(dh, g, u, p, dp2, dg);
    gmax = max(gmax, row_store_bf16_amax(dg, P.y_row + r * P.y_row_ld + col));
    gmax = max(gmax, row_store_bf16_amax(u, P.y_row + r * P.y_row_ld + I + col));
    if (P.y_col != nullptr) {
      col_store_bf16(dg, P.y_col, P.y_col_ld, col, tok0, lane);
      col_store_bf16(u, P.y_col, P.y_col_ld, I + col, tok0, lane);
    }
  }
  P.dp_part[r * P.dp_ld + 2 * tc.nt + hf] = dp2.x + dp2.y;
  if constexpr (OPK == OPK_F8) warp_amax_to(P.amax_out + tc.e, gmax, lane);
}

// The MXFP8 dgrad-down epilogue at BN = 256 stores its dGU codes with TMA,
// not with per-lane global stores: an epilogue lane owns one row, so a warp's
// global store touches 32 rows (32 L1 wavefronts per instruction), and with
// those the SM's L1 data path was the busiest unit of the kernel (LSU
// wavefronts at 65 % of peak beside the operand stream's 26 %, ncu).  Per
// epilogue warp, in shared memory:
//   out  : 4 KB, the chunk's dGU codes, row-wise dg | du (32 rows x 32 bytes
//          each) and column-wise dg | du (32 columns x 32 tokens each),
//          32-byte swizzle, stored by TMA while the next chunk is computed;
//   slots: the column quantiser's 32 x 20-word scratch.
// The saved g|u stay plain 32-byte loads: reading them by TMA as well (4 KB
// more per warp, a four-stage ring) measured slower.
struct DsTma {
  uint8_t* out;
  float* slots;
};

__device__ __forceinline__ void epi_dswiglu_tma(const GemmArgs& P, const TileCoord& tc, uint32_t tb, int q, int lane,
                                                int hf, const AccRelease& tempty, uint32_t tstage, const DsTma& d,
                                                const CUtensorMap* tmO1, const CUtensorMap* tmO2) {
  constexpr int COLS = 128;
  const int tok0 = tc.m0 + q * 32;
  const int64_t r = tok0 + lane;
  park_dh<OPK_MX>(P, tc, tb, hf, lane, tempty, tstage);
  const float p = P.probs_perm[r];
  const int I = P.I;
  const int j0 = tc.nt * 256 + hf * COLS;
  // this lane's row in the g|u tiles of the warp's four chunks (consecutive
  // tiles: gu_tile_offset)
  const uint16_t* gt = P.gu_save + gu_tile_offset(I, tok0, j0) + lane * 16;
  float2 dp2 = make_float2(0.f, 0.f);
  uint32_t sbg = 0, sbu = 0;
  // the saved g|u of chunk c + 1 are requested (as raw bf16 pairs) before
  // chunk c's math, so their latency overlaps it: 64 experts top-8 0.932
  // (paired), the Mixtral layer unchanged
  uint32_t gw[16], uw[16];
  ld_global_nc_v8(gt, gw);
  ld_global_nc_v8(gt + 512, gw + 8);
  ld_global_nc_v8(gt + 1024, uw);
  ld_global_nc_v8(gt + 1536, uw + 8);
#pragma unroll 1
  for (int c = 0; c < COLS / 32; ++c) {
    const int col = j0 + c * 32;
    float dh[32], g[32], u[32], dg[32];
    unpark_dh(tstage, c, dh);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      g[2 * j] = u2f(gw[j] << 16);
      g[2 * j + 1] = u2f(gw[j] & 0xffff0000u);
      u[2 * j] = u2f(uw[j] << 16);
      u[2 * j + 1] = u2f(uw[j] & 0xffff0000u);
    }
    if (c + 1 < COLS / 32) {
      const uint16_t* nt = gt + (c + 1) * 2048;
      ld_global_nc_v8(nt, gw);
      ld_global_nc_v8(nt + 512, gw + 8);
      ld_global_nc_v8(nt + 1024, uw);
      ld_global_nc_v8(nt + 1536, uw + 8);
    }
    dswiglu32(dh, g, u, p, dp2, dg);
    // the previous chunk's code stores have finished reading the staging tiles
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
    sbg |= row_quant32_staged(dg, d.out, lane) << (8 * c);
    sbu |= row_quant32_staged(u, d.out + 1024, lane) << (8 * c);
    col_quant32_slots<true>(dg, d.slots, 20, d.out + 2048, P.sc_out, 0, P.sc_rows, col, tok0, lane);
    col_quant32_slots<true>(u, d.slots, 20, d.out + 3072, P.sc_out, 0, P.sc_rows, I + col, tok0, lane);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tmO1, d.out, col, tok0);
      tma_store_2d(tmO1, d.out + 1024, I + col, tok0);
      tma_store_2d(tmO2, d.out + 2048, tok0, col);
      tma_store_2d(tmO2, d.out + 3072, tok0, I + col);
      bulk_commit_group();
    }
  }
  // the row's four scale bytes of each half are adjacent (j0 and I are
  // multiples of 128, so the first block index is a multiple of 4)
  *reinterpret_cast<uint32_t*>(P.s_out + sf_mma_offset(r, j0 >> 5, P.s_out_rows)) = sbg;
  *reinterpret_cast<uint32_t*>(P.s_out + sf_mma_offset(r, (I + j0) >> 5, P.s_out_rows)) = sbu;
  P.dp_part[r * P.dp_ld + 2 * tc.nt + hf] = dp2.x + dp2.y;
}

template <int BN, int EPI, bool KG, bool PAIR, int OPK>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                const __grid_constant__ CUtensorMap tmO1, const __grid_constant__ CUtensorMap tmO2, const GemmArgs P) {
  using C = Cfg<BN, EPI, PAIR, OPK, KG>;
  constexpr int CG = C::CG;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ctrl = smem + C::kStages * C::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint64_t* tempty = tfull + C::kAcc;
  uint64_t* drained = tempty + C::kAcc;
  uint64_t* sfready = drained + 1;                  // scale factors of a stage are in TMEM
  uint64_t* cdrained = sfready + C::kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(cdrained + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* never_set = reinterpret_cast<int*>(tmem_slot + 2);
  int* s_poff = reinterpret_cast<int*>(tmem_slot + 4);
  float* xpose = reinterpret_cast<float*>(ctrl + C::kCtrlBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t limit_ns = P.wait_limit_ns != 0 ? P.wait_limit_ns : kWaitLimitNs;
  // In a CTA pair, rank 0 issues the MMAs for both CTAs; rank 1 feeds its half.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int E = P.E;
  for (int i = threadIdx.x; i <= E; i += kThreads) s_poff[i] = P.poff[i];
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      // in a pair, rank 0's full barrier also counts the bytes rank 1's copies
      // complete on it (rank 1's own full barriers are unused)
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < C::kAcc; ++a) {
      mbar_init(&tfull[a], 1);
      // the epilogue warps' arrivals (8) + in a pair the MMA thread's arrive.expect_tx
      // for the 8 x 4 bytes rank 1's warps store
      mbar_init(&tempty[a], PAIR ? 9 : 8);
    }
    mbar_init(drained, 1);
    for (int st = 0; st < C::kStages; ++st) mbar_init(&sfready[st], 1);
    mbar_init(cdrained, 1);
    *abort_flag = 0;
    *never_set = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (PAIR) {
      tma_prefetch_desc(&tmSA);
      tma_prefetch_desc(&tmSB);
    }
    if (C::kDsTma || C::kTmaOut) {
      tma_prefetch_desc(&tmO1);
      tma_prefetch_desc(&tmO2);
    }
  }
  __syncthreads();

  // Group offsets must be aligned to the tile height, monotone, inside capacity.
  bool ok = true;
  const int64_t cap = KG ? P.a_cols : P.M;
  const int align = KG ? C::kKElems : C::kTileM;
  for (int e = 0; e < E; ++e) {
    const int a = s_poff[e], b = s_poff[e + 1];
    if (a < 0 || (a % align) || b < a) ok = false;
  }
  if ((s_poff[E] % align) || s_poff[E] > cap) ok = false;
  if (!ok) {
    if (threadIdx.x == 0) report(P.status, MXG_ERR_OFFSETS);
    return;
  }

  if (warp == 1) {
    tmem_alloc<CG>(tmem_slot, 512);
    tmem_relinquish<CG>();
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // both CTAs' barriers initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int ntn = KG ? P.N / BN : (EPI == EPI_SWIGLU ? P.I / (BN / 2) : P.N / BN);
  const int mtn_kg = P.M / C::kTileM;
  const int64_t total = KG ? static_cast<int64_t>(E) * mtn_kg * ntn
                           : static_cast<int64_t>(s_poff[E] / C::kTileM) * ntn;
  const int64_t tile0 = PAIR ? blockIdx.x / 2 : blockIdx.x;
  const int64_t tstep = PAIR ? gridDim.x / 2 : gridDim.x;

  // Tile t -> expert, this CTA's first row (m0), column tile, contraction range.
  auto decode = [&](int64_t t) {
    TileCoord tc;
    if (KG) {
      // The operand with the larger per-expert footprint is streamed once: its
      // tile index varies slowest and the other operand's tiles (which stay in
      // L2) vary fastest.
      const int64_t tpe = static_cast<int64_t>(mtn_kg) * ntn;
      tc.e = static_cast<int>(t / tpe);
      const int local = static_cast<int>(t - tc.e * tpe);
      int mt;
      if (P.M >= P.N) {
        mt = local / ntn;
        tc.nt = local % ntn;
      } else {
        tc.nt = local / mtn_kg;
        mt = local % mtn_kg;
      }
      tc.m0 = mt * C::kTileM + static_cast<int>(rank) * BM;
      tc.kbeg = s_poff[tc.e];
      tc.num_k = (s_poff[tc.e + 1] - s_poff[tc.e]) / C::kKElems;
    } else {
      int e = 0;
      while (e + 1 < E && static_cast<int64_t>(s_poff[e + 1] / C::kTileM) * ntn <= t) ++e;
      const int local = static_cast<int>(t - static_cast<int64_t>(s_poff[e] / C::kTileM) * ntn);
      const int mcount = (s_poff[e + 1] - s_poff[e]) / C::kTileM;
      tc.e = e;
      tc.nt = local / mcount;
      tc.m0 = s_poff[e] + (local - tc.nt * mcount) * C::kTileM + static_cast<int>(rank) * BM;
      tc.kbeg = 0;
      tc.num_k = P.K / C::kKElems;
    }
    return tc;
  };
  auto fail = [&]() {
    report(P.status, MXG_ERR_TIMEOUT);
    *abort_flag = 1;
  };
  // the barrier the epilogue releases accumulators on (rank 0's, in a pair)
  uint32_t* landing = reinterpret_cast<uint32_t*>(tmem_slot + 4) + 264;   // after s_poff (E <= 256)

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && P.debug_stall == 0) {
      uint32_t stage = 0, phase = 0;
      bool aborted = false;
      const uint32_t full0 = PAIR ? map_to_rank(smem_u32(full), 0) : 0u;   // rank 0's full barriers
      for (int64_t t = tile0; t < total && !aborted; t += tstep) {
        const TileCoord tc = decode(t);
        const int a_row = tc.m0;
        // b_row0: first B row this CTA loads (b_row1: the up rows of a gate-up
        // tile); sfb0/sfb1: first rows of the tile's two 128-row scale atoms
        // (BN = 256; every CTA of a pair loads both)
        int b_row0, b_row1 = 0, sfb0, sfb1;
        if (KG) {
          sfb0 = tc.nt * BN;
          sfb1 = sfb0 + 128;
          b_row0 = sfb0 + static_cast<int>(rank) * C::kBRows;
        } else if (EPI == EPI_SWIGLU) {
          sfb0 = tc.e * P.b_rows_per_expert + tc.nt * (BN / 2);  // gate rows
          sfb1 = sfb0 + P.I;                                     // up rows
          b_row0 = (PAIR && rank == 1) ? sfb1 : sfb0;             // in a pair, rank 1 holds the up half
          b_row1 = sfb1;
        } else {
          sfb0 = tc.e * P.b_rows_per_expert + tc.nt * BN;
          sfb1 = sfb0 + 128;
          b_row0 = sfb0 + static_cast<int>(rank) * C::kBRows;
        }
        for (int kb = 0; kb < tc.num_k; ++kb) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1, abort_flag, limit_ns)) {
            fail();
            aborted = true;
            break;
          }
          uint8_t* sA = smem + stage * C::kStageBytes;
          uint8_t* sB = sA + C::kABytes;
          uint8_t* sSfa = sB + C::kBBytes;
          uint8_t* sSfb = sSfa + C::kSfaBytes;
          const int kx = tc.kbeg + kb * C::kKElems;
          const int64_t kc = kx >> 7;
          if (PAIR) {
            // scale atoms are rows of the scale tensors' maps (128 x u32 = 512 B)
            const int sa_atom = static_cast<int>(kc * (P.a_rows >> 7) + (a_row >> 7));
            const int sb_atom0 = static_cast<int>(kc * (P.b_rows >> 7) + (sfb0 >> 7));
            const int sb_atom1 = static_cast<int>(kc * (P.b_rows >> 7) + (sfb1 >> 7));
            if (rank == 0) {
              mbar_arrive_expect_tx(&full[stage], 2 * C::kTx);   // both CTAs' bytes
              tma_load_2d(sA, &tmA, kx, a_row, &full[stage]);
              tma_load_2d(sB, &tmB, kx, b_row0, &full[stage]);
              if constexpr (OPK == OPK_MX) {
                tma_load_2d(sSfa, &tmSA, 0, sa_atom, &full[stage]);
                tma_load_2d(sSfb, &tmSB, 0, sb_atom0, &full[stage]);
                if (EPI == EPI_SWIGLU) tma_load_2d(sSfb + 512, &tmSB, 0, sb_atom1, &full[stage]);
              }
            } else {
              const uint32_t bar0 = full0 + stage * 8;
              tma_load_2d_pair(sA, &tmA, kx, a_row, bar0);
              tma_load_2d_pair(sB, &tmB, kx, b_row0, bar0);
              if constexpr (OPK == OPK_MX) {
                tma_load_2d_pair(sSfa, &tmSA, 0, sa_atom, bar0);
                tma_load_2d_pair(sSfb, &tmSB, 0, sb_atom0, bar0);
                if (EPI == EPI_SWIGLU) tma_load_2d_pair(sSfb + 512, &tmSB, 0, sb_atom1, bar0);
              }
            }
          } else {
            mbar_arrive_expect_tx(&full[stage], C::kTx);
            tma_load_2d(sA, &tmA, kx, a_row, &full[stage]);
            if constexpr (OPK == OPK_MX) bulk_load(sSfa, P.sa + (kc * (P.a_rows >> 7) + (a_row >> 7)) * 512, 512, &full[stage]);
            if (EPI == EPI_SWIGLU) {
              tma_load_2d(sB, &tmB, kx, b_row0, &full[stage]);
              tma_load_2d(sB + 128 * 128, &tmB, kx, b_row1, &full[stage]);
              if constexpr (OPK == OPK_MX) {
                bulk_load(sSfb, P.sb + (kc * (P.b_rows >> 7) + (b_row0 >> 7)) * 512, 512, &full[stage]);
                bulk_load(sSfb + 512, P.sb + (kc * (P.b_rows >> 7) + (b_row1 >> 7)) * 512, 512, &full[stage]);
              }
            } else {
              tma_load_2d(sB, &tmB, kx, b_row0, &full[stage]);
              if constexpr (OPK == OPK_MX) bulk_load(sSfb, P.sb + (kc * (P.b_rows >> 7) + (sfb0 >> 7)) * 512, BN * 4, &full[stage]);
            }
          }
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (aborted) {  // let copies already in flight land before the CTA exits
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000ull) __nanosleep(1000);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0 && rank == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool aborted = false, committed = false;
      for (int64_t t = tile0; t < total && !aborted; t += tstep) {
        const TileCoord tc = decode(t);
        if (tc.num_k == 0) continue;
        const bool got = PAIR ? mbar_wait_bounded_cluster(&tempty[acc], acc_phase ^ 1, abort_flag, limit_ns)
                              : mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, abort_flag, limit_ns);
        if (!got) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t d_t = tmem + acc * BN;
        for (int kb = 0; kb < tc.num_k; ++kb) {
          // MXFP8: the copier thread has seen the stage's data land and its
          // scale factors are in TMEM slot `stage`; bf16: wait for the data
          bool in;
          if constexpr (OPK != OPK_MX)
            in = PAIR ? mbar_wait_bounded_cluster(&full[stage], phase, abort_flag, limit_ns)
                      : mbar_wait_bounded(&full[stage], phase, abort_flag, limit_ns);
          else
            in = mbar_wait_bounded(&sfready[stage], phase, abort_flag, limit_ns);
          if (!in) {
            fail();
            aborted = true;
            break;
          }
          tc_fence_after();
          uint8_t* sA = smem + stage * C::kStageBytes;
          uint8_t* sB = sA + C::kABytes;
          const uint64_t adesc = smem_desc(smem_u32(sA), 0, 1024, kLayoutSwizzle128B);
          const uint64_t bdesc = smem_desc(smem_u32(sB), 0, 1024, kLayoutSwizzle128B);
          if constexpr (OPK == OPK_BF16) {
            // four K = 16 steps of 32 bytes per 128-byte stage row
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_bf16<CG>(d_t, adesc + 2 * k, bdesc + 2 * k, idesc_bf16(C::kTileM, BN), (kb | k) != 0 ? 1u : 0u);
          } else if constexpr (OPK == OPK_F8) {
            // four K = 32 steps of E4M3 without scale factors
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_f8<CG>(d_t, adesc + 2 * k, bdesc + 2 * k, idesc_f8_e4m3(C::kTileM, BN), (kb | k) != 0 ? 1u : 0u);
          } else {
            const uint32_t sfa_t = tmem + C::kSfCol + stage * C::kSfSlot;
            const uint32_t sfb_t = sfa_t + 4;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_mxf8<CG>(d_t, adesc + 2 * k, bdesc + 2 * k, idesc_mxf8_e4m3(C::kTileM, BN, k, k), sfa_t, sfb_t,
                           (kb | k) != 0 ? 1u : 0u);
          }
          mma_commit<CG>(&empty[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (aborted) break;
        mma_commit<CG>(&tfull[acc]);
        if (PAIR) mbar_arrive_expect_tx(&tempty[acc], 8 * 4);
        committed = true;
        if (++acc == C::kAcc) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // rank 1's release stores for the last tile have landed in this CTA's
      // shared memory before the CTA exits
      if (PAIR && committed) mbar_wait_bounded(&tempty[acc], acc_phase ^ 1, never_set, limit_ns);
      // all MMAs issued by this thread are complete before TMEM is released
      mma_commit<CG>(drained);
      mbar_wait_bounded(drained, 0, never_set, limit_ns);
    }
  } else if (warp == 2) {
    // ------------------------------------------------- scale-factor copier
    // Waits for each stage's data and copies its scale factors into the
    // stage's TMEM slot.  Kept off the MMA thread: a barrier wait followed by
    // a shared->TMEM copy on the issuing thread starves the tensor pipe.
    if (OPK == OPK_MX && lane == 0 && rank == 0) {
      uint32_t stage = 0, phase = 0;
      bool aborted = false;
      for (int64_t t = tile0; t < total && !aborted; t += tstep) {
        const TileCoord tc = decode(t);
        for (int kb = 0; kb < tc.num_k; ++kb) {
          const bool in = PAIR ? mbar_wait_bounded_cluster(&full[stage], phase, abort_flag, limit_ns)
                               : mbar_wait_bounded(&full[stage], phase, abort_flag, limit_ns);
          if (!in) {
            fail();
            aborted = true;
            break;
          }
          uint8_t* sSfa = smem + stage * C::kStageBytes + C::kABytes + C::kBBytes;
          uint8_t* sSfb = sSfa + C::kSfaBytes;
          const uint32_t sfa_t = tmem + C::kSfCol + stage * C::kSfSlot;
          tmem_cp_32x128b_warpx4<CG>(sfa_t, smem_desc(smem_u32(sSfa), 0, 128, kLayoutNone));
#pragma unroll
          for (int i = 0; i < BN / 128; ++i)
            tmem_cp_32x128b_warpx4<CG>(sfa_t + 4 + 4 * i, smem_desc(smem_u32(sSfb + 512 * i), 0, 128, kLayoutNone));
          mma_commit<CG>(&sfready[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // every copy issued by this thread has landed before TMEM is released
      mma_commit<CG>(cdrained);
      mbar_wait_bounded(cdrained, 0, never_set, limit_ns);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    // warps 4..11: TMEM lane quadrant q = warp % 4, column half hf.
    const int q = warp & 3;
    const int hf = (warp - 4) >> 2;
    const int row = q * 32 + lane;
    float* my_xpose = xpose + (warp - 4) * 32 * 33;
    uint32_t acc = 0, acc_phase = 0;
    DsTma dt{};
    if constexpr (C::kDsTma) {
      uint8_t* base = reinterpret_cast<uint8_t*>(xpose);
      const int w = warp - 4;
      dt.out = base + w * 4096;
      dt.slots = reinterpret_cast<float*>(base + 8 * 4096 + w * 32 * 20 * 4);
    }
    for (int64_t t = tile0; t < total; t += tstep) {
      const TileCoord tc = decode(t);
      if (tc.num_k == 0) {
        // token-grouped tile of an expert without tokens: exact zeros (an fp32
        // gradient buffer being accumulated into stays as it is)
        if constexpr (EPI == EPI_ACC_F32) continue;
        uint16_t* drow = P.d + static_cast<int64_t>(tc.e) * P.M * P.N + static_cast<int64_t>(tc.m0 + row) * P.N +
                         tc.nt * BN + hf * (BN / 2);
#pragma unroll 4
        for (int c = 0; c < BN / 16; ++c) reinterpret_cast<uint4*>(drow)[c] = make_uint4(0u, 0u, 0u, 0u);
        continue;
      }
      if constexpr (EPI == EPI_ACC_F32) {
        // the gradient rows this thread will read-modify-write come into L2
        // while the tile's MMAs run, so the epilogue's loads hit L2 instead of
        // waiting on HBM
        const float* pr = P.dacc + static_cast<int64_t>(tc.e) * P.M * P.N +
                          static_cast<int64_t>(tc.m0 + row) * P.N + tc.nt * BN + hf * (BN / 2);
#pragma unroll
        for (int j = 0; j < BN / 2 / 32; ++j) prefetch_l2(pr + 32 * j);
      }
      bool got = mbar_wait_bounded(&tfull[acc], acc_phase, abort_flag, limit_ns);
      got = __all_sync(0xffffffffu, got);
      if (!got) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      AccRelease rel;
      rel.peer = PAIR && rank == 1;
      rel.bar = rel.peer ? map_to_rank(smem_u32(&tempty[acc]), 0) : smem_u32(&tempty[acc]);
      rel.land = rel.peer ? map_to_rank(smem_u32(&landing[warp - 4]), 0) : 0u;
      if constexpr (EPI == EPI_SWIGLU) {
        epi_swiglu<BN, OPK>(P, tc, tb, q, lane, hf, rel, xpose + (warp - 4) * 32 * 20,
                            C::kSwTma && P.gu_save != nullptr);
      } else if constexpr (EPI == EPI_DSWIGLU) {
        const uint32_t tstage = tmem + (static_cast<uint32_t>(q * 32) << 16) + C::kDsCol + hf * 64;
        if constexpr (C::kDsTma) {
          epi_dswiglu_tma(P, tc, tb, q, lane, hf, rel, tstage, dt, &tmO1, &tmO2);
        } else if constexpr (BN == 256) {
          epi_dswiglu_staged<OPK>(P, tc, tb, q, lane, hf, rel, tstage);
        } else {
          epi_dswiglu<BN>(P, tc, tb, q, lane, hf, rel, my_xpose);
        }
      } else if (C::kTmaOut && (KG || P.cmb_out == nullptr)) {
        epi_tma_out<BN, KG, EPI == EPI_ACC_F32>(P, tc, tb, q, hf, rel, lane,
                                               reinterpret_cast<uint8_t*>(xpose) + (warp - 4) * 2048, &tmO1);
      } else if constexpr (EPI == EPI_ACC_F32) {
        epi_acc_f32<BN>(P, tc, tb, row, hf, rel, lane);
      } else if constexpr (C::kTmaOut) {     // fused combine: rows by TMA, completed before the counters
        epi_bf16<BN, KG, OPK>(P, tc, tb, row, hf, rel, lane, reinterpret_cast<uint8_t*>(xpose) + (warp - 4) * 2048,
                              &tmO1);
      } else {
        epi_bf16<BN, KG, OPK>(P, tc, tb, row, hf, rel, lane);
      }
      if (++acc == C::kAcc) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if constexpr (C::kDsTma || C::kTmaOut || C::kSwTma) {
      // the TMA stores have completed before the CTA exits
      if (lane == 0) bulk_wait_group<0>();
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // the peer is done with the pair's TMEM too
  tc_fence_after();
  if (warp == 1) tmem_dealloc<CG>(tmem, 512);
}

// ------------------------------------------------------------------- host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D uint8 tensor map over [rows][cols] with a 128-byte-wide swizzled box.
bool encode_u8(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, uint32_t box_cols,
               uint32_t box_rows) {
  EncodeTiledFn enc = get_encode();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols)};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 tensor map over [rows][cols] with a 64-element (128-byte) wide
// swizzled box.
bool encode_bf16(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D tensor map over [rows][cols] elements of `esize` bytes, rows
// `row_bytes` apart, with a box_cols x box_rows box and the given swizzle.
bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int64_t cols, int64_t rows,
               int64_t row_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle sw,
               CUtensorMapL2promotion l2) {
  EncodeTiledFn enc = get_encode();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, l2,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [atoms][128] uint32 view of a tensor-core scale buffer (512-byte atoms);
// a box of `box_rows` consecutive atoms.  B's two 128-row atoms of a 256-wide
// tile are adjacent unless the tile pairs gate and up rows, and then come in
// one copy: measured on GB300, one TMA copy fewer per stage and CTA made the
// step 2.8 % faster (13.99 -> 13.58 ms), most on the weight gradients.
bool encode_atoms(CUtensorMap* m, const void* base, int64_t atoms, uint32_t box_rows = 1) {
  EncodeTiledFn enc = get_encode();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {128, static_cast<cuuint64_t>(atoms)};
  const cuuint64_t strides[1] = {512};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <int BN, int EPI, bool KG, bool PAIR, int OPK = OPK_MX>
cudaError_t launch_impl(const GemmArgs& g, cudaStream_t s) {
  using C = Cfg<BN, EPI, PAIR, OPK, KG>;
  CUtensorMap ta, tb;
  const int b_box = (EPI == EPI_SWIGLU && !PAIR) ? 128 : C::kBRows;
  if (OPK == OPK_BF16) {
    if (!encode_bf16(&ta, g.a, g.a_cols, g.a_rows, BM)) return cudaErrorInvalidValue;
    if (!encode_bf16(&tb, g.b, g.b_cols, g.b_rows, b_box)) return cudaErrorInvalidValue;
  } else {
    if (!encode_u8(&ta, g.a, g.a_cols, g.a_rows, BK, BM)) return cudaErrorInvalidValue;
    if (!encode_u8(&tb, g.b, g.b_cols, g.b_rows, BK, b_box)) return cudaErrorInvalidValue;
  }
  auto kern = gemm_kernel<BN, EPI, KG, PAIR, OPK>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (err != cudaSuccess) return err;
  const int64_t units = PAIR ? num_sms() / 2 : num_sms();     // CTAs, or CTA pairs
  int64_t n = g.tiles_upper < units ? g.tiles_upper : units;
  if (n < 1) n = 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(static_cast<unsigned>(PAIR ? 2 * n : n));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  if (PAIR) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  // scale tensors as rows of 512-byte atoms, for the CTA pair's TMA loads
  CUtensorMap tsa = ta, tsb = tb;
  if (PAIR && OPK == OPK_MX) {
    if (!encode_atoms(&tsa, g.sa, (g.a_rows / 128) * (g.a_cols / 128))) return cudaErrorInvalidValue;
    if (!encode_atoms(&tsb, g.sb, (g.b_rows / 128) * (g.b_cols / 128), EPI == EPI_SWIGLU ? 1 : 2))
      return cudaErrorInvalidValue;
  }
  // MXFP8 dSwiGLU at BN = 256: the row-wise dGU codes ([rows][2I]) and the
  // column-wise ones ([2I][token capacity]), 32 x 32-byte boxes, 32-byte swizzle
  CUtensorMap tq = ta, tqc = ta;
  // token-grouped pair tiles: the [E·M][N] output (bf16 dW, or the fp32
  // main_grad added into), 32-row x 64-byte boxes, 64-byte swizzle
  // MXFP8 gate-up: the saved g|u in 32 x 32 tiles (gu_tile_offset)
  if (C::kSwTma && g.gu_save != nullptr && (g.M % 32 != 0 || g.I % 32 != 0)) return cudaErrorInvalidValue;
  if (C::kTmaOut) {
    const bool acc = EPI == EPI_ACC_F32;
    // token-grouped: [E·M][N] with rows N apart; row-grouped: [M][N] with rows ldd apart
    const int64_t rows = KG ? static_cast<int64_t>(g.E) * g.M : g.M;
    const int64_t ld = KG ? g.N : g.ldd;
    if (!encode_2d(&tq, acc ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   acc ? static_cast<const void*>(g.dacc) : static_cast<const void*>(g.d), g.N, rows,
                   ld * (acc ? 4 : 2), acc ? 16 : 32, 32, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE))
      return cudaErrorInvalidValue;
  }
  if (C::kDsTma) {
    if (!encode_2d(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.q_out, g.q_out_ld, g.M, g.q_out_ld, 32, 32,
                   CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE) ||
        !encode_2d(&tqc, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.qc_out, g.qc_ld, g.sc_rows, g.qc_ld, 32, 32,
                   CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE))
      return cudaErrorInvalidValue;
  }
  err = cudaLaunchKernelEx(&cfg, kern, ta, tb, tsa, tsb, tq, tqc, g);
  count_launch();
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

bool tma_map_bf16(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, uint32_t box_rows) {
  return encode_bf16(m, base, cols, rows, box_rows);
}

int gemm_pick_bn(int epi, int N) {
  if (epi == EPI_SWIGLU) return 256;
  return N % 256 == 0 ? 256 : 128;
}

int dswiglu_partials(int I) { return 2 * (I / gemm_pick_bn(EPI_DSWIGLU, I)); }

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t s) {
  if (g.bf16) {  // BF16 path: CTA-pair tiles only
    if (!g.pair) return cudaErrorInvalidValue;
    if (g.epi == EPI_SWIGLU) return launch_impl<256, EPI_SWIGLU, false, true, OPK_BF16>(g, s);
    if (g.epi == EPI_DSWIGLU) return launch_impl<256, EPI_DSWIGLU, false, true, OPK_BF16>(g, s);
    if (g.kgroup) return launch_impl<256, EPI_BF16, true, true, OPK_BF16>(g, s);
    return launch_impl<256, EPI_BF16, false, true, OPK_BF16>(g, s);
  }
  if (g.fp8) {  // FP8 path (per-tensor scales): CTA-pair tiles only
    if (!g.pair || g.amax_a == nullptr || g.amax_b == nullptr) return cudaErrorInvalidValue;
    if (g.epi == EPI_SWIGLU) return launch_impl<256, EPI_SWIGLU, false, true, OPK_F8>(g, s);
    if (g.epi == EPI_DSWIGLU) return launch_impl<256, EPI_DSWIGLU, false, true, OPK_F8>(g, s);
    if (g.kgroup) return launch_impl<256, EPI_BF16, true, true, OPK_F8>(g, s);
    return launch_impl<256, EPI_BF16, false, true, OPK_F8>(g, s);
  }
  if (g.pair) {  // CTA-pair tiles, 256 x 256
    if (g.epi == EPI_SWIGLU) return launch_impl<256, EPI_SWIGLU, false, true>(g, s);
    if (g.epi == EPI_DSWIGLU) return launch_impl<256, EPI_DSWIGLU, false, true>(g, s);
    if (g.kgroup && g.epi == EPI_ACC_F32) return launch_impl<256, EPI_ACC_F32, true, true>(g, s);
    if (g.kgroup) return launch_impl<256, EPI_BF16, true, true>(g, s);
    return launch_impl<256, EPI_BF16, false, true>(g, s);
  }
  const int bn = gemm_pick_bn(g.epi, g.epi == EPI_DSWIGLU ? g.I : g.N);
  if (g.epi == EPI_SWIGLU) return launch_impl<256, EPI_SWIGLU, false, false>(g, s);
  if (g.epi == EPI_DSWIGLU)
    return bn == 256 ? launch_impl<256, EPI_DSWIGLU, false, false>(g, s) : launch_impl<128, EPI_DSWIGLU, false, false>(g, s);
  if (g.kgroup && g.epi == EPI_ACC_F32)
    return bn == 256 ? launch_impl<256, EPI_ACC_F32, true, false>(g, s) : launch_impl<128, EPI_ACC_F32, true, false>(g, s);
  if (g.kgroup)
    return bn == 256 ? launch_impl<256, EPI_BF16, true, false>(g, s) : launch_impl<128, EPI_BF16, true, false>(g, s);
  return bn == 256 ? launch_impl<256, EPI_BF16, false, false>(g, s) : launch_impl<128, EPI_BF16, false, false>(g, s);
}

}  // namespace mxg
