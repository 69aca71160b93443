// Internal launchers shared by the C-ABI layer (api.cu) and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

namespace mxg {

void count_launch();

// ---------------------------------------------------------------- quantiser
struct QuantParams {
  const uint16_t* x;          // bf16 source
  int64_t ld_x;               // source row stride (elements)
  int64_t x_batch_stride;     // elements between batches (blockIdx.z)
  const int32_t* src_rows;    // nullable: row p reads source row src_rows[p]/src_div; -1 = zero row
  int32_t src_div;
  const float* probs;         // nullable: probs_perm[p] = probs[src_rows[p]] (0 for padding)
  float* probs_perm;
  int32_t rows;               // rows per batch (multiple of 32)
  int32_t cols;               // columns (multiple of 128)
  int32_t batch;
  const int32_t* rows_valid;  // nullable device scalar: row blocks at or past it are skipped
  uint8_t* q_row;             // nullable: [batch*rows][cols]
  uint8_t* s_row;
  int64_t sf_row_rows;        // rows of the row-wise matrix (MMA layout)
  uint8_t* q_col;             // nullable: [batch*cols][ld_col], rows of x become columns
  uint8_t* s_col;
  int64_t ld_col;
  int64_t sf_col_rows;        // rows of the column-wise matrix (MMA layout)
  int32_t layout;             // MXG_LAYOUT_*
  // bf16 pass-through (the BF16 path): the staged rows copied out unchanged
  uint16_t* b_row;            // nullable: [batch*rows][cols] (gathered copy)
  uint16_t* b_col;            // nullable: [batch*cols][ld_col] (transposed copy)
  // per-tensor FP8 (the FP8 path): when pt_amax is set, codes are E4M3(v * s)
  // with s = fp8_scale(pt_amax[g]) for the tile's tensor g (the row group of
  // pt_group_off [pt_groups + 1] that holds the tile, else the batch index);
  // q_row / q_col get the codes, no scales are written
  const float* pt_amax;
  const int32_t* pt_group_off;
  int32_t pt_groups;
  // grouped rows without a row map (the standalone grouped quantiser): padded
  // row p of group g (grp_poff[g] <= p < grp_poff[g+1]) reads source row
  // grp_off[g] + (p - grp_poff[g]) while that is below grp_off[g+1], else it
  // is a zero padding row; set rows_valid = grp_poff + groups
  const int32_t* grp_off;
  const int32_t* grp_poff;
  int32_t groups;
};
cudaError_t launch_quant(const QuantParams& p, cudaStream_t s);
// Two tensors quantised by one launch when their modes match (else two launches);
// the outputs are those of launch_quant(a) then launch_quant(b).
cudaError_t launch_quant2(const QuantParams& a, const QuantParams& b, cudaStream_t s);

// Padded layout of grouped rows: poff[g] = sum over g' < g of the group sizes
// off[g'+1] - off[g'] each rounded up to `align`.  off must start at 0, be
// monotone and end at `rows`, and the padded total must fit `cap` rows;
// otherwise MXG_ERR_OFFSETS goes to status and poff is all zeros (nothing is
// then quantised).
cudaError_t launch_group_pad(const int32_t* off, int groups, int rows, int align, int64_t cap, int32_t* poff,
                             int32_t* status, cudaStream_t s);

// Largest magnitude of each tensor of a bf16 matrix batch (per-tensor FP8):
// rows optionally gathered like QuantParams; a tensor is a row group of
// group_off [groups + 1] (rows 32-aligned in groups) or a batch.  amax holds
// fp32 values and must be zeroed by the caller (the kernel takes maxima).
struct AmaxParams {
  const uint16_t* x;
  int64_t ld_x;
  int64_t x_batch_stride;
  const int32_t* src_rows;    // nullable: row p reads source row src_rows[p]/src_div; -1 = zero row
  int32_t src_div;
  int32_t rows;               // rows per batch (multiple of 32)
  int32_t cols;               // multiple of 256
  int32_t batch;
  const int32_t* rows_valid;  // nullable device scalar
  const int32_t* group_off;   // nullable
  int32_t groups;
  float* amax;
};
cudaError_t launch_amax(const AmaxParams& p, cudaStream_t s);

// ------------------------------------------------------------ route/permute
cudaError_t launch_topk(const float* logits, int T, int E, int k, int32_t* ids, float* probs, cudaStream_t s);

struct PermuteParams {
  const int32_t* ids;
  int32_t R, E;
  int32_t* counts;            // scratch [nblk][E]
  int32_t* bases;             // scratch [nblk][E]
  int32_t* offsets;           // [E+1]
  int32_t* padded_offsets;    // [E+1]
  int32_t pad;                // group alignment in rows (128 or 256)
  int32_t* split_sizes;       // [E]
  int32_t* src_of_row;        // nullable [R] (unpadded)
  int32_t* row_of_src;        // nullable [R] (unpadded)
  int32_t* prow_src;          // nullable [m_cap] padded row -> flat index (prefilled with -1)
  int32_t* prow_of_src;       // nullable [R] flat index -> padded row
  int32_t* status;
};
int permute_num_blocks(int R);
cudaError_t launch_permute(const PermuteParams& p, cudaStream_t s);

// 2-D TMA map over a bf16 matrix [rows][cols] (row stride cols * 2 bytes):
// boxes of 64 columns (one 128-byte swizzled row) x box_rows rows; reads
// past the matrix's edges fill zeros.
bool tma_map_bf16(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, uint32_t box_rows);

// Router logits on the tensor cores and the top-k route (router_mma.cu):
// logits fp32 [T][E] = x [T][H] W_r [E][H]^T, then ids / probs as the route.
// When counts is given (zeroed by the caller), every CTA also adds its
// tokens' expert counts into counts[f / kPermuteChunk][e] (f = t*k + j): the
// permute's histogram, so the permute can start from its scan.
cudaError_t launch_router_mma(const uint16_t* x, const uint16_t* w, int T, int H, int E, int k, float* logits,
                              int32_t* ids, float* probs, int32_t* counts, int32_t* status, cudaStream_t s);
constexpr int kPermuteChunk = 4096;
// The permute's scan and scatter after an external histogram (counts filled).
cudaError_t launch_permute_from_counts(const PermuteParams& p, cudaStream_t s);

// ------------------------------------------------------------------ combine
// y[t] = sum_j src[prow_of_src[t*k + j]] (fp32 in slot order, one bf16
// rounding).  Negative entries are skipped; entries >= src_rows are skipped
// and reported as MXG_ERR_INDEX through status (nullable).
cudaError_t launch_combine(const uint16_t* src, const int32_t* prow_of_src, int T, int k, int H, uint16_t* out,
                           cudaStream_t s, int64_t src_rows = INT64_MAX, int32_t* status = nullptr);
// dst row r = src row index[r] / div (rows of row_bytes bytes, a multiple of
// 4); an index outside [0, src_rows * div) gives a zero row and MXG_ERR_INDEX.
cudaError_t launch_gather_rows(const void* src, int64_t src_rows, int64_t row_bytes, const int32_t* index, int div,
                               int64_t rows, void* dst, int32_t* status, cudaStream_t s);
// Pre-quantised rows into the padded row layout: padded row p takes codes
// row f = src[p] of q (cols bytes) and its cols/32 canonical scale bytes,
// written as codes [rows][cols] and tensor-core-layout scales (sf_rows rows);
// f < 0 (padding) gives zero codes and scales.  probs_perm[p] = probs[f]
// (0 for padding) when probs is given.
cudaError_t launch_place_rows(const uint8_t* q, const uint8_t* s, int64_t src_rows, const int32_t* src, int64_t rows,
                              const int32_t* rows_valid, int cols, uint8_t* q_out, uint8_t* s_out, int64_t sf_rows,
                              const float* probs, float* probs_perm, int32_t* status, cudaStream_t st);
// ids[r] = the group of row r, from split sizes [E] (rows of group e follow
// those of e - 1); sizes that are negative or do not sum to R give
// MXG_ERR_OFFSETS and ids -1 for the rows no group covers.
cudaError_t launch_expand_splits(const int32_t* split_sizes, int E, int64_t R, int32_t* ids, int32_t* status,
                                 cudaStream_t s);
cudaError_t launch_dprob(const float* part, int ld, const int32_t* prow_of_src, int R, float* dprobs,
                         cudaStream_t s);

// --------------------------------------------------------------------- GEMM
enum Epi { EPI_BF16 = 0, EPI_SWIGLU = 1, EPI_DSWIGLU = 2, EPI_ACC_F32 = 3 };

struct GemmArgs {
  int epi;
  bool kgroup;
  bool pair;                  // CTA-pair 256 x 256 tiles (row groups 256-aligned)
  const uint8_t* a;           // codes
  const uint8_t* sa;
  int64_t a_rows;             // rows of the A matrix (SF layout, tensor map)
  int64_t a_cols;             // contraction extent stored in A (K, or token capacity)
  const uint8_t* b;
  const uint8_t* sb;
  int64_t b_rows;
  int64_t b_cols;
  const int32_t* poff;
  int32_t E;
  int32_t M;                  // K-grouped: rows of each D_e; M-grouped: row capacity
  int32_t N;                  // output columns (SwiGLU: 2I)
  int32_t K;                  // M-grouped contraction length
  int32_t b_rows_per_expert;  // M-grouped
  int32_t I;                  // SwiGLU / dSwiGLU intermediate size
  uint16_t* d;
  int64_t ldd;
  const float* probs_perm;
  uint16_t* gu_save;
  uint8_t* q_out;
  uint8_t* s_out;
  int64_t q_out_ld;
  int64_t s_out_rows;
  uint8_t* qc_out;
  uint8_t* sc_out;
  int64_t qc_ld;
  int64_t sc_rows;
  float* dp_part;
  int32_t dp_ld;
  int32_t* status;
  // BF16 path: A and B hold bf16 values (a_cols / b_cols count elements), no
  // scale factors; the fused epilogues write bf16 instead of MXFP8
  bool bf16;
  uint16_t* y_row;            // [rows][..] bf16 row-major output (h, or dGU)
  int64_t y_row_ld;
  uint16_t* y_col;            // [cols][..] bf16 transposed output (h^T, or dGU^T)
  int64_t y_col_ld;
  // FP8 path: E4M3 operands with one power-of-two scale per expert tensor (no scale
  // factors); the epilogue multiplies by fp8_dequant(amax_a[e]) *
  // fp8_dequant(amax_b[e]) and writes bf16 like the BF16 path, adding the
  // largest magnitude of the bf16 h / dGU it writes into amax_out[e]
  bool fp8;
  const float* amax_a;
  const float* amax_b;
  float* amax_out;
  float* dacc;                // EPI_ACC_F32 (token-grouped): fp32 [E][M][N] that the tile is added into
  // Combine fused into a row-grouped bf16 epilogue: out[t] = sum over the k
  // rows of token t (slot order) of D, written by whichever thread stores the
  // last of them (counters [T][N/BN][2], zero before the launch; they are left
  // at zero again).  Null: no combine.
  uint16_t* cmb_out;          // [T][N] bf16
  const int32_t* cmb_prow_src;     // [M] padded row -> flat index t*k + j (-1: padding)
  const int32_t* cmb_prow_of_src;  // [T*k] flat index -> padded row
  int32_t* cmb_count;
  int32_t cmb_k;
  int64_t tiles_upper;        // host bound on the number of tiles (grid sizing)
  uint64_t wait_limit_ns;     // bound on every wait inside the kernel (0: default)
  int32_t debug_stall;        // test hook: the producer issues no copies
};
int gemm_pick_bn(int epi, int N);
int dswiglu_partials(int I);   // d(prob) partial sums per row (two per column tile)
cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t s);

}  // namespace mxg
