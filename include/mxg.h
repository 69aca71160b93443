/*
 * mxg — grouped MXFP8 MoE expert MLP for GB300 (sm_103a).  C ABI.
 *
 * The path: top-k routing, a permute of tokens into per-expert groups with one
 * count per expert (split_sizes), MXFP8 quantisation (E4M3 values, one E8M0
 * scale per 32 consecutive values along the contraction axis), a grouped
 * gate-up GEMM fused with ScaledSwiGLU (x routing probability) and
 * re-quantisation, a grouped down GEMM, and an unpermute/combine — plus the
 * backward (dgrad and wgrad grouped GEMMs; the wgrad operands are quantised
 * column-wise over tokens).
 *
 * Sources (web pages about the BioNeMo Mixtral MoE recipe):
 *   [Grouped]  "BioNeMo Uses Grouped Kernels and MXFP8" (toolai.io)
 *   [Overhead] "How BioNeMo cuts overhead in biological AI training"
 *              (roboticlifestyle.com)
 *
 * Conventions for every call:
 *   - Returns an mxg_status; 0 (MXG_OK) means the work was enqueued.
 *   - Asynchronous on the caller's CUDA stream (`stream` is a cudaStream_t,
 *     0 = legacy default stream).  No call synchronises the host.
 *   - No call allocates device or host memory.  Every buffer is a device
 *     pointer owned by the caller; scratch is passed in explicitly, sized by
 *     the matching *_bytes() query.
 *   - Argument errors are detected on the host before anything is launched and
 *     returned as MXG_ERR_ARG / MXG_ERR_SHAPE / MXG_ERR_ALIGN /
 *     MXG_ERR_WORKSPACE.  Errors only visible on the device (an expert id out
 *     of range, inconsistent group offsets, a kernel wait that timed out) are
 *     written to the caller's `dev_status` int32 (device memory, zero it before
 *     the call; the first error wins) and the affected kernels skip the bad
 *     work instead of faulting.
 *   - bf16 tensors are passed as uint16_t bit patterns.  All matrices are
 *     row-major and dense unless stated otherwise.
 *   - Device pointers must be 32-byte aligned (MXG_ERR_ALIGN otherwise): the
 *     GEMM epilogues read and write whole 32-byte sectors.  Allocations from
 *     cudaMalloc and torch's caching allocator satisfy this.
 */
#ifndef MXG_H_
#define MXG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MXG_OK = 0,
  MXG_ERR_ARG = 1,        /* null pointer, non-positive size, bad enum value        */
  MXG_ERR_SHAPE = 2,      /* a dimension violates the call's divisibility rules      */
  MXG_ERR_ALIGN = 3,      /* a device pointer is not 32-byte aligned                 */
  MXG_ERR_ARCH = 4,       /* current device is not sm_103 / library not built for it */
  MXG_ERR_WORKSPACE = 5,  /* caller's scratch/saved buffer is too small              */
  MXG_ERR_CUDA = 6,       /* a CUDA runtime call or kernel launch failed             */
  /* device-detected, reported through dev_status */
  MXG_ERR_EXPERT_ID = 16, /* an expert id outside [0, E)                             */
  MXG_ERR_OFFSETS = 17,   /* group offsets not monotone / not 128-aligned / too big  */
  MXG_ERR_TIMEOUT = 18,   /* a bounded wait inside a kernel gave up                  */
  MXG_ERR_INDEX = 19      /* a row index outside the buffer it indexes               */
} mxg_status;

/* Layout of MXFP8 scale bytes. */
enum {
  /* row-wise: s[r][c/32]; column-wise (transposed): sT[c][r/32] */
  MXG_LAYOUT_CANONICAL = 0,
  /* the tensor-core operand layout: for a matrix with R rows (multiple of 128)
     and contraction length K (multiple of 128), the scale of (row r, 32-block
     b) sits at byte
        ((b/4)*(R/128) + r/128)*512 + (r%32)*16 + ((r/32)%4)*4 + (b%4)
     i.e. 512-byte atoms of 128 rows x 4 blocks, laid out K-chunk-major. */
  MXG_LAYOUT_MMA = 1
};

/* Text for a status code (static storage). */
const char* mxg_status_string(int status);

/* 1 if the library's kernels can run on the current device (sm_103). */
int mxg_device_supported(void);

/* Number of kernel launches the library has enqueued since load (monotone
   counter kept on the host; used to report launches per step). */
uint64_t mxg_launch_count(void);

/* ----------------------------------------------------------------------------
 * Top-k routing.  [Grouped] Fig. 1: a top-2 router sends each token to two of
 * eight experts and the outputs are combined as a weighted sum.
 *   logits  fp32 [T][E] (device)
 *   ids     int32 [T][k] out: the k largest logits per token, descending,
 *           ties to the lower expert id
 *   probs   fp32 [T][k] out: softmax over the chosen k logits (renormalised)
 * Requires 1 <= k <= E <= 256, k <= 32.
 */
int mxg_route_topk(const float* logits, int T, int E, int k, int32_t* ids, float* probs, void* stream);

/* ----------------------------------------------------------------------------
 * Router front end: logits = x W_r^T (one linear layer H -> E, no bias) and the
 * top-k route of mxg_route_topk on them, in one kernel.  [Grouped] Fig. 1 (a
 * router picks two of eight experts per token); the page does not spell the
 * router out, the single bias-free linear layer is the reading taken.  The
 * contraction runs on the tensor cores (bf16 operands, fp32 accumulators,
 * 128 tokens per CTA); the route is taken on the fp32 logits.
 *   x         bf16 [T][H] (device)
 *   w_router  bf16 [E][H] (device)
 *   logits    fp32 [T][E] out, accumulated in fp32 from the bf16 products
 *   ids, probs  as mxg_route_topk
 * Requires H % 128 == 0, 1 <= k <= E <= 256, k <= 32.  x, w_router 32-byte
 * aligned.  A kernel wait that gives up (no status word here) leaves the
 * affected tokens' ids at -1, which a following permute reports.
 */
int mxg_router_fwd(const uint16_t* x, const uint16_t* w_router, int T, int H, int E, int k, float* logits,
                   int32_t* ids, float* probs, void* stream);

/* Router front end fused with the permute: the logits and route of
 * mxg_router_fwd, and the permute of mxg_route_permute on the chosen ids, with
 * the permute's per-chunk expert histogram accumulated by the router kernel
 * itself (the route output feeds the histogram without a second pass over the
 * ids).  [Grouped] Fig. 1 (router, top-2 of 8) and "Grouping fragmented expert
 * workloads" (split_sizes).
 *   x, w_router, logits, ids, probs   as mxg_router_fwd
 *   split_sizes, src_of_row, row_of_src, padded_offsets, ws, ws_bytes,
 *   dev_status                        as mxg_route_permute (ws sized by
 *                                     mxg_route_permute_workspace_bytes)
 * Results equal mxg_router_fwd followed by mxg_route_permute, bit for bit.
 * Requires H % 128 == 0, 1 <= k <= E <= 256, k <= 32. */
int mxg_router_fwd_permute(const uint16_t* x, const uint16_t* w_router, int T, int H, int E, int k, float* logits,
                           int32_t* ids, float* probs, int32_t* split_sizes, int32_t* src_of_row, int32_t* row_of_src,
                           int32_t* padded_offsets, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Scratch for mxg_router_bwd (bytes). */
size_t mxg_router_bwd_workspace_bytes(int T, int H, int E, int k);

/* ----------------------------------------------------------------------------
 * Router backward.  The choice of experts carries no gradient; the
 * probabilities are a softmax over the chosen logits, so
 *   dlogit[t, ids[t,j]] = probs[t,j] * (dprobs[t,j] - sum_i probs[t,i] dprobs[t,i])
 * (0 for experts not chosen), then
 *   dx[t]     += sum_j dlogit[t, ids[t,j]] * W_r[ids[t,j]]   (in place, bf16)
 *   dw_router  = sum_t dlogits[t]^T x[t]                     (fp32, overwritten)
 *   x, w_router  bf16 as in mxg_router_fwd
 *   ids, probs   the route of mxg_router_fwd; dprobs fp32 [T][k] (the MLP's
 *                d(probs) output)
 *   dx           bf16 [T][H] in/out: the router's term is added to it (pass the
 *                MLP's dx to get the layer's input gradient)
 *   dw_router    fp32 [E][H] out
 *   workspace    >= mxg_router_bwd_workspace_bytes(T, H, E, k) bytes
 * dw_router is a fixed-order sum (deterministic).  Expert ids outside [0, E)
 * are skipped and reported as MXG_ERR_EXPERT_ID through dev_status.
 * Requires H % 128 == 0, 1 <= k <= E <= 256, k <= 32.
 */
int mxg_router_bwd(const uint16_t* x, const uint16_t* w_router, const int32_t* ids, const float* probs,
                   const float* dprobs, int T, int H, int E, int k, uint16_t* dx, float* dw_router, void* workspace,
                   size_t workspace_bytes, int32_t* dev_status, void* stream);

/* ----------------------------------------------------------------------------
 * Permute index: counting sort of the flat index f = t*k + j by expert id,
 * stable in f (bit-exact, deterministic).  [Grouped] "Grouping fragmented
 * expert workloads" (split_sizes: one token count per expert); [Overhead]
 * "Grouping the expert work".
 *   ids             int32 [T][k] (device)
 *   split_sizes     int32 [E] out: rows per expert
 *   src_of_row      int32 [T*k] out: flat source index f of permuted row r
 *   row_of_src      int32 [T*k] out: permuted row of flat index f (inverse)
 *   padded_offsets  int32 [E+1] out: exclusive scan of split sizes each rounded
 *                   up to a multiple of 128 (the grouped kernels' row layout)
 *   ws              scratch of mxg_route_permute_workspace_bytes(T,k,E) bytes
 * Ids outside [0,E) set MXG_ERR_EXPERT_ID in dev_status; such entries are
 * dropped (their row_of_src is -1).
 */
size_t mxg_route_permute_workspace_bytes(int T, int k, int E);
int mxg_route_permute(const int32_t* ids, int T, int k, int E, int32_t* split_sizes, int32_t* src_of_row,
                      int32_t* row_of_src, int32_t* padded_offsets, void* ws, size_t ws_bytes,
                      int32_t* dev_status, void* stream);

/* Permute without caller scratch.  No counterpart in the paper: an addition for
 * callers that cannot allocate device memory where they route tokens (code
 * inside another framework's memory pool, or a runtime that hands out only the
 * input and output buffers), so they cannot provide the `ws` buffer above.
 * Same inputs, outputs, results and error reporting as mxg_route_permute; the
 * scratch is a fixed 256 KB (MXG_NOALLOC_SCRATCH_BYTES) array in device memory
 * that every GPU loading this library holds until the process exits.
 *   - At most mxg_route_permute_noalloc_max_entries(E) routed entries (T*k);
 *     larger calls return MXG_ERR_WORKSPACE without launching (16,773,120
 *     entries for E = 8, 2,093,056 for E = 64, 520,192 for E = 256).
 *   - The first call on each device looks up the array's device address (a
 *     host-side runtime query, no allocation).
 *   - All calls share the one array.  Calls whose kernels overlap on the GPU
 *     (different streams without ordering) race and give wrong results;
 *     serialise them.  Nothing needs clearing between calls: every scratch
 *     entry is written before it is read.
 *   - Calls no cudaMalloc, cudaFree or other allocating routine. */
#define MXG_NOALLOC_SCRATCH_BYTES 262144
size_t mxg_route_permute_noalloc_max_entries(int E);
int mxg_route_permute_noalloc(const int32_t* ids, int T, int k, int E, int32_t* split_sizes, int32_t* src_of_row,
                              int32_t* row_of_src, int32_t* padded_offsets, int32_t* dev_status, void* stream);

/* ----------------------------------------------------------------------------
 * Measurement entry (no counterpart in the paper's API): the MXFP8 tensor-core
 * ceiling of the current GPU.  One CTA per SM runs `steps` steps of four
 * block-scaled E4M3 MMAs (tcgen05 kind::mxf8f6f4, 128 x 256 x 32 each, fp32
 * accumulators in TMEM) on operands resident in shared memory, the scale
 * factors copied into TMEM per stage as the grouped GEMM does; nothing is read
 * from or written to global memory except dev_status.  The operand values are
 * fixed small E4M3 codes and the results are discarded.
 * [Grouped] "Reducing memory pressure with MXFP8": the recipe's gain comes
 * from 8-bit tensor-core math; the dense MXFP8 rate is measured here so the
 * GEMMs' fraction of peak has a denominator taken on the same GPU.
 *   steps      > 0; every step is 4 * 2 * 128 * 256 * 32 flop per SM
 *   flops      host out: the flop count of the launch (SM count x steps x 4 x
 *              2 * 128 * 256 * 32); time the launch with events on `stream`
 *   dev_status device int32; MXG_ERR_TIMEOUT if a bounded wait gave up
 * The kernel holds all 512 TMEM columns of every SM while it runs: launch it
 * alone, not concurrently with other tensor-core kernels. */
int mxg_bench_mxfp8_mma_peak(int steps, double* flops, int32_t* dev_status, void* stream);

/* ----------------------------------------------------------------------------
 * MXFP8 quantisation of a bf16 matrix x [rows][cols].  [Grouped] "Reducing
 * memory pressure with MXFP8", Fig. 3; [Overhead] "How MXFP8 reduces memory
 * use".  Scale rule (OCP MX): e = floor(log2(max|v| over the block)) - 8,
 * clamped to [-127,127] (an all-zero block gets e = -127); scale byte e+127;
 * codes = E4M3(v * 2^-e), round to nearest even, saturate to +-448.
 *   q_row/s_row  (nullable) row-wise: blocks of 32 along cols.
 *                q_row uint8 [rows][cols]; s_row per `layout`.
 *   q_col/s_col  (nullable) column-wise: blocks of 32 consecutive rows,
 *                stored transposed: q_col uint8 [cols][rows]; s_col per layout.
 * Requires rows % 32 == 0 and cols % 128 == 0; the MMA layout also requires
 * rows % 128 == 0.
 */
int mxg_mxfp8_quantize(const uint16_t* x, int rows, int cols, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                       uint8_t* s_col, int layout, void* stream);

/* ----------------------------------------------------------------------------
 * MXFP8 quantisation of rows that come in groups (the tokens of each expert,
 * one count per expert: [Grouped] "Grouping fragmented expert workloads"),
 * with the column-wise blocks of 32 rows restarting at every group's first
 * row, as the weight-gradient operands need them ([Grouped] "Fusing precision
 * conversion and expert computation": MXFP8 in the backward too; the blocks
 * run over tokens because the weight gradients contract over tokens).  Scale
 * rule as mxg_mxfp8_quantize.
 *   x               bf16 [rows][cols] (device), the groups one after another
 *   group_offsets   int32 [groups+1] (device): 0 = off[0] <= ... <= off[groups]
 *                   = rows; group g is rows [off[g], off[g+1])
 *   padded_offsets  int32 [groups+1] out (device): the output row layout;
 *                   group g occupies padded rows [poff[g], poff[g+1]), its
 *                   size rounded up to A rows, A = 32 (MXG_LAYOUT_CANONICAL) or
 *                   128 (MXG_LAYOUT_MMA, the grouped GEMMs' tile height)
 *   q_row/s_row     (nullable) row-wise (blocks along cols): codes uint8
 *                   [cap][cols], scales per `layout` (R = cap rows)
 *   q_col/s_col     (nullable) column-wise, transposed: codes uint8
 *                   [cols][cap], blocks of 32 consecutive padded rows (never
 *                   straddling groups); scales per `layout` (R = cols rows,
 *                   K = cap)
 *   cap             = mxg_mxfp8_grouped_rows_capacity(rows, groups, layout)
 * Padding rows inside a group's padded range are zero codes (and zero scale
 * bytes where a whole block is padding); rows at or past poff[groups] are not
 * written.  Requires cols % 128 == 0, 1 <= groups <= 2^20.  Offsets that do not
 * start at 0, decrease, or do not end at `rows` set MXG_ERR_OFFSETS in
 * dev_status; padded_offsets is then all zeros and nothing is quantised.
 * Two launches (the padded offsets, then the quantiser). */
size_t mxg_mxfp8_grouped_rows_capacity(int rows, int groups, int layout);
int mxg_mxfp8_quantize_grouped(const uint16_t* x, int rows, int cols, const int32_t* group_offsets, int groups,
                               int32_t* padded_offsets, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                               uint8_t* s_col, int layout, int32_t* dev_status, void* stream);

/* ----------------------------------------------------------------------------
 * Row gather: dst row r = src row index[r] / div, for rows of row_bytes bytes
 * (a multiple of 4).  The dispatch and return steps around grouped tokens:
 * x in permuted order (index = src_of_row, div = k), the per-row routing
 * probabilities (index = src_of_row, div = 1, row_bytes = 4), the rows an
 * expert-parallel exchange brings back, or dprobs[t][j] = dprob_rows[
 * row_of_src[t*k+j]] ([Grouped] "Grouping fragmented expert workloads": tokens
 * are grouped per expert before the grouped GEMMs and returned after).
 *   src    device, src_rows rows;  index int32 [rows] (device)
 *   dst    device, rows rows (must not overlap src)
 * An index outside [0, src_rows * div) gives a zero row and MXG_ERR_INDEX in
 * dev_status.  Pointers 4-byte aligned (16-byte aligned rows go as 16-byte
 * vectors).  HBM-bound: one read and one write per byte. */
int mxg_gather_rows(const void* src, int64_t src_rows, int64_t row_bytes, const int32_t* index, int div,
                    int64_t rows, void* dst, int32_t* dev_status, void* stream);

/* ----------------------------------------------------------------------------
 * Combine (unpermute + sum): y[t] = sum_j rows[row_of_src[t*k + j]] for
 * j = 0..k-1, accumulated in fp32 in slot order, one bf16 rounding.  The
 * weighted sum of [Grouped] Fig. 1 with the routing probability already
 * applied to each row (inside ScaledSwiGLU, "Fusing precision conversion and
 * expert computation"), so this is a plain sum.  The MLP calls run it (or
 * its fused form) themselves; this entry serves rows that come back from
 * elsewhere (an expert-parallel return, or mxg_grouped_mlp_fwd_grouped).
 *   rows        bf16 [src_rows][H] (device);  row_of_src int32 [T*k] (device;
 *               a negative entry is skipped; one >= src_rows is skipped and
 *               reported as MXG_ERR_INDEX)
 *   y           bf16 [T][H] out
 * Requires H % 8 == 0, k <= 32; rows and y 16-byte aligned. */
int mxg_combine(const uint16_t* rows, int64_t src_rows, const int32_t* row_of_src, int T, int k, int H, uint16_t* y,
                int32_t* dev_status, void* stream);

/* ----------------------------------------------------------------------------
 * Grouped MXFP8 GEMM, row-grouped (the GroupedLinear forward/dgrad shape;
 * [Grouped] "Grouping fragmented expert workloads"): for each expert e, rows
 * [padded_offsets[e], padded_offsets[e+1]) of A are multiplied by expert e's
 * B: D[r][n] = sum_k deq(A)[r][k] * deq(B_e)[n][k], stored as bf16.
 *   a, sa   uint8 codes [m_cap][K] + scales (MXG_LAYOUT_MMA, R = m_cap)
 *   b, sb   uint8 codes [E*N][K] + scales (MXG_LAYOUT_MMA, R = E*N)
 *   padded_offsets int32 [E+1] (device): 128-aligned, monotone, last <= m_cap
 *   d       bf16 [m_cap][N]; rows outside the groups are not written
 * Requires K % 128 == 0, N % 128 == 0, m_cap % 128 == 0.
 */
int mxg_grouped_gemm(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                     const int32_t* padded_offsets, int E, int m_cap, int N, int K, uint16_t* d,
                     int32_t* dev_status, void* stream);

/* Test hook for failure detection (no counterpart in the paper): runs
 * mxg_grouped_gemm with every kernel wait bounded by `wait_limit_ns` and a
 * producer that never issues its copies, so the first wait of the MMA warp
 * runs out.  The kernel then records MXG_ERR_TIMEOUT in dev_status, stops,
 * waits for its own work, frees its tensor memory and returns; the CUDA
 * context stays usable.  `d` is left unwritten.  Same argument rules as
 * mxg_grouped_gemm; wait_limit_ns must be non-zero. */
int mxg_debug_grouped_gemm_stall(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                                 const int32_t* padded_offsets, int E, int m_cap, int N, int K, uint16_t* d,
                                 uint64_t wait_limit_ns, int32_t* dev_status, void* stream);

/* Grouped MXFP8 GEMM, contraction-grouped (the weight-gradient shape): for
 * each expert e, D_e[m][n] = sum over tokens t in [padded_offsets[e],
 * padded_offsets[e+1]) of deq(A)[m][t] * deq(B)[n][t].  A and B are stored
 * token-contiguous (the column-wise quantiser's output).
 *   a, sa  uint8 [M][t_cap] + scales (MMA layout, R = M, K = t_cap)
 *   b, sb  uint8 [N][t_cap] + scales (MMA layout, R = N, K = t_cap)
 *   d      bf16 [E][M][N]; an expert with no tokens gets exact zeros.
 * Requires M % 128 == 0, N % 128 == 0, t_cap % 128 == 0.
 */
int mxg_grouped_gemm_wgrad(const uint8_t* a, const uint8_t* sa, const uint8_t* b, const uint8_t* sb,
                           const int32_t* padded_offsets, int E, int M, int N, int t_cap, uint16_t* d,
                           int32_t* dev_status, void* stream);

/* ----------------------------------------------------------------------------
 * The whole grouped expert MLP.  [Grouped] "Fusing precision conversion and
 * expert computation" and Fig. 4; [Overhead] "Why fused operations matter".
 *   forward : permute -> quantise x (and W, both orientations) -> gate-up GEMM
 *             with fused h = p * SiLU(g) * u and MXFP8 re-quantisation of h ->
 *             down GEMM -> combine y[t] = sum_j Y[row(t,j)].  The routing
 *             probability is applied once, inside the activation.
 *   backward: quantise dy -> dgrad-down GEMM with fused dSwiGLU (emits dGU in
 *             both MXFP8 orientations and d(prob)) -> wgrad-down -> dgrad-gate-up
 *             -> wgrad-gate-up -> combine dx, reduce dprobs.
 * Weight layout: w_gate_up [E][2I][H] (rows 0..I-1 gate, I..2I-1 up),
 * w_down [E][H][I]; bf16 master weights, no bias.
 * Shapes: H % 128 == 0, I % 128 == 0, 1 <= k <= E <= 256.
 * `saved` (mxg_mlp_saved_bytes) is written by the forward and read by the
 * backward; `workspace` (mxg_mlp_workspace_bytes) is scratch for either call.
 */
typedef struct {
  int32_t T, H, I, E, k;
  const uint16_t* x;         /* bf16 [T][H]                                  */
  const int32_t* ids;        /* int32 [T][k] expert ids (e.g. from route_topk) */
  const float* probs;        /* fp32 [T][k] routing probabilities            */
  const uint16_t* w_gate_up; /* bf16 [E][2I][H]                              */
  const uint16_t* w_down;    /* bf16 [E][H][I]                               */
  uint16_t* y;               /* out bf16 [T][H]                              */
  int32_t* split_sizes;      /* out int32 [E]                                */
  void* saved;               /* caller-owned, kept for the backward          */
  uint64_t saved_bytes;
  void* workspace;
  uint64_t workspace_bytes;
  int32_t save_for_backward; /* 0: inference (skips what only backward needs) */
  int32_t* dev_status;
  /* Optional weight cache (NULL: quantise w_gate_up / w_down in this call).
   * When given, the forward skips the weight quantisation stage and reads the
   * MXFP8 weights written by mxg_mlp_quantize_weights(); w_gate_up and w_down
   * may then be NULL, and `saved` needs only mxg_mlp_saved_bytes_cached(). */
  const void* weight_cache;
  uint64_t weight_cache_bytes;
} mxg_mlp_fwd_args;

typedef struct {
  int32_t T, H, I, E, k;
  const uint16_t* dy;        /* bf16 [T][H] upstream gradient               */
  const void* saved;         /* written by the forward with save_for_backward */
  uint64_t saved_bytes;
  uint16_t* dx;              /* out bf16 [T][H]                              */
  uint16_t* dw_gate_up;      /* out bf16 [E][2I][H]                          */
  uint16_t* dw_down;         /* out bf16 [E][H][I]                           */
  float* dprobs;             /* out fp32 [T][k]                              */
  void* workspace;
  uint64_t workspace_bytes;
  int32_t* dev_status;
  /* The weight cache the forward used (NULL if it quantised the weights
   * itself); it must be unchanged since that forward. */
  const void* weight_cache;
  uint64_t weight_cache_bytes;
  /* Optional fp32 gradient accumulators (main_grad), both or neither.  When
   * given, the weight gradients are added into them in fp32 straight from the
   * GEMM accumulators (a buffer's element belongs to one output tile, so the
   * update is deterministic) and dw_gate_up / dw_down are not written (they
   * may be NULL).  Experts without tokens leave their slices unchanged. */
  float* main_grad_gate_up;  /* in/out fp32 [E][2I][H]                       */
  float* main_grad_down;     /* in/out fp32 [E][H][I]                        */
} mxg_mlp_bwd_args;

/* The forward and backward are sequences of stages, each one kernel launch
 * (the permute is three).  *_stage() runs a single stage with the same
 * arguments and checks; running every stage in order equals the full call.
 * Used to time each kernel with events on the caller's stream. */
enum {
  MXG_FWD_PERMUTE = 0,       /* histogram -> scan -> stable scatter (3 launches)       */
  MXG_FWD_QUANT_WEIGHTS = 1, /* W_gate_up then W_down, both orientations (2 launches) */
  MXG_FWD_QUANT_X = 2,       /* gather x to the padded layout + quantise               */
  MXG_FWD_GATE_UP = 3,       /* gate-up GEMM + ScaledSwiGLU + requantise               */
  MXG_FWD_DOWN = 4,          /* down GEMM                                              */
  MXG_FWD_COMBINE = 5,       /* y[t] = sum_j Y[row(t, j)] (MXFP8: fused into DOWN for long K) */
  MXG_FWD_NUM_STAGES = 6
};
enum {
  MXG_BWD_QUANT_DY = 0,      /* gather dy + quantise, both orientations               */
  MXG_BWD_DGRAD_DOWN = 1,    /* dH GEMM + fused dSwiGLU                                */
  MXG_BWD_WGRAD_DOWN = 2,    /* dW_down GEMM (token-grouped)                           */
  MXG_BWD_DGRAD_GATE_UP = 3, /* dX GEMM                                                */
  MXG_BWD_WGRAD_GATE_UP = 4, /* dW_gate_up GEMM (token-grouped)                        */
  MXG_BWD_COMBINE_DX = 5,    /* dx[t] = sum_j dX[row(t, j)] (MXFP8: fused for long K) */
  MXG_BWD_DPROBS = 6,        /* dprobs[t, j] from the per-tile partials                */
  MXG_BWD_NUM_STAGES = 7
};
int mxg_grouped_mlp_fwd_stage(const mxg_mlp_fwd_args* args, int stage, void* stream);
int mxg_grouped_mlp_bwd_stage(const mxg_mlp_bwd_args* args, int stage, void* stream);

/* The MLP keeps each expert's rows in a padded layout whose groups start on a
 * multiple of mxg_mlp_group_align() rows (256: one CTA-pair GEMM tile);
 * mxg_mlp_row_capacity() is the number of padded rows it reserves. */
int mxg_mlp_group_align(void);
size_t mxg_mlp_row_capacity(int T, int k, int E);
size_t mxg_mlp_saved_bytes(int T, int H, int I, int E, int k);
size_t mxg_mlp_workspace_bytes(int T, int H, int I, int E, int k);
int mxg_grouped_mlp_fwd(const mxg_mlp_fwd_args* args, void* stream);
int mxg_grouped_mlp_bwd(const mxg_mlp_bwd_args* args, void* stream);

/* ----------------------------------------------------------------------------
 * The grouped expert MLP on tokens that arrive already grouped by expert: the
 * pages' GroupedLinear call, experts(tokens, split_sizes), one count per
 * expert and one weight per expert ([Grouped] "Grouping fragmented expert
 * workloads"), e.g. rows an expert-parallel dispatcher delivered or a caller
 * that permuted them itself.  Same forward as mxg_grouped_mlp_fwd with each
 * row its own token (T = R, k = 1) and its expert given by position:
 *   x            bf16 [R][H]: expert e's rows are [sum_{e'<e} split_sizes[e'],
 *                + split_sizes[e]) (empty experts allowed)
 *   split_sizes  int32 [E] (device, input); negative sizes or a sum other
 *                than R set MXG_ERR_OFFSETS in dev_status (rows no expert
 *                covers are then skipped and reported as MXG_ERR_EXPERT_ID)
 *   probs        fp32 [R]: each row's routing probability, applied once in
 *                ScaledSwiGLU
 *   y            bf16 [R][H] out: each row's expert output (not combined;
 *                mxg_combine sums a token's rows)
 *   saved        mxg_mlp_grouped_saved_bytes(R, H, I, E) bytes
 *   workspace    mxg_mlp_grouped_workspace_bytes(R, H, I, E) bytes
 *   w_gate_up, w_down, save_for_backward, dev_status, weight_cache: as
 *                mxg_mlp_fwd_args.
 * The backward is mxg_grouped_mlp_bwd with T = R, k = 1, this `saved`, and a
 * workspace of the same size: dy [R][H] -> dx [R][H] (per row), dW, dprobs
 * [R].  Same shape rules and errors as mxg_grouped_mlp_fwd. */
typedef struct {
  int32_t R, H, I, E;
  const uint16_t* x;           /* bf16 [R][H], grouped by expert             */
  const int32_t* split_sizes;  /* int32 [E] rows per expert (device, input)  */
  const float* probs;          /* fp32 [R]                                   */
  const uint16_t* w_gate_up;   /* bf16 [E][2I][H]                            */
  const uint16_t* w_down;      /* bf16 [E][H][I]                             */
  uint16_t* y;                 /* out bf16 [R][H]                            */
  void* saved;
  uint64_t saved_bytes;
  void* workspace;
  uint64_t workspace_bytes;
  int32_t save_for_backward;
  int32_t* dev_status;
  const void* weight_cache;
  uint64_t weight_cache_bytes;
} mxg_mlp_grouped_fwd_args;
size_t mxg_mlp_grouped_saved_bytes(int R, int H, int I, int E);
size_t mxg_mlp_grouped_workspace_bytes(int R, int H, int I, int E);
int mxg_grouped_mlp_fwd_grouped(const mxg_mlp_grouped_fwd_args* args, void* stream);

/* The same forward on grouped rows that arrive already quantised: row-wise
 * MXFP8 codes and E8M0 scales (blocks of 32 along H), e.g. what an
 * expert-parallel dispatcher shipped instead of bf16 rows (about half the
 * bytes).  Inference only: the weight gradient of W_gate_up needs x quantised
 * in blocks of 32 tokens of each expert's group, which row-wise codes cannot
 * give, so there is no backward for this call.  [Grouped] "Reducing memory
 * pressure with MXFP8" (MXFP8 operands) and "Grouping fragmented expert
 * workloads" (tokens grouped with split_sizes).
 *   xq   uint8 [R][H] E4M3 codes (device, 32-byte aligned)
 *   xs   uint8 [R][H/32] E8M0 scales, canonical layout (device, 4-byte aligned)
 *   the rest as mxg_mlp_grouped_fwd_args without x and save_for_backward;
 *   saved and workspace sized by the mxg_mlp_grouped_* queries.
 * Given the codes and scales mxg_mxfp8_quantize writes for x's rows, y equals
 * mxg_grouped_mlp_fwd_grouped's bit for bit. */
typedef struct {
  int32_t R, H, I, E;
  const uint8_t* xq;           /* E4M3 codes [R][H], grouped by expert       */
  const uint8_t* xs;           /* E8M0 scales [R][H/32]                      */
  const int32_t* split_sizes;  /* int32 [E] (device, input)                  */
  const float* probs;          /* fp32 [R]                                   */
  const uint16_t* w_gate_up;   /* bf16 [E][2I][H]                            */
  const uint16_t* w_down;      /* bf16 [E][H][I]                             */
  uint16_t* y;                 /* out bf16 [R][H]                            */
  void* saved;
  uint64_t saved_bytes;
  void* workspace;
  uint64_t workspace_bytes;
  int32_t* dev_status;
  const void* weight_cache;
  uint64_t weight_cache_bytes;
} mxg_mlp_grouped_fwd_mx_args;
int mxg_grouped_mlp_fwd_grouped_mx(const mxg_mlp_grouped_fwd_mx_args* args, void* stream);

/* Weight cache: the four MXFP8 weight tensors the MLP needs (W_gate_up
 * quantised along H and along 2I, W_down along I and along H, codes and
 * tensor-core scale layout), written once per weight update and reused by
 * every forward / backward until the weights change (micro-batches of one
 * optimizer step).  This is the forward's weight stage on its own ("Fusing
 * precision conversion and expert computation": the recipe converts the bf16
 * master weights to MXFP8 before the GEMMs).
 *   mxg_mlp_weight_cache_bytes: bytes of the cache (0 for unsupported shapes).
 *   mxg_mlp_quantize_weights: w_gate_up bf16 [E][2I][H], w_down bf16 [E][H][I]
 *     (device) -> cache (device, caller-owned, >= cache_bytes).  Async on
 *     `stream`; MXG_ERR_SHAPE / MXG_ERR_ALIGN / MXG_ERR_WORKSPACE before any
 *     launch.
 *   mxg_mlp_saved_bytes_cached: the `saved` size when the forward is given a
 *     weight cache (the transposed weights then live in the cache only). */
size_t mxg_mlp_weight_cache_bytes(int H, int I, int E);
int mxg_mlp_quantize_weights(const uint16_t* w_gate_up, const uint16_t* w_down, int H, int I, int E, void* cache,
                             size_t cache_bytes, void* stream);
size_t mxg_mlp_saved_bytes_cached(int T, int H, int I, int E, int k);
/* Debug view into a weight cache (device pointer; NULL on bad arguments) for
 * the tests: 0 / 1 = W_gate_up along H: codes uint8 [E*2I][H] / scales
 * (tensor-core layout, E*2I rows x H/32 blocks); 2 / 3 = W_down along I:
 * [E*H][I] / (E*H rows x I/32); 4 / 5 = W_gate_up along 2I, transposed:
 * [E*H][2I] / (E*H rows x 2I/32); 6 / 7 = W_down along H, transposed:
 * [E*I][H] / (E*I rows x H/32). */
const void* mxg_mlp_weight_cache_view(const void* cache, int H, int I, int E, int which);

/* ----------------------------------------------------------------------------
 * The same grouped expert MLP in BF16: bf16 operands on the tensor cores with
 * fp32 accumulation, no quantisation; h and dGU are kept in bf16.  The like-
 * for-like reference of the MXFP8 path ([Grouped] "Training benchmark", Fig.
 * 5, compares the recipe's BF16 and MXFP8 runs).  Arguments, stages, outputs,
 * ownership and errors as mxg_grouped_mlp_fwd / _bwd, with `saved` and
 * `workspace` sized by the two _bf16_ queries (a saved buffer of one precision
 * cannot be passed to the other's backward; weight_cache and the main_grad
 * pointers must be NULL: MXG_ERR_ARG otherwise).  Requires H % 256 == 0 and
 * I % 256 == 0 (every GEMM runs as 256 x 256 CTA-pair tiles; expert groups
 * start on multiples of 256 padded rows).
 */
size_t mxg_mlp_bf16_saved_bytes(int T, int H, int I, int E, int k);
size_t mxg_mlp_bf16_workspace_bytes(int T, int H, int I, int E, int k);
int mxg_grouped_mlp_bf16_fwd(const mxg_mlp_fwd_args* args, void* stream);
int mxg_grouped_mlp_bf16_bwd(const mxg_mlp_bwd_args* args, void* stream);
int mxg_grouped_mlp_bf16_fwd_stage(const mxg_mlp_fwd_args* args, int stage, void* stream);
int mxg_grouped_mlp_bf16_bwd_stage(const mxg_mlp_bwd_args* args, int stage, void* stream);

/* ----------------------------------------------------------------------------
 * The same grouped expert MLP in per-tensor FP8: E4M3 operands with one
 * power-of-two scale per expert tensor (the MX rule with the whole tensor as
 * its block, "current scaling": e = floor(log2 amax) - 8 of the tensor, a
 * tensor being an expert's weight matrix or its rows of x, h, dy or dGU;
 * codes E4M3(v * 2^-e), round to nearest even, saturating) on the tensor
 * cores (kind::f8f6f4, fp32 accumulation scaled by both tensors' 2^e).  The FP8
 * variant of the recipe ([Grouped] "Reducing memory pressure with MXFP8": FP8
 * and MXFP8 differ in scaling granularity).  h and dGU are written in bf16 by
 * the GEMM epilogues, which also take their per-expert amax, and quantised by
 * a following pass (the gate-up and dgrad-down stages are two launches plus a
 * memset; the quantise stages are a memset, an amax pass and the quantiser).
 * Arguments, outputs, ownership and errors as mxg_grouped_mlp_fwd / _bwd with
 * `saved` / `workspace` sized by the _fp8_ queries; weight_cache and the
 * main_grad pointers must be NULL (MXG_ERR_ARG).  Requires H % 256 == 0 and
 * I % 256 == 0.
 */
size_t mxg_mlp_fp8_saved_bytes(int T, int H, int I, int E, int k);
size_t mxg_mlp_fp8_workspace_bytes(int T, int H, int I, int E, int k);
int mxg_grouped_mlp_fp8_fwd(const mxg_mlp_fwd_args* args, void* stream);
int mxg_grouped_mlp_fp8_bwd(const mxg_mlp_bwd_args* args, void* stream);
int mxg_grouped_mlp_fp8_fwd_stage(const mxg_mlp_fwd_args* args, int stage, void* stream);
int mxg_grouped_mlp_fp8_bwd_stage(const mxg_mlp_bwd_args* args, int stage, void* stream);
/* Debug views into an FP8 `saved` buffer (device pointers; NULL on bad
 * arguments) for the tests: 0 = x's codes transposed (uint8 [H][m_cap], the
 * padded row layout of mxg_mlp_row_capacity), 1..4 = amax of x, W_gate_up,
 * W_down, h per expert (fp32 [E]), 5 = padded_offsets (int32 [E+1]). */
const void* mxg_mlp_fp8_saved_view(const void* saved, int T, int H, int I, int E, int k, int which);

/* Debug views into `saved` (device pointers; NULL on bad arguments) used by the
 * tests to compare intermediates: 0 = GU (the gate-up GEMM output before the
 * activation, m_cap x 2I bf16 values, m_cap = mxg_mlp_row_capacity) in 32 x 32
 * tiles: the tile of rows 32rb.. and gate columns 32cb.. (cb < I/32) starts at
 * element (rb*I/32 + cb)*2048 and holds the gate block, then the up block of
 * the same columns, each as two 16-column halves of 32 rows x 16 values (row r
 * of half h at h*512 + r*16), 1 =
 * padded_offsets (int32 [E+1], multiples of mxg_mlp_group_align()), 2 =
 * row_of_src in the padded layout (int32 [T*k]), 3 / 4 = x's token-column-wise
 * codes (uint8 [H][m_cap]) / scales (tensor-core layout, H rows x m_cap/32
 * blocks), 5 / 6 = the same for h (I rows). */
const void* mxg_mlp_saved_view(const void* saved, int T, int H, int I, int E, int k, int which);
/* Debug views into the MXFP8 `workspace` (device pointers; NULL on bad
 * arguments): after a backward, the dSwiGLU epilogue's re-quantised dGU, 0 / 1 =
 * row-wise codes (uint8 [m_cap][2I]) / scales (tensor-core layout, m_cap rows
 * x 2I/32 blocks), 2 / 3 = token-column-wise codes (uint8 [2I][m_cap]) /
 * scales (2I rows x m_cap/32 blocks); 4 = the down GEMM's rows before the
 * combine (bf16 [m_cap][H], after a forward), 5 = the dgrad-gate-up GEMM's rows
 * before the combine (bf16 [m_cap][H], after a backward).  Valid until the
 * workspace is reused. */
const void* mxg_mlp_workspace_view(const void* workspace, int T, int H, int I, int E, int k, int which);

#ifdef __cplusplus
}
#endif
#endif /* MXG_H_ */
