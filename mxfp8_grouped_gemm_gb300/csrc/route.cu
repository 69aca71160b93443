// Top-k routing and the bit-exact permute (histogram -> scan -> stable scatter).
//
// Routing: BioNeMo Uses Grouped Kernels and MXFP8, Fig. 1 (a top-2 router sends
// each token to two of eight experts; outputs combined as a weighted sum).
// Permute: same page, "Grouping fragmented expert workloads" (split_sizes,
// one count per expert).  Within an expert, rows keep the order of the flat
// index t*k + j, so the result is deterministic and needs no atomics to
// decide the order.
#include <cfloat>

#include "common.cuh"
#include "kernels.h"

namespace mxg {

namespace {

// ----------------------------------------------------------------- top-k ----
// One warp per token (see warp_topk_softmax).
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                   int32_t* __restrict__ ids, float* __restrict__ probs) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  warp_topk_softmax(logits + static_cast<int64_t>(warp) * E, E, k, lane, ids + static_cast<int64_t>(warp) * k,
                    probs + static_cast<int64_t>(warp) * k);
}

// One thread per token while E k <= 64 (thread_topk_softmax: the same ids and
// probabilities as the warp route, bit for bit).
__global__ void __launch_bounds__(256) topk_thread_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                          int32_t* __restrict__ ids, float* __restrict__ probs) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  int sel[8];
  thread_topk_softmax(logits + static_cast<int64_t>(t) * E, E, k, ids + static_cast<int64_t>(t) * k,
                      probs + static_cast<int64_t>(t) * k, sel);
}

// --------------------------------------------------------------- permute ----
constexpr int kChunk = kPermuteChunk;     // flat entries per CTA
constexpr int kThreads = 256;             // the scan
constexpr int kWide = 1024;               // count and scatter: a chunk in four passes
constexpr int kMaxE = 256;

__global__ void __launch_bounds__(kWide) count_kernel(const PermuteParams P) {
  __shared__ int hist[kMaxE];
  for (int e = threadIdx.x; e < P.E; e += kWide) hist[e] = 0;
  __syncthreads();
  const int base = blockIdx.x * kChunk;
  for (int i = threadIdx.x; i < kChunk; i += kWide) {
    const int f = base + i;
    if (f >= P.R) break;
    const int e = P.ids[f];
    if (e < 0 || e >= P.E) report(P.status, MXG_ERR_EXPERT_ID);
    else atomicAdd(&hist[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < P.E; e += kWide) P.counts[blockIdx.x * P.E + e] = hist[e];
}

// One CTA: per-expert totals, exclusive scans (plain and padded) and the
// per-(chunk, expert) starting rows.
__global__ void __launch_bounds__(kThreads) scan_kernel(const PermuteParams P, int nblk) {
  __shared__ int tot[kMaxE];
  __shared__ int off[kMaxE + 1];
  __shared__ int poff[kMaxE + 1];
  for (int e = threadIdx.x; e < P.E; e += kThreads) {
    int run = 0;
    for (int b = 0; b < nblk; ++b) {
      P.bases[b * P.E + e] = run;
      run += P.counts[b * P.E + e];
    }
    tot[e] = run;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    off[0] = 0;
    poff[0] = 0;
    for (int e = 0; e < P.E; ++e) {
      off[e + 1] = off[e] + tot[e];
      poff[e + 1] = poff[e] + (tot[e] + P.pad - 1) / P.pad * P.pad;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= P.E; e += kThreads) {
    P.offsets[e] = off[e];
    P.padded_offsets[e] = poff[e];
    if (e < P.E) P.split_sizes[e] = tot[e];
  }
  for (int e = threadIdx.x; e < P.E; e += kThreads)
    for (int b = 0; b < nblk; ++b) P.bases[b * P.E + e] += off[e];
}

// Stable scatter of one chunk: each pass takes kWide consecutive entries;
// within a warp, entries of the same expert are ranked by __match_any_sync,
// warps ahead in the pass by their per-expert counts, and earlier passes and
// chunks by the running base of each expert.
__global__ void __launch_bounds__(kWide) scatter_kernel(const PermuteParams P) {
  constexpr int kWarps = kWide / 32;
  __shared__ int run[kMaxE];
  __shared__ int off[kMaxE + 1];
  __shared__ int poff[kMaxE + 1];
  __shared__ int wcnt[kWarps][kMaxE];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < P.E; e += kWide) run[e] = P.bases[blockIdx.x * P.E + e];
  for (int e = threadIdx.x; e <= P.E; e += kWide) {
    off[e] = P.offsets[e];
    poff[e] = P.padded_offsets[e];
  }
  const unsigned lt_mask = (1u << lane) - 1u;
  const int base = blockIdx.x * kChunk;
  for (int it = 0; it < kChunk / kWide; ++it) {
    const int f = base + it * kWide + threadIdx.x;
    int e = -1;
    if (f < P.R) {
      e = P.ids[f];
      if (e < 0 || e >= P.E) e = -1;
    }
    for (int i = threadIdx.x; i < kWarps * P.E; i += kWide) (&wcnt[0][0])[(i / P.E) * kMaxE + i % P.E] = 0;
    __syncthreads();
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & lt_mask);
    if (e >= 0 && rank == 0) wcnt[warp][e] = __popc(peers);
    __syncthreads();
    if (e >= 0) {
      int pre = 0;
      for (int w = 0; w < warp; ++w) pre += wcnt[w][e];
      const int r = run[e] + pre + rank;
      const int pr = poff[e] + (r - off[e]);
      if (P.src_of_row) P.src_of_row[r] = f;
      if (P.row_of_src) P.row_of_src[f] = r;
      if (P.prow_src) P.prow_src[pr] = f;
      if (P.prow_of_src) P.prow_of_src[f] = pr;
    } else if (f < P.R) {
      if (P.row_of_src) P.row_of_src[f] = -1;
      if (P.prow_of_src) P.prow_of_src[f] = -1;
    }
    __syncthreads();
    for (int ee = threadIdx.x; ee < P.E; ee += kWide) {
      int s = 0;
      for (int w = 0; w < kWarps; ++w) s += wcnt[w][ee];
      run[ee] += s;
    }
    __syncthreads();
    if (base + (it + 1) * kWide >= P.R) break;
  }
}

}  // namespace

cudaError_t launch_topk(const float* logits, int T, int E, int k, int32_t* ids, float* probs, cudaStream_t s) {
  if (E * k <= 64) {
    const int grid = (T + 255) / 256;
    if (grid == 0) return cudaSuccess;
    topk_thread_kernel<<<grid, 256, 0, s>>>(logits, T, E, k, ids, probs);
    count_launch();
    return cudaGetLastError();
  }
  const int warps_per_block = 8;
  const int grid = (T + warps_per_block - 1) / warps_per_block;
  if (grid == 0) return cudaSuccess;
  topk_kernel<<<grid, warps_per_block * 32, 0, s>>>(logits, T, E, k, ids, probs);
  count_launch();
  return cudaGetLastError();
}

int permute_num_blocks(int R) { return (R + kChunk - 1) / kChunk; }

cudaError_t launch_permute_from_counts(const PermuteParams& p, cudaStream_t s) {
  const int nblk = permute_num_blocks(p.R);
  if (nblk == 0) return cudaSuccess;
  scan_kernel<<<1, kThreads, 0, s>>>(p, nblk);
  count_launch();
  scatter_kernel<<<nblk, kWide, 0, s>>>(p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_permute(const PermuteParams& p, cudaStream_t s) {
  const int nblk = permute_num_blocks(p.R);
  if (nblk == 0) return cudaSuccess;
  count_kernel<<<nblk, kWide, 0, s>>>(p);
  count_launch();
  scan_kernel<<<1, kThreads, 0, s>>>(p, nblk);
  count_launch();
  scatter_kernel<<<nblk, kWide, 0, s>>>(p);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mxg
