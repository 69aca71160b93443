// Router front end: logits = x W_r^T fused with the top-k route, and its
// backward (dlogits, the router's term of dx, dW_r).
//
// BioNeMo Uses Grouped Kernels and MXFP8, Fig. 1: a router picks two of eight
// experts per token and the experts' outputs are summed with its weights.  The
// router itself is read as one bias-free linear layer H -> E on the token's
// hidden state; the route on its logits is the one of warp_topk_softmax.
//
// Backward: the choice of experts carries no gradient; with p = softmax over
// the k chosen logits, dlogit_j = p_j (dp_j - sum_i p_i dp_i), zero for the
// experts not chosen.  dx gets sum_j dlogit_j W_r[e_j] added in place;
// dW_r = dlogits^T x is reduced over fixed token chunks in a fixed order.
#include <climits>

#include "api_common.h"
#include "common.cuh"
#include "kernels.h"

namespace mxg {

namespace {

// ------------------------------------------------------------------ forward
// The forward (logits on the tensor cores, the route, optionally the
// permute's histogram) is router_mma.cu; H must be a multiple of this.
constexpr int kHChunk = 128;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ----------------------------------------------------------------- backward
// One warp per token: the chosen logits' gradients (kept for dW_r), then the
// token's dx row gets sum_j dlogit_j W_r[e_j] added (fp32, rounded to bf16 once).
__global__ void __launch_bounds__(256) router_dx_kernel(const uint16_t* __restrict__ w,
                                                       const int32_t* __restrict__ ids,
                                                       const float* __restrict__ probs,
                                                       const float* __restrict__ dprobs, int T, int H, int E, int k,
                                                       uint16_t* __restrict__ dx, float* __restrict__ dsel,
                                                       int32_t* __restrict__ status) {
  const int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  float p = 0.f, dp = 0.f;
  int e = 0;
  if (lane < k) {
    p = probs[t * k + lane];
    dp = dprobs[t * k + lane];
    e = ids[t * k + lane];
  }
  float inner = p * dp;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) inner += __shfl_xor_sync(0xffffffffu, inner, off);
  float d = lane < k ? p * (dp - inner) : 0.f;
  if (lane < k && (e < 0 || e >= E)) {
    report(status, MXG_ERR_EXPERT_ID);
    d = 0.f;
    e = 0;
  }
  if (lane < k) dsel[t * k + lane] = d;
  uint16_t* row = dx + t * H;
  for (int c = lane; c < H / 8; c += 32) {
    float v[8];
    const uint4 q = *reinterpret_cast<const uint4*>(row + c * 8);
    const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = bf16_lo(qw[i]);
      v[2 * i + 1] = bf16_hi(qw[i]);
    }
    for (int j = 0; j < k; ++j) {
      const int ej = __shfl_sync(0xffffffffu, e, j);
      const float dj = __shfl_sync(0xffffffffu, d, j);
      const uint4 r = *reinterpret_cast<const uint4*>(w + static_cast<int64_t>(ej) * H + c * 8);
      const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] = fmaf(dj, bf16_lo(rw[i]), v[2 * i]);
        v[2 * i + 1] = fmaf(dj, bf16_hi(rw[i]), v[2 * i + 1]);
      }
    }
    *reinterpret_cast<uint4*>(row + c * 8) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                                       pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
  }
}

constexpr int kDwCols = 128;      // hidden columns per CTA (two per thread)
constexpr int kDwThreads = kDwCols / 2;
constexpr int kDwExperts = 32;    // experts per CTA (grid z covers the rest)
// tokens per partial sum: 256 puts 512 CTAs of the one-pass backward on the
// Mixtral tokens (measured against 512: 0.170 vs 0.175 ms there, 0.167 vs
// 0.176 ms at 64 experts top-8, and twice as fast for a few thousand tokens)
constexpr int kDwTokChunk = 256;
constexpr int kDwUnroll = 8;      // tokens whose x values are loaded together

// Partial dW_r over one token chunk for 128 columns and up to 32 experts, in
// shared memory (each thread owns its two columns, so no two threads touch
// the same word).  x is read 8 tokens at a time so the loads overlap.
__global__ void __launch_bounds__(kDwThreads) router_dw_partial_kernel(const uint16_t* __restrict__ x,
                                                                      const int32_t* __restrict__ ids,
                                                                      const float* __restrict__ dsel, int T, int H,
                                                                      int E, int k, float* __restrict__ part) {
  __shared__ float2 acc[kDwExperts][kDwThreads];
  const int tid = threadIdx.x;
  const int hp = blockIdx.x * kDwThreads + tid;          // column pair
  const int e0 = blockIdx.z * kDwExperts;
  const int ne = min(kDwExperts, E - e0);
  for (int ee = 0; ee < ne; ++ee) acc[ee][tid] = make_float2(0.f, 0.f);
  const uint32_t* x2 = reinterpret_cast<const uint32_t*>(x);
  const int ta = blockIdx.y * kDwTokChunk;
  const int tb = min(T, ta + kDwTokChunk);
  for (int t = ta; t < tb; t += kDwUnroll) {
    uint32_t xv[kDwUnroll];
#pragma unroll
    for (int u = 0; u < kDwUnroll; ++u)
      xv[u] = t + u < tb ? x2[static_cast<int64_t>(t + u) * (H / 2) + hp] : 0u;
#pragma unroll
    for (int u = 0; u < kDwUnroll; ++u) {
      if (t + u >= tb) break;
      const float xl = bf16_lo(xv[u]), xh = bf16_hi(xv[u]);
      const int64_t f0 = static_cast<int64_t>(t + u) * k;
      for (int j = 0; j < k; ++j) {
        const int e = ids[f0 + j] - e0;
        if (e >= 0 && e < ne) {
          const float d = dsel[f0 + j];
          float2 a = acc[e][tid];
          a.x = fmaf(d, xl, a.x);
          a.y = fmaf(d, xh, a.y);
          acc[e][tid] = a;
        }
      }
    }
  }
  for (int ee = 0; ee < ne; ++ee) {
    const int64_t o = (static_cast<int64_t>(blockIdx.y) * E + e0 + ee) * H + 2 * hp;
    *reinterpret_cast<float2*>(part + o) = acc[ee][tid];
  }
}

// The backward in one pass while k <= 8: a CTA takes a chunk of kDwTokChunk
// tokens, 512 hidden columns (two per thread) and a group of EG experts
// (blockIdx.z).  It first computes each token's chosen-logit gradients
// d_j = p_j (dp_j - sum_i p_i dp_i) (the sum in the warp route's butterfly
// order, as router_dx_kernel) into shared memory, both as the token's dense
// row over the group's experts (zeros elsewhere) and as its (expert, d) list.
// Then per token every thread adds d_e x[t] into its 2 EG register
// accumulators: adding the zeros of the unchosen experts is exact (the sums
// start at +0 and never become -0), so each expert's sum runs over the same
// tokens in the same order as router_dw_partial_kernel, bit for bit, without
// its dependent shared-memory updates.  Group 0 also adds sum_j d_j W_r[e_j]
// into the token's dx (in slot order, as router_dx_kernel).
constexpr int kFzCols = 512;
constexpr int kFzThreads = kFzCols / 2;
constexpr int kFzMaxK = 8;

template <int EG>
__global__ void __launch_bounds__(kFzThreads) router_bwd_fused_kernel(
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ w, const int32_t* __restrict__ ids,
    const float* __restrict__ probs, const float* __restrict__ dprobs, int T, int H, int E, int k,
    uint16_t* __restrict__ dx, float* __restrict__ part, int32_t* __restrict__ status) {
  extern __shared__ float fz_smem[];
  float (*s_dd)[EG] = reinterpret_cast<float (*)[EG]>(fz_smem);                          // [chunk][EG]
  float (*s_d)[kFzMaxK] = reinterpret_cast<float (*)[kFzMaxK]>(fz_smem + kDwTokChunk * EG);
  int (*s_e)[kFzMaxK] = reinterpret_cast<int (*)[kFzMaxK]>(fz_smem + kDwTokChunk * (EG + kFzMaxK));
  const int tid = threadIdx.x;
  const int e0 = blockIdx.z * EG;
  const int ta = blockIdx.y * kDwTokChunk;
  const int nt = min(kDwTokChunk, T - ta);
  const bool do_dx = blockIdx.z == 0;
  for (int tl = tid; tl < nt; tl += kFzThreads) {
    const int64_t t = ta + tl;
    float p[kFzMaxK], dp[kFzMaxK], a[32];
    int e[kFzMaxK];
#pragma unroll
    for (int j = 0; j < kFzMaxK; ++j) {
      p[j] = j < k ? probs[t * k + j] : 0.f;
      dp[j] = j < k ? dprobs[t * k + j] : 0.f;
      e[j] = j < k ? ids[t * k + j] : 0;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) a[i] = i < kFzMaxK ? p[i] * dp[i] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int i = 0; i < off; ++i) a[i] = a[i] + a[i + off];
    const float inner = a[0];
#pragma unroll
    for (int ee = 0; ee < EG; ++ee) s_dd[tl][ee] = 0.f;
#pragma unroll
    for (int j = 0; j < kFzMaxK; ++j) {
      if (j >= k) break;
      float d = p[j] * (dp[j] - inner);
      int ej = e[j];
      if (ej < 0 || ej >= E) {
        if (do_dx && blockIdx.x == 0) report(status, MXG_ERR_EXPERT_ID);
        d = 0.f;
        ej = -1;
      } else if (ej >= e0 && ej < e0 + EG) {
        s_dd[tl][ej - e0] = d;
      }
      s_d[tl][j] = d;
      s_e[tl][j] = ej;
    }
  }
  __syncthreads();
  const int hp = blockIdx.x * kFzThreads + tid;          // column pair
  if (hp >= H / 2) return;
  const uint32_t* x2 = reinterpret_cast<const uint32_t*>(x);
  const uint32_t* w2 = reinterpret_cast<const uint32_t*>(w);
  uint32_t* dx2 = reinterpret_cast<uint32_t*>(dx);
  float2 acc[EG];
#pragma unroll
  for (int ee = 0; ee < EG; ++ee) acc[ee] = make_float2(0.f, 0.f);
  // sixteen tokens' x and dx words requested together, then added up
  // (measured: 4 tokens 0.230 ms, 16 tokens 0.174 ms on the Mixtral tokens;
  // a two-buffer pipeline of 8 + 8 ran 0.232 ms)
  constexpr int U = 16;
  for (int tl = 0; tl < nt; tl += U) {
    uint32_t xv[U], dv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t t = ta + tl + u;
      xv[u] = tl + u < nt ? x2[t * (H / 2) + hp] : 0u;
      dv[u] = do_dx && tl + u < nt ? dx2[t * (H / 2) + hp] : 0u;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (tl + u >= nt) break;
      const float xl = bf16_lo(xv[u]), xh = bf16_hi(xv[u]);
#pragma unroll
      for (int ee = 0; ee < EG; ++ee) {
        const float d = s_dd[tl + u][ee];
        acc[ee].x = fmaf(d, xl, acc[ee].x);
        acc[ee].y = fmaf(d, xh, acc[ee].y);
      }
      if (do_dx) {
        float vl = bf16_lo(dv[u]), vh = bf16_hi(dv[u]);
        for (int j = 0; j < k; ++j) {
          const int ej = s_e[tl + u][j];
          const float dj = s_d[tl + u][j];
          const uint32_t wv = w2[static_cast<int64_t>(ej < 0 ? 0 : ej) * (H / 2) + hp];
          vl = fmaf(dj, bf16_lo(wv), vl);
          vh = fmaf(dj, bf16_hi(wv), vh);
        }
        dx2[static_cast<int64_t>(ta + tl + u) * (H / 2) + hp] = pack_bf16x2(vl, vh);
      }
    }
  }
#pragma unroll
  for (int ee = 0; ee < EG; ++ee)
    if (e0 + ee < E)
      *reinterpret_cast<float2*>(part + (static_cast<int64_t>(blockIdx.y) * E + e0 + ee) * H + 2 * hp) = acc[ee];
}

// dW_r[e][h] = sum over token chunks, in chunk order.
__global__ void __launch_bounds__(256) router_dw_reduce_kernel(const float* __restrict__ part, int nchunks, int E,
                                                              int H, float* __restrict__ dw) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<int64_t>(E) * H) return;
  float s = 0.f;
  for (int c = 0; c < nchunks; ++c) s += part[static_cast<int64_t>(c) * E * H + i];
  dw[i] = s;
}

inline int64_t align256(int64_t v) { return (v + 255) / 256 * 256; }
inline int dw_chunks(int T) { return (T + kDwTokChunk - 1) / kDwTokChunk; }

bool router_shape_ok(int T, int H, int E, int k, int hmult) {
  return T > 0 && H > 0 && H % hmult == 0 && k >= 1 && E >= k && E <= 256 && k <= 32;
}

}  // namespace

}  // namespace mxg

using namespace mxg;

extern "C" int mxg_router_fwd(const uint16_t* x, const uint16_t* w_router, int T, int H, int E, int k, float* logits,
                              int32_t* ids, float* probs, void* stream) {
  if (!x || !w_router || !logits || !ids || !probs) return MXG_ERR_ARG;
  if (T <= 0 || H <= 0 || E <= 0 || k <= 0) return MXG_ERR_ARG;
  if (!router_shape_ok(T, H, E, k, kHChunk)) return MXG_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w_router)) & 31u) return MXG_ERR_ALIGN;
  api::NvtxRange nvtx("mxg.router_fwd");
  return api::cuda_status(launch_router_mma(x, w_router, T, H, E, k, logits, ids, probs, nullptr, nullptr,
                                            static_cast<cudaStream_t>(stream)));
}

extern "C" int mxg_router_fwd_permute(const uint16_t* x, const uint16_t* w_router, int T, int H, int E, int k,
                                      float* logits, int32_t* ids, float* probs, int32_t* split_sizes,
                                      int32_t* src_of_row, int32_t* row_of_src, int32_t* padded_offsets, void* ws,
                                      size_t ws_bytes, int32_t* dev_status, void* stream) {
  if (!x || !w_router || !logits || !ids || !probs || !split_sizes || !src_of_row || !row_of_src ||
      !padded_offsets || !ws || !dev_status)
    return MXG_ERR_ARG;
  if (T <= 0 || H <= 0 || E <= 0 || k <= 0) return MXG_ERR_ARG;
  if (!router_shape_ok(T, H, E, k, kHChunk)) return MXG_ERR_SHAPE;
  const int64_t R = static_cast<int64_t>(T) * k;
  if (R > INT32_MAX) return MXG_ERR_SHAPE;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w_router) |
                        reinterpret_cast<uintptr_t>(ids) | reinterpret_cast<uintptr_t>(split_sizes) |
                        reinterpret_cast<uintptr_t>(src_of_row) | reinterpret_cast<uintptr_t>(row_of_src) |
                        reinterpret_cast<uintptr_t>(padded_offsets) | reinterpret_cast<uintptr_t>(ws);
  if (mis & 31u) return MXG_ERR_ALIGN;
  if (ws_bytes < mxg_route_permute_workspace_bytes(T, k, E)) return MXG_ERR_WORKSPACE;
  api::NvtxRange nvtx("mxg.router_fwd_permute");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t nblk = permute_num_blocks(static_cast<int>(R));
  const int64_t cb = api::align_up(4 * nblk * E, api::kAlign);
  PermuteParams p{};
  p.ids = ids;
  p.R = static_cast<int32_t>(R);
  p.E = E;
  p.counts = api::at<int32_t>(ws, 0);
  p.bases = api::at<int32_t>(ws, cb);
  p.offsets = api::at<int32_t>(ws, 2 * cb);
  p.padded_offsets = padded_offsets;
  p.pad = 128;
  p.split_sizes = split_sizes;
  p.src_of_row = src_of_row;
  p.row_of_src = row_of_src;
  p.status = dev_status;
  // the router kernel adds every routed entry into its chunk's histogram row
  if (cudaMemsetAsync(p.counts, 0, 4 * nblk * E, s) != cudaSuccess) return MXG_ERR_CUDA;
  if (launch_router_mma(x, w_router, T, H, E, k, logits, ids, probs, p.counts, dev_status, s) != cudaSuccess)
    return MXG_ERR_CUDA;
  return api::cuda_status(launch_permute_from_counts(p, s));
}

extern "C" size_t mxg_router_bwd_workspace_bytes(int T, int H, int E, int k) {
  if (T <= 0 || H <= 0 || E <= 0 || k <= 0) return 0;
  return static_cast<size_t>(align256(4ll * T * k) + 4ll * dw_chunks(T) * E * H);
}

extern "C" int mxg_router_bwd(const uint16_t* x, const uint16_t* w_router, const int32_t* ids, const float* probs,
                              const float* dprobs, int T, int H, int E, int k, uint16_t* dx, float* dw_router,
                              void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (!x || !w_router || !ids || !probs || !dprobs || !dx || !dw_router || !workspace || !dev_status)
    return MXG_ERR_ARG;
  if (T <= 0 || H <= 0 || E <= 0 || k <= 0) return MXG_ERR_ARG;
  if (!router_shape_ok(T, H, E, k, kDwCols)) return MXG_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w_router) | reinterpret_cast<uintptr_t>(dx) |
       reinterpret_cast<uintptr_t>(workspace)) & 31u)
    return MXG_ERR_ALIGN;
  if (workspace_bytes < mxg_router_bwd_workspace_bytes(T, H, E, k)) return MXG_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* dsel = static_cast<float*>(workspace);
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align256(4ll * T * k));
  if (k <= kFzMaxK) {
    // one pass: dx and the dW_r partials (graph replay on the Mixtral tokens,
    // T = 16384, H = 4096, E = 8, top-2: 0.174 ms against 0.254 ms for the
    // two-kernel pass below; 64 experts top-8: 0.177 against 0.333 ms)
    const int eg = E <= 8 ? 8 : 16;
    const dim3 grid((H / 2 + kFzThreads - 1) / kFzThreads, dw_chunks(T), (E + eg - 1) / eg);
    const int smem = kDwTokChunk * (eg + 2 * kFzMaxK) * 4;
    auto kern = eg == 8 ? router_bwd_fused_kernel<8> : router_bwd_fused_kernel<16>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return MXG_ERR_CUDA;
    kern<<<grid, kFzThreads, smem, s>>>(x, w_router, ids, probs, dprobs, T, H, E, k, dx, part, dev_status);
    count_launch();
  } else {
    const int dx_grid = static_cast<int>((static_cast<int64_t>(T) * 32 + 255) / 256);
    router_dx_kernel<<<dx_grid, 256, 0, s>>>(w_router, ids, probs, dprobs, T, H, E, k, dx, dsel, dev_status);
    count_launch();
    const dim3 pgrid(H / kDwCols, dw_chunks(T), (E + kDwExperts - 1) / kDwExperts);
    router_dw_partial_kernel<<<pgrid, kDwThreads, 0, s>>>(x, ids, dsel, T, H, E, k, part);
    count_launch();
  }
  const int rgrid = static_cast<int>((static_cast<int64_t>(E) * H + 255) / 256);
  router_dw_reduce_kernel<<<rgrid, 256, 0, s>>>(part, dw_chunks(T), E, H, dw_router);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? MXG_OK : MXG_ERR_CUDA;
}
