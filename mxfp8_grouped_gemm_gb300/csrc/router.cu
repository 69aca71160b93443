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
#include "common.cuh"
#include "kernels.h"

namespace mxg {

namespace {

// ------------------------------------------------------------------ forward
constexpr int kHChunk = 128;               // hidden columns staged per step
constexpr int kRowWords = kHChunk / 2 + 1; // bf16x2 words per staged row (odd: no bank conflicts)
constexpr int kFwdThreads = 256;
constexpr int kTokBlock = 4;               // tokens per thread block of logits
constexpr int kExpBlock = 2;               // experts per thread block of logits
constexpr int kMaxBlocks = 4;              // blocks per thread

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Tokens per CTA: as many as keep every thread at <= 4 blocks of 4 tokens x 2
// experts, and few enough that the grid covers the GPU twice over.
int router_tokens_per_cta(int T, int E) {
  const int eg = (E + kExpBlock - 1) / kExpBlock;
  int tt = kFwdThreads * kMaxBlocks * kTokBlock / eg;
  tt = tt > 256 ? 256 : tt;
  const int spread = T / (2 * 152) / 32 * 32;
  if (tt > spread) tt = spread;
  tt = tt / 32 * 32;
  return tt < 32 ? 32 : tt;
}

size_t router_fwd_smem(int TT, int E) {
  return static_cast<size_t>(TT + E) * kRowWords * 4 + static_cast<size_t>(TT) * E * 4;
}

// One CTA: TT tokens.  The x rows and all E router rows are staged 128
// columns at a time; each thread accumulates blocks of 4 tokens x 2 experts
// (8 logits, fp32, each a sequential sum over the columns), so one staged x
// word feeds two experts and one router word four tokens.
__global__ void __launch_bounds__(kFwdThreads) router_fwd_kernel(const uint16_t* __restrict__ x,
                                                                const uint16_t* __restrict__ w, int T, int H, int E,
                                                                int k, int TT, float* __restrict__ logits,
                                                                int32_t* __restrict__ ids, float* __restrict__ probs) {
  extern __shared__ uint32_t sm[];
  uint32_t* sx = sm;
  uint32_t* sw = sx + TT * kRowWords;
  float* sl = reinterpret_cast<float*>(sw + E * kRowWords);
  const int t0 = blockIdx.x * TT;
  const int tid = threadIdx.x;
  const int eg = (E + kExpBlock - 1) / kExpBlock;
  const int nblocks = (TT / kTokBlock) * eg;
  float acc[kMaxBlocks][kTokBlock][kExpBlock];
#pragma unroll
  for (int b = 0; b < kMaxBlocks; ++b)
#pragma unroll
    for (int i = 0; i < kTokBlock; ++i)
#pragma unroll
      for (int j = 0; j < kExpBlock; ++j) acc[b][i][j] = 0.f;

  for (int h0 = 0; h0 < H; h0 += kHChunk) {
    for (int i = tid; i < TT * (kHChunk / 8); i += kFwdThreads) {
      const int r = i / (kHChunk / 8), c = i % (kHChunk / 8);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (t0 + r < T) v = *reinterpret_cast<const uint4*>(x + static_cast<int64_t>(t0 + r) * H + h0 + c * 8);
      uint32_t* d = sx + r * kRowWords + c * 4;
      d[0] = v.x;
      d[1] = v.y;
      d[2] = v.z;
      d[3] = v.w;
    }
    for (int i = tid; i < E * (kHChunk / 8); i += kFwdThreads) {
      const int r = i / (kHChunk / 8), c = i % (kHChunk / 8);
      const uint4 v = *reinterpret_cast<const uint4*>(w + static_cast<int64_t>(r) * H + h0 + c * 8);
      uint32_t* d = sw + r * kRowWords + c * 4;
      d[0] = v.x;
      d[1] = v.y;
      d[2] = v.z;
      d[3] = v.w;
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < kMaxBlocks; ++b) {
      const int pb = tid + b * kFwdThreads;
      if (pb < nblocks) {
        const int tg = pb / eg, e0 = (pb - tg * eg) * kExpBlock;
        const uint32_t* xr = sx + tg * kTokBlock * kRowWords;
        const uint32_t* wr0 = sw + e0 * kRowWords;
        const uint32_t* wr1 = sw + (e0 + 1 < E ? e0 + 1 : e0) * kRowWords;   // odd E: duplicate, discarded
#pragma unroll 4
        for (int q = 0; q < kHChunk / 2; ++q) {
          const uint32_t w0 = wr0[q], w1 = wr1[q];
          const float w0l = bf16_lo(w0), w0h = bf16_hi(w0), w1l = bf16_lo(w1), w1h = bf16_hi(w1);
#pragma unroll
          for (int i = 0; i < kTokBlock; ++i) {
            const uint32_t xv = xr[i * kRowWords + q];
            const float xl = bf16_lo(xv), xh = bf16_hi(xv);
            acc[b][i][0] = fmaf(xh, w0h, fmaf(xl, w0l, acc[b][i][0]));
            acc[b][i][1] = fmaf(xh, w1h, fmaf(xl, w1l, acc[b][i][1]));
          }
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int b = 0; b < kMaxBlocks; ++b) {
    const int pb = tid + b * kFwdThreads;
    if (pb < nblocks) {
      const int tg = pb / eg, e0 = (pb - tg * eg) * kExpBlock;
#pragma unroll
      for (int i = 0; i < kTokBlock; ++i) {
        const int tk = tg * kTokBlock + i;
#pragma unroll
        for (int j = 0; j < kExpBlock; ++j) {
          if (e0 + j >= E) continue;
          sl[tk * E + e0 + j] = acc[b][i][j];
          if (t0 + tk < T) logits[static_cast<int64_t>(t0 + tk) * E + e0 + j] = acc[b][i][j];
        }
      }
    }
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  for (int tk = warp; tk < TT; tk += kFwdThreads / 32) {
    const int64_t t = t0 + tk;
    if (t >= T) break;
    warp_topk_softmax(sl + tk * E, E, k, lane, ids + t * k, probs + t * k);
  }
}

// Few experts (E <= 8, the router matrix in <= 96 KB of shared memory): one
// warp takes four tokens at a time and streams their rows straight from HBM,
// 16 bytes per lane per load, against the staged router rows (each staged
// router word feeds four tokens); lane partial sums are reduced across the
// warp and the route is taken on the warp's logits.
constexpr int kStreamMaxE = 8;
constexpr int kStreamTok = 4;
constexpr size_t kStreamMaxW = 96 * 1024;

__global__ void __launch_bounds__(kFwdThreads) router_fwd_stream_kernel(const uint16_t* __restrict__ x,
                                                                       const uint16_t* __restrict__ w, int T, int H,
                                                                       int E, int k, float* __restrict__ logits,
                                                                       int32_t* __restrict__ ids,
                                                                       float* __restrict__ probs) {
  extern __shared__ uint4 sw4[];                      // [E][H/8]
  __shared__ float srow[kFwdThreads / 32][kStreamTok][kStreamMaxE];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hc = H / 8;
  for (int i = tid; i < E * hc; i += kFwdThreads)
    sw4[i] = reinterpret_cast<const uint4*>(w)[i];
  __syncthreads();
  const int64_t groups = (T + kStreamTok - 1) / kStreamTok;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * (kFwdThreads / 32) + warp; g < groups;
       g += static_cast<int64_t>(gridDim.x) * (kFwdThreads / 32)) {
    const int64_t t0 = g * kStreamTok;
    float acc[kStreamTok][kStreamMaxE];
#pragma unroll
    for (int u = 0; u < kStreamTok; ++u)
#pragma unroll
      for (int e = 0; e < kStreamMaxE; ++e) acc[u][e] = 0.f;
#pragma unroll 2
    for (int c = lane; c < hc; c += 32) {
      float xv[kStreamTok][8];
#pragma unroll
      for (int u = 0; u < kStreamTok; ++u) {
        uint4 xq = make_uint4(0u, 0u, 0u, 0u);
        if (t0 + u < T) xq = reinterpret_cast<const uint4*>(x + (t0 + u) * H)[c];
        const uint32_t xw[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          xv[u][2 * i] = bf16_lo(xw[i]);
          xv[u][2 * i + 1] = bf16_hi(xw[i]);
        }
      }
#pragma unroll
      for (int e = 0; e < kStreamMaxE; ++e) {
        if (e < E) {
          const uint4 wq = sw4[e * hc + c];
          const uint32_t ww[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float wl = bf16_lo(ww[i]), wh = bf16_hi(ww[i]);
#pragma unroll
            for (int u = 0; u < kStreamTok; ++u) acc[u][e] = fmaf(xv[u][2 * i + 1], wh, fmaf(xv[u][2 * i], wl, acc[u][e]));
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kStreamTok; ++u)
#pragma unroll
      for (int e = 0; e < kStreamMaxE; ++e) {
        if (e < E) {
          float v = acc[u][e];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
          if (lane == 0) srow[warp][u][e] = v;
        }
      }
    __syncwarp();
    for (int u = 0; u < kStreamTok; ++u) {
      const int64_t t = t0 + u;
      if (t >= T) break;
      if (lane < E) logits[t * E + lane] = srow[warp][u][lane];
      warp_topk_softmax(srow[warp][u], E, k, lane, ids + t * k, probs + t * k);
    }
    __syncwarp();
  }
}

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
constexpr int kDwTokChunk = 512;  // tokens per partial sum
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
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t wbytes = static_cast<size_t>(E) * H * 2;
  if (E <= kStreamMaxE && wbytes <= kStreamMaxW) {
    if (cudaFuncSetAttribute(router_fwd_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(wbytes)) != cudaSuccess)
      return MXG_ERR_CUDA;
    const int64_t groups = (T + kStreamTok - 1) / kStreamTok;
    int grid = static_cast<int>((groups + kFwdThreads / 32 - 1) / (kFwdThreads / 32));
    if (grid > 2 * 152) grid = 2 * 152;
    router_fwd_stream_kernel<<<grid, kFwdThreads, wbytes, s>>>(x, w_router, T, H, E, k, logits, ids, probs);
  } else {
    const int tt = router_tokens_per_cta(T, E);
    const size_t smem = router_fwd_smem(tt, E);
    if (cudaFuncSetAttribute(router_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MXG_ERR_CUDA;
    const int grid = (T + tt - 1) / tt;
    router_fwd_kernel<<<grid, kFwdThreads, smem, s>>>(x, w_router, T, H, E, k, tt, logits, ids, probs);
  }
  count_launch();
  return cudaGetLastError() == cudaSuccess ? MXG_OK : MXG_ERR_CUDA;
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
  const int dx_grid = static_cast<int>((static_cast<int64_t>(T) * 32 + 255) / 256);
  router_dx_kernel<<<dx_grid, 256, 0, s>>>(w_router, ids, probs, dprobs, T, H, E, k, dx, dsel, dev_status);
  count_launch();
  const dim3 pgrid(H / kDwCols, dw_chunks(T), (E + kDwExperts - 1) / kDwExperts);
  router_dw_partial_kernel<<<pgrid, kDwThreads, 0, s>>>(x, ids, dsel, T, H, E, k, part);
  count_launch();
  const int rgrid = static_cast<int>((static_cast<int64_t>(E) * H + 255) / 256);
  router_dw_reduce_kernel<<<rgrid, 256, 0, s>>>(part, dw_chunks(T), E, H, dw_router);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? MXG_OK : MXG_ERR_CUDA;
}
