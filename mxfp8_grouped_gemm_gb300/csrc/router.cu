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
constexpr int kTokPerCta = 32;             // tokens per CTA
constexpr int kHChunk = 128;               // hidden columns staged per step
constexpr int kRowWords = kHChunk / 2 + 1; // bf16x2 words per staged row (odd: no bank conflicts)
constexpr int kFwdThreads = 256;
constexpr int kMaxPairs = kTokPerCta * 256 / kFwdThreads;   // (token, expert) pairs per thread, E <= 256

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

size_t router_fwd_smem(int E) {
  return static_cast<size_t>(kTokPerCta + E) * kRowWords * 4 + static_cast<size_t>(kTokPerCta) * E * 4;
}

// One CTA: 32 tokens.  The x rows and all E router rows are staged 128 columns
// at a time; thread i accumulates the logits of pairs i, i+256, ... (pair =
// token * E + expert) in fp32, each as a sequential sum over the columns.
__global__ void __launch_bounds__(kFwdThreads) router_fwd_kernel(const uint16_t* __restrict__ x,
                                                                const uint16_t* __restrict__ w, int T, int H, int E,
                                                                int k, float* __restrict__ logits,
                                                                int32_t* __restrict__ ids, float* __restrict__ probs) {
  extern __shared__ uint32_t sm[];
  uint32_t* sx = sm;
  uint32_t* sw = sx + kTokPerCta * kRowWords;
  float* sl = reinterpret_cast<float*>(sw + E * kRowWords);
  const int t0 = blockIdx.x * kTokPerCta;
  const int tid = threadIdx.x;
  const int npairs = kTokPerCta * E;
  float acc[kMaxPairs];
#pragma unroll
  for (int i = 0; i < kMaxPairs; ++i) acc[i] = 0.f;

  for (int h0 = 0; h0 < H; h0 += kHChunk) {
    for (int i = tid; i < kTokPerCta * (kHChunk / 8); i += kFwdThreads) {
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
    for (int i = 0; i < kMaxPairs; ++i) {
      const int pr = tid + i * kFwdThreads;
      if (pr < npairs) {
        const int tk = pr / E, e = pr - tk * E;
        const uint32_t* xr = sx + tk * kRowWords;
        const uint32_t* wr = sw + e * kRowWords;
        float a = acc[i];
#pragma unroll 8
        for (int q = 0; q < kHChunk / 2; ++q) {
          const uint32_t xv = xr[q], wv = wr[q];
          a = fmaf(bf16_lo(xv), bf16_lo(wv), a);
          a = fmaf(bf16_hi(xv), bf16_hi(wv), a);
        }
        acc[i] = a;
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < kMaxPairs; ++i) {
    const int pr = tid + i * kFwdThreads;
    if (pr < npairs) {
      const int tk = pr / E, e = pr - tk * E;
      sl[tk * E + e] = acc[i];
      if (t0 + tk < T) logits[static_cast<int64_t>(t0 + tk) * E + e] = acc[i];
    }
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  for (int tk = warp; tk < kTokPerCta; tk += kFwdThreads / 32) {
    const int64_t t = t0 + tk;
    if (t >= T) break;
    warp_topk_softmax(sl + tk * E, E, k, lane, ids + t * k, probs + t * k);
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

constexpr int kDwCols = 128;      // hidden columns per CTA (one per thread)
constexpr int kDwExperts = 32;    // experts per CTA (grid z covers the rest)
constexpr int kDwTokChunk = 512;  // tokens per partial sum

// Partial dW_r over one token chunk for 128 columns and up to 32 experts, in
// shared memory (each thread owns its column, so no two threads touch the
// same word).
__global__ void __launch_bounds__(kDwCols) router_dw_partial_kernel(const uint16_t* __restrict__ x,
                                                                   const int32_t* __restrict__ ids,
                                                                   const float* __restrict__ dsel, int T, int H,
                                                                   int E, int k, float* __restrict__ part) {
  __shared__ float acc[kDwExperts][kDwCols];
  const int tid = threadIdx.x;
  const int h = blockIdx.x * kDwCols + tid;
  const int e0 = blockIdx.z * kDwExperts;
  const int ne = min(kDwExperts, E - e0);
  for (int ee = 0; ee < ne; ++ee) acc[ee][tid] = 0.f;
  const int ta = blockIdx.y * kDwTokChunk;
  const int tb = min(T, ta + kDwTokChunk);
  for (int t = ta; t < tb; ++t) {
    const float xv = bf16_bits_to_float(x[static_cast<int64_t>(t) * H + h]);
    for (int j = 0; j < k; ++j) {
      const int e = ids[static_cast<int64_t>(t) * k + j] - e0;
      if (e >= 0 && e < ne) acc[e][tid] = fmaf(dsel[static_cast<int64_t>(t) * k + j], xv, acc[e][tid]);
    }
  }
  for (int ee = 0; ee < ne; ++ee)
    part[(static_cast<int64_t>(blockIdx.y) * E + e0 + ee) * H + h] = acc[ee][tid];
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
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w_router)) & 15u) return MXG_ERR_ALIGN;
  const size_t smem = router_fwd_smem(E);
  if (cudaFuncSetAttribute(router_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MXG_ERR_CUDA;
  const int grid = (T + kTokPerCta - 1) / kTokPerCta;
  router_fwd_kernel<<<grid, kFwdThreads, smem, static_cast<cudaStream_t>(stream)>>>(x, w_router, T, H, E, k, logits,
                                                                                  ids, probs);
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
       reinterpret_cast<uintptr_t>(workspace)) & 15u)
    return MXG_ERR_ALIGN;
  if (workspace_bytes < mxg_router_bwd_workspace_bytes(T, H, E, k)) return MXG_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* dsel = static_cast<float*>(workspace);
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + align256(4ll * T * k));
  const int dx_grid = static_cast<int>((static_cast<int64_t>(T) * 32 + 255) / 256);
  router_dx_kernel<<<dx_grid, 256, 0, s>>>(w_router, ids, probs, dprobs, T, H, E, k, dx, dsel, dev_status);
  count_launch();
  const dim3 pgrid(H / kDwCols, dw_chunks(T), (E + kDwExperts - 1) / kDwExperts);
  router_dw_partial_kernel<<<pgrid, kDwCols, 0, s>>>(x, ids, dsel, T, H, E, k, part);
  count_launch();
  const int rgrid = static_cast<int>((static_cast<int64_t>(E) * H + 255) / 256);
  router_dw_reduce_kernel<<<rgrid, 256, 0, s>>>(part, dw_chunks(T), E, H, dw_router);
  count_launch();
  return cudaGetLastError() == cudaSuccess ? MXG_OK : MXG_ERR_CUDA;
}
