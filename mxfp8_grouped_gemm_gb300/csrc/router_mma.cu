// Router logits on the tensor cores, fused with the top-k route and
// (optionally) the permute's expert histogram.
//
// BioNeMo Uses Grouped Kernels and MXFP8, Fig. 1: a router picks two of
// eight experts per token.  Read as one bias-free linear layer H -> E on the
// token's hidden state, the logits are a [T, H] x [H, E] contraction.  A
// cluster of S CTAs (S = 1, 2 or 4) takes 128 tokens; CTA s contracts its
// share of H: TMA streams its x rows and the router rows 64 columns at a time
// into a shared-memory ring (each cluster starting at its own column, so the
// clusters do not all read the same router rows at once), one thread issues
// tcgen05.mma kind::f16 (bf16 operands, fp32 accumulators; M = 128 tokens,
// N = E rounded up to a multiple of 16, the extra router rows read as zeros),
// and the partial logits land in TMEM with one token per lane.  Four epilogue
// warps stage them in the then idle ring; after a cluster barrier each CTA
// sums the S partials of its 128 / S tokens in rank order through distributed
// shared memory and takes their route (warp_topk_softmax).  Splitting H over
// a cluster puts 2-4x more CTAs on the x stream than one per 128 tokens and
// shares the per-token route work among them.  The contraction is at most
// 1 GFLOP per layer, so the kernel is bound by streaming x from HBM.
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace mxg {
namespace {

constexpr int kRtM = 128;          // tokens per cluster: one TMEM lane each
constexpr int kRtK = 64;           // bf16 contraction elements per stage (one 128-byte swizzled row)
constexpr int kRtThreads = 192;    // warp 0 TMA, warp 1 TMEM + MMA, warps 2-5 epilogue
constexpr int kRtMaxSplit = 4;

template <int NP>
struct RtCfg {
  // up to 64 experts two CTAs share an SM
  static constexpr int kRing = NP <= 64 ? 98304 : 196608;
  static constexpr int kABytes = kRtM * kRtK * 2;
  static constexpr int kBBytes = NP * kRtK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = kRing / kStageBytes > 8 ? 8 : kRing / kStageBytes;
  static constexpr uint32_t kTmemCols = NP < 32 ? 32 : NP;
  static constexpr int kCtrl = 256;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kCtrl;
  static constexpr int kLogBytes = kRtM * NP * 4;      // the partial logits of 128 tokens
  static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned (128-byte swizzle atoms)");
  static_assert(kStages >= 2, "ring depth");
  // the partials, and the summed logits of a CTA's share of tokens (S >= 2)
  static_assert(kStages * kStageBytes >= kLogBytes + kLogBytes / 2, "the ring holds the logits");
  static_assert(kSmem <= 232448, "shared memory budget");
};

template <int NP>
__global__ void __launch_bounds__(kRtThreads, NP <= 64 ? 2 : 1)
    router_mma_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, int T, int H,
                      int E, int k, int S, float* __restrict__ logits, int32_t* __restrict__ ids,
                      float* __restrict__ probs, int32_t* __restrict__ counts, int32_t* status) {
  using C = RtCfg<NP>;
  extern __shared__ uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* never_set = abort_flag + 1;
  int* bad = reinterpret_cast<int*>(tmem_slot + 3);     // this CTA's partials are missing (read by the cluster)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = S > 1 ? cluster_ctarank() : 0u;
  const int tile = blockIdx.x / S;
  const int t0 = tile * kRtM;
  // this CTA's contraction steps [kb_lo, kb_lo + nloc)
  const int nk = H / kRtK;
  const int kb_lo = static_cast<int>(static_cast<int64_t>(rank) * nk / S);
  const int nloc = static_cast<int>(static_cast<int64_t>(rank + 1) * nk / S) - kb_lo;
  // Every cluster reads the same router rows: started at the same step, all
  // of them would ask for the same few L2 lines at once.  Each starts at its
  // own step of its range and wraps around.
  const int kb0 = static_cast<int>((static_cast<int64_t>(tile) * 5) % nloc);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    *abort_flag = 0;
    *never_set = 0;
    *bad = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  __syncthreads();
  if (warp == 1) {
    tmem_alloc<1>(tmem_slot, C::kTmemCols);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  float* slog = reinterpret_cast<float*>(sm);                         // [128 tokens][E] partials
  float* sfin = reinterpret_cast<float*>(sm + C::kLogBytes);          // [128 / S tokens][E] sums (S >= 2)

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int kb = 0; kb < nloc; ++kb) {
        const int st = kb % C::kStages;
        const uint32_t ph = (kb / C::kStages) & 1u;
        if (kb >= C::kStages && !mbar_wait_bounded(&empty[st], ph ^ 1u, abort_flag, kWaitLimitNs)) {
          report(status, MXG_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        uint8_t* sA = sm + st * C::kStageBytes;
        const int kc = (kb_lo + (kb0 + kb) % nloc) * kRtK;
        mbar_arrive_expect_tx(&full[st], C::kStageBytes);
        tma_load_2d(sA, &tmX, kc, t0, &full[st]);
        tma_load_2d(sA + C::kABytes, &tmW, kc, 0, &full[st]);
      }
      if (*abort_flag) {  // let copies already in flight land before the ring is reused
        const uint64_t g0 = globaltimer_ns();
        while (globaltimer_ns() - g0 < 1000000ull) __nanosleep(1000);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      for (int kb = 0; kb < nloc; ++kb) {
        const int st = kb % C::kStages;
        const uint32_t ph = (kb / C::kStages) & 1u;
        if (!mbar_wait_bounded(&full[st], ph, abort_flag, kWaitLimitNs)) {
          report(status, MXG_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        uint8_t* sA = sm + st * C::kStageBytes;
        const uint64_t adesc = smem_desc(smem_u32(sA), 0, 1024, kLayoutSwizzle128B);
        const uint64_t bdesc = smem_desc(smem_u32(sA + C::kABytes), 0, 1024, kLayoutSwizzle128B);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)      // K = 16 per MMA, 32 bytes of each 128-byte row
          mma_bf16<1>(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc_bf16(kRtM, NP), (kb | kk) != 0 ? 1u : 0u);
        mma_commit<1>(&empty[st]);
      }
      // arrives once every MMA issued above has completed (also after an abort)
      mma_commit<1>(tfull);
    }
  } else {
    // ------------------------------------------- epilogue: stage the partials
    // warps 2..5 read TMEM lane quadrant warp % 4: token row = 32 (warp % 4) + lane
    const int q = warp & 3;
    const int row = q * 32 + lane;
    bool got = mbar_wait_bounded(tfull, 0, never_set, kWaitLimitNs);
    got = __all_sync(0xffffffffu, got) && *abort_flag == 0;
    tc_fence_after();
    // The ring is idle once every MMA has completed (all its loads were consumed).
    if (got) {
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < NP; c += 16) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(taddr + c, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (c + i < E) slog[row * E + c + i] = __uint_as_float(r[i]);
      }
    } else if (lane == 0) {
      *bad = 1;
      report(status, MXG_ERR_TIMEOUT);
    }
  }

  // every CTA of the cluster has staged its partials
  tc_fence_before();
  if (S > 1) cluster_sync();
  else __syncthreads();

  const int tpc = kRtM / S;                 // tokens this CTA routes: [rank * tpc, (rank + 1) * tpc)
  const int tk0 = static_cast<int>(rank) * tpc;
  bool any_bad = false;
  if (warp >= 2) {
    const int i = threadIdx.x - 64;         // 0..127
    if (S > 1) {
      // partial sums in rank order (the same order whichever CTA adds them)
      for (int s = 0; s < S; ++s) any_bad |= ld_shared_cluster_s32(map_to_rank(smem_u32(bad), s)) != 0;
      for (int idx = i; idx < tpc * E; idx += kRtM) {
        const int tk = tk0 + idx / E, e = idx - (idx / E) * E;
        const uint32_t a = smem_u32(slog + tk * E + e);
        float v = 0.f;
        for (int s = 0; s < S; ++s) v += ld_shared_cluster_f32(map_to_rank(a, s));
        sfin[idx] = v;
        if (t0 + tk < T) logits[static_cast<int64_t>(t0 + tk) * E + e] = v;
      }
    } else {
      any_bad = *bad != 0;
      for (int idx = i; idx < kRtM * E; idx += kRtM) {
        const int tk = idx / E;
        if (t0 + tk < T) logits[static_cast<int64_t>(t0 + tk) * E + (idx - tk * E)] = slog[idx];
      }
    }
  }
  // no CTA reads another's shared memory after this point
  if (S > 1) cluster_sync();
  else __syncthreads();

  if (warp >= 2) {
    const float* fin = S > 1 ? sfin : slog;
    if (E * k <= 64) {
      // one token per thread: E k compares instead of k rounds of warp shuffles
      // (measured: Mixtral's 8 experts top-2 0.0395 -> 0.0278 ms; at 64 experts
      // top-8 the serial passes lose to the warp: 0.0387 -> 0.0436 ms)
      for (int tl = threadIdx.x - 64; tl < tpc; tl += kRtM) {
        const int64_t tt = static_cast<int64_t>(t0) + tk0 + tl;
        if (tt >= T) break;
        if (any_bad) {                             // no logits: mark the token unrouted
          for (int j = 0; j < k; ++j) {
            ids[tt * k + j] = -1;
            probs[tt * k + j] = 0.f;
          }
          continue;
        }
        int sel[8];
        thread_topk_softmax(fin + tl * E, E, k, ids + tt * k, probs + tt * k, sel);
        if (counts != nullptr)
          for (int j = 0; j < k; ++j) atomicAdd(counts + ((tt * k + j) / kPermuteChunk) * E + sel[j], 1);
      }
    } else {
      for (int tl = warp - 2; tl < tpc; tl += 4) {
        const int64_t tt = static_cast<int64_t>(t0) + tk0 + tl;
        if (tt >= T) break;
        if (any_bad) {                             // no logits: mark the tokens unrouted
          if (lane < k) {
            ids[tt * k + lane] = -1;
            probs[tt * k + lane] = 0.f;
          }
          continue;
        }
        const int e = warp_topk_softmax(fin + tl * E, E, k, lane, ids + tt * k, probs + tt * k);
        if (counts != nullptr && lane < k) atomicAdd(counts + ((tt * k + lane) / kPermuteChunk) * E + e, 1);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<1>(tmem, C::kTmemCols);
}

template <int NP>
cudaError_t launch_np(const CUtensorMap& mx, const CUtensorMap& mw, int T, int H, int E, int k, float* logits,
                      int32_t* ids, float* probs, int32_t* counts, int32_t* status, cudaStream_t s) {
  using C = RtCfg<NP>;
  auto kern = router_mma_kernel<NP>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (err != cudaSuccess) return err;
  // split H over a cluster until the x stream has about one CTA per SM slot
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int tiles = (T + kRtM - 1) / kRtM;
  const int nk = H / kRtK;
  int S = 1;
  while (S < kRtMaxSplit && 2 * S <= nk && static_cast<int64_t>(tiles) * S < static_cast<int64_t>(sms)) S *= 2;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * S));
  cfg.blockDim = dim3(kRtThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(S);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, kern, mx, mw, T, H, E, k, S, logits, ids, probs, counts, status);
  count_launch();
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_mma(const uint16_t* x, const uint16_t* w, int T, int H, int E, int k, float* logits,
                              int32_t* ids, float* probs, int32_t* counts, int32_t* status, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int NP = E <= 16 ? 16 : E <= 32 ? 32 : E <= 64 ? 64 : E <= 128 ? 128 : 256;
  CUtensorMap mx, mw;
  if (!tma_map_bf16(&mx, x, H, T, kRtM) || !tma_map_bf16(&mw, w, H, E, static_cast<uint32_t>(NP)))
    return cudaErrorInvalidValue;
  switch (NP) {
    case 16: return launch_np<16>(mx, mw, T, H, E, k, logits, ids, probs, counts, status, s);
    case 32: return launch_np<32>(mx, mw, T, H, E, k, logits, ids, probs, counts, status, s);
    case 64: return launch_np<64>(mx, mw, T, H, E, k, logits, ids, probs, counts, status, s);
    case 128: return launch_np<128>(mx, mw, T, H, E, k, logits, ids, probs, counts, status, s);
    default: return launch_np<256>(mx, mw, T, H, E, k, logits, ids, probs, counts, status, s);
  }
}

}  // namespace mxg
