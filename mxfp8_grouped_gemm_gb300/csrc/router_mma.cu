// Router logits on the tensor cores, fused with the top-k route and
// (optionally) the permute's expert histogram.
//
// BioNeMo Uses Grouped Kernels and MXFP8, Fig. 1: a router picks two of
// eight experts per token.  Read as one bias-free linear layer H -> E on the
// token's hidden state, the logits are a [T, H] x [H, E] contraction: one CTA
// takes 128 tokens, TMA streams its x rows and the router rows 64 columns at
// a time into a shared-memory ring (each CTA starting at its own column so
// the CTAs do not all read the same router rows at once), one thread issues
// tcgen05.mma kind::f16
// (bf16 operands, fp32 accumulators; M = 128 tokens, N = E rounded up to a
// multiple of 16, the extra router rows read as zeros), and the accumulators
// land in TMEM with one token per lane.  Four epilogue warps read them back
// (one token per thread), stage the logits in the then idle ring, and take
// the route of each token (warp_topk_softmax).  The contraction is at most
// 1 GFLOP per layer, so the kernel is bound by streaming x from HBM.
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace mxg {
namespace {

constexpr int kRtM = 128;          // tokens per CTA: one TMEM lane each
constexpr int kRtK = 64;           // bf16 contraction elements per stage (one 128-byte swizzled row)
constexpr int kRtThreads = 192;    // warp 0 TMA, warp 1 TMEM + MMA, warps 2-5 epilogue
constexpr int kRtRing = 196608;    // ring bytes at most

template <int NP>
struct RtCfg {
  static constexpr int kABytes = kRtM * kRtK * 2;
  static constexpr int kBBytes = NP * kRtK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = kRtRing / kStageBytes > 8 ? 8 : kRtRing / kStageBytes;
  static constexpr uint32_t kTmemCols = NP < 32 ? 32 : NP;
  static constexpr int kCtrl = 256;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kCtrl;
  static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned (128-byte swizzle atoms)");
  static_assert(kStages * kStageBytes >= kRtM * NP * 4, "the ring holds the logits of 128 tokens");
  static_assert(kSmem <= 232448, "shared memory budget");
};

template <int NP>
__global__ void __launch_bounds__(kRtThreads, 1)
    router_mma_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW, int T, int H,
                      int E, int k, float* __restrict__ logits, int32_t* __restrict__ ids, float* __restrict__ probs,
                      int32_t* __restrict__ counts, int32_t* status) {
  using C = RtCfg<NP>;
  extern __shared__ uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfull + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* never_set = abort_flag + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRtM;
  const int nk = H / kRtK;
  // Every CTA reads the same router rows: started at the same contraction
  // step, all of them would ask for the same few L2 lines at once.  Each CTA
  // starts at its own step and wraps around.
  const int kb0 = static_cast<int>((static_cast<int64_t>(blockIdx.x) * 5) % nk);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    *abort_flag = 0;
    *never_set = 0;
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int kb = 0; kb < nk; ++kb) {
        const int st = kb % C::kStages;
        const uint32_t ph = (kb / C::kStages) & 1u;
        if (kb >= C::kStages && !mbar_wait_bounded(&empty[st], ph ^ 1u, abort_flag, kWaitLimitNs)) {
          report(status, MXG_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        uint8_t* sA = sm + st * C::kStageBytes;
        const int kc = (kb0 + kb) % nk * kRtK;
        mbar_arrive_expect_tx(&full[st], C::kStageBytes);
        tma_load_2d(sA, &tmX, kc, t0, &full[st]);
        tma_load_2d(sA + C::kABytes, &tmW, kc, 0, &full[st]);
      }
      if (*abort_flag) {  // let copies already in flight land before the CTA exits
        const uint64_t g0 = globaltimer_ns();
        while (globaltimer_ns() - g0 < 1000000ull) __nanosleep(1000);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      for (int kb = 0; kb < nk; ++kb) {
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
    // ------------------------------------------------------------ epilogue
    // warps 2..5 read TMEM lane quadrant warp % 4: token row = 32 (warp % 4) + lane
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int64_t t = static_cast<int64_t>(t0) + row;
    bool got = mbar_wait_bounded(tfull, 0, never_set, kWaitLimitNs);
    got = __all_sync(0xffffffffu, got) && *abort_flag == 0;
    tc_fence_after();
    // The ring is idle once every MMA has completed (all its loads were
    // consumed): it holds the CTA's logits, [128 tokens][E] fp32.
    float* slog = reinterpret_cast<float*>(sm);
    if (got) {
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
      for (int c = 0; c < NP; c += 16) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(taddr + c, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int e = c + i;
          if (e < E) {
            const float v = __uint_as_float(r[i]);
            slog[row * E + e] = v;
            if (t < T) logits[t * E + e] = v;
          }
        }
      }
    } else {
      report(status, MXG_ERR_TIMEOUT);
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");     // the four epilogue warps' logits are staged
    for (int tk = warp - 2; tk < kRtM; tk += 4) {
      const int64_t tt = static_cast<int64_t>(t0) + tk;
      if (tt >= T) break;
      if (!got) {                                      // no logits: mark the tokens unrouted
        if (lane < k) {
          ids[tt * k + lane] = -1;
          probs[tt * k + lane] = 0.f;
        }
        continue;
      }
      warp_topk_softmax(slog + tk * E, E, k, lane, ids + tt * k, probs + tt * k);
      if (counts != nullptr && lane < k) {           // lane j wrote ids[tt*k + j] itself
        const int e = ids[tt * k + lane];
        const int64_t f = tt * k + lane;
        atomicAdd(counts + (f / kPermuteChunk) * E + e, 1);
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
  cudaError_t err = cudaFuncSetAttribute(router_mma_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (err != cudaSuccess) return err;
  const int grid = (T + kRtM - 1) / kRtM;
  router_mma_kernel<NP><<<grid, kRtThreads, C::kSmem, s>>>(mx, mw, T, H, E, k, logits, ids, probs, counts, status);
  count_launch();
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
