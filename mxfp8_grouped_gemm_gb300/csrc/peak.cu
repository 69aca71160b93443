// MXFP8 tensor-core ceiling on this GPU: a loop of block-scaled E4M3 MMAs
// (tcgen05.mma.kind::mxf8f6f4.block_scale, 128 x 256 x 32 per instruction)
// on operands that stay resident in shared memory, with the per-stage scale
// factors copied into TMEM by a second thread exactly as the grouped GEMM's
// copier warp does.  No global-memory traffic: the launch measures what the
// tensor pipe retires per clock, the denominator the GEMMs are compared with.
//
// The page ("BioNeMo Uses Grouped Kernels and MXFP8", "Reducing memory
// pressure with MXFP8") motivates MXFP8 by the throughput of 8-bit tensor-core
// math; the vendor's dense MXFP8 figure is a datasheet number, so it is
// measured here instead.
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace mxg {
namespace {

constexpr int kPeakStages = 3;
constexpr int kPeakA = 128 * 128;                // A codes: 128 rows x 128 K bytes
constexpr int kPeakB = 256 * 128;                // B codes: 256 rows x 128 K bytes
constexpr int kPeakSf = 3 * 512;                 // scale atoms: A (128 rows), B (256 rows)
constexpr int kPeakStageBytes = kPeakA + kPeakB + 2048;   // stages stay 1024-byte aligned
static_assert(kPeakSf <= 2048 && kPeakStageBytes % 1024 == 0, "stage layout");
constexpr int kPeakSmem = kPeakStages * kPeakStageBytes + 1024 + 256;
constexpr int kPeakMmasPerStep = 4;              // K = 128 per step, 32 per MMA
constexpr double kPeakFlopPerMma = 2.0 * 128 * 256 * 32;

__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int steps, int32_t* status) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint64_t* copied = reinterpret_cast<uint64_t*>(sm + kPeakStages * kPeakStageBytes);
  uint64_t* consumed = copied + kPeakStages;
  uint64_t* mma_done = consumed + kPeakStages;
  uint64_t* copy_done = mma_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(copy_done + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* never_set = abort + 1;   // the final drains wait whatever happened before

  // operands: small finite E4M3 codes, scale bytes 127 (2^0)
  for (int i = threadIdx.x; i < kPeakStages * kPeakStageBytes; i += blockDim.x) {
    const int o = i % kPeakStageBytes;
    sm[i] = o < kPeakA + kPeakB ? static_cast<uint8_t>((i * 7 + 3) & 0x3f) : uint8_t{127};
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPeakStages; ++s) {
      mbar_init(&copied[s], 1);
      mbar_init(&consumed[s], 1);
    }
    mbar_init(mma_done, 1);
    mbar_init(copy_done, 1);
    *abort = 0;
    *never_set = 0;
    fence_barrier_init();
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  if (threadIdx.x < 32) {
    tmem_alloc<1>(tmem_slot, 512);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 32) {
    // scale-factor copier: stage s's A atom and B's two atoms into its TMEM slot
    for (int s = 0; s < steps; ++s) {
      const int st = s % kPeakStages;
      if (s >= kPeakStages &&
          !mbar_wait_bounded(&consumed[st], ((s / kPeakStages) - 1) & 1, abort, kWaitLimitNs)) {
        report(status, MXG_ERR_TIMEOUT);
        *abort = 1;
        break;
      }
      const uint8_t* sf = sm + st * kPeakStageBytes + kPeakA + kPeakB;
      const uint32_t slot = tmem + 256 + st * 12;
#pragma unroll
      for (int a = 0; a < 3; ++a)
        tmem_cp_32x128b_warpx4<1>(slot + 4 * a, smem_desc(smem_u32(sf + 512 * a), 0, 128, kLayoutNone));
      mma_commit<1>(&copied[st]);
    }
    mma_commit<1>(copy_done);   // own copies finished before TMEM is released
    if (!mbar_wait_bounded(copy_done, 0, never_set, kWaitLimitNs)) report(status, MXG_ERR_TIMEOUT);
  } else if (threadIdx.x == 0) {
    // MMA issuer: four K = 32 MMAs per stage into one 128 x 256 fp32 accumulator
    for (int s = 0; s < steps; ++s) {
      const int st = s % kPeakStages;
      if (!mbar_wait_bounded(&copied[st], (s / kPeakStages) & 1, abort, kWaitLimitNs)) {
        report(status, MXG_ERR_TIMEOUT);
        *abort = 1;
        break;
      }
      tc_fence_after();
      const uint8_t* a = sm + st * kPeakStageBytes;
      const uint64_t adesc = smem_desc(smem_u32(a), 0, 1024, kLayoutSwizzle128B);
      const uint64_t bdesc = smem_desc(smem_u32(a + kPeakA), 0, 1024, kLayoutSwizzle128B);
      const uint32_t slot = tmem + 256 + st * 12;
#pragma unroll
      for (int k = 0; k < kPeakMmasPerStep; ++k)
        mma_mxf8<1>(tmem, adesc + 2 * k, bdesc + 2 * k, idesc_mxf8_e4m3(128, 256, k, k), slot, slot + 4,
                    (s | k) != 0 ? 1u : 0u);
      mma_commit<1>(&consumed[st]);
    }
    mma_commit<1>(mma_done);
    if (!mbar_wait_bounded(mma_done, 0, never_set, kWaitLimitNs)) report(status, MXG_ERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) tmem_dealloc<1>(tmem, 512);
}

}  // namespace
}  // namespace mxg

using namespace mxg;

extern "C" int mxg_bench_mxfp8_mma_peak(int steps, double* flops, int32_t* dev_status, void* stream) {
  if (steps <= 0 || !flops || !dev_status) return MXG_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(dev_status) & 3u) != 0) return MXG_ERR_ALIGN;
  int dev = 0, nsm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MXG_ERR_CUDA;
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MXG_ERR_CUDA;
  if (cudaFuncSetAttribute(mma_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeakSmem) != cudaSuccess)
    return MXG_ERR_CUDA;
  mma_peak_kernel<<<nsm, 128, kPeakSmem, static_cast<cudaStream_t>(stream)>>>(steps, dev_status);
  count_launch();
  if (cudaGetLastError() != cudaSuccess) return MXG_ERR_CUDA;
  *flops = static_cast<double>(nsm) * steps * kPeakMmasPerStep * kPeakFlopPerMma;
  return MXG_OK;
}
