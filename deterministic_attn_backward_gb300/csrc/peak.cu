// peak.cu -- dense bf16 tensor throughput of this build's own tcgen05 path.
//
// The backward's throughput is quoted as a fraction of the dense bf16 tensor
// peak.  Besides the measured copy of a library GEMM, that peak is measured
// here with the same instructions the backward kernel uses: one CTA per SM,
// one thread issuing back-to-back tcgen05.mma of M = 128, N = 256, K = 16
// (bf16 operands, f32 accumulation in tensor memory), both operands resident
// in shared memory (A 128 x 64, B 256 x 64, K-major, 128-byte swizzle).  No
// global memory is touched, so the result is the tensor pipe's issue rate at
// the clock the GPU runs at.  Work: gridDim.x * iters * 4 MMAs of
// 2 * 128 * 256 * 16 flops each.
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace dab {
namespace {

constexpr int kPeakThreads = 128;
constexpr int kOffA = 0;                     // [128][64] bf16
constexpr int kOffB = 128 * 128;             // [256][64] bf16
constexpr int kOffBar = kOffB + 256 * 128;
constexpr int kPeakSmem = kOffBar + 64;

__global__ void __launch_bounds__(kPeakThreads, 1) peak_kernel(int iters, WsHeader* hdr,
                                                                unsigned long long timeout_ns) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kOffBar + 16);
  const uint32_t sbase = smem_u32(smem);
  if ((sbase & 1023u) != 0u) {
    if (threadIdx.x == 0) raise_error(hdr, kStatusBounds, kDetailAlign);
    return;
  }
  // Operands: small finite values (the products are not inspected).
  for (int i = threadIdx.x; i < kOffBar / 16; i += kPeakThreads)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0x3c003c00u, 0x3c003c00u, 0u, 0u);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (threadIdx.x < 32) {
    tmem_alloc(tslot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *tslot;
  if (threadIdx.x == 0) {
    const uint64_t a0 = desc_kmajor(sbase + kOffA, 0, 128);
    const uint64_t b0 = desc_kmajor(sbase + kOffB, 0, 256);
    constexpr uint32_t kId = idesc_bf16(128, 256, 0, 0);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        mma_ss(tb, a0 + koff_kmajor(k, 128), b0 + koff_kmajor(k, 256), kId, (it | k) != 0);
    }
    mma_commit(bar);
    drain_wait(bar, 0, hdr, timeout_ns, 5);
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(tb, 256);
  }
}

}  // namespace

int peak_smem_bytes() { return kPeakSmem; }
const void* peak_kernel_ptr() { return reinterpret_cast<const void*>(&peak_kernel); }
int peak_threads() { return kPeakThreads; }

}  // namespace dab
