// selftest.cu -- one-CTA check of the five tensor-core operand forms the
// backward kernel uses, on single 128-row tiles, with the same shared-memory
// layouts, descriptors and tensor-memory placements:
//   out0 = X Y^T        A K-major smem, B K-major smem     (S^T, dP^T)
//   out1 = P Y          A bf16 in tensor memory, B MN-major (dV)
//   out2 = Z Y          A K-major (thread-written), B MN-major (dK)
//   out3 = X^T Z  (d=128) / Z^T X (d=64)  both MN-major     (dQ^T / dQ)
// X, Y: [128][d] bf16 (loaded by TMA); Z, P: [128][128] bf16 (written by
// threads into the swizzled layout / into tensor memory).  Outputs f32.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace dab {
namespace {

struct STBars {
  uint64_t xy_full, written, mma_a, read_a, mma_b, drain;
};

template <int HD>
__global__ void __launch_bounds__(192, 1)
    selftest_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_y,
                    const __nv_bfloat16* __restrict__ z, const __nv_bfloat16* __restrict__ pm,
                    float* out0, float* out1, float* out2, float* out3, WsHeader* hdr) {
  constexpr int T = kTile * HD * 2;
  constexpr int kOffX = 0, kOffY = T, kOffZ = 2 * T, kOffBar = 2 * T + 32768;
  extern __shared__ __align__(1024) uint8_t smem[];
  STBars* bars = reinterpret_cast<STBars*>(smem + kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kOffBar + 64);
  int* abort_flag = reinterpret_cast<int*>(smem + kOffBar + 68);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if ((sbase & 1023u) != 0u) {
    if (threadIdx.x == 0) raise_error(hdr, kStatusBounds, kDetailAlign);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&bars->xy_full, 1);
    mbar_init(&bars->written, 4);
    mbar_init(&bars->mma_a, 1);
    mbar_init(&bars->read_a, 4);
    mbar_init(&bars->mma_b, 1);
    mbar_init(&bars->drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *tslot;
  const WaitCtl wc{abort_flag, hdr, 2000000000ull};
  constexpr uint32_t kCol0 = 0, kCol1 = 128, kCol2 = 256, kColP = 448, kCol3 = 0;

  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars->xy_full, 2 * T);
      for (int db = 0; db < HD / 64; ++db) {
        tma_load_2d(smem + kOffX + db * 16384, &tm_x, &bars->xy_full, db * 64, 0);
        tma_load_2d(smem + kOffY + db * 16384, &tm_y, &bars->xy_full, db * 64, 0);
      }
      drain_wait(&bars->xy_full, 0, hdr, 2000000000ull, 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t sX = sbase + kOffX, sY = sbase + kOffY, sZ = sbase + kOffZ;
      bool ok = mbar_wait(&bars->xy_full, 0, wc, 1) && mbar_wait(&bars->written, 0, wc, 2);
      if (ok) {
        tc_fence_after();
        for (int k = 0; k < HD / 16; ++k)
          mma_ss(tb + kCol0, desc_kmajor(sX, k, 128), desc_kmajor(sY, k, 128),
                 idesc_bf16(128, 128, 0, 0), k > 0);
        for (int k = 0; k < 8; ++k)
          mma_ts(tb + kCol1, tb + kColP + 8 * k, desc_mnmajor(sY, k, 128), idesc_bf16(128, HD, 0, 1),
                 k > 0);
        for (int k = 0; k < 8; ++k)
          mma_ss(tb + kCol2, desc_kmajor(sZ, k, 128), desc_mnmajor(sY, k, 128),
                 idesc_bf16(128, HD, 0, 1), k > 0);
        mma_commit(&bars->mma_a);
        ok = mbar_wait(&bars->read_a, 0, wc, 3);
      }
      if (ok) {
        tc_fence_after();
        for (int k = 0; k < 8; ++k) {
          if (HD == 128)
            mma_ss(tb + kCol3, desc_mnmajor(sX, k, 128), desc_mnmajor(sZ, k, 128),
                   idesc_bf16(128, 128, 1, 1), k > 0);
          else
            mma_ss(tb + kCol3, desc_mnmajor(sZ, k, 128), desc_mnmajor(sX, k, 128),
                   idesc_bf16(128, 64, 1, 1), k > 0);
        }
        mma_commit(&bars->mma_b);
      }
      mma_commit(&bars->drain);
      drain_wait(&bars->drain, 0, hdr, 2000000000ull, 2);
    }
    __syncwarp();
  } else {
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lo = (uint32_t)(quad * 32) << 16;
    // Z row r -> swizzled [2][128][64] layout; P row r -> tensor memory (bf16 pairs).
    uint8_t* sz = smem + kOffZ;
    for (int cc = 0; cc < 16; ++cc) {
      const uint4 val = reinterpret_cast<const uint4*>(z + r * 128)[cc];
      const int qb = cc >> 3, c8 = cc & 7;
      *reinterpret_cast<uint4*>(sz + qb * 16384 + r * 128 + ((c8 ^ (r & 7)) << 4)) = val;
    }
    for (int ch = 0; ch < 4; ++ch) {
      uint32_t w[16];
      const uint32_t* src = reinterpret_cast<const uint32_t*>(pm + r * 128 + 32 * ch);
      for (int e = 0; e < 16; ++e) w[e] = src[e];
      tmem_st16(tb + lo + kColP + 16 * ch, w);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars->written);
    if (warp_wait(&bars->mma_a, 0, wc, 4)) {
      tc_fence_after();
      uint32_t v[32];
      for (int ch = 0; ch < 4; ++ch) {
        tmem_ld32(tb + lo + kCol0 + 32 * ch, v);
        for (int e = 0; e < 32; ++e) out0[r * 128 + 32 * ch + e] = __uint_as_float(v[e]);
      }
      for (int ch = 0; ch < HD / 32; ++ch) {
        tmem_ld32(tb + lo + kCol1 + 32 * ch, v);
        for (int e = 0; e < 32; ++e) out1[r * HD + 32 * ch + e] = __uint_as_float(v[e]);
        tmem_ld32(tb + lo + kCol2 + 32 * ch, v);
        for (int e = 0; e < 32; ++e) out2[r * HD + 32 * ch + e] = __uint_as_float(v[e]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->read_a);
      if (warp_wait(&bars->mma_b, 0, wc, 5)) {
        tc_fence_after();
        constexpr int n3 = (HD == 128) ? 128 : 64;
        for (int ch = 0; ch < n3 / 32; ++ch) {
          tmem_ld32(tb + lo + kCol3 + 32 * ch, v);
          for (int e = 0; e < 32; ++e) out3[r * n3 + 32 * ch + e] = __uint_as_float(v[e]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

}  // namespace

template <int HD>
int selftest_smem_bytes() {
  return 2 * kTile * HD * 2 + 32768 + 128;
}
template <int HD>
const void* selftest_kernel_ptr() {
  return reinterpret_cast<const void*>(&selftest_kernel<HD>);
}
template int selftest_smem_bytes<64>();
template int selftest_smem_bytes<128>();
template const void* selftest_kernel_ptr<64>();
template const void* selftest_kernel_ptr<128>();

}  // namespace dab
