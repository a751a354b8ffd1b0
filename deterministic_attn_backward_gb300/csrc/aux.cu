// aux.cu -- the two bandwidth-bound kernels around the main backward kernel.
//
// preprocess: D_r = sum_k dO_rk O_rk in f32 (the row term of
//             dS = P o (dP - D)), LSE_r * log2(e) for the base-2 softmax
//             recomputation, and the reset of everything the main kernel
//             needs at zero (status word, dispatch counters, dQ semaphores;
//             the f32 dQ accumulator too for the unordered atomic schedule).
// convert:    dQ = bf16(scale * (dQacc_0 + dQacc_1 + ...)), the accumulation
//             buffers added in index order.  The ordered schedules do the same
//             arithmetic inside the main kernel by default; this pass serves
//             the atomic schedule and callers that ask for a separate pass.
// Both are grid-stride loops over 16-byte vectors, sized to a multiple of the
// SM count by the host.
#include <cuda_bf16.h>
#include <cstdint>

#include "common.cuh"

namespace dab {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// Sum of the bf16 products of two 16-byte vectors (8 elements each), in f32.
// bf16 x bf16 products are exact in f32; they are added in element order.
__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 b) {
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
  const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc = fmaf(__uint_as_float(aw[i] << 16), __uint_as_float(bw[i] << 16), acc);
    acc = fmaf(__uint_as_float(aw[i] & 0xFFFF0000u), __uint_as_float(bw[i] & 0xFFFF0000u), acc);
  }
  return acc;
}

// One row of HD bf16 is HD/8 vectors; a warp covers 32 / (HD/8) rows at once.
// D and LSE2 = -LSE * log2(e) are laid out per head with S_pad = 128 *
// ceil(S / 128) rows; the rows past S of a partial last tile get D = 0 and
// LSE2 = -infinity, so that every P the main kernel forms for them is exactly
// 0.  (Negated, so that the main kernel forms scale*log2(e) * s + LSE2 with
// one packed fma per pair of columns.)
template <int HD>
__global__ void __launch_bounds__(256) preprocess_kernel(
    const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
    const float* __restrict__ lse, float* __restrict__ D, float* __restrict__ lse2,
    uint32_t* __restrict__ sem, int n_sem, WsHeader* __restrict__ hdr,
    float4* __restrict__ dqacc, long long dq_vec4, int BH, int S, int S_pad) {
  const int rows = BH * S;
  constexpr int kLanesPerRow = HD / 8;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  const int lane = threadIdx.x & 31;
  const long long gwarp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  const long long gtid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nthreads = (long long)gridDim.x * blockDim.x;

  if (gtid == 0) {
    hdr->status = 0u;
    hdr->detail = 0u;
    hdr->ticket = 0u;
    hdr->conv_ticket = 0u;
  }
  for (long long i = gtid; i < n_sem; i += nthreads) sem[i] = 0u;
  if (S_pad > S) {
    const long long npad = (long long)BH * (S_pad - S);
    for (long long i = gtid; i < npad; i += nthreads) {
      const long long idx = (i / (S_pad - S)) * S_pad + S + i % (S_pad - S);
      D[idx] = 0.f;
      lse2[idx] = -INFINITY;
    }
  }
  if (dqacc != nullptr) {
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (long long i = gtid; i < dq_vec4; i += nthreads) dqacc[i] = z;
  }

  const int sub = lane / kLanesPerRow;   // row within the warp's group
  const int part = lane % kLanesPerRow;  // 16-byte piece of the row
  // kGroups row groups per warp and pass, all loads issued before the sums
  constexpr int kGroups = 4;
  for (long long r0 = gwarp * kRowsPerWarp * kGroups; r0 < rows;
       r0 += nwarps * kRowsPerWarp * kGroups) {
    uint4 a[kGroups], b[kGroups];
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      const long long row = r0 + g * kRowsPerWarp + sub;
      if (row < rows) {
        a[g] = reinterpret_cast<const uint4*>(o + row * HD)[part];
        b[g] = reinterpret_cast<const uint4*>(dout + row * HD)[part];
      } else {
        a[g] = make_uint4(0u, 0u, 0u, 0u);
        b[g] = a[g];
      }
    }
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      const long long row = r0 + g * kRowsPerWarp + sub;
      float acc = dot8_bf16(a[g], b[g]);
#pragma unroll
      for (int off = kLanesPerRow / 2; off > 0; off >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (row < rows && part == 0) {
        // padded per-head index (rows < 2^31: 32-bit arithmetic)
        const int ir = (int)row;
        const int idx = (S_pad == S) ? ir : (ir / S) * S_pad + ir % S;
        D[idx] = acc;
        lse2[idx] = -(lse[row] * kLog2e);
      }
    }
  }
}

// dQ = bf16(scale * sum of the accumulation buffers), tile by tile.  The
// buffers that received a contribution (min(ways, contributors of the Q
// tile): N for the full mask, j + 1 for causal, the tables' count under a
// block mask, 0 -> dQ = 0) are added in index order, times scale, rounded to
// bf16 (RN-even): the arithmetic of the main kernel's tail, so both give the
// same bits.  kCM: chunk-major tiles [d/4][128 rows][4] (every head padded
// to whole tiles), read 16 bytes per thread over consecutive rows, staged in
// shared memory and written row by row.  Otherwise (atomic, d = 128):
// row-major accumulator [B*H*S][d], 16-byte vectors.
template <int HD, bool kCM>
__global__ void __launch_bounds__(256) convert_kernel(const float4* __restrict__ acc,
                                                      __nv_bfloat16* __restrict__ dq, int ntiles,
                                                      float scale, long long acc_stride_vec4,
                                                      int ways, int causal, int N, int S,
                                                      const int* __restrict__ count) {
  constexpr int kChunks = HD / 4;
  constexpr int kRowBytes = HD * 2 + 16;
  __shared__ __align__(16) uint8_t stage[kCM ? kTile * kRowBytes : 16];
  for (int T = blockIdx.x; T < ntiles; T += gridDim.x) {
    const int bh = T / N, j = T % N;
    int nacc = ways < N ? ways : N;
    if (count != nullptr || causal) {
      const int c = (count != nullptr) ? count[j] : j + 1;
      if (c < nacc) nacc = c;
    }
    const int rows = min(kTile, S - j * kTile);
    if constexpr (!kCM) {
      const size_t e0 = ((size_t)bh * S + (size_t)j * kTile) * HD;
      const float4* a = acc + e0 / 4;
      uint2* out = reinterpret_cast<uint2*>(dq + e0);
      for (int i = threadIdx.x; i < rows * kChunks; i += blockDim.x) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (nacc > 0) {
          float4 w[kAccWays];
#pragma unroll
          for (int m = 0; m < kAccWays; ++m)
            if (m < nacc) w[m] = a[i + (long long)m * acc_stride_vec4];
          v = w[0];
#pragma unroll
          for (int m = 1; m < kAccWays; ++m) {
            if (m < nacc) {
              v.x += w[m].x; v.y += w[m].y; v.z += w[m].z; v.w += w[m].w;
            }
          }
        }
        out[i] = make_uint2(pack_bf16x2(scale * v.x, scale * v.y), pack_bf16x2(scale * v.z, scale * v.w));
      }
    } else {
      const float4* a = acc + (size_t)T * (kTile * kChunks);
      for (int u = threadIdx.x; u < kTile * kChunks; u += blockDim.x) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (nacc > 0) {
          // all loads first (at most kAccWays buffers), then the sum in the
          // fixed order buffer 0, 1, ...
          float4 w[kAccWays];
#pragma unroll
          for (int m = 0; m < kAccWays; ++m)
            if (m < nacc) w[m] = a[u + (long long)m * acc_stride_vec4];
          v = w[0];
#pragma unroll
          for (int m = 1; m < kAccWays; ++m) {
            if (m < nacc) {
              v.x += w[m].x; v.y += w[m].y; v.z += w[m].z; v.w += w[m].w;
            }
          }
          v.x *= scale; v.y *= scale; v.z *= scale; v.w *= scale;
        }
        const int row = u % kTile, ch = u / kTile;
        *reinterpret_cast<uint2*>(stage + row * kRowBytes + ch * 8) =
            make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
      }
      __syncthreads();
      uint4* out = reinterpret_cast<uint4*>(dq + ((size_t)bh * S + (size_t)j * kTile) * HD);
      for (int w = threadIdx.x; w < rows * (HD / 8); w += blockDim.x) {
        const int row = w / (HD / 8), piece = w % (HD / 8);
        out[w] = *reinterpret_cast<const uint4*>(stage + row * kRowBytes + piece * 16);
      }
      __syncthreads();
    }
  }
}

// The first device error among `n` (status, detail) pairs, written to the
// header `hdr` (status 0 when every pair is 0).  One thread: n is the number
// of head groups of a host-buffer call.
__global__ void status_collect_kernel(const uint32_t* __restrict__ slots, int n,
                                      WsHeader* __restrict__ hdr) {
  uint32_t st = 0u, det = 0u;
  for (int i = 0; i < n; ++i) {
    if (slots[2 * i] != 0u) {
      st = slots[2 * i];
      det = slots[2 * i + 1];
      break;
    }
  }
  hdr->status = st;
  hdr->detail = det;
}

// Schedule tables of a block mask (one CTA): for each KV tile i its visible Q
// tiles in visit order (ascending, or descending for DESCENDING_Q) and their
// number; for each Q tile j the rank of each visible KV tile in ascending KV
// order and the number of contributors.  Visible: flag (j, i) set and, for
// the causal mask, i <= j.
__global__ void block_tables_kernel(const uint8_t* __restrict__ tiles, int N, int causal,
                                    int descending, uint16_t* __restrict__ list,
                                    uint16_t* __restrict__ rank, int* __restrict__ nact,
                                    int* __restrict__ count) {
  auto vis = [&](int j, int i) { return tiles[(size_t)j * N + i] != 0 && (!causal || i <= j); };
  for (int x = threadIdx.x; x < N; x += blockDim.x) {
    int n = 0;
    for (int t = 0; t < N; ++t) {
      const int j = descending ? N - 1 - t : t;
      if (vis(j, x)) list[(size_t)x * N + n++] = (uint16_t)j;
    }
    nact[x] = n;
    int r = 0;
    for (int i = 0; i < N; ++i) {
      const bool v = vis(x, i);
      rank[(size_t)x * N + i] = v ? (uint16_t)r : (uint16_t)0xFFFFu;
      r += v ? 1 : 0;
    }
    count[x] = r;
  }
}

}  // namespace

cudaError_t launch_block_tables(const uint8_t* tiles, int N, int causal, int descending,
                                uint16_t* list, uint16_t* rank, int* nact, int* count,
                                cudaStream_t stream) {
  block_tables_kernel<<<1, 256, 0, stream>>>(tiles, N, causal, descending, list, rank, nact, count);
  return cudaGetLastError();
}

cudaError_t launch_preprocess(int HD, const void* o, const void* dout, const float* lse, float* D,
                              float* lse2, uint32_t* sem, int n_sem, WsHeader* hdr, float* dqacc,
                              long long dq_elems, int BH, int S, int S_pad, int grid,
                              cudaStream_t stream) {
  float4* z = reinterpret_cast<float4*>(dqacc);
  const long long nv = dqacc ? dq_elems / 4 : 0;
  if (HD == 128) {
    preprocess_kernel<128><<<grid, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse, D, lse2,
        sem, n_sem, hdr, z, nv, BH, S, S_pad);
  } else {
    preprocess_kernel<64><<<grid, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse, D, lse2,
        sem, n_sem, hdr, z, nv, BH, S, S_pad);
  }
  return cudaGetLastError();
}

cudaError_t launch_status_collect(const uint32_t* slots, int n, void* hdr, cudaStream_t stream) {
  status_collect_kernel<<<1, 1, 0, stream>>>(slots, n, static_cast<WsHeader*>(hdr));
  return cudaGetLastError();
}

cudaError_t launch_convert(const float* dqacc, int chunk_major, void* dq, int ntiles, float scale,
                           long long acc_stride, int ways, int causal, int N, int S, int d, int grid,
                           const int* count, cudaStream_t stream) {
  const float4* a = reinterpret_cast<const float4*>(dqacc);
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(dq);
  const long long st4 = acc_stride / 4;
  if (d == 64)
    convert_kernel<64, true><<<grid, 256, 0, stream>>>(a, out, ntiles, scale, st4, ways, causal, N, S, count);
  else if (chunk_major)
    convert_kernel<128, true><<<grid, 256, 0, stream>>>(a, out, ntiles, scale, st4, ways, causal, N, S, count);
  else
    convert_kernel<128, false><<<grid, 256, 0, stream>>>(a, out, ntiles, scale, st4, ways, causal, N, S, count);
  return cudaGetLastError();
}

}  // namespace dab
