// bwd.cu -- persistent attention backward kernel for GB300 (sm_103a).
//
// One CTA per SM.  A CTA takes work units (one KV tile's chain, or a pair of
// chains for the causal symmetric shift) and, for every step (KV tile i,
// Q tile j) of a chain, computes on the tensor cores (tcgen05, operands in
// shared memory or tensor memory, f32 accumulators in tensor memory):
//     S^T  = K_i Q_j^T                      (128 x 128, contraction over d)
//     P^T  = exp(scale S^T - LSE_j)         (softmax warps; causal mask)
//     dP^T = V_i dO_j^T
//     dV_i += P^T dO_j                      (P^T read from tensor memory)
//     dS^T = P^T o (dP^T - D_j)             (softmax warps -> shared memory)
//     dK_i += dS^T Q_j
//     dQ_j partial = dS K_i                 (Q rows on tensor-memory lanes)
// dK_i and dV_i stay in tensor memory for the whole chain (the KV-chain
// constraint of the DASH DAG model, technical summary section 2.1) and are
// written once at its end.  The dQ partial is added to an f32 accumulator in
// global memory by the reducer warps: for the deterministic schedules in the
// fixed order rank(i, j) (technical summary section 1: a fixed accumulation
// order for dQ), gated by per-(head, Q tile, eighth, buffer) semaphores; for
// ATOMIC with unordered float adds.  The partial is dQ (Q rows on
// tensor-memory lanes) and the accumulator is stored chunk-major per 128-row
// tile, [d/4][128 rows][4] f32, so that a thread adds 16 bytes at a time and
// a warp's 32 rows of a chunk form 512 contiguous bytes.  The one exception,
// ATOMIC at d = 128, keeps a row-major accumulator [B*H*S][d] with the
// partial as dQ^T (d on lanes): a reducer thread holds one d index over 64 Q
// rows and a warp's 32 one-float adds are one 128-byte segment of a row.  For
// the deterministic schedules the same kernel then converts dQ to bf16 in
// its tail: a CTA without units left converts the dQ tiles whose semaphores
// show every contribution in.
//
// Warp roles (20 warps):
//   warp 0      TMA producer (K_i, V_i per chain; Q_j, dO_j, LSE_j, D_j per
//               step, double-buffered) and tensor-memory allocation
//   warp 1      MMA issuer of S^T and dP^T (one thread)
//   warp 2      MMA issuer of dV, the dQ partial and dK (one thread)
//   warp 3      dQ publisher (ordered schedules): releases each contribution
//               once the reducers' adds are in
//   warps 4-11  softmax / dS, two warpgroups of 64 Q columns each (thread =
//               KV row), and the chain epilogue (dV by one, dK by the other)
//   warps 12-19 dQ reducer, one eighth of the dQ tile and one semaphore each
//   all warps   after the last unit: the dQ convert of finished tiles
// Every wait is bounded: on expiry the kernel records DAB_ERR_TIMEOUT in the
// workspace and every role drains and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"
#include "tile_sched.h"

namespace dab {
namespace {

// 20 warps: five per SM sub-partition, 96 registers per thread.
constexpr int kThreads = 640;
constexpr int kSoftmaxWarp0 = 4;    // warps 4-7: Q columns 0-63, warps 8-11: 64-127
constexpr int kReducerWarp0 = 12;   // warps 12-19: two reducer warpgroups

template <int HD>
struct Cfg {
  static constexpr int kTileBytes = kTile * HD * 2;        // one 128 x HD bf16 tile
  static constexpr int kBlockBytes = kTile * 128;          // one [128 rows][64] block
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffQ = 2 * kTileBytes;             // 2 stages
  static constexpr int kOffDO = 4 * kTileBytes;            // 2 stages
  static constexpr int kOffDS = 6 * kTileBytes;            // [2][128][64] bf16
  static constexpr int kOffLse = kOffDS + 32768;           // [2][128] f32
  static constexpr int kOffDD = kOffLse + 1024;            // [2][128] f32
  static constexpr int kOffBar = kOffDD + 1024;
  static constexpr int kOffMisc = kOffBar + 256;
  static constexpr int kOffPub = kOffMisc + 64;            // [2][8] (semaphore, value) to release
  static constexpr int kSmemBytes = kOffPub + 2 * 8 * 8;
  // Tensor memory columns (512 allocated).
  static constexpr uint32_t kColDV = 0;
  static constexpr uint32_t kColDK = HD;
  static constexpr uint32_t kColS = 2 * HD;                // S^T, then P^T (bf16, 64 cols)
  static constexpr uint32_t kColDP = 2 * HD + 128;
  static constexpr uint32_t kColDQ = (HD == 128) ? kColDP : 384;  // d=128 reuses dP
  static constexpr int kChunks = HD / 4;                   // 16-byte chunks of a dQ row
  // Instruction descriptors.
  static constexpr uint32_t kIdS = idesc_bf16(128, 128, 0, 0);   // S^T, dP^T
  static constexpr uint32_t kIdAcc = idesc_bf16(128, HD, 0, 1);  // dV, dK
  static constexpr uint32_t kIdDQ = idesc_bf16(128, HD, 1, 1);  // dQ = dS K, or dQ^T = K^T dS^T (d = 128)
};

struct Bars {
  uint64_t kv_full, kv_empty;
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full, dp_full, p_full, ds_full;
  uint64_t dv_done, ds_free, dq_full, dq_empty;
  uint64_t acc_full, acc_empty;
  uint64_t unit_full[2], unit_empty[2];
  uint64_t drain, drain2;
  uint64_t pub_full[2], pub_empty[2]; // reducers -> publisher, publisher -> reducers
};
static_assert(sizeof(Bars) <= 256, "barrier block");

struct Misc {
  uint32_t tmem_base;
  int abort;
  int ring[2];
  int conv;  // dQ tile being finalised in the tail, or -1
};
static_assert(sizeof(Misc) <= 64, "misc block");

static __device__ __noinline__ bool sem_wait(const uint32_t* sem, uint32_t target, const WaitCtl& w,
                                      uint32_t detail) {
  uint64_t t0 = 0;
  uint32_t it = 0;
  while (true) {
    if (ld_acquire_gpu(sem) == target) return true;
    if (it == 0) t0 = globaltimer_ns();
    if ((++it & 15u) == 0u) {
      if (*w.abort) return false;
      if (ld_volatile(&w.hdr->status) != 0u) {
        *w.abort = 1;
        return false;
      }
      if (globaltimer_ns() - t0 > w.timeout_ns) {
        raise_error(w.hdr, kStatusTimeout, kDetailSem | (detail & 0xFFFFFFu));
        *w.abort = 1;
        return false;
      }
    }
  }
}

// Schedule of unit u (one KV tile's chain, or a causal shift pair): the
// fixed schedules of tile_sched.h, or under a block mask the tables built
// from the tile flags (the KV tile's visible Q tiles in visit order; ranks in
// ascending KV order, shared by serial and descending as without a mask).
__device__ __forceinline__ int k_unit_steps(const BwdParams& p, int u) {
  return p.block ? p.blk_nact[u] : unit_steps(p.sched, p.mask, p.N, u);
}
__device__ __forceinline__ Step k_step(const BwdParams& p, int u, int t, int steps) {
  if (!p.block) return step(p.sched, p.mask, p.N, u, t);
  Step s;
  s.kv = u;
  s.q = p.blk_list[(size_t)u * p.N + t];
  s.chain_first = (t == 0);
  s.chain_last = (t == steps - 1);
  return s;
}
__device__ __forceinline__ int k_rank(const BwdParams& p, int i, int j) {
  if (!p.block) return rank(p.sched, p.mask, p.N, i, j);
  return p.sched == kSchedAtomic ? -1 : (int)p.blk_rank[(size_t)j * p.N + i];
}

// Bounded wait for a dQ semaphore to reach its final value, polled gently:
// the waiting CTA has no other work, and the CTAs still running share the L2.
static __device__ __noinline__ bool final_wait(const uint32_t* sem, uint32_t target,
                                               const WaitCtl& w, uint32_t detail) {
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_gpu(sem) != target) {
    if (*w.abort) return false;
    if (ld_volatile(&w.hdr->status) != 0u) {
      *w.abort = 1;
      return false;
    }
    if (globaltimer_ns() - t0 > w.timeout_ns) {
      raise_error(w.hdr, kStatusTimeout, kDetailSem | (detail & 0xFFFFFFu));
      *w.abort = 1;
      return false;
    }
    __nanosleep(200);
  }
  return true;
}

// dQ finalisation in the kernel's tail (ordered schedules).  A CTA that has
// run out of units claims whole dQ tiles (bh, j) from a second counter, in
// head order and, within a head, in the order the schedule completes them.
// A tile is final once every (sub-tile, buffer) semaphore holds the number of
// contributions that buffer receives: for c contributors and W buffers,
// buffer m < min(c, W) receives (c - 1 - m) / W + 1 of them.  Every unit has
// been claimed by a running CTA before any tile is, and no unit waits for a
// tile, so these waits always end.  The arithmetic is the convert pass's:
// the buffers added in index order, times scale, rounded to bf16 (RN-even),
// so dQ has the same bits whichever of the two wrote it.  The ordered
// schedules' tiles are chunk-major: read 16 bytes per thread (coalesced), the
// bf16 result goes through shared memory (free once the roles are done) and
// out row by row.
template <int HD, bool kRagged>
__device__ __forceinline__ void tail_convert(const BwdParams& p, Misc* misc, uint8_t* smem,
                                             const WaitCtl& wc) {
  constexpr int kChunks = HD / 4;
  constexpr int kRowBytes = HD * 2 + 16;                 // padded bf16 row in shared memory
  const int tid = threadIdx.x;
  const int ntiles = p.BH * p.N;
  const size_t stride4 = (size_t)p.acc_stride / 4;
  while (true) {
    if (tid == 0) {
      const int T = misc->abort ? ntiles : (int)atomicAdd(&p.hdr->conv_ticket, 1u);
      misc->conv = (T < ntiles) ? T : -1;
    }
    __syncthreads();
    const int T = misc->conv;
    if (T < 0) break;
    const int bh = T / p.N, jj = T % p.N;
    const int j = (p.sched == kSchedDescending) ? p.N - 1 - jj : jj;
    const int c = p.block ? p.blk_count[j] : (p.mask == kMaskCausal ? j + 1 : p.N);
    const int nacc = c < p.acc_ways ? c : p.acc_ways;
    int ok = 1;
    if (tid < kSubTiles * nacc) {
      const int sub = tid / nacc, way = tid % nacc;
      const size_t sem_idx = (((size_t)bh * p.N + j) * kSubTiles + sub) * p.acc_ways + way;
      const uint32_t target = (uint32_t)((c - 1 - way) / p.acc_ways + 1);
      ok = final_wait(p.sem + sem_idx, target, wc, (uint32_t)sem_idx) ? 1 : 0;
    }
    if (!__syncthreads_and(ok)) break;
    fence_acq_rel_gpu();
    // rows of the tile inside the head (a partial last tile stops at S)
    const int rows = kRagged ? min(kTile, p.S - j * kTile) : kTile;
    // chunk-major tile: chunk units u = chunk * 128 + row, consecutive
    // threads on consecutive rows (coalesced 16-byte loads); the bf16
    // result is staged in shared memory (free once the roles are done)
    // and written row by row
    const float4* acc = reinterpret_cast<const float4*>(p.dqacc) + ((size_t)bh * p.N + j) * (kTile * kChunks);
    for (int u = tid; u < kTile * kChunks; u += kThreads) {
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (nacc > 0) {
        float4 w[kAccWays];
#pragma unroll
        for (int m = 0; m < kAccWays; ++m)
          if (m < nacc) w[m] = __ldcg(acc + u + m * stride4);
        v = w[0];
#pragma unroll
        for (int m = 1; m < kAccWays; ++m) {
          if (m < nacc) {
            v.x += w[m].x; v.y += w[m].y; v.z += w[m].z; v.w += w[m].w;
          }
        }
        v.x *= p.scale; v.y *= p.scale; v.z *= p.scale; v.w *= p.scale;
      }
      const int row = u % kTile, ch = u / kTile;
      *reinterpret_cast<uint2*>(smem + row * kRowBytes + ch * 8) =
          make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
    }
    __syncthreads();
    uint4* out = reinterpret_cast<uint4*>(p.dq + ((size_t)bh * p.S + (size_t)j * kTile) * HD);
    for (int w = tid; w < rows * (HD / 8); w += kThreads) {
      const int row = w / (HD / 8), piece = w % (HD / 8);
      out[w] = *reinterpret_cast<const uint4*>(smem + row * kRowBytes + piece * 16);
    }
    __syncthreads();  // misc->conv and the staging rows are rewritten for the next tile
  }
}

// kRagged: S is not a multiple of the tile, so the last tile of each head is
// partial (masked keys, rows never written).  A separate instance, so that the
// common case carries none of those checks.  kCM: the dQ accumulation tiles
// are chunk-major [d/4][128][4] (every schedule at d = 64, the ordered ones at
// d = 128); otherwise row-major [row][d] (the atomic schedule at d = 128).
template <int HD, bool kRagged, bool kCM>
__global__ void __launch_bounds__(kThreads, 1) bwd_kernel(const __grid_constant__ BwdParams p) {
  using C = Cfg<HD>;
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kOffBar);
  Misc* misc = reinterpret_cast<Misc*>(smem + C::kOffMisc);
  float* s_lse = reinterpret_cast<float*>(smem + C::kOffLse);  // -LSE*log2(e) of the stage's Q rows
  float* s_dd = reinterpret_cast<float*>(smem + C::kOffDD);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Operand tiles need 1024-byte-aligned swizzle atoms.
  if ((sbase & 1023u) != 0u) {
    if (threadIdx.x == 0) raise_error(p.hdr, kStatusBounds, kDetailAlign);
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    mbar_init(&bars->kv_empty, 2);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->q_full[s], 1);
      mbar_init(&bars->q_empty[s], 2 + 8);
      mbar_init(&bars->unit_full[s], 1);
      mbar_init(&bars->unit_empty[s], 2 + 8 + 8 + 1);
      mbar_init(&bars->pub_full[s], 8);
      mbar_init(&bars->pub_empty[s], 1);
    }
    mbar_init(&bars->s_full, 1);
    mbar_init(&bars->dp_full, 1);
    mbar_init(&bars->p_full, 8);
    mbar_init(&bars->ds_full, 8);
    mbar_init(&bars->dv_done, 1);
    mbar_init(&bars->ds_free, 1);
    mbar_init(&bars->dq_full, 1);
    mbar_init(&bars->dq_empty, 8);
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->acc_empty, 8);
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->drain2, 1);
    misc->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&misc->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = misc->tmem_base;
  const WaitCtl wc{&misc->abort, p.hdr, p.timeout_ns};
  const bool deterministic = p.sched != kSchedAtomic;
  const bool is_static = static_dispatch(p.sched);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&p.tm_q);
      prefetch_tensormap(&p.tm_k);
      prefetch_tensormap(&p.tm_v);
      prefetch_tensormap(&p.tm_do);
      int s = 0, chain = 0, uidx = 0, prevU = -1;
      int issued[2] = {0, 0};
      bool ok = true;
      while (ok) {
        int U;
        if (is_static) {
          U = (uidx == 0) ? (int)blockIdx.x : prevU + (int)gridDim.x;
        } else {
          U = (int)atomicAdd(&p.hdr->ticket, 1u);
        }
        if (U >= p.total_units) U = -1;
        prevU = U;
        const int slot = uidx & 1;
        if (uidx >= 2 && !mbar_wait(&bars->unit_empty[slot], ((uidx >> 1) - 1) & 1, wc, 1)) break;
        misc->ring[slot] = U;
        mbar_arrive(&bars->unit_full[slot]);
        ++uidx;
        if (U < 0) break;
        const int bh = U / p.units_per_head, u = U % p.units_per_head;
        const int steps = k_unit_steps(p, u);
        for (int t = 0; t < steps; ++t) {
          const Step st = k_step(p, u, t, steps);
          if (st.chain_first) {
            if (chain > 0 && !mbar_wait(&bars->kv_empty, (chain - 1) & 1, wc, 2)) { ok = false; break; }
            mbar_arrive_expect_tx(&bars->kv_full, 2 * C::kTileBytes);
            const int row = bh * p.S + st.kv * kTile;
#pragma unroll
            for (int db = 0; db < HD / 64; ++db) {
              tma_load_2d(smem + C::kOffK + db * C::kBlockBytes, &p.tm_k, &bars->kv_full, db * 64, row);
              tma_load_2d(smem + C::kOffV + db * C::kBlockBytes, &p.tm_v, &bars->kv_full, db * 64, row);
            }
            ++chain;
          }
          const int stage = s & 1;
          if (s >= 2 && !mbar_wait(&bars->q_empty[stage], ((s >> 1) - 1) & 1, wc, 3)) { ok = false; break; }
          mbar_arrive_expect_tx(&bars->q_full[stage], 2 * C::kTileBytes + 1024);
          const int row = bh * p.S + st.q * kTile;
          uint8_t* sq = smem + C::kOffQ + stage * C::kTileBytes;
          uint8_t* sdo = smem + C::kOffDO + stage * C::kTileBytes;
#pragma unroll
          for (int db = 0; db < HD / 64; ++db) {
            tma_load_2d(sq + db * C::kBlockBytes, &p.tm_q, &bars->q_full[stage], db * 64, row);
            tma_load_2d(sdo + db * C::kBlockBytes, &p.tm_do, &bars->q_full[stage], db * 64, row);
          }
          // -LSE*log2(e) and D are padded to whole tiles per head (-inf / 0 past S)
          const size_t prow = (size_t)bh * (p.N * kTile) + (size_t)st.q * kTile;
          bulk_load(s_lse + stage * 128, p.lse2 + prow, 512, &bars->q_full[stage]);
          bulk_load(s_dd + stage * 128, p.D + prow, 512, &bars->q_full[stage]);
          ++issued[stage];
          ++s;
        }
      }
      // Teardown: every issued copy must land before the CTA may exit.
      if (chain > 0) drain_wait(&bars->kv_full, (chain - 1) & 1, p.hdr, p.timeout_ns, 1);
      for (int st = 0; st < 2; ++st)
        if (issued[st] > 0) drain_wait(&bars->q_full[st], (issued[st] - 1) & 1, p.hdr, p.timeout_ns, 2);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Two issuing threads on two SM sub-partitions.  With one thread, S^T of
    // the next step queued behind that thread's wait for dS of the current
    // step; split, each chain of products is issued as soon as its own
    // inputs are ready:
    //   warp 1, the "forward" products of every step: S^T = K Q^T once dV of
    //     the previous step has read P from the S columns, then dP^T = V dO^T
    //     once its columns are free (d = 128: the reducers have drained the
    //     previous dQ partial, which shares them; d = 64: the softmax has
    //     read the previous dP);
    //   warp 2, the "backward" products: dV += P^T dO once the softmax has
    //     written P, then the dQ partial (dQ = dS K; dQ^T = K^T dS^T for the
    //     atomic schedule's row-major accumulator at d = 128) and
    //     dK += dS^T Q once it has written dS.
    // A commit tracks only the MMAs of the thread that issues it, so the
    // barriers that release a Q/dO stage and the K/V tiles take one commit
    // from each issuer.
    if (lane == 0) {
      const bool fwd = (warp == 1);
      // Descriptors of every operand at K step 0, built once; step k adds a
      // compile-time offset.
      const uint64_t dK_k = desc_kmajor(sbase + C::kOffK, 0, 128);
      const uint64_t dK_mn = desc_mnmajor(sbase + C::kOffK, 0, 128);
      const uint64_t dV_k = desc_kmajor(sbase + C::kOffV, 0, 128);
      const uint64_t dDS_k = desc_kmajor(sbase + C::kOffDS, 0, 128);
      const uint64_t dDS_mn = desc_mnmajor(sbase + C::kOffDS, 0, 128);
      // stage 1 lies one tile above stage 0: its descriptors differ by a constant
      const uint64_t dQ_k0 = desc_kmajor(sbase + C::kOffQ, 0, 128);
      const uint64_t dQ_mn0 = desc_mnmajor(sbase + C::kOffQ, 0, 128);
      const uint64_t dDO_k0 = desc_kmajor(sbase + C::kOffDO, 0, 128);
      const uint64_t dDO_mn0 = desc_mnmajor(sbase + C::kOffDO, 0, 128);
      constexpr uint64_t kStageOff = C::kTileBytes >> 4;
      const uint32_t tS = tbase + C::kColS, tDP = tbase + C::kColDP, tDV = tbase + C::kColDV;
      const uint32_t tDK = tbase + C::kColDK, tDQ = tbase + C::kColDQ;
      int s = 0, chain = 0, uidx = 0;
      bool ok = true;
      while (ok) {
        const int slot = uidx & 1;
        if (!mbar_wait(&bars->unit_full[slot], (uidx >> 1) & 1, wc, fwd ? 10 : 22)) break;
        const int U = misc->ring[slot];
        mbar_arrive(&bars->unit_empty[slot]);
        ++uidx;
        if (U < 0) break;
        const int u = U % p.units_per_head;
        const int steps = k_unit_steps(p, u);
        for (int t = 0; t < steps; ++t) {
          const Step st = k_step(p, u, t, steps);
          const int stage = s & 1;
          if (fwd) {
            if (st.chain_first && !mbar_wait(&bars->kv_full, chain & 1, wc, 11)) { ok = false; break; }
            if (!mbar_wait(&bars->q_full[stage], (s >> 1) & 1, wc, 12)) { ok = false; break; }
            if (s > 0 && !mbar_wait(&bars->dv_done, (s - 1) & 1, wc, 13)) { ok = false; break; }
            tc_fence_after();
            {
              const uint64_t q0 = dQ_k0 + (uint64_t)stage * kStageOff;
#pragma unroll
              for (int k = 0; k < HD / 16; ++k)
                mma_ss(tS, dK_k + koff_kmajor(k, 128), q0 + koff_kmajor(k, 128), C::kIdS, k > 0);
              mma_commit(&bars->s_full);
            }
            if (s > 0 && !mbar_wait(HD == 128 ? &bars->dq_empty : &bars->ds_full, (s - 1) & 1, wc, 14)) {
              ok = false;
              break;
            }
            tc_fence_after();
            {
              const uint64_t o0 = dDO_k0 + (uint64_t)stage * kStageOff;
#pragma unroll
              for (int k = 0; k < HD / 16; ++k)
                mma_ss(tDP, dV_k + koff_kmajor(k, 128), o0 + koff_kmajor(k, 128), C::kIdS, k > 0);
              mma_commit(&bars->dp_full);
            }
            mma_commit(&bars->q_empty[stage]);
            if (st.chain_last) {
              mma_commit(&bars->kv_empty);
              ++chain;
            }
          } else {
            // dV += P^T dO; P^T from tensor memory, its two 64-column halves
            // packed at the start of each half of the S columns
            if (!mbar_wait(&bars->p_full, s & 1, wc, 15)) { ok = false; break; }
            if (st.chain_first && chain > 0 && !mbar_wait(&bars->acc_empty, (chain - 1) & 1, wc, 16)) { ok = false; break; }
            tc_fence_after();
            {
              const uint64_t o0 = dDO_mn0 + (uint64_t)stage * kStageOff;
              const uint32_t acc0 = st.chain_first ? 0u : 1u;
#pragma unroll
              for (int k = 0; k < kTile / 16; ++k)
                mma_ts(tDV, tS + (k >> 2) * 64 + (k & 3) * 8, o0 + koff_mnmajor(k), C::kIdAcc,
                       k == 0 ? acc0 : 1u);
            }
            mma_commit(&bars->dv_done);
            // dQ partial (dQ = dS K, or dQ^T = K^T dS^T for a row-major accumulator)
            if (!mbar_wait(&bars->ds_full, s & 1, wc, 17)) { ok = false; break; }
            if (HD == 64 && s > 0 && !mbar_wait(&bars->dq_empty, (s - 1) & 1, wc, 18)) { ok = false; break; }
            tc_fence_after();
            // dQ = dS K (lanes = Q rows) for a chunk-major accumulator,
            // dQ^T = K^T dS^T (lanes = d) for a row-major one
            if (kCM) {
#pragma unroll
              for (int k = 0; k < kTile / 16; ++k)
                mma_ss(tDQ, dDS_mn + koff_mnmajor(k), dK_mn + koff_mnmajor(k), C::kIdDQ, k > 0);
            } else {
#pragma unroll
              for (int k = 0; k < kTile / 16; ++k)
                mma_ss(tDQ, dK_mn + koff_mnmajor(k), dDS_mn + koff_mnmajor(k), C::kIdDQ, k > 0);
            }
            mma_commit(&bars->dq_full);
            // dK += dS^T Q
            {
              const uint64_t q0 = dQ_mn0 + (uint64_t)stage * kStageOff;
              const uint32_t acc0 = st.chain_first ? 0u : 1u;
#pragma unroll
              for (int k = 0; k < kTile / 16; ++k)
                mma_ss(tDK, dDS_k + koff_kmajor(k, 128), q0 + koff_mnmajor(k), C::kIdAcc, k == 0 ? acc0 : 1u);
            }
            mma_commit(&bars->q_empty[stage]);
            mma_commit(&bars->ds_free);
            if (st.chain_last) {
              mma_commit(&bars->acc_full);
              mma_commit(&bars->kv_empty);
              ++chain;
            }
          }
          ++s;
        }
      }
      // Teardown: wait until every MMA this thread issued has completed.
      uint64_t* dr = fwd ? &bars->drain : &bars->drain2;
      mma_commit(dr);
      drain_wait(dr, 0, p.hdr, p.timeout_ns, fwd ? 3 : 4);
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------ dQ publisher
    // Ordered schedules only (ATOMIC has no semaphores: this warp just
    // follows the units).  Every reducer warp arrives (release, CTA scope)
    // on pub_full after a warp barrier behind its adds of a step; this warp
    // acquires that phase and then, per eighth (lane k: eighth k), stores
    // rank + 1 with a gpu-scope release.  Release is cumulative: the adds
    // ordered before the arrive that the acquire observed are ordered before
    // the semaphore store for whoever acquires it.  So the reducer warps do
    // not wait for their adds to be performed before draining and adding the
    // next partial.  (Without the release the dQ bits changed between runs.)
    const uint2* slots = reinterpret_cast<const uint2*>(smem + C::kOffPub);
    int s = 0, uidx = 0;
    bool ok = true;
    while (ok) {
      const int slot = uidx & 1;
      if (!warp_wait(&bars->unit_full[slot], (uidx >> 1) & 1, wc, 51)) break;
      const int U = misc->ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->unit_empty[slot]);
      ++uidx;
      if (U < 0) break;
      const int steps = k_unit_steps(p, U % p.units_per_head);
      for (int t = 0; t < steps; ++t) {
        if (deterministic) {
          if (!warp_wait(&bars->pub_full[s & 1], (s >> 1) & 1, wc, 53)) { ok = false; break; }
          if (lane < kSubTiles) {
            const uint2 e = slots[(s & 1) * kSubTiles + lane];
            // a release store: the reducers' adds precede it in causality
            // order (their CTA-scope release, this warp's acquire), so it
            // publishes them at gpu scope without a separate fence
            st_release_gpu(p.sem + e.x, e.y);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->pub_empty[s & 1]);
        }
        ++s;
      }
    }
  } else if (warp >= kSoftmaxWarp0 && warp < kReducerWarp0) {
    // ------------------------------------------------------ softmax / dS
    // Two warpgroups; warpgroup h owns Q columns 64h .. 64h+63 of the tile.
    const int h = (warp - kSoftmaxWarp0) >> 2;
    const int quad = warp & 3;                 // tensor-memory lane quadrant
    const int r = quad * 32 + lane;            // KV row of the tile
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    uint8_t* sds = smem + C::kOffDS + h * 16384;
    int s = 0, chain = 0, uidx = 0;
    bool ok = true;
    while (ok) {
      const int slot = uidx & 1;
      if (!warp_wait(&bars->unit_full[slot], (uidx >> 1) & 1, wc, 30)) break;
      const int U = misc->ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->unit_empty[slot]);
      ++uidx;
      if (U < 0) break;
      const int bh = U / p.units_per_head, u = U % p.units_per_head;
      const int steps = k_unit_steps(p, u);
      if (steps == 0) {
        // A KV tile that no visible Q tile meets (block mask): dK = dV = 0.
        if (!kRagged || u * kTile + r < p.S) {
          const size_t row = (size_t)bh * p.S + (size_t)u * kTile + r;
          uint4* dst = reinterpret_cast<uint4*>((h == 0 ? p.dv : p.dk) + row * HD);
#pragma unroll
          for (int c = 0; c < HD / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      for (int t = 0; t < steps; ++t) {
        const Step st = k_step(p, u, t, steps);
        const int stage = s & 1;
        const float* lse = s_lse + stage * 128 + 64 * h;
        const float* dd = s_dd + stage * 128 + 64 * h;
        const bool diag = (p.mask == kMaskCausal) && (st.kv == st.q);
        // a key past the end of a partial last tile: its whole P row is 0
        // (applied to the packed words below; `key_out` only on such a tile)
        const bool key_out = (st.kv * kTile + r) >= p.S;
        const bool tail_kv = kRagged && (st.kv + 1) * kTile > p.S;  // uniform: a partial last KV tile
        if (!warp_wait(&bars->q_full[stage], (s >> 1) & 1, wc, 31)) { ok = false; break; }
        if (!warp_wait(&bars->s_full, s & 1, wc, 32)) { ok = false; break; }
        tc_fence_after();
        // P^T = exp2(S^T * scale*log2(e) - LSE*log2(e)), bf16 pairs written
        // over the columns this warpgroup has just read.  The stored values
        // are -LSE*log2(e), so each pair of columns is one packed fma.
        uint32_t pk[32];
        const unsigned long long c2 = f32x2_pack(p.scale_log2e, p.scale_log2e);
        // the loop in two copies, so that off-diagonal steps run it with no
        // per-element test or branch
        auto p_phase = [&](auto diag_tag) {
          constexpr bool kDiag = decltype(diag_tag)::value;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t v[32];
            tmem_ld32(tbase + lane_off + C::kColS + 64 * h + 32 * c, v);
            uint32_t w16[16];
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const int col = 32 * c + e;          // column within this half
              const float4 l4 = *reinterpret_cast<const float4*>(lse + col);
              float x0, x1, x2, x3;
              f32x2_unpack(fma_f32x2(f32x2_pack(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), c2,
                                     f32x2_pack(l4.x, l4.y)), x0, x1);
              f32x2_unpack(fma_f32x2(f32x2_pack(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3])), c2,
                                     f32x2_pack(l4.z, l4.w)), x2, x3);
              float p0 = ex2_approx(x0);
              float p1 = ex2_approx(x1);
              float p2 = ex2_approx(x2);
              float p3 = ex2_approx(x3);
              if (kDiag) {
                const int qc = 64 * h + col;       // Q column within the tile
                p0 = (r > qc) ? 0.f : p0;
                p1 = (r > qc + 1) ? 0.f : p1;
                p2 = (r > qc + 2) ? 0.f : p2;
                p3 = (r > qc + 3) ? 0.f : p3;
              }
              w16[e >> 1] = pack_bf16x2(p0, p1);
              w16[(e >> 1) + 1] = pack_bf16x2(p2, p3);
              pk[16 * c + (e >> 1)] = w16[e >> 1];
              pk[16 * c + (e >> 1) + 1] = w16[(e >> 1) + 1];
            }
            if (tail_kv && key_out) {
#pragma unroll
              for (int x = 0; x < 16; ++x) {
                w16[x] = 0u;
                pk[16 * c + x] = 0u;
              }
            }
            tmem_st16_nowait(tbase + lane_off + C::kColS + 64 * h + 16 * c, w16);
          }
        };
        if (diag) p_phase(std::true_type{});
        else p_phase(std::false_type{});
        tmem_st_wait_all();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full);
        // dS^T = P^T o (dP^T - D) -> shared memory block h (bf16, 128B-swizzled)
        if (!warp_wait(&bars->dp_full, s & 1, wc, 33)) { ok = false; break; }
        if (s > 0 && !warp_wait(&bars->ds_free, (s - 1) & 1, wc, 34)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[16];
          tmem_ld16(tbase + lane_off + C::kColDP + 64 * h + 16 * c, v);
          uint32_t w8[8];
#pragma unroll
          for (int e = 0; e < 16; e += 4) {
            const int col = 16 * c + e;
            const float4 d4 = *reinterpret_cast<const float4*>(dd + col);
            const uint32_t pa = pk[8 * c + (e >> 1)], pb = pk[8 * c + (e >> 1) + 1];
            float ds0, ds1, ds2, ds3;
            f32x2_unpack(mul_f32x2(f32x2_pack(__uint_as_float(pa << 16), __uint_as_float(pa & 0xFFFF0000u)),
                                   sub_f32x2(f32x2_pack(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                                             f32x2_pack(d4.x, d4.y))), ds0, ds1);
            f32x2_unpack(mul_f32x2(f32x2_pack(__uint_as_float(pb << 16), __uint_as_float(pb & 0xFFFF0000u)),
                                   sub_f32x2(f32x2_pack(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3])),
                                             f32x2_pack(d4.z, d4.w))), ds2, ds3);
            w8[e >> 1] = pack_bf16x2(ds0, ds1);
            w8[(e >> 1) + 1] = pack_bf16x2(ds2, ds3);
          }
          uint8_t* rowp = sds + r * 128;
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            const int cc = c * 2 + m;            // 16-byte chunk of the 128-byte row
            *reinterpret_cast<uint4*>(rowp + ((cc ^ (r & 7)) << 4)) =
                make_uint4(w8[4 * m], w8[4 * m + 1], w8[4 * m + 2], w8[4 * m + 3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars->ds_full);
          mbar_arrive(&bars->q_empty[stage]);
        }
        if (st.chain_last) {
          // Epilogue: warpgroup 0 writes dV_i = bf16(dV acc), warpgroup 1
          // writes dK_i = bf16(scale * dK acc).
          if (!warp_wait(&bars->acc_full, chain & 1, wc, 35)) { ok = false; break; }
          tc_fence_after();
          const size_t row = (size_t)bh * p.S + (size_t)st.kv * kTile + r;
          const bool row_in = !kRagged || st.kv * kTile + r < p.S;  // rows of a partial last tile
          __nv_bfloat16* out = (h == 0 ? p.dv : p.dk) + row * HD;
          const uint32_t col0 = (h == 0) ? C::kColDV : C::kColDK;
          const float sc = (h == 0) ? 1.0f : p.scale;
#pragma unroll
          for (int c = 0; c < HD / 16; ++c) {
            uint32_t v[16];
            tmem_ld16(tbase + lane_off + col0 + 16 * c, v);
            uint4* dst = reinterpret_cast<uint4*>(out + 16 * c);
#pragma unroll
            for (int m = 0; m < 2; ++m)
              if (row_in) dst[m] = make_uint4(
                  pack_bf16x2(sc * __uint_as_float(v[8 * m]), sc * __uint_as_float(v[8 * m + 1])),
                  pack_bf16x2(sc * __uint_as_float(v[8 * m + 2]), sc * __uint_as_float(v[8 * m + 3])),
                  pack_bf16x2(sc * __uint_as_float(v[8 * m + 4]), sc * __uint_as_float(v[8 * m + 5])),
                  pack_bf16x2(sc * __uint_as_float(v[8 * m + 6]), sc * __uint_as_float(v[8 * m + 7])));
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->acc_empty);
          ++chain;
        }
        ++s;
      }
    }
  } else if (warp >= kReducerWarp0) {
    // ------------------------------------------------------ dQ reducer
    // Two warpgroups, eight warps.  Warp (half, quad) drains its half of its
    // tensor-memory quadrant of the dQ partial into registers at once (so
    // the tensor memory is free for the next partial), then adds that
    // eighth of the tile into the f32 accumulator:
    //   chunk-major (dQ, lanes = Q rows): Q row 32*quad + lane, d columns
    //     (d/2)*half .. + d/2 - 1; each add is 16 bytes into the tile
    //     [d/4][128][4], a warp's 32 rows of a chunk are 512 contiguous bytes;
    //   row-major (atomic at d = 128; dQ^T, lanes = d): d index
    //     32*quad + lane, Q rows 64*half .. + 63; each add is one float, a
    //     warp's 32 adds of a row are 128 contiguous bytes.
    // For the ordered schedules every eighth of every accumulation buffer has
    // its own semaphore, so consecutive contributors to one dQ tile overlap
    // on different eighths and buffers while each element of a buffer still
    // receives its partial sums in rank order.  A buffer's first contribution
    // stores.  The release after the adds is the publisher's (warp 3).
    const int quad = warp & 3;                          // tensor-memory lane quadrant
    const int half = (warp - kReducerWarp0) >> 2;
    const int sub = half * 4 + quad;                    // sub-tile / semaphore index
    const int r = quad * 32 + lane;                     // Q row (chunk-major) or d index (row-major)
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    constexpr int kVals = (HD == 128) ? 64 : 32;        // values per thread per step
    uint2* slots = reinterpret_cast<uint2*>(smem + C::kOffPub);
    int s = 0, uidx = 0;
    bool ok = true;
    while (ok) {
      const int slot = uidx & 1;
      if (!warp_wait(&bars->unit_full[slot], (uidx >> 1) & 1, wc, 40)) break;
      const int U = misc->ring[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->unit_empty[slot]);
      ++uidx;
      if (U < 0) break;
      const int bh = U / p.units_per_head, u = U % p.units_per_head;
      const int steps = k_unit_steps(p, u);
      for (int t = 0; t < steps; ++t) {
        const Step st = k_step(p, u, t, steps);
        // everything but the values is computed before the drain
        // rank r -> buffer r mod ways, position r / ways within that buffer
        const int rank = deterministic ? k_rank(p, st.kv, st.q) : 0;
        const int way = rank % p.acc_ways, lrank = rank / p.acc_ways;
        const size_t sem_idx = (((size_t)bh * p.N + st.q) * kSubTiles + sub) * p.acc_ways + way;
        const bool store = deterministic && lrank == 0;  // a buffer's first contribution overwrites
        float* acc = p.dqacc + (size_t)way * (size_t)p.acc_stride;
        // chunk-major: this thread's row in its first chunk; row-major
        // (atomic, d = 128): this thread's column of Q rows 64*half ..
        constexpr bool cm = kCM;
        const size_t row0 = (size_t)bh * p.S + (size_t)st.q * kTile;
        float* base = cm ? acc + (((size_t)(bh * p.N + st.q) * C::kChunks + (size_t)half * (C::kChunks / 2)) * kTile + r) * 4
                         : acc + (row0 + (size_t)half * 64) * HD + r;
        // Rows past the end of a partial last Q tile: in a chunk-major tile
        // they lie in the tile's padding; in the row-major accumulator they
        // belong to the next head and are never touched (their partial sums
        // are zero).
        const int row_lim = p.S - st.q * kTile - half * 64;
        const int nvalid = !kRagged ? 64 : (row_lim < 0 ? 0 : (row_lim > 64 ? 64 : row_lim));
        if (!warp_wait(&bars->dq_full, s & 1, wc, 41)) { ok = false; break; }
        tc_fence_after();
        // d = 64: the first poll of this step's semaphore is in flight during
        // the drain.  (At d = 128 the drain frees dP's columns, and an acquire
        // ahead of it delays the drain: 1-5 % slower there, 2-4 % faster here.)
        uint32_t first = 0xFFFFFFFFu;
        if (HD == 64 && deterministic && lane == 0) first = ld_acquire_gpu(p.sem + sem_idx);
        uint32_t v[kVals];
#pragma unroll
        for (int c = 0; c < kVals / 32; ++c)
          tmem_ld32(tbase + lane_off + C::kColDQ + (uint32_t)(half * kVals + 32 * c),
                    *reinterpret_cast<uint32_t(*)[32]>(&v[32 * c]));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->dq_empty);
        if (deterministic) {
          int g = 1;
          if (lane == 0)
            g = (first == (uint32_t)lrank || sem_wait(p.sem + sem_idx, (uint32_t)lrank, wc, (uint32_t)sem_idx)) ? 1 : 0;
          g = __shfl_sync(0xffffffffu, g, 0);
          if (!g) { ok = false; break; }
          // Lane 0's acquire observed the previous rank's release; the warp
          // barrier orders that acquire before every lane's adds (or, with
          // DAB_BWD_PLAIN_ADD, loads), so each lane sees the previous rank's
          // sums and adds after them.
          __syncwarp();
        }
        // one straight-line loop per kind of add (no per-element branch)
        if (HD == 128 && !cm) {
          // row-major (atomic only): a warp's 32 adds of a row are 128
          // contiguous bytes
#pragma unroll
          for (int q = 0; q < 64; ++q)
            if (q < nvalid) red_add_f32(base + (size_t)q * HD, __uint_as_float(v[q]));
        } else {
          if (store) {
#pragma unroll
            for (int m = 0; m < kVals / 4; ++m)
              *reinterpret_cast<float4*>(base + (size_t)m * (kTile * 4)) =
                  make_float4(__uint_as_float(v[4 * m]), __uint_as_float(v[4 * m + 1]),
                              __uint_as_float(v[4 * m + 2]), __uint_as_float(v[4 * m + 3]));
          } else if (deterministic && p.plain_add) {
            // load + add + store: the same IEEE adds in the same order as the
            // red (only this contributor touches the sub-tile now); four
            // loads in flight before their stores
#pragma unroll
            for (int m0 = 0; m0 < kVals / 4; m0 += 4) {
              float4 b[4];
#pragma unroll
              for (int m = 0; m < 4; ++m) b[m] = ld_cg_v4_f32(base + (size_t)(m0 + m) * (kTile * 4));
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                const int e = 4 * (m0 + m);
                *reinterpret_cast<float4*>(base + (size_t)(m0 + m) * (kTile * 4)) =
                    make_float4(b[m].x + __uint_as_float(v[e]), b[m].y + __uint_as_float(v[e + 1]),
                                b[m].z + __uint_as_float(v[e + 2]), b[m].w + __uint_as_float(v[e + 3]));
              }
            }
          } else {
#pragma unroll
            for (int m = 0; m < kVals / 4; ++m)
              red_add_v4_f32(base + (size_t)m * (kTile * 4), __uint_as_float(v[4 * m]), __uint_as_float(v[4 * m + 1]),
                             __uint_as_float(v[4 * m + 2]), __uint_as_float(v[4 * m + 3]));
          }
        }
        if (deterministic) {
          // Hand the release of rank + 1 to the publisher.  The warp barrier
          // orders every lane's adds before lane 0's arrive (release, CTA
          // scope), so one arrive per warp carries the whole warp's adds
          // (256 arrives per step cost 1 % more).  The slot of this parity
          // is free once the publisher has released step s - 2.
          if (s >= 2 && !warp_wait(&bars->pub_empty[s & 1], ((s >> 1) - 1) & 1, wc, 44)) { ok = false; break; }
          if (lane == 0) slots[(s & 1) * kSubTiles + sub] = make_uint2((uint32_t)sem_idx, (uint32_t)lrank + 1u);
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->pub_full[s & 1]);
        }
        ++s;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
  // The tail convert reads chunk-major tiles: only the ordered schedules set
  // fuse_convert, and they always run a kCM instance.  (It is compiled into
  // the row-major instance too: without it that instance ran 3 % slower.)
  if (p.fuse_convert) tail_convert<HD, kRagged>(p, misc, smem, wc);
}

}  // namespace

template <int HD>
int bwd_smem_bytes() {
  return Cfg<HD>::kSmemBytes;
}

template <int HD>
const void* bwd_kernel_ptr(bool ragged, bool chunk_major) {
  static_assert(HD == 64 || HD == 128, "head dim");
  if (HD == 64 || chunk_major)
    return ragged ? reinterpret_cast<const void*>(&bwd_kernel<HD, true, true>)
                  : reinterpret_cast<const void*>(&bwd_kernel<HD, false, true>);
  return ragged ? reinterpret_cast<const void*>(&bwd_kernel<HD, true, (HD == 64)>)
                : reinterpret_cast<const void*>(&bwd_kernel<HD, false, (HD == 64)>);
}

template int bwd_smem_bytes<64>();
template int bwd_smem_bytes<128>();
template const void* bwd_kernel_ptr<64>(bool, bool);
template const void* bwd_kernel_ptr<128>(bool, bool);

}  // namespace dab
