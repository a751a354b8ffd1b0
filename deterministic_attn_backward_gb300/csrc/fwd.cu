// fwd.cu -- attention forward for GB300 (sm_103a): O = softmax(scale Q K^T) V
// and LSE, the inputs the backward pass consumes.
//
// One CTA per (head, 128-row Q tile), two passes over the visible KV tiles:
//   pass 1: S = Q K_c^T on the tensor cores; per Q row the maximum and the
//           sum of exp2(scale*log2(e) S - max) (online update) -> LSE;
//   pass 2: S again, P = exp2(scale*log2(e) S - LSE*log2(e)) in bf16 written
//           over the S columns just read, O += P V_c on the tensor cores.
// Recomputing S once avoids rescaling the O accumulator.  S is double
// buffered in tensor memory, so the tensor cores compute the next tile's S
// while the softmax warps work on the current one.  Two softmax warpgroups
// take 64 key columns of every tile each (thread = Q row); their running
// (max, sum) pairs are combined once, through shared memory, at the end of
// pass 1.
// With a block mask, KV tiles whose flag is zero are skipped by every role;
// a Q tile with no visible KV tile gets O = 0 and LSE = -infinity.
// Warps: 0 TMA producer, 1 MMA issuer, 4-11 softmax.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"
#include "tile_sched.h"

namespace dab {

__device__ WsHeader g_fwd_status;  // status word when the caller gives no workspace

namespace {

constexpr int kFwdThreads = 384;
constexpr int kFwdSoftmaxWarp0 = 4;  // warps 4-7: key columns 0-63, 8-11: 64-127
constexpr int kFwdSoftmaxWarps = 8;
// The barrier counts (s_free, p_full) and the named barrier of the (max, sum)
// combine expect exactly these warps: the block must hold all of them.
static_assert(kFwdThreads == 32 * (kFwdSoftmaxWarp0 + kFwdSoftmaxWarps), "forward warp roles");
constexpr float kLn2 = 0.6931471805599453f;

template <int HD>
struct FCfg {
  static constexpr int kTileBytes = kTile * HD * 2;
  static constexpr int kBlockBytes = kTile * 128;
  static constexpr int kOffQ = 0;
  static constexpr int kStages = 3;              // K, V tiles in flight
  static constexpr int kOffK = kTileBytes;       // kStages stages
  static constexpr int kOffV = (1 + kStages) * kTileBytes;
  static constexpr int kOffBar = (1 + 2 * kStages) * kTileBytes;
  static constexpr int kOffMisc = kOffBar + 256;
  static constexpr int kOffStat = kOffMisc + 16;  // [2 warpgroups][128 rows] (max, sum)
  static constexpr int kSmemBytes = kOffStat + 2 * 128 * 8;
  // Tensor memory: two S buffers (P written over the S columns just read),
  // then the O accumulator.
  static constexpr uint32_t kColS = 0;             // buffer b at kColS + 128 b
  static constexpr uint32_t kColO = 256;
  static constexpr uint32_t kIdS = idesc_bf16(128, 128, 0, 0);   // S = Q K^T
  static constexpr uint32_t kIdO = idesc_bf16(128, HD, 0, 1);    // O += P V
};

struct FBars {
  uint64_t q_full;
  uint64_t kv_full[3], kv_empty[3];
  uint64_t s_full[2];   // S of a tile in buffer b (MMA commit)
  uint64_t s_free[2];   // pass 1: the softmax warps have read buffer b
  uint64_t p_full[2];   // pass 2: P written over buffer b
  uint64_t o_done[2];   // pass 2: P V of buffer b completed
  uint64_t o_full, drain;
};
static_assert(sizeof(FBars) <= 256, "barrier block");

template <int HD>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_kernel(const __grid_constant__ FwdParams p,
                                                           WsHeader* hdr) {
  using C = FCfg<HD>;
  extern __shared__ __align__(1024) uint8_t smem[];
  FBars* bars = reinterpret_cast<FBars*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  int* abort_flag = reinterpret_cast<int*>(smem + C::kOffMisc + 4);
  float2* stat = reinterpret_cast<float2*>(smem + C::kOffStat);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (hdr == nullptr) hdr = &g_fwd_status;
  if ((sbase & 1023u) != 0u) {
    if (threadIdx.x == 0) raise_error(hdr, kStatusBounds, kDetailAlign);
    return;
  }
  const int bh = blockIdx.x / p.N, qi = blockIdx.x % p.N;
  const int nkv = (p.mask == kMaskCausal) ? qi + 1 : p.N;
  // KV tile c takes part unless the block mask hides it (uniform per CTA)
  auto visible = [&](int c) { return p.tiles == nullptr || p.tiles[(size_t)qi * p.N + c] != 0; };
  const unsigned long long timeout = 2000000000ull;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars->s_full[s], 1);
      mbar_init(&bars->s_free[s], kFwdSoftmaxWarps);
      mbar_init(&bars->p_full[s], kFwdSoftmaxWarps);
      mbar_init(&bars->o_done[s], 1);
    }
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  const WaitCtl wc{abort_flag, hdr, timeout};

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tensormap(&p.tm_q);
      prefetch_tensormap(&p.tm_k);
      prefetch_tensormap(&p.tm_v);
      mbar_arrive_expect_tx(&bars->q_full, C::kTileBytes);
      const int qrow = bh * p.S + qi * kTile;
#pragma unroll
      for (int db = 0; db < HD / 64; ++db)
        tma_load_2d(smem + C::kOffQ + db * C::kBlockBytes, &p.tm_q, &bars->q_full, db * 64, qrow);
      int it = 0, issued[C::kStages] = {};
      bool ok = true;
      for (int pass = 0; pass < 2 && ok; ++pass) {
        for (int c = 0; c < nkv; ++c) {
          if (!visible(c)) continue;
          const int st = it % C::kStages;
          if (it >= C::kStages && !mbar_wait(&bars->kv_empty[st], ((it / C::kStages) - 1) & 1, wc, 1)) { ok = false; break; }
          mbar_arrive_expect_tx(&bars->kv_full[st], (pass == 0 ? 1 : 2) * C::kTileBytes);
          const int krow = bh * p.S + c * kTile;
#pragma unroll
          for (int db = 0; db < HD / 64; ++db) {
            tma_load_2d(smem + C::kOffK + st * C::kTileBytes + db * C::kBlockBytes, &p.tm_k,
                        &bars->kv_full[st], db * 64, krow);
            if (pass == 1)
              tma_load_2d(smem + C::kOffV + st * C::kTileBytes + db * C::kBlockBytes, &p.tm_v,
                          &bars->kv_full[st], db * 64, krow);
          }
          ++issued[st];
          ++it;
        }
      }
      drain_wait(&bars->q_full, 0, hdr, timeout, 11);
      for (int st = 0; st < C::kStages; ++st)
        if (issued[st] > 0) drain_wait(&bars->kv_full[st], (issued[st] - 1) & 1, hdr, timeout, 12);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // Tile `it` (counted over both passes) uses KV stage and S buffer it & 1.
      // Before S overwrites a buffer, its previous use must be finished: the
      // softmax read it (pass 1: s_free) or P V read the P written over it
      // (pass 2: o_done).  In pass 2, S of the next tile is issued before P V
      // of the current one, so the tensor cores compute it while the softmax
      // warps form P.
      const uint32_t sQ = sbase + C::kOffQ;
      bool ok = mbar_wait(&bars->q_full, 0, wc, 20);
      int it = 0;
      int last_pass[2] = {-1, -1}, uses[2][2] = {{0, 0}, {0, 0}};  // uses[pass][buffer]
      int prev_it = -1;    // pass 2: the tile whose P V is still to issue
      int first2 = 0;      // index of the first pass-2 tile (its P V starts O)
      for (int pass = 0; pass < 2 && ok; ++pass) {
        if (pass == 1) first2 = it;
        for (int c = 0; c < nkv; ++c) {
          if (!visible(c)) continue;
          const int b = it & 1, st = it % C::kStages;
          const uint32_t sK = sbase + C::kOffK + st * C::kTileBytes;
          if (!mbar_wait(&bars->kv_full[st], (it / C::kStages) & 1, wc, 21)) { ok = false; break; }
          if (last_pass[b] == 0 && !mbar_wait(&bars->s_free[b], (uses[0][b] - 1) & 1, wc, 22)) { ok = false; break; }
          if (last_pass[b] == 1 && !mbar_wait(&bars->o_done[b], (uses[1][b] - 1) & 1, wc, 23)) { ok = false; break; }
          tc_fence_after();
          const uint32_t tS = tbase + C::kColS + 128u * b;
#pragma unroll
          for (int k = 0; k < HD / 16; ++k)
            mma_ss(tS, desc_kmajor(sQ, k, 128), desc_kmajor(sK, k, 128), C::kIdS, k > 0);
          mma_commit(&bars->s_full[b]);
          last_pass[b] = pass;
          ++uses[pass][b];
          if (pass == 0) mma_commit(&bars->kv_empty[st]);
          if (pass == 1 && prev_it >= 0) {  // P V of the previous tile
            const int pb = prev_it & 1;
            if (!mbar_wait(&bars->p_full[pb], (uses[1][pb] - 1) & 1, wc, 24)) { ok = false; break; }
            tc_fence_after();
            const int pst = prev_it % C::kStages;
            const uint32_t sV = sbase + C::kOffV + pst * C::kTileBytes;
            const uint32_t tP = tbase + C::kColS + 128u * pb;
#pragma unroll
            for (int k = 0; k < kTile / 16; ++k)
              mma_ts(tbase + C::kColO, tP + (k >> 2) * 64 + (k & 3) * 8, desc_mnmajor(sV, k, 128),
                     C::kIdO, !(prev_it == first2 && k == 0));
            mma_commit(&bars->o_done[pb]);
            mma_commit(&bars->kv_empty[pst]);
          }
          if (pass == 1) prev_it = it;
          ++it;
        }
      }
      if (ok && prev_it >= 0) {  // P V of the last tile
        const int pb = prev_it & 1;
        if (mbar_wait(&bars->p_full[pb], (uses[1][pb] - 1) & 1, wc, 25)) {
          tc_fence_after();
          const int pst = prev_it % C::kStages;
          const uint32_t sV = sbase + C::kOffV + pst * C::kTileBytes;
          const uint32_t tP = tbase + C::kColS + 128u * pb;
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k)
            mma_ts(tbase + C::kColO, tP + (k >> 2) * 64 + (k & 3) * 8, desc_mnmajor(sV, k, 128), C::kIdO,
                   !(prev_it == first2 && k == 0));
          mma_commit(&bars->o_done[pb]);
          mma_commit(&bars->kv_empty[pst]);
        } else {
          ok = false;
        }
      }
      if (ok) mma_commit(&bars->o_full);
      mma_commit(&bars->drain);
      drain_wait(&bars->drain, 0, hdr, timeout, 13);
    }
    __syncwarp();
  } else if (warp >= kFwdSoftmaxWarp0) {
    // Softmax: warpgroup h takes key columns 64 h .. 64 h + 63 of every tile;
    // thread = Q row r of the tile.
    const int h = (warp - kFwdSoftmaxWarp0) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const bool causal = (p.mask == kMaskCausal);
    float m = -INFINITY, l = 0.f;
    int it = 0, nvis = 0;
    bool ok = true;
    for (int c = 0; c < nkv && ok; ++c) {
      if (!visible(c)) continue;
      ++nvis;
      const int b = it & 1;
      if (!warp_wait(&bars->s_full[b], (it >> 1) & 1, wc, 30)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_off + C::kColS + 128u * b + 64 * h + 32 * ch, v);
        float x[32];
        float cmax = -INFINITY;
        // masks apply only on the causal diagonal tile and a partial last tile
        const bool masked = (causal && c == qi) || (c + 1) * kTile > p.S;
        if (masked) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int col = 64 * h + 32 * ch + e;
            x[e] = __uint_as_float(v[e]) * p.scale_log2e;
            if (causal && c == qi && col > r) x[e] = -INFINITY;
            if (c * kTile + col >= p.S) x[e] = -INFINITY;   // past the end of a partial last tile
            cmax = fmaxf(cmax, x[e]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            x[e] = __uint_as_float(v[e]) * p.scale_log2e;
            cmax = fmaxf(cmax, x[e]);
          }
        }
        // A half row may have seen no visible key yet (its keys all masked):
        // then the sum stays exactly 0 (no -inf - -inf).
        const float mn = fmaxf(m, cmax);
        const float base = (mn == -INFINITY) ? 0.f : mn;
        float sum = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) sum += ex2_approx(x[e] - base);
        l = l * ex2_approx(m - base) + sum;
        m = mn;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_free[b]);
      ++it;
    }
    // Combine the two warpgroups' (max, sum) of each row.  Every softmax warp
    // reaches this barrier, also after a failed wait.
    stat[h * 128 + r] = make_float2(m, l);
    named_bar_sync(1, 32 * kFwdSoftmaxWarps);
    const float2 s0 = stat[r], s1 = stat[128 + r];
    const float mt = fmaxf(s0.x, s1.x);
    float lse2 = -INFINITY;
    if (mt != -INFINITY) {
      const float lt = s0.y * ex2_approx(s0.x - mt) + s1.y * ex2_approx(s1.x - mt);
      lse2 = mt + __log2f(lt);
    }
    for (int c = 0; c < nkv && ok; ++c) {
      if (!visible(c)) continue;
      const int b = it & 1;
      if (!warp_wait(&bars->s_full[b], (it >> 1) & 1, wc, 31)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tS = tbase + lane_off + C::kColS + 128u * b + 64 * h;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t v[32];
        tmem_ld32(tS + 32 * ch, v);
        uint32_t w16[16];
        const bool masked = (causal && c == qi) || (c + 1) * kTile > p.S;
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int col = 64 * h + 32 * ch + e;
          float p0 = ex2_approx(fmaf(__uint_as_float(v[e]), p.scale_log2e, -lse2));
          float p1 = ex2_approx(fmaf(__uint_as_float(v[e + 1]), p.scale_log2e, -lse2));
          if (masked) {
            if (causal && c == qi) {
              if (col > r) p0 = 0.f;
              if (col + 1 > r) p1 = 0.f;
            }
            if (c * kTile + col >= p.S) p0 = 0.f;
            if (c * kTile + col + 1 >= p.S) p1 = 0.f;
          }
          w16[e >> 1] = pack_bf16x2(p0, p1);
        }
        // P over the columns this thread has read (packed: 16 words per 32 keys)
        tmem_st16_nowait(tS + 16 * ch, w16);
      }
      tmem_st_wait_all();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[b]);
      ++it;
    }
    if (ok && warp_wait(&bars->o_full, 0, wc, 33)) {
      tc_fence_after();
      const size_t row = (size_t)bh * p.S + (size_t)qi * kTile + r;
      const bool row_in = qi * kTile + r < p.S;  // rows of a partial last tile
#pragma unroll
      for (int ch = 0; ch < HD / 64; ++ch) {    // this warpgroup's half of the O columns
        const int col0 = h * (HD / 2) + 32 * ch;
        uint32_t v[32];
        tmem_ld32(tbase + lane_off + C::kColO + col0, v);
        if (nvis == 0) {  // nothing visible: O = 0 (the accumulator was never written)
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        uint4* dst = reinterpret_cast<uint4*>(p.o + row * HD + col0);
#pragma unroll
        for (int mm = 0; mm < 4; ++mm)
          if (row_in) dst[mm] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * mm]), __uint_as_float(v[8 * mm + 1])),
                               pack_bf16x2(__uint_as_float(v[8 * mm + 2]), __uint_as_float(v[8 * mm + 3])),
                               pack_bf16x2(__uint_as_float(v[8 * mm + 4]), __uint_as_float(v[8 * mm + 5])),
                               pack_bf16x2(__uint_as_float(v[8 * mm + 6]), __uint_as_float(v[8 * mm + 7])));
      }
      if (row_in && h == 0) p.lse[row] = lse2 * kLn2;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace

int fwd_threads() { return kFwdThreads; }

template <int HD>
int fwd_smem_bytes() {
  return FCfg<HD>::kSmemBytes;
}
template <int HD>
const void* fwd_kernel_ptr() {
  return reinterpret_cast<const void*>(&fwd_kernel<HD>);
}
template int fwd_smem_bytes<64>();
template int fwd_smem_bytes<128>();
template const void* fwd_kernel_ptr<64>();
template const void* fwd_kernel_ptr<128>();

}  // namespace dab
