// fwd.cu -- attention forward for GB300 (sm_103a): O = softmax(scale Q K^T) V
// and LSE, the inputs the backward pass consumes.
//
// One pass over the visible KV tiles with an online softmax.  A CTA owns two
// 128-row Q tiles of one head, A = 2p and B = 2p + 1 (B absent when the head
// has an odd number of tiles), and walks the KV tiles either of them sees; K
// and V are loaded once for both.  Per Q tile X and KV tile c the tensor
// cores compute S_X = Q_X K_c^T into tensor memory, the softmax warpgroup of
// X turns it into P (bf16, written over the S columns) and the tensor cores
// accumulate O_X += P V_c in tensor memory.  The two Q tiles alternate on the
// tensor cores, so the softmax of one overlaps the products of the other.
//
// Online softmax (thread = Q row, all 128 key columns of the tile): the row
// keeps m, the running maximum used as the exponent offset, and l, the sum
// of exp2(x - m) over the keys so far (x = scale*log2(e) * s).  When a tile
// raises the row maximum by more than kRescale (in log2 units) or m is still
// -infinity, the thread rescales its O row and l by exp2(m - m_new) and takes
// m = m_new; otherwise P may exceed 1 by up to 2^kRescale, which bf16 and the
// f32 accumulators hold without loss.  O and l share the scale history, so
// O / l and LSE = (m + log2 l) ln 2 are exact up to rounding.
//
// Warps: 0 TMA producer, 1 MMA issuer, 4-7 softmax of Q tile A, 8-11 softmax
// of Q tile B.  Tensor memory: S_A 0-127, S_B 128-255, O_A and O_B from 256.
// With a block mask each Q tile skips the KV tiles its flags hide; a Q tile
// with no visible KV tile gets O = 0 and LSE = -infinity.
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
constexpr int kFwdSoftmaxWarp0 = 4;  // warps 4-7: Q tile A, warps 8-11: Q tile B
constexpr int kFwdSoftmaxWarps = 8;
static_assert(kFwdThreads == 32 * (kFwdSoftmaxWarp0 + kFwdSoftmaxWarps), "forward warp roles");
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescale = 8.0f;     // log2 units: P stays below 2^8

template <int HD>
struct FCfg {
  static constexpr int kTileBytes = kTile * HD * 2;
  static constexpr int kBlockBytes = kTile * 128;
  static constexpr int kStages = (HD == 128) ? 2 : 3;  // K, V tiles in flight
  static constexpr int kOffQ = 0;                       // Q_A, Q_B
  static constexpr int kOffK = 2 * kTileBytes;
  static constexpr int kOffV = (2 + kStages) * kTileBytes;
  static constexpr int kOffBar = (2 + 2 * kStages) * kTileBytes;
  static constexpr int kOffMisc = kOffBar + 256;
  static constexpr int kSmemBytes = kOffMisc + 16;
  static constexpr uint32_t kColS = 0;                  // Q tile x at kColS + 128 x
  static constexpr uint32_t kColO = 256;                // Q tile x at kColO + HD x
  static constexpr uint32_t kIdS = idesc_bf16(128, 128, 0, 0);   // S = Q K^T
  static constexpr uint32_t kIdO = idesc_bf16(128, HD, 0, 1);    // O += P V
};

struct FBars {
  uint64_t q_full;
  uint64_t kv_full[3], kv_empty[3];
  uint64_t s_full[2];   // S of Q tile x (MMA commit)
  uint64_t p_full[2];   // P of Q tile x written (softmax warps)
  uint64_t o_done[2];   // P V of Q tile x completed (MMA commit)
  uint64_t drain;
};
static_assert(sizeof(FBars) <= 256, "barrier block");

// The CTA's pair of Q tiles: CTAs are ordered longest causal range first.
__device__ __forceinline__ void fwd_pair(const FwdParams& p, int& bh, int& qa, int& nq) {
  const int npairs = (p.N + 1) / 2;
  const int pr = npairs - 1 - (int)(blockIdx.x / p.BH);
  bh = (int)(blockIdx.x % p.BH);
  qa = 2 * pr;
  nq = (qa + 1 < p.N) ? 2 : 1;
}

template <int HD>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_kernel(const __grid_constant__ FwdParams p,
                                                           WsHeader* hdr) {
  using C = FCfg<HD>;
  extern __shared__ __align__(1024) uint8_t smem[];
  FBars* bars = reinterpret_cast<FBars*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  int* abort_flag = reinterpret_cast<int*>(smem + C::kOffMisc + 4);
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (hdr == nullptr) hdr = &g_fwd_status;
  if ((sbase & 1023u) != 0u) {
    if (threadIdx.x == 0) raise_error(hdr, kStatusBounds, kDetailAlign);
    return;
  }
  int bh, qa, nq;
  fwd_pair(p, bh, qa, nq);
  const bool causal = (p.mask == kMaskCausal);
  // KV tiles the CTA walks: those either Q tile may see
  const int nkv = causal ? qa + nq : p.N;
  // does Q tile x (0: A, 1: B) see KV tile c
  auto sees = [&](int x, int c) {
    const int qi = qa + x;
    if (x >= nq) return false;
    if (causal && c > qi) return false;
    return p.tiles == nullptr || p.tiles[(size_t)qi * p.N + c] != 0;
  };
  auto any = [&](int c) { return sees(0, c) || sees(1, c); };
  const unsigned long long timeout = 2000000000ull;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars->s_full[x], 1);
      mbar_init(&bars->p_full[x], 4);
      mbar_init(&bars->o_done[x], 1);
    }
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
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&p.tm_q);
      prefetch_tensormap(&p.tm_k);
      prefetch_tensormap(&p.tm_v);
      mbar_arrive_expect_tx(&bars->q_full, nq * C::kTileBytes);
      for (int x = 0; x < nq; ++x) {
        const int qrow = bh * p.S + (qa + x) * kTile;
#pragma unroll
        for (int db = 0; db < HD / 64; ++db)
          tma_load_2d(smem + C::kOffQ + x * C::kTileBytes + db * C::kBlockBytes, &p.tm_q, &bars->q_full,
                      db * 64, qrow);
      }
      int it = 0;
      for (int c = 0; c < nkv; ++c) {
        if (!any(c)) continue;
        const int st = it % C::kStages;
        if (it >= C::kStages && !mbar_wait(&bars->kv_empty[st], ((it / C::kStages) - 1) & 1, wc, 1)) break;
        mbar_arrive_expect_tx(&bars->kv_full[st], 2 * C::kTileBytes);
        const int krow = bh * p.S + c * kTile;
#pragma unroll
        for (int db = 0; db < HD / 64; ++db) {
          tma_load_2d(smem + C::kOffK + st * C::kTileBytes + db * C::kBlockBytes, &p.tm_k, &bars->kv_full[st],
                      db * 64, krow);
          tma_load_2d(smem + C::kOffV + st * C::kTileBytes + db * C::kBlockBytes, &p.tm_v, &bars->kv_full[st],
                      db * 64, krow);
        }
        ++it;
      }
      drain_wait(&bars->q_full, 0, hdr, timeout, 11);
      // stage st took loads it' = st, st + kStages, ... < it
#pragma unroll
      for (int st = 0; st < C::kStages; ++st) {
        const int issued = (it - st + C::kStages - 1) / C::kStages;
        if (issued > 0) drain_wait(&bars->kv_full[st], (issued - 1) & 1, hdr, timeout, 12);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Per KV tile c (the CTA's it-th): for each Q tile x that sees c, P V of
    // x, then, once that product has read P (it lies over S_x), S of x's
    // next tile when that is c + 1 (a later one is issued at the start of
    // its own iteration).  The products of A and B alternate on the tensor
    // cores, so one tile's softmax runs while the other's products do.
    if (lane == 0) {
      // per Q tile x (scalars, not arrays, so that they stay in registers):
      // P V products issued, and whether S of the tile x processes next is
      // already issued
      int cnt0 = 0, cnt1 = 0;
      bool rdy0 = false, rdy1 = false;
      bool ok = mbar_wait(&bars->q_full, 0, wc, 20);
      auto issue_s = [&](int x, int c, int st) {
        const uint32_t sQ = sbase + C::kOffQ + x * C::kTileBytes;
        const uint32_t sK = sbase + C::kOffK + st * C::kTileBytes;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k)
          mma_ss(tbase + C::kColS + 128u * x, desc_kmajor(sQ, k, 128), desc_kmajor(sK, k, 128), C::kIdS, k > 0);
        mma_commit(&bars->s_full[x]);
      };
      int it = 0;
      for (int c = 0; c < nkv && ok; ++c) {
        if (!any(c)) continue;
        const int st = it % C::kStages;
        if (!mbar_wait(&bars->kv_full[st], (it / C::kStages) & 1, wc, 21)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const int cx = x ? cnt1 : cnt0;
          if (!sees(x, c) || (x ? rdy1 : rdy0)) continue;
          // S_x is free once the previous P V of x has completed
          if (cx > 0 && !mbar_wait(&bars->o_done[x], (cx - 1) & 1, wc, 22)) { ok = false; break; }
          tc_fence_after();
          issue_s(x, c, st);
        }
        if (!ok) break;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          if (!sees(x, c)) continue;
          const int cx = x ? cnt1 : cnt0;
          if (!mbar_wait(&bars->p_full[x], cx & 1, wc, 23)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sV = sbase + C::kOffV + st * C::kTileBytes;
          const uint32_t tSx = tbase + C::kColS + 128u * x, tOx = tbase + C::kColO + (uint32_t)HD * x;
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k)
            mma_ts(tOx, tSx + k * 8, desc_mnmajor(sV, k, 128), C::kIdO, (cx > 0 || k > 0) ? 1u : 0u);
          mma_commit(&bars->o_done[x]);
          if (x) { ++cnt1; rdy1 = false; } else { ++cnt0; rdy0 = false; }
          // S of x's next tile right away when it is c + 1 (its K is loaded
          // or on its way: the stage of c + 1 was freed by iteration c - 1)
          if (c + 1 < nkv && sees(x, c + 1) && any(c + 1)) {
            const int st1 = (it + 1) % C::kStages;
            if (!mbar_wait(&bars->kv_full[st1], ((it + 1) / C::kStages) & 1, wc, 24)) { ok = false; break; }
            if (!mbar_wait(&bars->o_done[x], cx & 1, wc, 25)) { ok = false; break; }
            tc_fence_after();
            issue_s(x, c + 1, st1);
            if (x) rdy1 = true; else rdy0 = true;
          }
        }
        if (!ok) break;
        mma_commit(&bars->kv_empty[st]);
        ++it;
      }
      mma_commit(&bars->drain);
      drain_wait(&bars->drain, 0, hdr, timeout, 13);
    }
    __syncwarp();
  } else if (warp >= kFwdSoftmaxWarp0) {
    // ------------------------------------------------------------ softmax
    // Warpgroup x owns Q tile x; thread = Q row r, all 128 key columns.
    const int x = (warp - kFwdSoftmaxWarp0) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const int qi = qa + x;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    const uint32_t tS = tbase + lane_off + C::kColS + 128u * x;
    const uint32_t tO = tbase + lane_off + C::kColO + (uint32_t)HD * x;
    float m = -INFINITY, l = 0.f;
    int cnt = 0;
    bool ok = (x < nq);
    const unsigned long long c2 = f32x2_pack(p.scale_log2e, p.scale_log2e);
    for (int c = 0; c < nkv && ok; ++c) {
      if (!sees(x, c)) continue;
      if (!warp_wait(&bars->s_full[x], cnt & 1, wc, 30)) { ok = false; break; }
      tc_fence_after();
      // x = scale*log2(e) * s for the 128 keys (all four loads in flight
      // before one wait), -infinity where hidden: keys after the query on the
      // causal diagonal tile, keys past S on a partial last tile
      uint32_t v[128];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) tmem_ld32_nowait(tS + 32 * ch, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * ch]));
      tmem_ld_wait();
      const bool masked = (causal && c == qi) || (c + 1) * kTile > p.S;
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
      // two copies of the loop, so that the tiles without hidden keys run
      // straight-line code with no per-element test or branch
      if (!masked) {
#pragma unroll
        for (int e = 0; e < 128; e += 2) {
          float a, b;
          f32x2_unpack(mul_f32x2(f32x2_pack(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), c2), a, b);
          v[e] = __float_as_uint(a);
          v[e + 1] = __float_as_uint(b);
          mx[(e >> 1) & 7] = fmaxf(mx[(e >> 1) & 7], fmaxf(a, b));
        }
      } else {
        const int lim = min((causal && c == qi) ? r + 1 : kTile, p.S - c * kTile);  // keys < lim visible
#pragma unroll
        for (int e = 0; e < 128; e += 2) {
          float a, b;
          f32x2_unpack(mul_f32x2(f32x2_pack(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), c2), a, b);
          a = (e < lim) ? a : -INFINITY;
          b = (e + 1 < lim) ? b : -INFINITY;
          v[e] = __float_as_uint(a);
          v[e + 1] = __float_as_uint(b);
          mx[(e >> 1) & 7] = fmaxf(mx[(e >> 1) & 7], fmaxf(a, b));
        }
      }
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      // rescale when the maximum grew past the allowance (warp-uniform: the
      // tensor-memory accesses are warp-collective; a lane that does not need
      // it rescales by its own factor, which is also exact)
      const bool need = (mt > m + kRescale) || (m == -INFINITY && mt != -INFINITY);
      if (__any_sync(0xffffffffu, need)) {
        const float mn = fmaxf(m, mt);
        const float alpha = (m == -INFINITY) ? 0.f : ex2_approx(m - mn);
        l *= alpha;
        if (cnt > 0) {
          // P V of the previous tile completed before S of this one was
          // issued (the S columns held its P), so O is stable here
          const unsigned long long a2 = f32x2_pack(alpha, alpha);
#pragma unroll 1
          for (int ch = 0; ch < HD / 8; ++ch) {
            uint32_t o[8];
            tmem_ld8(tO + 8 * ch, o);
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              float a, b;
              f32x2_unpack(mul_f32x2(f32x2_pack(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), a2), a, b);
              o[e] = __float_as_uint(a);
              o[e + 1] = __float_as_uint(b);
            }
            tmem_st8(tO + 8 * ch, o);
          }
        }
        if (mn != -INFINITY) m = mn;
      }
      // P = exp2(x - m) (a hidden key gives exp2(-inf) = 0), in bf16 over
      // the S columns: keys 32 ch .. 32 ch + 31 -> columns 16 ch .. 16 ch + 15
      const float mb = (m == -INFINITY) ? 0.f : m;
      const unsigned long long nm2 = f32x2_pack(-mb, -mb);
      float sm[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) sm[i] = 0.f;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t w16[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float a, b;
          f32x2_unpack(add_f32x2(f32x2_pack(__uint_as_float(v[32 * ch + e]), __uint_as_float(v[32 * ch + e + 1])), nm2),
                       a, b);
          const float p0 = ex2_approx(a), p1 = ex2_approx(b);
          sm[(e >> 1) & 7] += p0 + p1;
          w16[e >> 1] = pack_bf16x2(p0, p1);
        }
        tmem_st16_nowait(tS + 16 * ch, w16);
      }
      const float sum0 = (sm[0] + sm[1]) + (sm[2] + sm[3]), sum1 = (sm[4] + sm[5]) + (sm[6] + sm[7]);
      l += sum0 + sum1;
      tmem_st_wait_all();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[x]);
      ++cnt;
    }
    if (ok || x >= nq) {
      if (x < nq && (cnt == 0 || warp_wait(&bars->o_done[x], (cnt - 1) & 1, wc, 33))) {
        tc_fence_after();
        const size_t row = (size_t)bh * p.S + (size_t)qi * kTile + r;
        const bool row_in = qi * kTile + r < p.S;  // rows of a partial last tile
        const float inv = (cnt > 0 && l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
        for (int ch = 0; ch < HD / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * ch, o);
          if (cnt == 0) {  // nothing visible: O = 0 (the accumulator was never written)
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0u;
          }
          uint4* dst = reinterpret_cast<uint4*>(p.o + row * HD + 32 * ch);
#pragma unroll
          for (int mm = 0; mm < 4; ++mm)
            if (row_in)
              dst[mm] = make_uint4(pack_bf16x2(inv * __uint_as_float(o[8 * mm]), inv * __uint_as_float(o[8 * mm + 1])),
                                   pack_bf16x2(inv * __uint_as_float(o[8 * mm + 2]), inv * __uint_as_float(o[8 * mm + 3])),
                                   pack_bf16x2(inv * __uint_as_float(o[8 * mm + 4]), inv * __uint_as_float(o[8 * mm + 5])),
                                   pack_bf16x2(inv * __uint_as_float(o[8 * mm + 6]), inv * __uint_as_float(o[8 * mm + 7])));
        }
        if (row_in) p.lse[row] = (cnt > 0 && l > 0.f) ? (m + __log2f(l)) * kLn2 : -INFINITY;
      }
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
int fwd_ctas(int BH, int N) { return BH * ((N + 1) / 2); }

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
