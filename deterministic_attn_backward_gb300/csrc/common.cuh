// common.cuh -- kernel parameter blocks, workspace header and the bounded
// waits shared by the kernels of the attention library.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace dab {

// Status codes written to the workspace status word (same values as the
// public dab_status_t).
enum : uint32_t { kStatusOk = 0, kStatusTimeout = 5, kStatusBounds = 6 };

// Workspace header (first 256 bytes of the workspace).
struct WsHeader {
  uint32_t status;   // 0 or the first device error
  uint32_t detail;   // where it happened (see kDetail*)
  uint32_t ticket;   // dynamic unit dispatch counter
  uint32_t conv_ticket;  // dQ tiles claimed for finalisation in the kernel's tail
  uint32_t pad[60];
};

// Detail codes: the high byte says which wait ran out, the rest is context.
enum : uint32_t {
  kDetailMbar = 0x01000000u,     // an on-chip pipeline wait (low bits: barrier id)
  kDetailSem = 0x02000000u,      // a dQ semaphore wait (low bits: the tile)
  kDetailAlign = 0x03000000u,    // shared memory misaligned
  kDetailDrain = 0x04000000u,    // teardown drain
};

constexpr int kTile = 128;  // rows of a KV tile and of a Q tile

// The ordered schedules accumulate dQ in kAccWays interleaved f32 buffers:
// the partial of rank r goes to buffer r mod kAccWays, in rank order within
// the buffer, and the dQ convert adds the buffers in index order.  A
// contributor then waits for rank r - kAccWays instead of r - 1, which hides
// the latency of the cross-SM hand-off; the summation order stays fixed.
constexpr int kAccWays = 4;
constexpr int kSubTiles = 8;  // semaphores (and reducer warps) per dQ tile per buffer

struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;  // [B*H*S, d] bf16, box 64 x 128, 128B swizzle
  const float* lse2;                    // [B*H*S_pad] -LSE * log2(e)
  const float* D;                       // [B*H*S_pad]
  float* dqacc;                         // [acc_ways][B*H*S_pad*d] f32 (see bwd.cu)
  long long acc_stride;                 // floats between two accumulation buffers
  int acc_ways;                         // kAccWays (ordered schedules) or 1 (atomic)
  __nv_bfloat16* dk;                    // [B*H*S, d]
  __nv_bfloat16* dv;
  uint32_t* sem;                        // [B*H, N]
  WsHeader* hdr;
  int BH, S, N;
  int sched, mask;
  int units_per_head, total_units;
  float scale, scale_log2e;
  unsigned long long timeout_ns;
  int plain_add;                        // ordered schedules: load + add + store instead of red
  // Ordered schedules: the main kernel also writes dQ = bf16(scale * sum of
  // the buffers), tile by tile, in its tail (no separate convert pass).
  int fuse_convert;
  __nv_bfloat16* dq;                    // [B*H*S, d]
  // Block mask (block != 0): the schedule comes from tables built on the
  // device from the tile flags, shared by all heads.
  int block;
  const uint16_t* blk_list;             // [N][N]: KV tile i's visible Q tiles, visit order
  const uint16_t* blk_rank;             // [N][N]: rank of KV tile i in dQ_j's order, at [j][i]
  const int* blk_nact;                  // [N]: visible Q tiles of KV tile i
  const int* blk_count;                 // [N]: contributors of Q tile j
};

struct FwdParams {
  CUtensorMap tm_q, tm_k, tm_v;
  __nv_bfloat16* o;
  float* lse;
  int BH, S, N;
  int mask;
  float scale_log2e;
  const uint8_t* tiles;                 // block mask [N][N] (query tile, key tile), or null
};

// Record the first device error (later ones are dropped).
__device__ __forceinline__ void raise_error(WsHeader* hdr, uint32_t code, uint32_t detail) {
  if (atomicCAS(&hdr->status, 0u, code) == 0u) {
    atomicExch(&hdr->detail, detail);
  }
}

// Shared state every waiting thread of a CTA watches.
struct WaitCtl {
  volatile int* abort;        // CTA-wide flag in shared memory
  WsHeader* hdr;
  unsigned long long timeout_ns;
};

// Wait for phase `parity` of an mbarrier.  Returns false when the CTA is
// aborting or the wait ran out (then the error is recorded and the CTA-wide
// abort flag is set).  Never traps.
static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, const WaitCtl& w,
                                            uint32_t id) {
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++it & 31u) == 0u) {
      if (*w.abort) return false;
      if (globaltimer_ns() - t0 > w.timeout_ns) {
        raise_error(w.hdr, kStatusTimeout, kDetailMbar | id);
        *w.abort = 1;
        return false;
      }
      if ((it & 1023u) == 0u && ld_volatile(&w.hdr->status) != 0u) {
        *w.abort = 1;  // another CTA failed: stop waiting
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtl& w,
                                          uint32_t id) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, w, id);
}

// All lanes of the warp wait; the warp continues only if every lane saw the
// phase complete (a uniform decision, required before .sync.aligned
// tensor-memory instructions).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& w,
                                          uint32_t id) {
  const bool ok = mbar_wait(bar, parity, w, id);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait that ignores the abort flag (teardown drains).
static __device__ __noinline__ void drain_wait(uint64_t* bar, uint32_t parity, WsHeader* hdr,
                                        unsigned long long timeout_ns, uint32_t id) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > timeout_ns) {
      raise_error(hdr, kStatusTimeout, kDetailDrain | id);
      return;
    }
  }
}

// Start-address offset, in the descriptor's 16-byte units, of K step k of a
// K-major operand with `rows` rows (64-column blocks), and of an MN-major
// operand (16 K rows of 128 bytes per step).  Adding them to a descriptor
// built for k = 0 gives the descriptor of step k (the start address is the
// low field and never carries into the next one for shared addresses).
__host__ __device__ constexpr uint64_t koff_kmajor(int k, int rows) {
  return (uint64_t)(((k >> 2) * rows * 128 + (k & 3) * 32) >> 4);
}
__host__ __device__ constexpr uint64_t koff_mnmajor(int k) { return (uint64_t)((k * 2048) >> 4); }

// K-major operand: rows x (64-column blocks); K step k (16 elements).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int k, int rows) {
  return sdesc_sw128(base + (k >> 2) * rows * 128 + (k & 3) * 32, 16, 1024);
}
// MN-major operand stored as [MN/64 blocks][K rows][64]; K step k (16 rows).
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int k, int rows) {
  return sdesc_sw128(base + k * 2048, rows * 128, 1024);
}

}  // namespace dab
