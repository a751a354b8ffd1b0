// api.cu -- the C ABI of libdab.so (declared in include/dab.h): argument
// checks, workspace layout, TMA tensor maps and kernel launches.  Host code
// only; the arithmetic is in the kernels.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "dab.h"
#include "dab_selftest.h"
#include "tile_sched.h"

namespace dab {
// kernels (bwd.cu, fwd.cu, aux.cu, selftest.cu)
template <int HD> int bwd_smem_bytes();
template <int HD> const void* bwd_kernel_ptr(bool ragged, bool chunk_major);
int fwd_threads();
int fwd_ctas(int BH, int N);
template <int HD> int fwd_smem_bytes();
template <int HD> const void* fwd_kernel_ptr();
template <int HD> int selftest_smem_bytes();
template <int HD> const void* selftest_kernel_ptr();
int peak_smem_bytes();
const void* peak_kernel_ptr();
int peak_threads();
cudaError_t launch_preprocess(int HD, const void* o, const void* dout, const float* lse, float* D,
                              float* lse2, uint32_t* sem, int n_sem, WsHeader* hdr, float* dqacc,
                              long long dq_elems, int BH, int S, int S_pad, int grid, cudaStream_t stream);
cudaError_t launch_convert(const float* dqacc, int chunk_major, void* dq, int ntiles, float scale, long long acc_stride,
                           int ways, int causal, int N, int S, int d, int grid, const int* count,
                           cudaStream_t stream);
cudaError_t launch_block_tables(const uint8_t* tiles, int N, int causal, int descending,
                                uint16_t* list, uint16_t* rank, int* nact, int* count,
                                cudaStream_t stream);
}  // namespace dab

namespace {

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s
constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int sms = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
thread_local char g_last_error[256] = "";

// Record a failed CUDA call for dab_last_error_string() and map it.
dab_status_t cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(e), (int)e);
  return DAB_ERR_CUDA;
}

// Per-device set-up: capability check and the dynamic shared-memory limits
// of the kernels.  Returns false if the device cannot run them.
bool device_setup(int* dev_out, int* sms_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    di.ready = true;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return false;
    di.sms = prop.multiProcessorCount;
    di.supported = (prop.major == 10 && prop.minor == 3);
    if (di.supported) {
      bool ok = true;
      for (bool ragged : {false, true}) {
        ok &= cudaFuncSetAttribute(dab::bwd_kernel_ptr<64>(ragged, true), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   dab::bwd_smem_bytes<64>()) == cudaSuccess;
        for (bool cm : {false, true})
          ok &= cudaFuncSetAttribute(dab::bwd_kernel_ptr<128>(ragged, cm), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     dab::bwd_smem_bytes<128>()) == cudaSuccess;
      }
      ok &= cudaFuncSetAttribute(dab::fwd_kernel_ptr<64>(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 dab::fwd_smem_bytes<64>()) == cudaSuccess;
      ok &= cudaFuncSetAttribute(dab::fwd_kernel_ptr<128>(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 dab::fwd_smem_bytes<128>()) == cudaSuccess;
      ok &= cudaFuncSetAttribute(dab::selftest_kernel_ptr<64>(),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 dab::selftest_smem_bytes<64>()) == cudaSuccess;
      ok &= cudaFuncSetAttribute(dab::peak_kernel_ptr(),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 dab::peak_smem_bytes()) == cudaSuccess;
      ok &= cudaFuncSetAttribute(dab::selftest_kernel_ptr<128>(),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 dab::selftest_smem_bytes<128>()) == cudaSuccess;
      di.supported = ok;
    }
  }
  if (dev_out) *dev_out = dev;
  if (sms_out) *sms_out = di.sms;
  return di.supported;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// [rows, d] bf16 row-major, box of 64 columns x 128 rows, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, long long rows, int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Any sequence length: the last 128-row tile of a head may be partial.  B, H
// or S of zero is an empty problem (nothing to compute, DAB_OK).
dab_status_t check_shape(int B, int H, int S, int d) {
  if (B < 0 || H < 0 || S < 0) return DAB_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return DAB_ERR_INVALID_ARG;
  if ((long long)B * H * (((long long)S + 127) / 128 * 128) >= (1ll << 31)) return DAB_ERR_INVALID_ARG;
  return DAB_OK;
}

bool empty_problem(int B, int H, int S) { return (long long)B * H * S == 0; }

// An empty backward launches no kernel; it still clears the status and detail
// words of a workspace it is given, so that dab_check_status reports this call.
dab_status_t clear_status(void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (workspace == nullptr || !aligned16(workspace) || ws_bytes < 8) return DAB_OK;
  const cudaError_t e = cudaMemsetAsync(workspace, 0, 8, stream);
  return e == cudaSuccess ? DAB_OK : cuda_fail(e, "status reset");
}

int tiles_of(int S) { return (S + 127) / 128; }

dab_status_t check_enums(dab_mask_t mask, dab_sched_t sched) {
  if ((int)mask < 0 || (int)mask > 1) return DAB_ERR_INVALID_ARG;
  if ((int)sched < 0 || (int)sched > 3) return DAB_ERR_INVALID_ARG;
  return DAB_OK;
}

// The entry points that run a backward also take DAB_SCHED_AUTO.
dab_status_t check_enums_auto(dab_mask_t mask, dab_sched_t sched) {
  return sched == DAB_SCHED_AUTO ? check_enums(mask, DAB_SCHED_SERIAL) : check_enums(mask, sched);
}

// DAB_SCHED_AUTO -> the schedule that dab_sched_select picks for `ctas` CTAs
// (the SM count of the current device when ctas <= 0).
dab_status_t resolve_sched(dab_mask_t mask, int B, int H, int S, int ctas, dab_sched_t* sched) {
  if (*sched != DAB_SCHED_AUTO) return DAB_OK;
  if (ctas <= 0) {
    int sms = 0;
    if (!device_setup(nullptr, &sms)) return DAB_ERR_UNSUPPORTED;
    ctas = sms;
  }
  const int pick = dab_sched_select(mask, B, H, S, ctas);
  if (pick < 0) return DAB_ERR_INVALID_ARG;
  *sched = static_cast<dab_sched_t>(pick);
  return DAB_OK;
}

int acc_ways(dab_sched_t sched) { return sched == DAB_SCHED_ATOMIC ? 1 : dab::kAccWays; }

// Layout of the f32 dQ accumulation tiles.  Chunk-major ([d/4][128 rows][4]
// per 128-row tile: a warp's 16-byte adds of one chunk are 512 contiguous
// bytes) for the ordered schedules and for d = 64.  The atomic schedule at
// d = 128 keeps row-major [row][d] with one-float adds of whole rows: its
// unpaced vector reds ran 3 % slower than scalar ones, while the ordered
// schedules gain 1-2 % (8 % with DAB_BWD_PLAIN_ADD) from the vector form.
int acc_chunk_major(int d, dab_sched_t sched) { return (d == 64 || sched != DAB_SCHED_ATOMIC) ? 1 : 0; }

bool layout(int B, int H, int S, int d, dab_sched_t sched, dab_ws_layout_t* L) {
  if (check_shape(B, H, S, d) != DAB_OK) return false;
  const size_t BH = (size_t)B * H, N = (size_t)tiles_of(S);
  const size_t rows_pad = BH * N * 128;  // D, LSE2 and dQ per head padded to whole tiles
  const size_t ways = (size_t)acc_ways(sched);
  size_t off = 0;
  L->status = off;
  off += 256;
  L->sem = off;
  off = round_up(off + BH * N * dab::kSubTiles * ways * 4, 256);  // per tile, sub-tile, buffer
  L->D = off;
  off = round_up(off + rows_pad * 4, 256);
  L->lse2 = off;
  off = round_up(off + rows_pad * 4, 256);
  L->dqacc = off;  // chunk-major tiles, every head padded to whole tiles
  off = round_up(off + ways * rows_pad * (size_t)d * 4, 256);
  L->total = off;
  return true;
}

// Block-mask schedule tables, after the ordinary workspace regions.
struct BlockTables {
  size_t list, rank, nact, count, total;
};
BlockTables block_tables_layout(const dab_ws_layout_t& L, int N) {
  BlockTables T;
  const size_t n2 = (size_t)N * N;
  T.list = round_up(L.total, 256);
  T.rank = T.list + 2 * n2;
  T.nact = round_up(T.rank + 2 * n2, 16);
  T.count = T.nact + 4 * (size_t)N;
  T.total = round_up(T.count + 4 * (size_t)N, 256);
  return T;
}

int elementwise_grid(int sms, long long work) {
  long long g = (long long)sms * 8;
  const long long need = (work + 255) / 256;
  if (need < g) g = need;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

extern "C" {

const char* dab_last_error_string(void) { return g_last_error; }

const char* dab_status_string(dab_status_t s) {
  switch (s) {
    case DAB_OK: return "DAB_OK";
    case DAB_ERR_INVALID_ARG: return "DAB_ERR_INVALID_ARG";
    case DAB_ERR_UNSUPPORTED: return "DAB_ERR_UNSUPPORTED";
    case DAB_ERR_WORKSPACE: return "DAB_ERR_WORKSPACE";
    case DAB_ERR_CUDA: return "DAB_ERR_CUDA";
    case DAB_ERR_TIMEOUT: return "DAB_ERR_TIMEOUT";
    case DAB_ERR_DEVICE_BOUNDS: return "DAB_ERR_DEVICE_BOUNDS";
  }
  return "DAB_ERR_UNKNOWN";
}

dab_status_t dab_bwd_workspace_layout(int B, int H, int S, int d, dab_mask_t mask, dab_sched_t sched,
                                      dab_ws_layout_t* L) {
  if (L == nullptr || check_enums_auto(mask, sched) != DAB_OK) return DAB_ERR_INVALID_ARG;
  // every deterministic schedule has the same layout, so AUTO needs no device
  if (sched == DAB_SCHED_AUTO) sched = DAB_SCHED_DESCENDING_Q;
  return layout(B, H, S, d, sched, L) ? DAB_OK : DAB_ERR_INVALID_ARG;
}

size_t dab_bwd_workspace_size(int B, int H, int S, int d, dab_mask_t mask, dab_sched_t sched) {
  dab_ws_layout_t L;
  if (dab_bwd_workspace_layout(B, H, S, d, mask, sched, &L) != DAB_OK) return 0;
  return L.total;
}

static dab_status_t fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                             int H, int S, int d, float scale, dab_mask_t mask, void* workspace,
                             size_t ws_bytes, cudaStream_t stream, const uint8_t* tiles) {
  if (check_shape(B, H, S, d) != DAB_OK) return DAB_ERR_INVALID_ARG;
  if (empty_problem(B, H, S)) return DAB_OK;
  if ((int)mask < 0 || (int)mask > 1) return DAB_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return DAB_ERR_INVALID_ARG;
  if (!(scale > 0.f)) return DAB_ERR_INVALID_ARG;
  if (workspace != nullptr && (ws_bytes < 256 || !aligned16(workspace))) return DAB_ERR_WORKSPACE;
  int sms = 0;
  if (!device_setup(nullptr, &sms)) return DAB_ERR_UNSUPPORTED;
  const long long rows = (long long)B * H * S;
  dab::FwdParams p;
  std::memset(&p, 0, sizeof(p));
  if (!make_map(&p.tm_q, q, rows, d) || !make_map(&p.tm_k, k, rows, d) || !make_map(&p.tm_v, v, rows, d))
    return DAB_ERR_CUDA;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.BH = B * H;
  p.S = S;
  p.N = tiles_of(S);
  p.mask = (int)mask;
  p.scale_log2e = scale * 1.4426950408889634f;
  p.tiles = tiles;
  dab::WsHeader* hdr = static_cast<dab::WsHeader*>(workspace);
  if (hdr != nullptr && cudaMemsetAsync(hdr, 0, 16, stream) != cudaSuccess) return DAB_ERR_CUDA;
  const dim3 grid((unsigned)dab::fwd_ctas(p.BH, p.N)), block((unsigned)dab::fwd_threads());
  void* args[] = {&p, &hdr};
  cudaError_t e;
  if (d == 128)
    e = cudaLaunchKernel(dab::fwd_kernel_ptr<128>(), grid, block, args, dab::fwd_smem_bytes<128>(), stream);
  else
    e = cudaLaunchKernel(dab::fwd_kernel_ptr<64>(), grid, block, args, dab::fwd_smem_bytes<64>(), stream);
  return e == cudaSuccess ? DAB_OK : cuda_fail(e, "forward launch");
}

dab_status_t dab_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                          int H, int S, int d, float scale, dab_mask_t mask, void* workspace,
                          size_t ws_bytes, cudaStream_t stream) {
  return fwd_impl(q, k, v, o, lse, B, H, S, d, scale, mask, workspace, ws_bytes, stream, nullptr);
}

dab_status_t dab_attn_fwd_block(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int H, int S, int d, float scale, const uint8_t* tiles,
                                int causal, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (tiles == nullptr || (causal != 0 && causal != 1) || (S % 128) != 0) return DAB_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, B, H, S, d, scale, causal ? DAB_MASK_CAUSAL : DAB_MASK_FULL,
                  workspace, ws_bytes, stream, tiles);
}

dab_status_t dab_bwd_preprocess(const void* o, const float* lse, const void* dout, int B, int H, int S,
                                int d, dab_mask_t mask, dab_sched_t sched, void* workspace,
                                size_t ws_bytes, cudaStream_t stream) {
  if (check_shape(B, H, S, d) != DAB_OK || check_enums_auto(mask, sched) != DAB_OK) return DAB_ERR_INVALID_ARG;
  if (empty_problem(B, H, S)) return DAB_OK;
  if (!aligned16(o) || !aligned16(lse) || !aligned16(dout)) return DAB_ERR_INVALID_ARG;
  if (sched == DAB_SCHED_AUTO) sched = DAB_SCHED_DESCENDING_Q;  // same preprocessing for all ordered schedules
  dab_ws_layout_t L;
  layout(B, H, S, d, sched, &L);
  if (workspace == nullptr || !aligned16(workspace)) return DAB_ERR_WORKSPACE;
  if (ws_bytes < L.total) return DAB_ERR_WORKSPACE;
  int sms = 0;
  if (!device_setup(nullptr, &sms)) return DAB_ERR_UNSUPPORTED;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const long long rows = (long long)B * H * S;
  const long long rows_pad = (long long)B * H * tiles_of(S) * 128;
  const int n_sem = B * H * tiles_of(S) * dab::kSubTiles * acc_ways(sched);
  float* dqacc = (sched == DAB_SCHED_ATOMIC) ? reinterpret_cast<float*>(ws + L.dqacc) : nullptr;
  const int grid = elementwise_grid(sms, rows * (d / 8));
  cudaError_t e = dab::launch_preprocess(
      d, o, dout, lse, reinterpret_cast<float*>(ws + L.D), reinterpret_cast<float*>(ws + L.lse2),
      reinterpret_cast<uint32_t*>(ws + L.sem), n_sem, reinterpret_cast<dab::WsHeader*>(ws + L.status),
      dqacc, rows_pad * d, B * H, S, tiles_of(S) * 128, grid, stream);
  return e == cudaSuccess ? DAB_OK : cuda_fail(e, "preprocess launch");
}

// The backward; `tiles` (device, [N][N]) selects the block-mask schedules.
static dab_status_t bwd_impl(const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                             int H, int S, int d, float scale, dab_mask_t mask, dab_sched_t sched,
                             void* workspace, size_t ws_bytes, cudaStream_t stream,
                             const dab_bwd_opts_t* opts, const uint8_t* tiles) {
  if (check_shape(B, H, S, d) != DAB_OK || check_enums_auto(mask, sched) != DAB_OK) return DAB_ERR_INVALID_ARG;
  if (empty_problem(B, H, S)) return clear_status(workspace, ws_bytes, stream);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return DAB_ERR_INVALID_ARG;
  if (!(scale > 0.f)) return DAB_ERR_INVALID_ARG;
  const bool block = tiles != nullptr;
  if (block && (S % 128) != 0) return DAB_ERR_INVALID_ARG;  // block masks cover whole tiles
  if (block) {
    if (sched == DAB_SCHED_AUTO) sched = DAB_SCHED_DESCENDING_Q;
    if (sched == DAB_SCHED_SHIFT) return DAB_ERR_UNSUPPORTED;  // no shift walk over a block mask
  } else {
    const dab_status_t st = resolve_sched(mask, B, H, S, (opts && opts->grid > 0) ? opts->grid : 0, &sched);
    if (st != DAB_OK) return st;
  }
  const int N = tiles_of(S);
  if (sched == DAB_SCHED_SHIFT && mask == DAB_MASK_CAUSAL && (N % 2) != 0) return DAB_ERR_UNSUPPORTED;
  dab_ws_layout_t L;
  layout(B, H, S, d, sched, &L);
  const BlockTables T = block_tables_layout(L, N);
  if (workspace == nullptr || !aligned16(workspace) || ws_bytes < (block ? T.total : L.total))
    return DAB_ERR_WORKSPACE;
  int sms = 0;
  if (!device_setup(nullptr, &sms)) return DAB_ERR_UNSUPPORTED;

  const uint32_t flags = opts ? opts->flags : 0u;
  const unsigned long long timeout =
      (opts && opts->spin_timeout_ns) ? (unsigned long long)opts->spin_timeout_ns : kDefaultTimeoutNs;
  const int uph = block ? N : dab::units_per_head((int)sched, (int)mask, N);
  const long long total_ll = (long long)B * H * uph;
  if (total_ll >= (1ll << 31)) return DAB_ERR_INVALID_ARG;
  const int total = (int)total_ll;
  int grid = (opts && opts->grid > 0) ? opts->grid : sms;
  if (grid > sms) grid = sms;  // one CTA per SM, all resident
  if (grid > total) grid = total;
  if (!block && dab::gang_size((int)sched, (int)mask, N) > grid) return DAB_ERR_UNSUPPORTED;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (!(flags & DAB_BWD_SKIP_PREPROCESS)) {
    dab_status_t st = dab_bwd_preprocess(o, lse, dout, B, H, S, d, mask, sched, workspace, ws_bytes, stream);
    if (st != DAB_OK) return st;
  }
  if (block) {
    const cudaError_t e = dab::launch_block_tables(
        tiles, N, mask == DAB_MASK_CAUSAL ? 1 : 0, sched == DAB_SCHED_DESCENDING_Q ? 1 : 0,
        reinterpret_cast<uint16_t*>(ws + T.list), reinterpret_cast<uint16_t*>(ws + T.rank),
        reinterpret_cast<int*>(ws + T.nact), reinterpret_cast<int*>(ws + T.count), stream);
    if (e != cudaSuccess) return cuda_fail(e, "block table launch");
  }

  dab::BwdParams p;
  std::memset(&p, 0, sizeof(p));
  const long long rows = (long long)B * H * S;
  if (!make_map(&p.tm_q, q, rows, d) || !make_map(&p.tm_k, k, rows, d) || !make_map(&p.tm_v, v, rows, d) ||
      !make_map(&p.tm_do, dout, rows, d))
    return DAB_ERR_CUDA;
  p.lse2 = reinterpret_cast<const float*>(ws + L.lse2);
  p.D = reinterpret_cast<const float*>(ws + L.D);
  p.dqacc = reinterpret_cast<float*>(ws + L.dqacc);
  p.acc_ways = acc_ways(sched);
  p.acc_stride = (long long)B * H * N * 128 * d;  // floats per buffer (padded tiles)
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.sem = reinterpret_cast<uint32_t*>(ws + L.sem);
  p.hdr = reinterpret_cast<dab::WsHeader*>(ws + L.status);
  p.BH = B * H;
  p.S = S;
  p.N = N;
  p.sched = (int)sched;
  p.mask = (int)mask;
  p.units_per_head = uph;
  p.total_units = total;
  p.scale = scale;
  p.scale_log2e = scale * 1.4426950408889634f;
  p.timeout_ns = timeout;
  p.plain_add = (flags & DAB_BWD_PLAIN_ADD) ? 1 : 0;
  // The ordered schedules finalise dQ in the main kernel's tail unless the
  // caller asks for the separate pass (or skips the main kernel or the convert).
  p.fuse_convert = (sched != DAB_SCHED_ATOMIC &&
                    !(flags & (DAB_BWD_SEPARATE_CONVERT | DAB_BWD_SKIP_CONVERT | DAB_BWD_SKIP_MAIN)))
                       ? 1 : 0;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  if (block) {
    p.block = 1;
    p.blk_list = reinterpret_cast<const uint16_t*>(ws + T.list);
    p.blk_rank = reinterpret_cast<const uint16_t*>(ws + T.rank);
    p.blk_nact = reinterpret_cast<const int*>(ws + T.nact);
    p.blk_count = reinterpret_cast<const int*>(ws + T.count);
  }

  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(640);
  cfg.dynamicSmemBytes = (d == 128) ? dab::bwd_smem_bytes<128>() : dab::bwd_smem_bytes<64>();
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident together
  attr[0].val.cooperative =
      ((flags & DAB_BWD_SHARE_GPU) && !dab::static_dispatch((int)sched)) ? 0 : 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&p};
  cudaError_t e = cudaSuccess;
  if (!(flags & DAB_BWD_SKIP_MAIN)) {
    const bool ragged = (S % 128) != 0;
    const bool cm = acc_chunk_major(d, sched) != 0;
    e = cudaLaunchKernelExC(&cfg, d == 128 ? dab::bwd_kernel_ptr<128>(ragged, cm) : dab::bwd_kernel_ptr<64>(ragged, cm),
                            args);
    if (e != cudaSuccess) return cuda_fail(e, "main kernel launch");
  }

  if (!(flags & DAB_BWD_SKIP_CONVERT) && !p.fuse_convert) {
    const int ntiles = B * H * N;
    const int cgrid = ntiles < 8 * sms ? ntiles : 8 * sms;
    e = dab::launch_convert(p.dqacc, acc_chunk_major(d, sched), dq, ntiles, scale, p.acc_stride, p.acc_ways,
                            mask == DAB_MASK_CAUSAL ? 1 : 0, N, S, d, cgrid,
                            block ? p.blk_count : nullptr, stream);
    if (e != cudaSuccess) return cuda_fail(e, "convert launch");
  }
  return DAB_OK;
}

dab_status_t dab_attn_bwd_ex(const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                             int H, int S, int d, float scale, dab_mask_t mask, dab_sched_t sched,
                             void* workspace, size_t ws_bytes, cudaStream_t stream,
                             const dab_bwd_opts_t* opts) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, S, d, scale, mask, sched, workspace, ws_bytes,
                  stream, opts, nullptr);
}

size_t dab_bwd_block_workspace_size(int B, int H, int S, int d, dab_sched_t sched) {
  if (sched == DAB_SCHED_SHIFT) return 0;
  if (sched == DAB_SCHED_AUTO) sched = DAB_SCHED_DESCENDING_Q;
  dab_ws_layout_t L;
  if (check_enums(DAB_MASK_FULL, sched) != DAB_OK || !layout(B, H, S, d, sched, &L)) return 0;
  return block_tables_layout(L, tiles_of(S)).total;
}

dab_status_t dab_attn_bwd_block(const void* q, const void* k, const void* v, const void* o,
                                const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                int B, int H, int S, int d, float scale, const uint8_t* tiles,
                                int causal, dab_sched_t sched, void* workspace, size_t ws_bytes,
                                cudaStream_t stream) {
  if (tiles == nullptr || (causal != 0 && causal != 1)) return DAB_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, H, S, d, scale,
                  causal ? DAB_MASK_CAUSAL : DAB_MASK_FULL, sched, workspace, ws_bytes, stream, nullptr,
                  tiles);
}

dab_status_t dab_attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                          const void* dout, void* dq, void* dk, void* dv, int B, int H, int S, int d,
                          float scale, dab_mask_t mask, dab_sched_t sched, void* workspace,
                          size_t ws_bytes, cudaStream_t stream) {
  return dab_attn_bwd_ex(q, k, v, o, lse, dout, dq, dk, dv, B, H, S, d, scale, mask, sched, workspace,
                         ws_bytes, stream, nullptr);
}

dab_status_t dab_check_status(const void* workspace, cudaStream_t stream) {
  if (workspace == nullptr) return DAB_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DAB_ERR_CUDA;
  uint32_t hdr[2] = {0, 0};
  if (cudaMemcpy(hdr, workspace, sizeof(hdr), cudaMemcpyDeviceToHost) != cudaSuccess) return DAB_ERR_CUDA;
  if (hdr[0] == 0) return DAB_OK;
  if (hdr[0] == DAB_ERR_TIMEOUT || hdr[0] == DAB_ERR_DEVICE_BOUNDS) return (dab_status_t)hdr[0];
  return DAB_ERR_DEVICE_BOUNDS;
}

// ---------------------------------------------------------------- schedules
int dab_sched_units_per_head(dab_sched_t sched, dab_mask_t mask, int N) {
  if (check_enums(mask, sched) != DAB_OK || N < 1) return -1;
  if (sched == DAB_SCHED_SHIFT && mask == DAB_MASK_CAUSAL && (N % 2)) return -1;
  return dab::units_per_head((int)sched, (int)mask, N);
}

int dab_sched_unit_steps(dab_sched_t sched, dab_mask_t mask, int N, int u) {
  const int uph = dab_sched_units_per_head(sched, mask, N);
  if (uph < 0 || u < 0 || u >= uph) return -1;
  return dab::unit_steps((int)sched, (int)mask, N, u);
}

int dab_sched_step(dab_sched_t sched, dab_mask_t mask, int N, int u, int t, int* kv_tile, int* q_tile) {
  const int steps = dab_sched_unit_steps(sched, mask, N, u);
  if (steps < 0 || t < 0 || t >= steps) return -1;
  const dab::Step s = dab::step((int)sched, (int)mask, N, u, t);
  if (kv_tile) *kv_tile = s.kv;
  if (q_tile) *q_tile = s.q;
  return 0;
}

int dab_sched_rank(dab_sched_t sched, dab_mask_t mask, int N, int i, int j) {
  if (dab_sched_units_per_head(sched, mask, N) < 0) return -1;
  if (i < 0 || j < 0 || i >= N || j >= N) return -1;
  return dab::rank((int)sched, (int)mask, N, i, j);
}

int dab_sched_contributors(dab_mask_t mask, int N, int j) {
  if ((int)mask < 0 || (int)mask > 1 || j < 0 || j >= N) return -1;
  return dab::contributors((int)mask, N, j);
}

int dab_sched_gang_size(dab_sched_t sched, dab_mask_t mask, int N) {
  if (dab_sched_units_per_head(sched, mask, N) < 0) return -1;
  return dab::gang_size((int)sched, (int)mask, N);
}

// ---------------------------------------------------------------- selftest
dab_status_t dab_selftest_mma(int d, const void* x, const void* y, const void* z, const void* pm,
                              float* out0, float* out1, float* out2, float* out3, void* status_ws,
                              cudaStream_t stream) {
  if (d != 64 && d != 128) return DAB_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(z) || !aligned16(pm) || !aligned16(out0) ||
      !aligned16(out1) || !aligned16(out2) || !aligned16(out3) || !aligned16(status_ws))
    return DAB_ERR_INVALID_ARG;
  if (!device_setup(nullptr, nullptr)) return DAB_ERR_UNSUPPORTED;
  CUtensorMap mx, my;
  if (!make_map(&mx, x, 128, d) || !make_map(&my, y, 128, d)) return DAB_ERR_CUDA;
  if (cudaMemsetAsync(status_ws, 0, 16, stream) != cudaSuccess) return DAB_ERR_CUDA;
  dab::WsHeader* hdr = static_cast<dab::WsHeader*>(status_ws);
  const __nv_bfloat16* zz = static_cast<const __nv_bfloat16*>(z);
  const __nv_bfloat16* pp = static_cast<const __nv_bfloat16*>(pm);
  void* args[] = {&mx, &my, &zz, &pp, &out0, &out1, &out2, &out3, &hdr};
  cudaError_t e;
  if (d == 128)
    e = cudaLaunchKernel(dab::selftest_kernel_ptr<128>(), dim3(1), dim3(192), args,
                         dab::selftest_smem_bytes<128>(), stream);
  else
    e = cudaLaunchKernel(dab::selftest_kernel_ptr<64>(), dim3(1), dim3(192), args,
                         dab::selftest_smem_bytes<64>(), stream);
  return e == cudaSuccess ? DAB_OK : DAB_ERR_CUDA;
}

// ------------------------------------------------------------- tensor peak
int dab_mma_peak_grid(void) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return sms;
}

dab_status_t dab_mma_peak(int iters, void* status_ws, cudaStream_t stream) {
  if (iters < 1 || iters > (1 << 22) || !aligned16(status_ws)) return DAB_ERR_INVALID_ARG;
  if (!device_setup(nullptr, nullptr)) return DAB_ERR_UNSUPPORTED;
  const int grid = dab_mma_peak_grid();
  if (grid <= 0) return DAB_ERR_CUDA;
  if (cudaMemsetAsync(status_ws, 0, 16, stream) != cudaSuccess) return DAB_ERR_CUDA;
  dab::WsHeader* hdr = static_cast<dab::WsHeader*>(status_ws);
  unsigned long long timeout_ns = 4000000000ull;  // the longest allowed run is about 1 s
  void* args[] = {&iters, &hdr, &timeout_ns};
  const cudaError_t e = cudaLaunchKernel(dab::peak_kernel_ptr(), dim3(grid), dim3(dab::peak_threads()),
                                         args, dab::peak_smem_bytes(), stream);
  return e == cudaSuccess ? DAB_OK : DAB_ERR_CUDA;
}

}  // extern "C"
