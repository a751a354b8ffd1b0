// hostio.cu -- the attention backward on host buffers, copies overlapped
// with the computation.
//
// The heads are split into chunks of consecutive (b, h) heads.  On two copy
// streams owned by the library, the inputs of every chunk are copied to the
// device back to back, and the gradients of chunk c are copied back while
// chunk c+1 is computed; the backward of each chunk runs on the caller's
// stream as an ordinary dab_attn_bwd call on that range of heads (B = 1,
// H = heads in the chunk), so every chunk computes exactly what the whole
// call would for those heads.  Events order the three streams: the copies
// start after the work already queued on the caller's stream, and the
// caller's stream waits for the last copy back.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "dab.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kDefaultChunks = 8;

struct CopyStreams {
  cudaStream_t in = nullptr, out = nullptr;
};
std::mutex g_mu;
CopyStreams g_streams[kMaxDevices];

// The copy streams of the current device, created on first use.
bool copy_streams(CopyStreams* cs) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  CopyStreams& s = g_streams[dev];
  if (s.in == nullptr) {
    if (cudaStreamCreateWithFlags(&s.in, cudaStreamNonBlocking) != cudaSuccess) return false;
    if (cudaStreamCreateWithFlags(&s.out, cudaStreamNonBlocking) != cudaSuccess) {
      cudaStreamDestroy(s.in);
      s.in = nullptr;
      return false;
    }
  }
  *cs = s;
  return true;
}

size_t round_up(size_t x) { return (x + 255) / 256 * 256; }

// Device workspace of the host path: copies of the inputs and outputs, then
// the backward workspace of the largest chunk.
struct HostLayout {
  size_t q, k, v, o, dout, lse, dq, dk, dv, ws, ws_bytes, total;
  int chunks, per_chunk;
};

bool host_layout(int B, int H, int S, int d, dab_mask_t mask, dab_sched_t sched, int chunks,
                 HostLayout* L) {
  if (B < 1 || H < 1) return false;
  const long long bh = (long long)B * H;
  if (chunks <= 0) chunks = kDefaultChunks;
  if (chunks > bh) chunks = (int)bh;
  L->per_chunk = (int)((bh + chunks - 1) / chunks);
  L->chunks = (int)((bh + L->per_chunk - 1) / L->per_chunk);
  L->ws_bytes = dab_bwd_workspace_size(1, L->per_chunk, S, d, mask, sched);
  if (L->ws_bytes == 0 || dab_bwd_workspace_size(B, H, S, d, mask, sched) == 0) return false;
  const size_t t = round_up((size_t)bh * S * d * 2), r = round_up((size_t)bh * S * 4);
  size_t off = 0;
  for (size_t* f : {&L->q, &L->k, &L->v, &L->o, &L->dout}) {
    *f = off;
    off += t;
  }
  L->lse = off;
  off += r;
  for (size_t* f : {&L->dq, &L->dk, &L->dv}) {
    *f = off;
    off += t;
  }
  L->ws = off;
  L->total = off + round_up(L->ws_bytes);
  return true;
}

}  // namespace

extern "C" size_t dab_bwd_host_workspace_size(int B, int H, int S, int d, dab_mask_t mask,
                                              dab_sched_t sched, int chunks) {
  if (B >= 0 && H >= 0 && S >= 0 && (long long)B * H * S == 0)  // empty problem
    return dab_bwd_workspace_size(B, H, S, d, mask, sched) ? 256 : 0;
  HostLayout L;
  return host_layout(B, H, S, d, mask, sched, chunks, &L) ? L.total : 0;
}

extern "C" dab_status_t dab_attn_bwd_host(const void* q, const void* k, const void* v,
                                          const void* o, const float* lse, const void* dout,
                                          void* dq, void* dk, void* dv, int B, int H, int S, int d,
                                          float scale, dab_mask_t mask, dab_sched_t sched,
                                          void* dev_ws, size_t dev_ws_bytes, int chunks,
                                          cudaStream_t stream) {
  if (B >= 0 && H >= 0 && S >= 0 && (long long)B * H * S == 0)  // empty problem: nothing to do
    return dab_bwd_workspace_size(B, H, S, d, mask, sched) ? DAB_OK : DAB_ERR_INVALID_ARG;
  HostLayout L;
  if (!host_layout(B, H, S, d, mask, sched, chunks, &L)) return DAB_ERR_INVALID_ARG;
  for (const void* p : {q, k, v, o, static_cast<const void*>(lse), dout,
                        static_cast<const void*>(dq), static_cast<const void*>(dk),
                        static_cast<const void*>(dv)})
    if (p == nullptr) return DAB_ERR_INVALID_ARG;
  if (dev_ws == nullptr || (reinterpret_cast<uintptr_t>(dev_ws) & 255u) != 0 ||
      dev_ws_bytes < L.total)
    return DAB_ERR_WORKSPACE;
  CopyStreams cs;
  if (!copy_streams(&cs)) return DAB_ERR_CUDA;

  uint8_t* w = static_cast<uint8_t*>(dev_ws);
  const size_t head_t = (size_t)S * d * 2, head_r = (size_t)S * 4;
  const void* hin[5] = {q, k, v, o, dout};
  const size_t din[5] = {L.q, L.k, L.v, L.o, L.dout};
  void* hout[3] = {dq, dk, dv};
  const size_t dout_off[3] = {L.dq, L.dk, L.dv};

  std::vector<cudaEvent_t> ev(2 * L.chunks + 2, nullptr);
  for (auto& e : ev)
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
      for (auto& x : ev)
        if (x != nullptr) cudaEventDestroy(x);
      return DAB_ERR_CUDA;
    }
  cudaEvent_t start = ev[2 * L.chunks], done = ev[2 * L.chunks + 1];
  dab_status_t st = DAB_OK;
  auto ok = [&](cudaError_t e) {
    if (e != cudaSuccess && st == DAB_OK) st = DAB_ERR_CUDA;
    return e == cudaSuccess;
  };
  const long long bh = (long long)B * H;
  // copies start after what is already queued on the caller's stream
  if (ok(cudaEventRecord(start, stream)) && ok(cudaStreamWaitEvent(cs.in, start, 0)) &&
      ok(cudaStreamWaitEvent(cs.out, start, 0))) {
    for (int c = 0; c < L.chunks && st == DAB_OK; ++c) {  // all inputs, back to back
      const long long h0 = (long long)c * L.per_chunk;
      const long long nh = (h0 + L.per_chunk <= bh) ? L.per_chunk : bh - h0;
      for (int i = 0; i < 5; ++i)
        ok(cudaMemcpyAsync(w + din[i] + h0 * head_t, static_cast<const uint8_t*>(hin[i]) + h0 * head_t,
                           nh * head_t, cudaMemcpyHostToDevice, cs.in));
      ok(cudaMemcpyAsync(w + L.lse + h0 * head_r, reinterpret_cast<const uint8_t*>(lse) + h0 * head_r,
                         nh * head_r, cudaMemcpyHostToDevice, cs.in));
      ok(cudaEventRecord(ev[c], cs.in));
    }
    for (int c = 0; c < L.chunks && st == DAB_OK; ++c) {  // compute chunk c, then copy it back
      const long long h0 = (long long)c * L.per_chunk;
      const long long nh = (h0 + L.per_chunk <= bh) ? L.per_chunk : bh - h0;
      if (!ok(cudaStreamWaitEvent(stream, ev[c], 0))) break;
      auto dp = [&](size_t off) { return static_cast<void*>(w + off + h0 * head_t); };
      const dab_status_t r =
          dab_attn_bwd(dp(L.q), dp(L.k), dp(L.v), dp(L.o), reinterpret_cast<const float*>(w + L.lse + h0 * head_r),
                       dp(L.dout), dp(L.dq), dp(L.dk), dp(L.dv), 1, (int)nh, S, d, scale, mask, sched,
                       w + L.ws, L.ws_bytes, stream);
      if (r != DAB_OK) {
        st = r;
        break;
      }
      if (!ok(cudaEventRecord(ev[L.chunks + c], stream)) ||
          !ok(cudaStreamWaitEvent(cs.out, ev[L.chunks + c], 0)))
        break;
      for (int i = 0; i < 3; ++i)
        ok(cudaMemcpyAsync(static_cast<uint8_t*>(hout[i]) + h0 * head_t, w + dout_off[i] + h0 * head_t,
                           nh * head_t, cudaMemcpyDeviceToHost, cs.out));
    }
    // the caller's stream continues once everything has been copied back
    if (ok(cudaEventRecord(done, cs.out))) ok(cudaStreamWaitEvent(stream, done, 0));
  }
  for (auto& e : ev) cudaEventDestroy(e);  // released once the work using them completes
  return st;
}
