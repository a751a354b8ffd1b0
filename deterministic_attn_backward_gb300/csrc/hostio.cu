// hostio.cu -- the attention backward on host buffers, copies overlapped
// with the computation.
//
// The heads are split into chunks of consecutive (b, h) heads.  On two copy
// streams owned by the library, the inputs of every chunk are copied to the
// device back to back, and the gradients of chunk c are copied back while
// later chunks are computed.  The backward of each chunk is an ordinary
// dab_attn_bwd_ex call on that range of heads (B = 1, H = heads in the
// chunk), so every chunk computes exactly what the whole call would for those
// heads.  Even chunks run on the caller's stream and odd chunks on a third
// library stream, each stream with its own backward workspace, and the main
// kernel is launched with DAB_BWD_SHARE_GPU: the next chunk's CTAs start on
// the SMs that the current chunk's last, partly filled wave leaves idle.
// Events order the streams: everything starts after the work already queued
// on the caller's stream, and the caller's stream waits for the last copy
// back (which itself waits for every chunk's computation).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "dab.h"

namespace dab {
cudaError_t launch_status_collect(const uint32_t* slots, int n, void* hdr, cudaStream_t stream);
}

namespace {

constexpr int kMaxDevices = 64;
constexpr int kDefaultChunks = 8;

struct CopyStreams {
  cudaStream_t in = nullptr, out = nullptr, comp = nullptr;  // comp: odd chunks
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
    cudaStream_t st[3] = {nullptr, nullptr, nullptr};
    for (int i = 0; i < 3; ++i) {
      if (cudaStreamCreateWithFlags(&st[i], cudaStreamNonBlocking) != cudaSuccess) {
        for (int j = 0; j < i; ++j) cudaStreamDestroy(st[j]);
        return false;
      }
    }
    s.in = st[0];
    s.out = st[1];
    s.comp = st[2];
  }
  *cs = s;
  return true;
}

size_t round_up(size_t x) { return (x + 255) / 256 * 256; }

// Device workspace of the host path: a status header (the first device
// error of any chunk, collected at the end of the call, as dab_check_status
// reads it) and one (status, detail) slot per chunk, copies of the inputs
// and outputs, then the backward workspaces of the largest chunk, one per
// compute stream.
struct HostLayout {
  size_t slots, q, k, v, o, dout, lse, dq, dk, dv, ws[2], ws_bytes, total;
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
  L->slots = 256;  // after the status header at offset 0
  size_t off = L->slots + round_up((size_t)L->chunks * 8);
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
  L->ws[0] = off;
  L->ws[1] = off + round_up(L->ws_bytes);
  L->total = L->ws[1] + (L->chunks > 1 ? round_up(L->ws_bytes) : 0);
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
  if (B >= 0 && H >= 0 && S >= 0 && (long long)B * H * S == 0) {  // empty problem: no kernel
    if (dab_bwd_workspace_size(B, H, S, d, mask, sched) == 0) return DAB_ERR_INVALID_ARG;
    // the status header still reports this call
    if (dev_ws != nullptr && (reinterpret_cast<uintptr_t>(dev_ws) & 15u) == 0 && dev_ws_bytes >= 8 &&
        cudaMemsetAsync(dev_ws, 0, 8, stream) != cudaSuccess)
      return DAB_ERR_CUDA;
    return DAB_OK;
  }
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
  // everything starts after what is already queued on the caller's stream
  if (ok(cudaEventRecord(start, stream)) && ok(cudaStreamWaitEvent(cs.in, start, 0)) &&
      ok(cudaStreamWaitEvent(cs.out, start, 0)) && ok(cudaStreamWaitEvent(cs.comp, start, 0))) {
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
    dab_bwd_opts_t opts;
    opts.spin_timeout_ns = 0;
    opts.flags = DAB_BWD_SHARE_GPU;
    opts.grid = 0;
    for (int c = 0; c < L.chunks && st == DAB_OK; ++c) {  // compute chunk c, then copy it back
      const long long h0 = (long long)c * L.per_chunk;
      const long long nh = (h0 + L.per_chunk <= bh) ? L.per_chunk : bh - h0;
      cudaStream_t cstream = (c % 2 == 0) ? stream : cs.comp;
      if (!ok(cudaStreamWaitEvent(cstream, ev[c], 0))) break;
      auto dp = [&](size_t off) { return static_cast<void*>(w + off + h0 * head_t); };
      const dab_status_t r = dab_attn_bwd_ex(
          dp(L.q), dp(L.k), dp(L.v), dp(L.o), reinterpret_cast<const float*>(w + L.lse + h0 * head_r),
          dp(L.dout), dp(L.dq), dp(L.dk), dp(L.dv), 1, (int)nh, S, d, scale, mask, sched,
          w + L.ws[c % 2], L.ws_bytes, cstream, &opts);
      if (r != DAB_OK) {
        st = r;
        break;
      }
      // this chunk's status and detail words, before its workspace is reused
      if (!ok(cudaMemcpyAsync(w + L.slots + 8 * (size_t)c, w + L.ws[c % 2], 8,
                              cudaMemcpyDeviceToDevice, cstream)))
        break;
      if (!ok(cudaEventRecord(ev[L.chunks + c], cstream)) ||
          !ok(cudaStreamWaitEvent(cs.out, ev[L.chunks + c], 0)))
        break;
      for (int i = 0; i < 3; ++i)
        ok(cudaMemcpyAsync(static_cast<uint8_t*>(hout[i]) + h0 * head_t, w + dout_off[i] + h0 * head_t,
                           nh * head_t, cudaMemcpyDeviceToHost, cs.out));
    }
    // the caller's stream continues once everything has been copied back;
    // then the first device error of any chunk goes to the status header
    if (ok(cudaEventRecord(done, cs.out)) && ok(cudaStreamWaitEvent(stream, done, 0)) &&
        st == DAB_OK)
      ok(dab::launch_status_collect(reinterpret_cast<const uint32_t*>(w + L.slots), L.chunks, w,
                                    stream));
  }
  for (auto& e : ev) cudaEventDestroy(e);  // released once the work using them completes
  return st;
}
