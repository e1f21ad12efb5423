// attn_fwd_bwd_host: one forward + backward of the attention path whose
// inputs and results live in host memory. The heads are split into chunks;
// the host-to-device copies of a chunk, the kernels of the chunk before it
// and the device-to-host copies of the chunk before that run at the same
// time (the two directions use separate copy engines; on GB300 the host
// link carries about 210 GB/s one way and 336 GB/s both ways at once). The
// kernels are the library's own attn_fwd and attn_bwd, called per chunk;
// this file only orders copies and launches. The chunks alternate between
// the caller's stream and a second kernel stream, and each chunk's backward
// takes its own part of the workspace, so the kernels of two neighbouring
// chunks may run at once: the SMs that one launch's last, partial wave of
// work leaves idle take the next chunk's work instead. The declaration is
// in include/attn.h.
#include "attn.h"

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 64;
// Automatic split: about 24 MiB of inputs a chunk, at most 8 chunks. The
// first chunk's inputs and the last chunk's results are the part of the
// copies that nothing overlaps; smaller chunks shrink it but add per-copy
// and per-launch costs (for the base model's 96 x 8 heads of 256 rows, 100 MB
// of inputs: 4 chunks 0.81 ms, 8 chunks 0.87, 16 chunks 0.90, 1 chunk 1.06).
constexpr size_t kAutoChunkBytes = size_t(24) << 20;
constexpr int kAutoMaxChunks = 8;

// Streams and events of the pipeline, created once per device on first use
// and kept until exit. The events are re-recorded by every call: a wait
// enqueued on a stream takes the event's record at the time of the wait, so
// a later record does not disturb it. One copy stream per direction: a
// second stream in the same direction only shares the link (measured
// slower: 0.96 ms against 0.81 for the case above) and delays the first chunk.
struct Pipe {
  cudaStream_t h2d = nullptr;
  cudaStream_t d2h = nullptr;
  cudaStream_t kern = nullptr;  // kernels of the odd chunks (the even ones run on the caller's stream)
  cudaEvent_t start = nullptr;
  cudaEvent_t in_ready[kMaxChunks] = {};   // inputs of chunk c are on the device
  cudaEvent_t fwd_done[kMaxChunks] = {};   // O and lse of chunk c are written
  cudaEvent_t bwd_done[kMaxChunks] = {};   // dQ, dK, dV of chunk c are written
  cudaEvent_t drained[3] = {};
  bool ready = false;
};

std::mutex g_mu[kMaxDevices];  // one call at a time per device: the events are shared
Pipe g_pipe[kMaxDevices];

cudaError_t pipe_setup(Pipe& P) {
  if (P.ready) return cudaSuccess;
  // What an earlier, failed set-up made is kept and only the rest is made.
  cudaError_t e = cudaSuccess;
  auto stream = [&e](cudaStream_t& x) {
    if (e == cudaSuccess && x == nullptr) e = cudaStreamCreateWithFlags(&x, cudaStreamNonBlocking);
  };
  auto event = [&e](cudaEvent_t& x) {
    if (e == cudaSuccess && x == nullptr) e = cudaEventCreateWithFlags(&x, cudaEventDisableTiming);
  };
  stream(P.h2d);
  stream(P.d2h);
  stream(P.kern);
  event(P.start);
  for (int c = 0; c < kMaxChunks; ++c) {
    event(P.in_ready[c]);
    event(P.fwd_done[c]);
    event(P.bwd_done[c]);
  }
  for (int i = 0; i < 3; ++i) event(P.drained[i]);
  if (e == cudaSuccess) P.ready = true;
  return e;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Bytes of one head of a [BH, rows, cols] tensor with `elem`-byte elements.
size_t head_bytes(int rows, int cols, int elem) {
  return static_cast<size_t>(rows) * static_cast<size_t>(cols) * static_cast<size_t>(elem);
}

}  // namespace

extern "C" int attn_fwd_bwd_host(const void* hq, const void* hk, const void* hv, const void* hdO,
                                 void* ho, float* hlse, void* hdq, void* hdk, void* hdv,
                                 void* q, void* k, void* v, void* dO, void* o, float* lse,
                                 void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                                 int B, int h, int n, int m, int d_k, int d_v, int causal, float scale,
                                 int chunks, attn_stream_t stream) {
  // Everything that can be refused is refused before anything is enqueued.
  if (B < 0 || h < 0 || n < 0 || m < 1 || d_k < 1 || d_v < 1 || chunks < 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (d_k != d_v) return ATTN_ERR_UNSUPPORTED;
  if (d_k != 32 && d_k != 64 && d_k != 128) return ATTN_ERR_UNSUPPORTED;
  const long long BH_ll = static_cast<long long>(B) * h;
  if (BH_ll > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  if ((static_cast<long long>(n) + 255) / 256 > 65535) return ATTN_ERR_UNSUPPORTED;
  if ((static_cast<long long>(m) + 127) / 128 > 65535) return ATTN_ERR_UNSUPPORTED;
  const int BH = static_cast<int>(BH_ll);
  if (BH == 0) return ATTN_OK;
  // Without query rows (n = 0) only the key side takes part: dK = dV = 0.
  if (!hk || !hv || !hdk || !hdv || !k || !v || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (n > 0 && (!hq || !hdO || !hdq || !q || !dO || !o || !lse || !dq)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(o) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv))
    return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return ATTN_ERR_INVALID_ARG;
  const size_t ws_need = attn_bwd_workspace_bytes(B, h, n, m, d_k, d_v, causal);
  if (ws_need > 0 && (!workspace || !aligned16(workspace) || workspace_bytes < ws_need))
    return ATTN_ERR_INVALID_ARG;

  // Per-head bytes of every tensor.
  const size_t b_q = head_bytes(n, d_k, 2), b_k = head_bytes(m, d_k, 2), b_v = head_bytes(m, d_v, 2);
  const size_t b_o = head_bytes(n, d_v, 2), b_lse = head_bytes(n, 1, 4);
  if (chunks == 0) {
    const size_t in_bytes = static_cast<size_t>(BH) * (b_q + b_k + b_v + b_o);
    size_t c = in_bytes / kAutoChunkBytes;
    chunks = static_cast<int>(c < 1 ? 1 : (c > kAutoMaxChunks ? kAutoMaxChunks : c));
  }
  if (chunks > kMaxChunks) chunks = kMaxChunks;
  if (chunks > BH) chunks = BH;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu[dev]);
  Pipe& P = g_pipe[dev];
  if (pipe_setup(P) != cudaSuccess) return ATTN_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  // The copies into the device buffers start after the work already queued on
  // `stream` (which may still read them).
  if (cudaEventRecord(P.start, s) != cudaSuccess) return ATTN_ERR_CUDA;
  if (cudaStreamWaitEvent(P.h2d, P.start, 0) != cudaSuccess || cudaStreamWaitEvent(P.d2h, P.start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(P.kern, P.start, 0) != cudaSuccess)
    return ATTN_ERR_CUDA;  // nothing copied yet: no stream of the call is ahead of `stream`

  auto at = [](const void* base, size_t off) {
    return static_cast<void*>(static_cast<char*>(const_cast<void*>(base)) + off);
  };
  auto h2d = [&](void* dst, const void* src, size_t bytes, cudaStream_t cs) {
    return bytes == 0 || cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, cs) == cudaSuccess;
  };
  auto d2h = [&](void* dst, const void* src, size_t bytes, cudaStream_t cs) {
    return bytes == 0 || cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, cs) == cudaSuccess;
  };

  int status = ATTN_OK;
  // Stage 1: every chunk's inputs, in chunk order.
  for (int c = 0; c < chunks && status == ATTN_OK; ++c) {
    const int h0 = static_cast<int>(static_cast<long long>(BH) * c / chunks);
    const int h1 = static_cast<int>(static_cast<long long>(BH) * (c + 1) / chunks);
    const size_t nh = static_cast<size_t>(h1 - h0);
    cudaStream_t cs = P.h2d;
    const bool ok = h2d(at(q, h0 * b_q), at(hq, h0 * b_q), nh * b_q, cs) &&
                    h2d(at(k, h0 * b_k), at(hk, h0 * b_k), nh * b_k, cs) &&
                    h2d(at(v, h0 * b_v), at(hv, h0 * b_v), nh * b_v, cs) &&
                    h2d(at(dO, h0 * b_o), at(hdO, h0 * b_o), nh * b_o, cs) &&
                    cudaEventRecord(P.in_ready[c], cs) == cudaSuccess;
    if (!ok) status = ATTN_ERR_CUDA;
  }
  // Stage 2 and 3: per chunk, the kernels once its inputs landed, then its
  // results back on a device-to-host stream (O and lse right after the
  // forward, the gradients after the backward). A chunk's forward also waits
  // for the previous chunk's forward, so at most two chunks are in flight and
  // they finish in order: it runs beside the previous chunk's backward.
  for (int c = 0; c < chunks && status == ATTN_OK; ++c) {
    const int h0 = static_cast<int>(static_cast<long long>(BH) * c / chunks);
    const int h1 = static_cast<int>(static_cast<long long>(BH) * (c + 1) / chunks);
    const int nh = h1 - h0;
    cudaStream_t ks = (c & 1) ? P.kern : s;
    if (cudaStreamWaitEvent(ks, P.in_ready[c], 0) != cudaSuccess ||
        (c > 0 && cudaStreamWaitEvent(ks, P.fwd_done[c - 1], 0) != cudaSuccess)) {
      status = ATTN_ERR_CUDA;
      break;
    }
    // The workspace holds the whole batch's per-head scratch in head order;
    // this chunk takes the part of its own heads.
    void* ws_c = workspace;
    size_t ws_c_bytes = workspace_bytes;
    if (ws_need > 0) {
      ws_c = at(workspace, attn_bwd_workspace_bytes(h0, 1, n, m, d_k, d_v, causal));
      ws_c_bytes = attn_bwd_workspace_bytes(nh, 1, n, m, d_k, d_v, causal);
    }
    // A chunk is nh heads of one sequence each: no argument of the kernels
    // depends on how the heads group into sequences (there is no key padding here).
    float* lse_c = reinterpret_cast<float*>(at(lse, h0 * b_lse));
    const attn_stream_t kst = reinterpret_cast<attn_stream_t>(ks);
    status = attn_fwd(at(q, h0 * b_q), at(k, h0 * b_k), at(v, h0 * b_v), at(o, h0 * b_o), lse_c, nh, 1, n, m, d_k,
                      d_v, causal, scale, kst);
    if (status != ATTN_OK) break;
    if (cudaEventRecord(P.fwd_done[c], ks) != cudaSuccess) {
      status = ATTN_ERR_CUDA;
      break;
    }
    status = attn_bwd(at(q, h0 * b_q), at(k, h0 * b_k), at(v, h0 * b_v), at(o, h0 * b_o), lse_c, at(dO, h0 * b_o),
                      at(dq, h0 * b_q), at(dk, h0 * b_k), at(dv, h0 * b_v), nh, 1, n, m, d_k, d_v, causal, scale,
                      ws_c, ws_c_bytes, kst);
    if (status != ATTN_OK) break;
    if (cudaEventRecord(P.bwd_done[c], ks) != cudaSuccess) {
      status = ATTN_ERR_CUDA;
      break;
    }
    cudaStream_t cs = P.d2h;
    const size_t z = static_cast<size_t>(nh);
    const bool ok = cudaStreamWaitEvent(cs, P.fwd_done[c], 0) == cudaSuccess &&
                    (ho == nullptr || d2h(at(ho, h0 * b_o), at(o, h0 * b_o), z * b_o, cs)) &&
                    (hlse == nullptr || d2h(at(hlse, h0 * b_lse), lse_c, z * b_lse, cs)) &&
                    cudaStreamWaitEvent(cs, P.bwd_done[c], 0) == cudaSuccess &&
                    d2h(at(hdq, h0 * b_q), at(dq, h0 * b_q), z * b_q, cs) &&
                    d2h(at(hdk, h0 * b_k), at(dk, h0 * b_k), z * b_k, cs) &&
                    d2h(at(hdv, h0 * b_v), at(dv, h0 * b_v), z * b_v, cs);
    if (!ok) status = ATTN_ERR_CUDA;
  }
  // `stream` continues only after every copy of this call (also after an
  // error, so that no copy of this call outlives it unordered).
  const bool drained = cudaEventRecord(P.drained[0], P.h2d) == cudaSuccess &&
                       cudaEventRecord(P.drained[1], P.d2h) == cudaSuccess &&
                       cudaEventRecord(P.drained[2], P.kern) == cudaSuccess &&
                       cudaStreamWaitEvent(s, P.drained[0], 0) == cudaSuccess &&
                       cudaStreamWaitEvent(s, P.drained[1], 0) == cudaSuccess &&
                       cudaStreamWaitEvent(s, P.drained[2], 0) == cudaSuccess;
  if (!drained && status == ATTN_OK) status = ATTN_ERR_CUDA;
  return status;
}
