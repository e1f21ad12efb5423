// C ABI of the attention library: argument checks, TMA tensor-map encoding,
// kernel launches and the device error word. The declarations, with the
// meaning of every argument, are in include/attn.h.
#include "attn.h"
#include "attn_kernels.cuh"

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

namespace {

using attn::BwdHeadParams;
using attn::BwdParams;
using attn::BwdPostParams;
using attn::BwdPreParams;
using attn::FwdParams;

constexpr unsigned long long kDefaultWatchdogNs = 2000000000ull;  // 2 s per wait
constexpr int kMaxDevices = 64;

std::atomic<unsigned long long> g_watchdog_ns{kDefaultWatchdogNs};
std::atomic<int> g_inject{0};

// One device error word per device, allocated on first use and kept until exit.
std::mutex g_status_mu;
uint32_t* g_status[kMaxDevices] = {nullptr};

cudaError_t device_status_word(uint32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (g_status[dev] == nullptr) {
    uint32_t* p = nullptr;
    e = cudaMalloc(&p, sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    e = cudaMemset(p, 0, sizeof(uint32_t));
    if (e != cudaSuccess) {
      cudaFree(p);
      return e;
    }
    g_status[dev] = p;
  }
  *out = g_status[dev];
  return cudaSuccess;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// 3-D map over a [BH, S, d] bf16 tensor: box = (atom, box_rows, 1 head).
// Rows past S read as zero (out-of-bounds fill), so ragged tiles never touch
// the next head.
bool make_tile_map(CUtensorMap* map, const void* base, long long BH, long long S, int d,
                   int box_rows = 128) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const int atom = d >= 64 ? 64 : d;
  const CUtensorMapSwizzle sw = d >= 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(S),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(S) * d * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(atom), static_cast<cuuint32_t>(box_rows), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D map over a row-major bf16 array [d2][d1][d0] (d0 fastest): box =
// (64, box1, 1), 128-byte swizzle. Out-of-bounds reads are zero, stores clip.
bool make_map3(CUtensorMap* map, const void* base, long long d0, long long d1, long long d2, int box1) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d0), static_cast<cuuint64_t>(d1), static_cast<cuuint64_t>(d2)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d0) * 2, static_cast<cuuint64_t>(d0 * d1) * 2};
  cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(box1), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D map over the fp32 dQ accumulator [rows, d]: box = (32 columns, 128 rows),
// 128-byte swizzle (the layout the backward kernel stages its dQ tile in).
bool make_dq_map(CUtensorMap* map, const float* base, long long rows, int d) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 4};
  cuuint32_t box[2] = {32u, 128u};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr double kLog2e = 1.4426950408889634074;

// Shared checks of attn_fwd / attn_bwd. Returns ATTN_OK to proceed, or the
// status to return; *empty is set when there is nothing to compute.
int check_common(int B, int h, int n, int m, int d_k, int d_v, float scale, bool* empty) {
  *empty = false;
  if (B < 0 || h < 0 || n < 0 || m < 1 || d_k < 1 || d_v < 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (d_k != d_v) return ATTN_ERR_UNSUPPORTED;
  if (d_k != 32 && d_k != 64 && d_k != 128) return ATTN_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * h;
  if (BH > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  if ((static_cast<long long>(n) + 255) / 256 > 65535) return ATTN_ERR_UNSUPPORTED;
  if ((static_cast<long long>(m) + 127) / 128 > 65535) return ATTN_ERR_UNSUPPORTED;
  if (BH == 0 || n == 0) *empty = true;
  return ATTN_OK;
}

long long round_up(long long x, long long a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------- profiling

struct EventPair {
  cudaEvent_t begin = nullptr, end = nullptr;
  int kind = 0;
};

std::atomic<int> g_prof_on{0};
std::mutex g_prof_mu;
std::vector<EventPair> g_prof_pending;  // recorded, not yet read
std::vector<EventPair> g_prof_free;     // created, reusable
EventPair g_prof_open[attn::kNumKinds];  // begun, waiting for prof_end
double g_prof_ms[attn::kNumKinds] = {};
int g_prof_count[attn::kNumKinds] = {};

// Moves every pending pair's elapsed time into the per-kind totals.
cudaError_t prof_drain_locked() {
  for (EventPair& ep : g_prof_pending) {
    cudaError_t e = cudaEventSynchronize(ep.end);
    if (e != cudaSuccess) return e;
    float ms = 0.f;
    e = cudaEventElapsedTime(&ms, ep.begin, ep.end);
    if (e != cudaSuccess) return e;
    g_prof_ms[ep.kind] += ms;
    g_prof_count[ep.kind] += 1;
    g_prof_free.push_back(ep);
  }
  g_prof_pending.clear();
  return cudaSuccess;
}

}  // namespace

namespace attn {

void prof_begin(int kind, cudaStream_t stream) {
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  EventPair ep;
  if (!g_prof_free.empty()) {
    ep = g_prof_free.back();
    g_prof_free.pop_back();
  } else if (cudaEventCreate(&ep.begin) != cudaSuccess || cudaEventCreate(&ep.end) != cudaSuccess) {
    return;
  }
  ep.kind = kind;
  cudaEventRecord(ep.begin, stream);
  g_prof_open[kind] = ep;
}

void prof_end(int kind, cudaStream_t stream) {
  if (!g_prof_on.load(std::memory_order_relaxed)) return;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  EventPair ep = g_prof_open[kind];
  if (ep.begin == nullptr) return;
  g_prof_open[kind] = EventPair{};
  cudaEventRecord(ep.end, stream);
  g_prof_pending.push_back(ep);
}

}  // namespace attn

// ---------------------------------------------------------------- allocation-free backward
//
// Scratch of attn_bwd_noalloc: the fp32 dQ accumulator and the two padded
// per-row statistics live in this fixed device array instead of a
// caller-provided workspace. It exists once per device that loads the
// library and stays until the process exits.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
// Watchdog word for devices on which no attn_fwd/attn_bwd call has created
// the per-device error word yet (that word needs an allocation).
__device__ uint32_t g_noalloc_status;

std::once_flag g_noalloc_once[kMaxDevices];
void* g_noalloc_scratch_ptr[kMaxDevices] = {nullptr};
uint32_t* g_noalloc_status_ptr[kMaxDevices] = {nullptr};
cudaError_t g_noalloc_setup_err[kMaxDevices] = {cudaSuccess};

}  // namespace

extern "C" {

int attn_profile_enable(int on) {
  g_prof_on.store(on ? 1 : 0);
  return ATTN_OK;
}

int attn_profile_read(int kind, int* launches, double* total_ms) {
  if (kind < 0 || kind >= attn::kNumKinds) return ATTN_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (prof_drain_locked() != cudaSuccess) return ATTN_ERR_CUDA;
  if (launches) *launches = g_prof_count[kind];
  if (total_ms) *total_ms = g_prof_ms[kind];
  g_prof_count[kind] = 0;
  g_prof_ms[kind] = 0.0;
  return ATTN_OK;
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    default: return "ATTN_ERR_UNKNOWN";
  }
}

int attn_set_watchdog_ns(unsigned long long budget_ns) {
  g_watchdog_ns.store(budget_ns == 0 ? kDefaultWatchdogNs : budget_ns);
  return ATTN_OK;
}

int attn_debug_inject(int mode) {
  if (mode != 0 && mode != 1) return ATTN_ERR_INVALID_ARG;
  g_inject.store(mode);
  return ATTN_OK;
}

// A window side: negative or reaching past every position is open (-1).
static int window_side(int w, int n, int m) {
  if (w < 0) return -1;
  return (static_cast<long long>(w) >= static_cast<long long>(n) + m) ? -1 : w;
}

// attn_fwd / attn_fwd_varlen / attn_fwd_masked: kv_len (device, B ints, or
// nullptr) are the real keys of each sequence, which the kernels clamp to
// [0, m]; wl / wr the restricted-attention window (-1: open side).
static int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, const int* kv_len,
                    int B, int h, int n, int m, int d_k, int d_v, int causal, int wl, int wr, float scale,
                    attn_stream_t stream) {
  bool empty = false;
  int st = check_common(B, h, n, m, d_k, d_v, scale, &empty);
  if (st != ATTN_OK) return st;
  if (empty) return ATTN_OK;
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_INVALID_ARG;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return ATTN_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * h;
  CUtensorMap tq, tk, tv, to;
  wl = window_side(wl, n, m);
  wr = window_side(wr, n, m);
  const int bn = attn::fwd_key_tile(d_k, n, m, causal ? 1 : 0, wl >= 0 || wr >= 0);
  if (!make_tile_map(&tq, q, BH, n, d_k) || !make_tile_map(&tk, k, BH, m, d_k, bn) ||
      !make_tile_map(&tv, v, BH, m, d_v, bn) || !make_tile_map(&to, o, BH, n, d_v))
    return ATTN_ERR_CUDA;
  uint32_t* status = nullptr;
  if (device_status_word(&status) != cudaSuccess) return ATTN_ERR_CUDA;
  FwdParams p{};
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.n = n;
  p.m = m;
  p.causal = causal ? 1 : 0;
  p.neg = scale < 0.f ? 1 : 0;
  p.c = static_cast<float>(std::fabs(static_cast<double>(scale)) * kLog2e);
  p.num_qblocks = 0;  // set by the launcher for its query-tile configuration
  p.inject = g_inject.exchange(0);
  p.kv_len = kv_len;
  p.h = h;
  p.wl = wl;
  p.wr = wr;
  p.wd.status = status;
  p.wd.budget_ns = g_watchdog_ns.load();
  cudaError_t e = attn::launch_fwd(d_k, tq, tk, tv, to, p, static_cast<int>(BH),
                                   reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

size_t attn_bwd_workspace_bytes(int B, int h, int n, int m, int d_k, int d_v, int causal) {
  (void)m;
  (void)causal;
  if (B <= 0 || h <= 0 || n <= 0 || d_k <= 0) return 0;
  if (d_k == d_v && attn::bwd_head_supported(n, d_k)) return 0;  // whole-head kernel: no scratch
  const long long BH = static_cast<long long>(B) * h;
  const long long n_pad = round_up(n, 128);
  // dQ accumulator [BH, n_pad, d] + lse*log2(e) [BH, n_pad] + D [BH, n_pad], fp32
  return static_cast<size_t>(BH * n_pad * (static_cast<long long>(d_k) + 2) * 4);
}

// Short query sequences: the whole-head kernel (no scratch, one launch).
static int bwd_head_path(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dO, void* dq, void* dk, void* dv, const int* kv_len, long long BH,
                         int h, int n, int m, int d, int causal, int wl, int wr, float scale,
                         uint32_t* status, cudaStream_t stream) {
  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
  if (!make_tile_map(&tq, q, BH, n, d) || !make_tile_map(&tk, k, BH, m, d) ||
      !make_tile_map(&tv, v, BH, m, d) || !make_tile_map(&tdo, dO, BH, n, d) ||
      !make_tile_map(&tdq, dq, BH, n, d) || !make_tile_map(&tdk, dk, BH, m, d) ||
      !make_tile_map(&tdv, dv, BH, m, d))
    return ATTN_ERR_CUDA;
  BwdHeadParams p{};
  p.o = static_cast<const __nv_bfloat16*>(o);
  p.dO = static_cast<const __nv_bfloat16*>(dO);
  p.lse = lse;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.BH = static_cast<int>(BH);
  p.n = n;
  p.m = m;
  p.causal = causal ? 1 : 0;
  p.neg = scale < 0.f ? 1 : 0;
  p.c = static_cast<float>(std::fabs(static_cast<double>(scale)) * kLog2e);
  p.scale = scale;
  p.kv_len = kv_len;
  p.h = h;
  p.wl = wl;
  p.wr = wr;
  p.wd.status = status;
  p.wd.budget_ns = g_watchdog_ns.load();
  const cudaError_t e = attn::launch_bwd_head(d, tq, tk, tv, tdo, tdq, tdk, tdv, p, stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

static int bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv, const int* kv_len, int B, int h,
                    int n, int m, int d_k, int d_v, int causal, int wl, int wr, float scale, void* workspace,
                    size_t workspace_bytes, attn_stream_t stream) {
  bool empty = false;
  int st = check_common(B, h, n, m, d_k, d_v, scale, &empty);
  if (st != ATTN_OK) return st;
  wl = window_side(wl, n, m);
  wr = window_side(wr, n, m);
  if (!k || !v || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv)) return ATTN_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * h;
  if (empty) {
    // No query rows: every gradient is zero. dK and dV still have BH*m rows.
    if (BH == 0) return ATTN_OK;
    const size_t bytes = static_cast<size_t>(BH) * m * d_k * 2;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(dk, 0, bytes, s) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemsetAsync(dv, 0, bytes, s) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  if (!q || !o || !lse || !dO || !dq) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o) || !aligned16(dO) || !aligned16(dq)) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return ATTN_ERR_INVALID_ARG;
  const size_t ws_need = attn_bwd_workspace_bytes(B, h, n, m, d_k, d_v, causal);
  if (ws_need == 0) {
    uint32_t* status = nullptr;
    if (device_status_word(&status) != cudaSuccess) return ATTN_ERR_CUDA;
    return bwd_head_path(q, k, v, o, lse, dO, dq, dk, dv, kv_len, BH, h, n, m, d_k, causal, wl, wr, scale,
                         status, reinterpret_cast<cudaStream_t>(stream));
  }
  if (!workspace || !aligned16(workspace) || workspace_bytes < ws_need) return ATTN_ERR_INVALID_ARG;

  const long long n_pad = round_up(n, 128);
  float* ws = static_cast<float*>(workspace);
  float* dq_acc = ws;
  float* lse2 = dq_acc + BH * n_pad * d_k;
  float* Dsum = lse2 + BH * n_pad;

  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
  if (!make_tile_map(&tq, q, BH, n, d_k) || !make_tile_map(&tk, k, BH, m, d_k) ||
      !make_tile_map(&tv, v, BH, m, d_v) || !make_tile_map(&tdo, dO, BH, n, d_v) ||
      !make_dq_map(&tdq, dq_acc, BH * n_pad, d_k) || !make_tile_map(&tdk, dk, BH, m, d_k) ||
      !make_tile_map(&tdv, dv, BH, m, d_v))
    return ATTN_ERR_CUDA;
  uint32_t* status = nullptr;
  if (device_status_word(&status) != cudaSuccess) return ATTN_ERR_CUDA;

  BwdPreParams pre{};
  pre.o = static_cast<const __nv_bfloat16*>(o);
  pre.dO = static_cast<const __nv_bfloat16*>(dO);
  pre.lse = lse;
  pre.lse2 = lse2;
  pre.Dsum = Dsum;
  pre.dq_acc = dq_acc;
  pre.n = n;
  pre.n_pad = static_cast<int>(n_pad);
  pre.d = d_k;
  pre.BH = static_cast<int>(BH);

  BwdParams p{};
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.lse2 = lse2;
  p.Dsum = Dsum;
  p.dq_acc = dq_acc;
  p.n = n;
  p.m = m;
  p.n_pad = static_cast<int>(n_pad);
  p.causal = causal ? 1 : 0;
  p.neg = scale < 0.f ? 1 : 0;
  p.c = static_cast<float>(std::fabs(static_cast<double>(scale)) * kLog2e);
  p.scale = scale;
  p.num_kblocks = static_cast<int>((m + 127) / 128);
  p.kv_len = kv_len;
  p.h = h;
  p.wl = wl;
  p.wr = wr;
  p.wd.status = status;
  p.wd.budget_ns = g_watchdog_ns.load();

  BwdPostParams post{};
  post.dq_acc = dq_acc;
  post.dq = static_cast<__nv_bfloat16*>(dq);
  post.scale = scale;
  post.n = n;
  post.n_pad = static_cast<int>(n_pad);
  post.d = d_k;
  post.BH = static_cast<int>(BH);

  cudaError_t e = attn::launch_bwd(d_k, tq, tk, tv, tdk, tdv, tdo, tdq, pre, p, post, static_cast<int>(BH),
                                   reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int h, int n,
             int m, int d_k, int d_v, int causal, float scale, attn_stream_t stream) {
  return fwd_impl(q, k, v, o, lse, nullptr, B, h, n, m, d_k, d_v, causal, -1, -1, scale, stream);
}

int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* kv_len,
                    int B, int h, int n, int m, int d_k, int d_v, int causal, float scale,
                    attn_stream_t stream) {
  if ((reinterpret_cast<uintptr_t>(kv_len) & 3u) != 0) return ATTN_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, kv_len, B, h, n, m, d_k, d_v, causal, -1, -1, scale, stream);
}

int attn_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, const int* kv_len,
                    int B, int h, int n, int m, int d_k, int d_v, int causal, int window_left,
                    int window_right, float scale, attn_stream_t stream) {
  if ((reinterpret_cast<uintptr_t>(kv_len) & 3u) != 0) return ATTN_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, kv_len, B, h, n, m, d_k, d_v, causal, window_left, window_right, scale,
                  stream);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dO, void* dq, void* dk, void* dv, int B, int h, int n, int m, int d_k,
             int d_v, int causal, float scale, void* workspace, size_t workspace_bytes,
             attn_stream_t stream) {
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, nullptr, B, h, n, m, d_k, d_v, causal, -1, -1, scale,
                  workspace, workspace_bytes, stream);
}

int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv, const int* kv_len, int B, int h,
                    int n, int m, int d_k, int d_v, int causal, float scale, void* workspace,
                    size_t workspace_bytes, attn_stream_t stream) {
  if ((reinterpret_cast<uintptr_t>(kv_len) & 3u) != 0) return ATTN_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, kv_len, B, h, n, m, d_k, d_v, causal, -1, -1, scale,
                  workspace, workspace_bytes, stream);
}

int attn_bwd_masked(const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv, const int* kv_len, int B, int h,
                    int n, int m, int d_k, int d_v, int causal, int window_left, int window_right,
                    float scale, void* workspace, size_t workspace_bytes, attn_stream_t stream) {
  if ((reinterpret_cast<uintptr_t>(kv_len) & 3u) != 0) return ATTN_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o, lse, dO, dq, dk, dv, kv_len, B, h, n, m, d_k, d_v, causal, window_left,
                  window_right, scale, workspace, workspace_bytes, stream);
}

size_t attn_decode_workspace_bytes(int B, int h, int n, int m, int d_k, int d_v) {
  (void)d_v;
  if (B <= 0 || h <= 0 || n <= 0 || m <= 0 || d_k <= 0) return 0;
  const long long BH = static_cast<long long>(B) * h;
  int splits = 1, chunk = 0;
  attn::decode_split(BH, m, &splits, &chunk);
  return static_cast<size_t>(BH * splits * n * (static_cast<long long>(d_k) + 2) * 4);
}

int attn_decode(const void* q, const void* k, const void* v, void* o, float* lse, const int* kv_len, int B, int h,
                int n, int m, int d_k, int d_v, float scale, void* workspace, size_t workspace_bytes,
                attn_stream_t stream) {
  if (B < 0 || h < 0 || m < 1 || n < 1 || n > attn::kDecMaxN || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (d_k != d_v || (d_k != 32 && d_k != 64 && d_k != 128)) return ATTN_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * h;
  if (BH > 65535) return ATTN_ERR_UNSUPPORTED;  // grid y
  if (BH == 0) return ATTN_OK;
  if (!q || !k || !v || !o || !workspace) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(workspace))
    return ATTN_ERR_INVALID_ARG;
  if ((lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) ||
      (reinterpret_cast<uintptr_t>(kv_len) & 3u) != 0)
    return ATTN_ERR_INVALID_ARG;
  if (workspace_bytes < attn_decode_workspace_bytes(B, h, n, m, d_k, d_v)) return ATTN_ERR_INVALID_ARG;
  CUtensorMap tk, tv;
  if (!make_tile_map(&tk, k, BH, m, d_k, 64) || !make_tile_map(&tv, v, BH, m, d_v, 64)) return ATTN_ERR_CUDA;
  uint32_t* status = nullptr;
  if (device_status_word(&status) != cudaSuccess) return ATTN_ERR_CUDA;
  attn::DecParams p{};
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.part = static_cast<float*>(workspace);
  p.kv_len = kv_len;
  p.h = h;
  p.n = n;
  p.m = m;
  attn::decode_split(BH, m, &p.splits, &p.chunk);
  p.c = static_cast<float>(static_cast<double>(scale) * kLog2e);
  p.wd.status = status;
  p.wd.budget_ns = g_watchdog_ns.load();
  const cudaError_t e = attn::launch_decode(d_k, tk, tv, p, static_cast<int>(BH),
                                            reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Checks shared by the projections: head sizes 64 / 128 (whole 64-column
// boxes per head), widths that are multiples of the 64-column boxes.
static int check_proj(int B, int n, int d_model, int h, int d) {
  if (B < 0 || n < 0 || d_model < 1 || h < 1) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (d_model % 64 != 0) return ATTN_ERR_UNSUPPORTED;
  const long long hd = static_cast<long long>(h) * d;
  if (hd > 0x3fffffff || static_cast<long long>(B) * h > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

int attn_qkv_projection(const void* x_q, const void* x_kv, const void* w_qkv, void* q, void* k, void* v, int B,
                        int n, int m, int d_model, int h, int d, attn_stream_t stream) {
  int st = check_proj(B, n, d_model, h, d);
  if (st != ATTN_OK) return st;
  if (m < 0) return ATTN_ERR_INVALID_ARG;
  if ((static_cast<long long>(h) * d) % 128 != 0) return ATTN_ERR_UNSUPPORTED;  // tiles never straddle Q | K | V
  if (B == 0 || (n == 0 && m == 0)) return ATTN_OK;
  if (!x_q || !x_kv || !w_qkv || !q || !k || !v) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(x_q) || !aligned16(x_kv) || !aligned16(w_qkv) || !aligned16(q) || !aligned16(k) || !aligned16(v))
    return ATTN_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * h, hd = static_cast<long long>(h) * d;
  uint32_t* status = nullptr;
  if (device_status_word(&status) != cudaSuccess) return ATTN_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  CUtensorMap tw, tq, tk, tv;
  if (!make_map3(&tw, w_qkv, 3 * hd, d_model, 1, 64)) return ATTN_ERR_CUDA;
  if ((n > 0 && !make_tile_map(&tq, q, BH, n, d)) || (m > 0 && (!make_tile_map(&tk, k, BH, m, d) ||
                                                               !make_tile_map(&tv, v, BH, m, d))))
    return ATTN_ERR_CUDA;
  attn::ProjParams p{};
  p.mode = 0;
  p.B = B;
  p.K = d_model;
  p.h = h;
  p.d = d;
  p.wd.status = status;
  p.wd.budget_ns = g_watchdog_ns.load();
  const bool fused = x_q == x_kv && n == m;
  if (fused) {
    // self-attention: one GEMM against all of W^Q | W^K | W^V
    CUtensorMap tx;
    if (!make_map3(&tx, x_q, d_model, n, B, 128)) return ATTN_ERR_CUDA;
    p.S = n;
    p.N = static_cast<int>(3 * hd);
    p.n_base = 0;
    return attn::launch_proj(tx, tw, tq, tk, tv, p, s) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
  }
  // cross-attention: Q from x_q, K and V from x_kv
  if (n > 0) {
    CUtensorMap tx;
    if (!make_map3(&tx, x_q, d_model, n, B, 128)) return ATTN_ERR_CUDA;
    p.S = n;
    p.N = static_cast<int>(hd);
    p.n_base = 0;
    if (attn::launch_proj(tx, tw, tq, tq, tq, p, s) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  if (m > 0) {
    CUtensorMap tx;
    if (!make_map3(&tx, x_kv, d_model, m, B, 128)) return ATTN_ERR_CUDA;
    p.S = m;
    p.N = static_cast<int>(2 * hd);
    p.n_base = static_cast<int>(hd);
    if (attn::launch_proj(tx, tw, tk, tk, tv, p, s) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

int attn_out_projection(const void* o, const void* w_o, void* y, int B, int n, int d_model, int h, int d,
                        attn_stream_t stream) {
  int st = check_proj(B, n, d_model, h, d);
  if (st != ATTN_OK) return st;
  if (B == 0 || n == 0) return ATTN_OK;
  if (!o || !w_o || !y) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(w_o) || !aligned16(y)) return ATTN_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * h, hd = static_cast<long long>(h) * d;
  uint32_t* status = nullptr;
  if (device_status_word(&status) != cudaSuccess) return ATTN_ERR_CUDA;
  CUtensorMap to, tw, ty;
  if (!make_tile_map(&to, o, BH, n, d) || !make_map3(&tw, w_o, d_model, hd, 1, 64) ||
      !make_map3(&ty, y, d_model, n, B, 128))
    return ATTN_ERR_CUDA;
  attn::ProjParams p{};
  p.mode = 1;
  p.B = B;
  p.S = n;
  p.K = static_cast<int>(hd);
  p.N = d_model;
  p.h = h;
  p.d = d;
  p.n_base = 0;
  p.wd.status = status;
  p.wd.budget_ns = g_watchdog_ns.load();
  return attn::launch_proj(to, tw, ty, ty, ty, p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_CUDA;
}

// ---------------------------------------------------------------- projection backward

// Token splits of the QKV weight gradient: d_model x 3 h d outputs, the longer
// of the two token ranges in 64-token chunks.
static int qkv_bwd_splits(int B, int n, int m, int d_model, int h, int d) {
  const long long hd = static_cast<long long>(h) * d;
  const long long chunks = static_cast<long long>(B) * (((n > m ? n : m) + 63) / 64);
  return attn::proj_bwd_splits(d_model, static_cast<int>(3 * hd), chunks > 0x7fffffff ? 0x7fffffff
                                                                                     : static_cast<int>(chunks));
}

static int out_bwd_splits(int B, int n, int d_model, int h, int d) {
  const long long chunks = static_cast<long long>(B) * ((n + 63) / 64);
  return attn::proj_bwd_splits(h * d, d_model, chunks > 0x7fffffff ? 0x7fffffff : static_cast<int>(chunks));
}

size_t attn_qkv_projection_bwd_workspace_bytes(int B, int n, int m, int d_model, int h, int d) {
  if (check_proj(B, n, d_model, h, d) != ATTN_OK || m < 0 || (static_cast<long long>(h) * d) % 128 != 0) return 0;
  if (B == 0 || (n == 0 && m == 0)) return 0;
  const int z = qkv_bwd_splits(B, n, m, d_model, h, d);
  return static_cast<size_t>(z) * d_model * (3 * static_cast<size_t>(h) * d) * sizeof(float);
}

size_t attn_out_projection_bwd_workspace_bytes(int B, int n, int d_model, int h, int d) {
  if (check_proj(B, n, d_model, h, d) != ATTN_OK) return 0;
  if (B == 0 || n == 0) return 0;
  const int z = out_bwd_splits(B, n, d_model, h, d);
  return static_cast<size_t>(z) * (static_cast<size_t>(h) * d) * d_model * sizeof(float);
}

int attn_qkv_projection_bwd(const void* x_q, const void* x_kv, const void* w_qkv, const void* dq, const void* dk,
                            const void* dv, void* dx_q, void* dx_kv, void* dw_qkv, int B, int n, int m,
                            int d_model, int h, int d, void* workspace, size_t workspace_bytes,
                            attn_stream_t stream) {
  int st = check_proj(B, n, d_model, h, d);
  if (st != ATTN_OK) return st;
  if (m < 0) return ATTN_ERR_INVALID_ARG;
  if ((static_cast<long long>(h) * d) % 128 != 0) return ATTN_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * h, hd = static_cast<long long>(h) * d;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (B == 0) return ATTN_OK;
  if (!w_qkv || !dw_qkv || !aligned16(w_qkv) || !aligned16(dw_qkv)) return ATTN_ERR_INVALID_ARG;
  if (n == 0 && m == 0) {  // no token: the weight gradient is zero
    return cudaMemsetAsync(dw_qkv, 0, static_cast<size_t>(d_model) * 3 * hd * 2, s) == cudaSuccess ? ATTN_OK
                                                                                                    : ATTN_ERR_CUDA;
  }
  if (n > 0 && (!x_q || !dq || !dx_q || !aligned16(x_q) || !aligned16(dq) || !aligned16(dx_q)))
    return ATTN_ERR_INVALID_ARG;
  if (m > 0 && (!x_kv || !dk || !dv || !dx_kv || !aligned16(x_kv) || !aligned16(dk) || !aligned16(dv) ||
                !aligned16(dx_kv)))
    return ATTN_ERR_INVALID_ARG;
  const int z = qkv_bwd_splits(B, n, m, d_model, h, d);
  if (z <= 0) return ATTN_ERR_CUDA;
  const size_t need = static_cast<size_t>(z) * d_model * static_cast<size_t>(3 * hd) * sizeof(float);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
  uint32_t* status = nullptr;
  if (device_status_word(&status) != cudaSuccess) return ATTN_ERR_CUDA;
  // W rows as the K-major operand of dX; gradients K-major (dX) and MN-major (dW); x MN-major (dW)
  CUtensorMap tw, gq, gk, gv, gq64, gk64, gv64, xq64, xkv64, oq, okv;
  if (!make_map3(&tw, w_qkv, 3 * hd, d_model, 1, 128)) return ATTN_ERR_CUDA;
  if (n > 0 && (!make_tile_map(&gq, dq, BH, n, d) || !make_tile_map(&gq64, dq, BH, n, d, 64) ||
                !make_map3(&xq64, x_q, d_model, n, B, 64) || !make_map3(&oq, dx_q, d_model, n, B, 128)))
    return ATTN_ERR_CUDA;
  if (m > 0 && (!make_tile_map(&gk, dk, BH, m, d) || !make_tile_map(&gv, dv, BH, m, d) ||
                !make_tile_map(&gk64, dk, BH, m, d, 64) || !make_tile_map(&gv64, dv, BH, m, d, 64) ||
                !make_map3(&xkv64, x_kv, d_model, m, B, 64) || !make_map3(&okv, dx_kv, d_model, m, B, 128)))
    return ATTN_ERR_CUDA;
  attn::ProjBwdParams p{};
  p.kind = 0;
  p.B = B;
  p.N = d_model;
  p.h = h;
  p.d = d;
  p.a_heads = 1;
  p.wd.status = status;
  p.wd.budget_ns = g_watchdog_ns.load();
  const bool self = x_q == x_kv && n == m;
  if (self && dx_q == dx_kv) {
    // dx = Concat(dq | dk | dv) W_qkv^T: one reduction over all 3 h d columns
    p.S = n;
    p.K = static_cast<int>(3 * hd);
    p.k_base = 0;
    if (attn::launch_proj_bwd(gq, gk, gv, tw, tw, tw, oq, p, s) != cudaSuccess) return ATTN_ERR_CUDA;
  } else {
    if (n > 0) {
      p.S = n;
      p.K = static_cast<int>(hd);
      p.k_base = 0;
      if (attn::launch_proj_bwd(gq, gq, gq, tw, tw, tw, oq, p, s) != cudaSuccess) return ATTN_ERR_CUDA;
    }
    if (m > 0) {
      p.S = m;
      p.K = static_cast<int>(2 * hd);
      p.k_base = static_cast<int>(hd);
      if (attn::launch_proj_bwd(gk, gv, gv, tw, tw, tw, okv, p, s) != cudaSuccess) return ATTN_ERR_CUDA;
    }
  }
  // dW partials [z][d_model][3 h d], then their sum in split order
  float* ws = static_cast<float*>(workspace);
  attn::ProjBwdParams q{};
  q.kind = 1;
  q.B = B;
  q.M = d_model;
  q.h = h;
  q.d = d;
  q.a_heads = 0;
  q.b_heads = 1;
  q.splits = z;
  q.ws = ws;
  q.ws_ld = static_cast<int>(3 * hd);
  q.wd = p.wd;
  if (self) {
    q.S = n;
    q.N = static_cast<int>(3 * hd);
    q.n_base = 0;
    if (attn::launch_proj_bwd(xq64, xq64, xq64, gq64, gk64, gv64, tw, q, s) != cudaSuccess) return ATTN_ERR_CUDA;
  } else {
    const size_t pitch = static_cast<size_t>(3 * hd) * sizeof(float), rows = static_cast<size_t>(z) * d_model;
    if (n > 0) {
      q.S = n;
      q.N = static_cast<int>(hd);
      q.n_base = 0;
      if (attn::launch_proj_bwd(xq64, xq64, xq64, gq64, gq64, gq64, tw, q, s) != cudaSuccess) return ATTN_ERR_CUDA;
    } else if (cudaMemset2DAsync(ws, pitch, 0, static_cast<size_t>(hd) * sizeof(float), rows, s) != cudaSuccess) {
      return ATTN_ERR_CUDA;
    }
    if (m > 0) {
      q.S = m;
      q.N = static_cast<int>(2 * hd);
      q.n_base = static_cast<int>(hd);
      if (attn::launch_proj_bwd(xkv64, xkv64, xkv64, gk64, gk64, gv64, tw, q, s) != cudaSuccess)
        return ATTN_ERR_CUDA;
    } else if (cudaMemset2DAsync(ws + hd, pitch, 0, static_cast<size_t>(2 * hd) * sizeof(float), rows, s) !=
               cudaSuccess) {
      return ATTN_ERR_CUDA;
    }
  }
  return attn::launch_proj_reduce(ws, dw_qkv, static_cast<long long>(d_model) * 3 * hd, z, s) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_CUDA;
}

int attn_out_projection_bwd(const void* o, const void* w_o, const void* dy, void* d_o, void* dw_o, int B, int n,
                            int d_model, int h, int d, void* workspace, size_t workspace_bytes,
                            attn_stream_t stream) {
  int st = check_proj(B, n, d_model, h, d);
  if (st != ATTN_OK) return st;
  const long long BH = static_cast<long long>(B) * h, hd = static_cast<long long>(h) * d;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (B == 0) return ATTN_OK;
  if (!w_o || !dw_o || !aligned16(w_o) || !aligned16(dw_o)) return ATTN_ERR_INVALID_ARG;
  if (n == 0) {  // no token: the weight gradient is zero
    return cudaMemsetAsync(dw_o, 0, static_cast<size_t>(hd) * d_model * 2, s) == cudaSuccess ? ATTN_OK
                                                                                            : ATTN_ERR_CUDA;
  }
  if (!o || !dy || !d_o || !aligned16(o) || !aligned16(dy) || !aligned16(d_o)) return ATTN_ERR_INVALID_ARG;
  const int z = out_bwd_splits(B, n, d_model, h, d);
  if (z <= 0) return ATTN_ERR_CUDA;
  const size_t need = static_cast<size_t>(z) * static_cast<size_t>(hd) * d_model * sizeof(float);
  if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
  uint32_t* status = nullptr;
  if (device_status_word(&status) != cudaSuccess) return ATTN_ERR_CUDA;
  CUtensorMap tdy, tw, tdo, to64, tdy64;
  if (!make_map3(&tdy, dy, d_model, n, B, 128) || !make_map3(&tw, w_o, d_model, hd, 1, 128) ||
      !make_tile_map(&tdo, d_o, BH, n, d) || !make_tile_map(&to64, o, BH, n, d, 64) ||
      !make_map3(&tdy64, dy, d_model, n, B, 64))
    return ATTN_ERR_CUDA;
  // dO = dy (W^O)^T, written in the [B, h, n, d] layout
  attn::ProjBwdParams p{};
  p.kind = 0;
  p.B = B;
  p.S = n;
  p.K = d_model;
  p.N = static_cast<int>(hd);
  p.h = h;
  p.d = d;
  p.a_heads = 0;
  p.out_heads = 1;
  p.k_base = 0;
  p.wd.status = status;
  p.wd.budget_ns = g_watchdog_ns.load();
  if (attn::launch_proj_bwd(tdy, tdy, tdy, tw, tw, tw, tdo, p, s) != cudaSuccess) return ATTN_ERR_CUDA;
  // dW^O = Concat(o)^T dy: partials [z][h d][d_model], then their sum
  float* ws = static_cast<float*>(workspace);
  attn::ProjBwdParams q{};
  q.kind = 1;
  q.B = B;
  q.S = n;
  q.M = static_cast<int>(hd);
  q.N = d_model;
  q.h = h;
  q.d = d;
  q.a_heads = 1;
  q.b_heads = 0;
  q.n_base = 0;
  q.splits = z;
  q.ws = ws;
  q.ws_ld = d_model;
  q.wd = p.wd;
  if (attn::launch_proj_bwd(to64, to64, to64, tdy64, tdy64, tdy64, tdo, q, s) != cudaSuccess) return ATTN_ERR_CUDA;
  return attn::launch_proj_reduce(ws, dw_o, hd * d_model, z, s) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_get_device_status(attn_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  uint32_t* status = nullptr;
  if (device_status_word(&status) != cudaSuccess) return ATTN_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (v != 0 && cudaMemset(status, 0, sizeof(uint32_t)) != cudaSuccess) return ATTN_ERR_CUDA;
  // attn_bwd_noalloc reports into a word of its own while the word above does
  // not exist yet on the device (creating it allocates): read and clear it too
  uint32_t w = 0;
  if (cudaMemcpyFromSymbol(&w, g_noalloc_status, sizeof(w)) != cudaSuccess) return ATTN_ERR_CUDA;
  if (w != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(g_noalloc_status, &zero, sizeof(zero)) != cudaSuccess) return ATTN_ERR_CUDA;
  }
  return (v == 0 && w == 0) ? ATTN_OK : ATTN_ERR_TIMEOUT;
}

}  // extern "C"


extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                const float* lse, const void* dO, void* dq, void* dk, void* dv,
                                int B, int h, int n, int m, int d_k, int d_v, int causal,
                                float scale, attn_stream_t stream) {
  bool empty = false;
  int st = check_common(B, h, n, m, d_k, d_v, scale, &empty);
  if (st != ATTN_OK) return st;
  // Sizes whose scratch does not fit the fixed array are refused before anything else.
  if (!empty && attn_bwd_workspace_bytes(B, h, n, m, d_k, d_v, causal) > kNoAllocScratchBytes)
    return ATTN_ERR_UNSUPPORTED;
  if (!k || !v || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv)) return ATTN_ERR_INVALID_ARG;
  const long long BH = static_cast<long long>(B) * h;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (empty) {
    if (BH == 0) return ATTN_OK;
    const size_t bytes = static_cast<size_t>(BH) * m * d_k * 2;
    if (cudaMemsetAsync(dk, 0, bytes, s) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaMemsetAsync(dv, 0, bytes, s) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  if (!q || !o || !lse || !dO || !dq) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o) || !aligned16(dO) || !aligned16(dq)) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return ATTN_ERR_INVALID_ARG;

  // Set-up, once per device, with that device current: the device address of
  // the scratch array (and of the fallback watchdog word).
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::call_once(g_noalloc_once[dev], [dev] {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e == cudaSuccess) {
      g_noalloc_scratch_ptr[dev] = ptr;
      void* sp = nullptr;
      e = cudaGetSymbolAddress(&sp, g_noalloc_status);
      if (e == cudaSuccess) g_noalloc_status_ptr[dev] = static_cast<uint32_t*>(sp);
    }
    g_noalloc_setup_err[dev] = e;
  });
  if (g_noalloc_setup_err[dev] != cudaSuccess || g_noalloc_scratch_ptr[dev] == nullptr)
    return ATTN_ERR_CUDA;
  uint32_t* status = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_status_mu);
    status = g_status[dev];  // read only: never allocated here
  }
  if (status == nullptr) status = g_noalloc_status_ptr[dev];
  if (attn_bwd_workspace_bytes(B, h, n, m, d_k, d_v, causal) == 0)  // needs no scratch at all
    return bwd_head_path(q, k, v, o, lse, dO, dq, dk, dv, nullptr, BH, h, n, m, d_k, causal, -1, -1, scale,
                         status, s);

  const long long n_pad = round_up(n, 128);
  float* dq_acc = static_cast<float*>(g_noalloc_scratch_ptr[dev]);
  float* lse2 = dq_acc + BH * n_pad * d_k;
  float* Dsum = lse2 + BH * n_pad;

  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
  if (!make_tile_map(&tq, q, BH, n, d_k) || !make_tile_map(&tk, k, BH, m, d_k) ||
      !make_tile_map(&tv, v, BH, m, d_v) || !make_tile_map(&tdo, dO, BH, n, d_v) ||
      !make_dq_map(&tdq, dq_acc, BH * n_pad, d_k) || !make_tile_map(&tdk, dk, BH, m, d_k) ||
      !make_tile_map(&tdv, dv, BH, m, d_v))
    return ATTN_ERR_CUDA;

  BwdPreParams pre{};
  pre.o = static_cast<const __nv_bfloat16*>(o);
  pre.dO = static_cast<const __nv_bfloat16*>(dO);
  pre.lse = lse;
  pre.lse2 = lse2;
  pre.Dsum = Dsum;
  pre.dq_acc = dq_acc;
  pre.n = n;
  pre.n_pad = static_cast<int>(n_pad);
  pre.d = d_k;
  pre.BH = static_cast<int>(BH);

  BwdParams p{};
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.lse2 = lse2;
  p.Dsum = Dsum;
  p.dq_acc = dq_acc;
  p.n = n;
  p.m = m;
  p.n_pad = static_cast<int>(n_pad);
  p.causal = causal ? 1 : 0;
  p.neg = scale < 0.f ? 1 : 0;
  p.c = static_cast<float>(std::fabs(static_cast<double>(scale)) * kLog2e);
  p.scale = scale;
  p.num_kblocks = static_cast<int>((m + 127) / 128);
  p.kv_len = nullptr;
  p.h = h;
  p.wl = -1;
  p.wr = -1;
  p.wd.status = status;
  p.wd.budget_ns = g_watchdog_ns.load();

  BwdPostParams post{};
  post.dq_acc = dq_acc;
  post.dq = static_cast<__nv_bfloat16*>(dq);
  post.scale = scale;
  post.n = n;
  post.n_pad = static_cast<int>(n_pad);
  post.d = d_k;
  post.BH = static_cast<int>(BH);

  cudaError_t e = attn::launch_bwd(d_k, tq, tk, tv, tdk, tdv, tdo, tdq, pre, p, post, static_cast<int>(BH), s);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
