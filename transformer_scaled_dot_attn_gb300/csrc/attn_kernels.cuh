// Internal declarations shared by the attention kernels and the C-ABI host code.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace attn {

// Device error word values (0 = no error). The low byte names the wait site.
constexpr uint32_t kDevTimeout = 0x100u;
// A kernel could not place its shared-memory tiles (alignment); it did no work.
constexpr uint32_t kDevLayout = 0x200u;

// Sites, for diagnosis of a watchdog report.
enum WaitSite : uint32_t {
  kSiteQFull = 1, kSiteKFull, kSiteVFull, kSiteKEmpty, kSiteVEmpty, kSiteSFull,
  kSitePFull, kSiteOFull, kSiteDrain, kSiteBwdLoad, kSiteBwdS, kSiteBwdDP, kSiteBwdDS,
  kSiteBwdDQ, kSiteBwdFree, kSiteBwdFinal, kSiteExpTurn
};

struct Watchdog {
  uint32_t* status;      // device error word (global)
  uint64_t budget_ns;    // per-wait limit
};

constexpr uint32_t kWaitSleepNs = 20000;  // longest suspension per try in guarded_wait

// Bounded mbarrier wait. Returns false when the CTA is aborting or this wait
// ran out of time (in which case it raises the CTA abort flag and records the
// site in the device error word). Never traps, never spins forever.
__device__ __forceinline__ bool guarded_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             const Watchdog& wd, uint32_t site) {
  if (sm103::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = sm103::global_timer_ns();
  while (true) {
    // sleep in the barrier (woken by the phase completing) rather than spin:
    // spinning warps take issue slots from the warps that do the work
    if (sm103::mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
    if (*abort_flag) return false;
    if (sm103::global_timer_ns() - t0 > wd.budget_ns) {
      *abort_flag = 1;
      atomicCAS(wd.status, 0u, kDevTimeout | site);
      return false;
    }
  }
}

// Key padding: real keys of head bh, kv_len[b] for its sequence b = bh / h
// clamped to [0, m]; all m without a length array.
__device__ __forceinline__ int head_keys(const int* kv_len, int bh, int h, int m) {
  if (kv_len == nullptr) return m;
  return min(max(__ldg(kv_len + bh / h), 0), m);
}

// Keys [lo, hi) visible to query row i of a head with mb real keys: the
// causal mask (j <= i), key padding (j < mb) and the restricted-attention
// window i - wl <= j <= i + wr (a side given as -1 is open; the host clamps
// both to [-1, n + m]). hi <= lo: the row sees no key.
__device__ __forceinline__ void key_range(int i, int mb, int causal, int wl, int wr, int& lo, int& hi) {
  int h = mb;
  if (causal) h = min(h, i + 1);
  if (wr >= 0) h = min(h, i + wr + 1);
  lo = (wl >= 0) ? max(0, i - wl) : 0;
  hi = h;
}

// Query rows [lo, hi) that see some key of [k0, k1] (k1 < mb), the transpose
// of key_range for a key tile: rows i with i - wl <= k1, and i >= k0 when
// causal, and i + wr >= k0.
__device__ __forceinline__ void query_range(int k0, int k1, int n, int causal, int wl, int wr, int& lo,
                                            int& hi) {
  int l = 0;
  if (causal) l = max(l, k0);
  if (wr >= 0) l = max(l, k0 - wr);
  lo = l;
  hi = (wl >= 0) ? min(n, k1 + wl + 1) : n;
}

// Profiling hooks (implemented with the C ABI): bracket one kernel launch
// with CUDA events on `stream` when profiling is enabled; no-ops otherwise.
enum KernelKind : int {
  kKindFwd = 0, kKindBwdPre = 1, kKindBwdMain = 2, kKindBwdPost = 3, kKindDecode = 4, kKindDecodeMerge = 5,
  kKindProj = 6, kNumKinds = 7
};
void prof_begin(int kind, cudaStream_t stream);
void prof_end(int kind, cudaStream_t stream);

// ---------------------------------------------------------------- forward

struct FwdParams {
  __nv_bfloat16* o;   // [BH, n, d]
  float* lse;         // [BH, n] or nullptr
  int n, m;           // queries, keys per head
  int causal;
  int neg;            // scale < 0: the score MMA negates Q K^T so that c >= 0
  float c;            // |scale| * log2(e)
  int num_qblocks;    // query blocks (set by the launcher)
  int qb_fast;        // per-item forward grid: 1 = (query block, head), 0 = (head, query block)
  int inject;         // test hook: 1 = skip the first value-tile load
  const int* kv_len;  // [B] real keys per sequence (key padding) or nullptr
  int h;              // heads per sequence (kv_len is indexed by bh / h)
  int wl, wr;         // window: query i sees keys i - wl .. i + wr (-1: open side)
  Watchdog wd;
};

// Keys per tile the forward kernel streams for head size d and n queries
// (the K/V TMA box height).
int fwd_key_tile(int d, int n, int m, int causal, bool windowed);

cudaError_t launch_fwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& to,
                       const FwdParams& p, int BH, cudaStream_t stream);

// ---------------------------------------------------------------- backward

struct BwdPreParams {
  const __nv_bfloat16* o;   // [BH, n, d]
  const __nv_bfloat16* dO;  // [BH, n, d]
  const float* lse;         // [BH, n]
  float* lse2;              // [BH, n_pad]  -lse * log2(e)  (padding rows: -inf)
  float* Dsum;              // [BH, n_pad]  D_i = sum_c dO_ic O_ic (padding rows: 0)
  float* dq_acc;            // [BH, n_pad, d] zeroed here
  int n, n_pad, d, BH;
};

struct BwdParams {
  __nv_bfloat16* dk;        // [BH, m, d]
  __nv_bfloat16* dv;        // [BH, m, d]
  const float* lse2;        // [BH, n_pad]
  const float* Dsum;        // [BH, n_pad]
  float* dq_acc;            // [BH, n_pad, d]
  int n, m, n_pad;
  int causal, neg;
  float c;                  // |scale| * log2(e)
  float scale;              // signed scale, applied to dK
  int num_kblocks;          // ceil(m / 128)
  int BH;                   // heads (set by the launcher)
  int num_items;            // BH * num_kblocks work items (set by the launcher)
  int head_major;           // item order: head major (1) or key-tile major (0) (set by the launcher)
  const int* kv_len;        // [B] real keys per sequence (key padding) or nullptr
  int h;                    // heads per sequence
  int wl, wr;               // window (see FwdParams)
  Watchdog wd;
};

struct BwdPostParams {
  const float* dq_acc;      // [BH, n_pad, d]
  __nv_bfloat16* dq;        // [BH, n, d]
  float scale;
  int n, n_pad, d, BH;
};

// Whole-head backward (n <= 256, d <= 64): one launch, no workspace.
struct BwdHeadParams {
  const __nv_bfloat16* o;   // [BH, n, d]
  const __nv_bfloat16* dO;  // [BH, n, d]
  const float* lse;         // [BH, n], natural log
  __nv_bfloat16* dq;        // [BH, n, d]
  __nv_bfloat16* dk;        // [BH, m, d]
  __nv_bfloat16* dv;        // [BH, m, d]
  int BH, n, m;
  int causal, neg;
  float c;                  // |scale| * log2(e)
  float scale;              // signed scale, applied to dQ and dK
  const int* kv_len;        // [B] real keys per sequence (key padding) or nullptr
  int h;                    // heads per sequence
  int wl, wr;               // window (see FwdParams)
  Watchdog wd;
};
bool bwd_head_supported(int n, int d);
// tdq, tdk, tdv: maps over the bf16 outputs, the same shape of map as the inputs'.
cudaError_t launch_bwd_head(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tdk,
                            const CUtensorMap& tdv, const BwdHeadParams& p, cudaStream_t stream);

// tdq: 2-D fp32 map over the dQ accumulator [BH*n_pad, d], box 32 x 128, 128-byte swizzle.
// tdk, tdv: maps over the bf16 dK / dV outputs (the same shape of map as K's).
cudaError_t launch_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdk, const CUtensorMap& tdv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const BwdPreParams& pre,
                       const BwdParams& p, const BwdPostParams& post, int BH, cudaStream_t stream);

// ---------------------------------------------------------------- decoding

constexpr int kDecMaxN = 16;  // new queries per sequence in one decoding step

struct DecParams {
  const __nv_bfloat16* q;   // [BH, n, d]
  __nv_bfloat16* o;         // [BH, n, d]
  float* lse;               // [BH, n] or nullptr
  float* part;              // [BH, splits, n, d + 2] fp32: partial O, max, sum (log2 units)
  const int* kv_len;        // [B] cached positions per sequence or nullptr (all m)
  int h, n, m;              // heads per sequence, new queries, cache capacity
  int splits, chunk;        // key chunks per head and keys per chunk (set by decode_split)
  float c;                  // scale * log2(e)
  Watchdog wd;
};
// Key chunks of a decoding step over BH heads with capacity m.
void decode_split(long long BH, int m, int* splits, int* chunk);
// tk, tv: maps over the caches [BH, m, d] with 64-row boxes.
cudaError_t launch_decode(int d, const CUtensorMap& tk, const CUtensorMap& tv, const DecParams& p, int BH,
                          cudaStream_t stream);

// ---------------------------------------------------------------- projections

struct ProjParams {
  int mode;        // 0: A = token rows x [B, S, K] (map (K, S, B)), output scattered to Q | K | V
                   //    [B, h, S, d]; 1: A = O [B, h, S, d] (K = h d), output Y [B, S, N]
  int B, S, K, N;  // sequences, tokens per sequence, reduction, output columns of this launch
  int h, d;        // heads and head size of the [B, h, S, d] side
  int n_base;      // mode 0: first column of W (and of Q | K | V) this launch computes
  int tiles_s;     // set by the launcher
  int num_tiles;   // set by the launcher
  Watchdog wd;
};
// ta: A map (mode 0: (K, S, B), box (64, 128, 1); mode 1: O's (d, S, B h) map);
// tb: W map (Ntot, K, 1), box (64, 64, 1); to0..to2: Q, K, V maps (mode 0) or
// the Y map (N, S, B) in to0 (mode 1). 128-byte swizzle everywhere.
cudaError_t launch_proj(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to0,
                        const CUtensorMap& to1, const CUtensorMap& to2, ProjParams p, cudaStream_t stream);

struct ProjBwdParams {
  int kind;        // 0: out = A W^T (rows = tokens); 1: fp32 partials of A^T B over token splits
  int B, S;        // sequences, tokens per sequence
  int K;           // kind 0: reduction (multiple of 64)
  int N;           // output columns of this launch
  int M;           // kind 1: output rows (weight rows)
  int h, d;        // heads and head size of the [B, h, S, d] side
  int a_heads;     // A from [B, h, S, d] maps (kind 0: ta0 | ta1 | ta2 by column / (h d)); else rows (k, s, b)
  int b_heads;     // kind 1: B from [B, h, S, d] maps tb0 | tb1 | tb2 by column / (h d); else rows (n, s, b)
  int out_heads;   // kind 0: output into a [B, h, S, d] map; else rows [B, S, N]
  int k_base;      // kind 0: first W column of the reduction
  int n_base;      // kind 1: first column of the partial rows (and of the B side) this launch covers
  int splits;      // kind 1: token splits
  float* ws;       // kind 1: partials [splits][M][ws_ld] fp32
  int ws_ld;
  int tiles_s, tiles_m, chunks_s, chunks, cps, num_units;  // set by the launcher
  Watchdog wd;
};
// Maps (128-byte swizzle): kind 0: ta* (64, 128, 1) boxes, tb0 the W map
// (columns, rows) with (64, 128) boxes, to the output map (64, 128). kind 1:
// ta0 and tb* with (64, 64) boxes over (columns, tokens, sequence [x head]).
cudaError_t launch_proj_bwd(const CUtensorMap& ta0, const CUtensorMap& ta1, const CUtensorMap& ta2,
                            const CUtensorMap& tb0, const CUtensorMap& tb1, const CUtensorMap& tb2,
                            const CUtensorMap& to, ProjBwdParams p, cudaStream_t stream);
// Token splits of a weight gradient of M x N (0 when the device is unknown).
int proj_bwd_splits(int M, int N, int chunks);
// out (bf16) = sum over splits of part[z][0 .. count), count a multiple of 8.
cudaError_t launch_proj_reduce(const float* part, void* out, long long count, int splits, cudaStream_t stream);

}  // namespace attn
