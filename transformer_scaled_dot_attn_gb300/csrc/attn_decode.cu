// Incremental decoding: the n newest queries of each sequence against its
// cached keys and values ("Attention Is All You Need" §3: the decoder emits
// one symbol at a time, each step attending to the positions produced so far,
// itself included). Query i of n stands at position L - n + i of a sequence
// with L cached positions and sees the keys j <= L - n + i.
//
// A step reads every cached key and value once and does about one multiply-add
// per element read and query: it is bound by HBM, not by the tensor cores. So
// it runs on the FP32 pipes: the keys of a head are split into chunks, one CTA
// per (chunk, head) streams its chunk's K and V tiles through a TMA ring,
// computes the scores, an exact running maximum and the weights per query,
// and accumulates P.V; a second kernel merges the chunks' partial results
// (rescaled to the common maximum) into O and lse.
#include "attn_kernels.cuh"

#include <mutex>

namespace attn {
namespace {

using namespace sm103;

constexpr int kDecTK = 64;          // keys per tile (TMA box rows)
constexpr int kDecThreads = 128;
constexpr float kDecLn2 = 0.69314718055994530942f;

// NQ: the queries the layout holds (the kernel's compiled query count): the
// query, score and reduction areas are sized for it, so that steps with few
// queries fit three CTAs per SM.
template <int D, int NQ = kDecMaxN>
struct Dec {
  static constexpr int ATOM = D >= 64 ? 64 : D;            // bf16 per swizzle row
  static constexpr int NATOM = D / ATOM;                   // TMA boxes per tile
  static constexpr uint32_t BOX = kDecTK * ATOM * 2;
  static constexpr uint32_t TILE = kDecTK * D * 2;         // one K (or V) tile
  // Ring depth: a shallow ring per CTA and more CTAs per SM (four at d = 64,
  // three at d = 128 with one query) keep as many bytes in flight as a deep
  // ring with fewer CTAs, and give the SM more warps to cover the barriers
  // (n = 1 over 4096 cached d64: 4 stages 175 us, 3 stages 165 us; over 16384
  // cached d128: 3 stages 357 us, 2 stages 318 us). From four queries on, the
  // step is bound by the barriers more than by loads in flight: 2 stages and
  // five CTAs per SM at d = 64 (n = 4: 270 -> 260 us).
  static constexpr int STAGES = D <= 64 ? (NQ >= 4 ? 2 : 3) : 2;
  static constexpr int CP = D / 2;                         // column pairs (P.V phase)
  static constexpr int KG = kDecThreads / CP;              // key groups (P.V phase)
  static constexpr int KPG = kDecTK / KG;                  // keys per group
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = STAGES * TILE;
  static constexpr uint32_t OFF_Q = 2 * STAGES * TILE;                       // [n][D] fp32
  static constexpr uint32_t OFF_S = OFF_Q + NQ * D * 4;                     // [n][TK] fp32
  static constexpr uint32_t OFF_A = OFF_S + NQ * kDecTK * 4;                 // [n] fp32
  static constexpr uint32_t OFF_R = (OFF_A + NQ * 4 + 15) & ~15u;            // [KG][n][D] fp32
  static constexpr uint32_t SMEM = OFF_R + KG * NQ * D * 4 + 1024;          // + alignment slack
  static_assert(kDecThreads % CP == 0 && kDecTK % KG == 0, "thread mapping");
};

// Byte offset of the 16-byte chunk cc of row r in a tile written by a TMA map
// with the 128-byte (ATOM 64) or 64-byte (ATOM 32) swizzle.
template <int D>
__device__ __forceinline__ uint32_t dec_off(int r, int cc) {
  using C = Dec<D>;
  constexpr int CPA = C::ATOM / 8;
  const int a = cc / CPA, ca = cc % CPA;
  const int pc = (C::ATOM == 64) ? (ca ^ (r & 7)) : (ca ^ ((r >> 1) & 3));
  return a * C::BOX + r * (C::ATOM * 2) + (pc << 4);
}

__device__ __forceinline__ float dec_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Waits without looking at the abort flag (copies in flight must land before
// the CTA's shared memory goes away), bounded by the watchdog budget.
__device__ __forceinline__ void drain_wait_dec(uint64_t* bar, uint32_t parity, const Watchdog& wd) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > wd.budget_ns) {
      atomicCAS(wd.status, 0u, kDevTimeout | kSiteDrain);
      return;
    }
  }
}

// Bounded wait on a TMA phase that polls without a suspend hint: the step has
// no other work to hand the issue slots to, and a suspended thread resumes late.
__device__ __forceinline__ bool spin_wait_dec(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                              const Watchdog& wd, uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > wd.budget_ns) {
      *abort_flag = 1;
      atomicCAS(wd.status, 0u, kDevTimeout | site);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// NQ: queries the kernel is compiled for (n <= NQ; the smallest power of two
// that holds n), so that loops over the queries carry no idle iterations.
template <int D, int NQ>
__global__ void __launch_bounds__(kDecThreads)
attn_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const DecParams p) {
  using C = Dec<D, NQ>;
  constexpr int NU = (NQ + 3) / 4;   // queries per warp in the weight phase
  constexpr int QPT = (NQ + 1) / 2;  // queries per thread in the score phase (two threads per key)
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[C::STAGES];
  __shared__ int abort_word;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, bh = blockIdx.y;
  const int n = p.n;
  const int L = head_keys(p.kv_len, bh, p.h, p.m);  // cached positions of this sequence
  const int k_begin = split * p.chunk;
  const int k_end = min(L, k_begin + p.chunk);
  const int ntiles = k_end > k_begin ? (k_end - k_begin + kDecTK - 1) / kDecTK : 0;
  float* part = p.part + (static_cast<size_t>(bh) * p.splits + split) * n * (D + 2);
  if (ntiles == 0) {
    // no cached key in this chunk: an empty partial (the merge skips it)
    for (int i = tid; i < n; i += kDecThreads) {
      part[i * (D + 2) + D] = -INFINITY;
      part[i * (D + 2) + D + 1] = 0.f;
    }
    return;
  }
  volatile int* abort_flag = &abort_word;
  const Watchdog wd = p.wd;
  float* sQ = reinterpret_cast<float*>(smem + C::OFF_Q);
  float* sS = reinterpret_cast<float*>(smem + C::OFF_S);
  float* sA = reinterpret_cast<float*>(smem + C::OFF_A);
  float* sR = reinterpret_cast<float*>(smem + C::OFF_R);

  if (tid == 0) {
    for (int s = 0; s < C::STAGES; ++s) mbar_init(&full[s], 1);
    abort_word = 0;
    fence_mbar_init();
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
  }
  // the queries, scaled by c = scale * log2(e) so that scores are in log2 units
  for (int idx = tid; idx < n * D; idx += kDecThreads) {
    const uint16_t b = reinterpret_cast<const uint16_t*>(p.q)[static_cast<size_t>(bh) * n * D + idx];
    sQ[idx] = __uint_as_float(static_cast<uint32_t>(b) << 16) * p.c;
  }
  __syncthreads();
  auto load = [&](int t) {
    const int st = t % C::STAGES;
    mbar_arrive_expect_tx(&full[st], 2 * C::TILE);
    for (int a = 0; a < C::NATOM; ++a) {
      tma_load_3d(smem + C::OFF_K + st * C::TILE + a * C::BOX, &tm_k, &full[st], a * C::ATOM,
                  k_begin + t * kDecTK, bh);
      tma_load_3d(smem + C::OFF_V + st * C::TILE + a * C::BOX, &tm_v, &full[st], a * C::ATOM,
                  k_begin + t * kDecTK, bh);
    }
  };
  if (tid == 0)
    for (int t = 0; t < C::STAGES && t < ntiles; ++t) load(t);

  // running maximum and sum of query i = warp + 4 u, held by every lane of that warp
  float mrun[NU], lrun[NU];
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    mrun[u] = -INFINITY;
    lrun[u] = 0.f;
  }
  // P.V accumulators: columns 2 cp, 2 cp + 1 of every query, over key group kg;
  // the value pair sits in 16-byte chunk cc of its row, which the swizzle
  // moves by the row's index mod 8 (the same 8 offsets for every 8 rows)
  const int cp = tid % C::CP, kg = tid / C::CP;
  float acc[NQ][2];
#pragma unroll
  for (int i = 0; i < NQ; ++i) acc[i][0] = acc[i][1] = 0.f;
  uint32_t voff[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) voff[u] = dec_off<D>(u, cp / 4) + (cp % 4) * 4 - u * (C::ATOM * 2);

  int t = 0;
  for (; t < ntiles; ++t) {
    const int st = t % C::STAGES;
    const bool ok = spin_wait_dec(&full[st], (t / C::STAGES) & 1, abort_flag, wd, kSiteKFull);
    const uint8_t* sK = smem + C::OFF_K + st * C::TILE;
    const uint8_t* sV = smem + C::OFF_V + st * C::TILE;
    const int kbase = k_begin + t * kDecTK;
    if (ok) {
      if constexpr (QPT == 1) {
        // scores: thread = key j of the tile, queries i = tid / 64, + 2, ...
        // (n <= 2: one query per thread at most; the key row is loaded whole first)
        const int j = tid & (kDecTK - 1);
        const int key = kbase + j;
        uint4 kr[D / 8];
#pragma unroll
        for (int cc = 0; cc < D / 8; ++cc) kr[cc] = *reinterpret_cast<const uint4*>(sK + dec_off<D>(j, cc));
        for (int i = tid >> 6; i < n; i += kDecThreads / kDecTK) {
          const float* qi = sQ + i * D;
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int cc = 0; cc < D / 8; ++cc) {
            const uint32_t w[4] = {kr[cc].x, kr[cc].y, kr[cc].z, kr[cc].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 kf = bf16x2_to_f2(w[e]);
              s0 = fmaf(qi[cc * 8 + 2 * e], kf.x, s0);
              s1 = fmaf(qi[cc * 8 + 2 * e + 1], kf.y, s1);
            }
          }
          // key visible to query i: cached (key < k_end <= L) and not after its position
          const bool vis = key < k_end && key <= L - n + i;
          sS[i * kDecTK + j] = vis ? s0 + s1 : -INFINITY;
        }
      } else {
        // scores: thread = key j of the tile, queries i = tid / 64, + 2, ...;
        // each 16-byte chunk of the key row is unpacked once for all of them,
        // and the queries' sums interleave (n = 4 at d = 64: 313 -> 287 us
        // against a loop over the queries that unpacks the row for each).
        // Query rows past n read a real row of sQ and are not stored.
        const int j = tid & (kDecTK - 1);
        const int key = kbase + j;
        float sa[QPT], sb[QPT];
#pragma unroll
        for (int u = 0; u < QPT; ++u) sa[u] = sb[u] = 0.f;
        // (sixteen queries at d = 128: a partial unroll keeps the loop within the registers)
#pragma unroll(QPT * D > 512 ? 4 : D / 8)
        for (int cc = 0; cc < D / 8; ++cc) {
          const uint4 kw = *reinterpret_cast<const uint4*>(sK + dec_off<D>(j, cc));
          const float2 k0 = bf16x2_to_f2(kw.x), k1 = bf16x2_to_f2(kw.y);
          const float2 k2 = bf16x2_to_f2(kw.z), k3 = bf16x2_to_f2(kw.w);
#pragma unroll
          for (int u = 0; u < QPT; ++u) {
            const int i = (tid >> 6) + 2 * u;
            if (i < n) {
              const float4 qa = *reinterpret_cast<const float4*>(sQ + i * D + cc * 8);
              const float4 qb = *reinterpret_cast<const float4*>(sQ + i * D + cc * 8 + 4);
              sa[u] = fmaf(qa.x, k0.x, sa[u]);
              sb[u] = fmaf(qa.y, k0.y, sb[u]);
              sa[u] = fmaf(qa.z, k1.x, sa[u]);
              sb[u] = fmaf(qa.w, k1.y, sb[u]);
              sa[u] = fmaf(qb.x, k2.x, sa[u]);
              sb[u] = fmaf(qb.y, k2.y, sb[u]);
              sa[u] = fmaf(qb.z, k3.x, sa[u]);
              sb[u] = fmaf(qb.w, k3.y, sb[u]);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < QPT; ++u) {
          const int i = (tid >> 6) + 2 * u;
          if (i < n) sS[i * kDecTK + j] = (key < k_end && key <= L - n + i) ? sa[u] + sb[u] : -INFINITY;
        }
      }
    }
    // the wait's outcome joins the barrier after the scores: a thread whose
    // wait failed computes none, and every thread leaves the loop together
    if (__syncthreads_or(!ok)) break;
    // exact running maximum and the weights, one warp per query
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int i = warp + 4 * u;
      if (i < n) {
        const float s0 = sS[i * kDecTK + lane], s1 = sS[i * kDecTK + lane + 32];
        const float m_new = fmaxf(mrun[u], warp_max(fmaxf(s0, s1)));
        const float m_ref = (m_new == -INFINITY) ? 0.f : m_new;  // nothing visible yet: weights 0
        const float alpha = dec_ex2(mrun[u] - m_ref);
        const float p0 = dec_ex2(s0 - m_ref), p1 = dec_ex2(s1 - m_ref);
        sS[i * kDecTK + lane] = p0;
        sS[i * kDecTK + lane + 32] = p1;
        lrun[u] = lrun[u] * alpha + warp_sum(p0 + p1);
        mrun[u] = m_new;
        if (lane == 0) sA[i] = alpha;
      }
    }
    __syncthreads();
    // P.V over this thread's key group, four keys at a time (rows past n
    // hold weight 0 and contribute nothing)
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      const float a = (i < n) ? sA[i] : 1.f;
      acc[i][0] *= a;
      acc[i][1] *= a;
    }
#pragma unroll
    for (int j4 = 0; j4 < C::KPG; j4 += 4) {
      const int j0 = kg * C::KPG + j4;
      float2 vf[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = j0 + e;
        vf[e] = bf16x2_to_f2(*reinterpret_cast<const uint32_t*>(sV + j * (C::ATOM * 2) + voff[j & 7]));
      }
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
        const float4 pw = *reinterpret_cast<const float4*>(sS + i * kDecTK + j0);
        acc[i][0] = fmaf(pw.x, vf[0].x, acc[i][0]);
        acc[i][1] = fmaf(pw.x, vf[0].y, acc[i][1]);
        acc[i][0] = fmaf(pw.y, vf[1].x, acc[i][0]);
        acc[i][1] = fmaf(pw.y, vf[1].y, acc[i][1]);
        acc[i][0] = fmaf(pw.z, vf[2].x, acc[i][0]);
        acc[i][1] = fmaf(pw.z, vf[2].y, acc[i][1]);
        acc[i][0] = fmaf(pw.w, vf[3].x, acc[i][0]);
        acc[i][1] = fmaf(pw.w, vf[3].y, acc[i][1]);
      }
    }
    __syncthreads();  // stage st and the weights are free again
    if (tid == 0 && t + C::STAGES < ntiles) {
      fence_proxy_async_smem();  // this thread's generic reads of the stage come before the TMA write
      load(t + C::STAGES);
    }
  }
  if (t < ntiles) {
    // the watchdog fired at tile t: tiles t .. t + STAGES - 1 (those loaded)
    // were not waited for by every thread; let their copies land before the CTA exits
    if (tid == 0)
      for (int x = t; x < t + C::STAGES && x < ntiles; ++x)
        drain_wait_dec(&full[x % C::STAGES], (x / C::STAGES) & 1, wd);
    __syncthreads();
    return;
  }
  // combine the key groups' accumulators
#pragma unroll
  for (int i = 0; i < NQ; ++i)
    if (i < n) {
      sR[(kg * NQ + i) * D + 2 * cp] = acc[i][0];
      sR[(kg * NQ + i) * D + 2 * cp + 1] = acc[i][1];
    }
  __syncthreads();
  for (int idx = tid; idx < n * D; idx += kDecThreads) {
    const int i = idx / D, c = idx % D;
    float o = 0.f;
#pragma unroll
    for (int g = 0; g < C::KG; ++g) o += sR[(g * NQ + i) * D + c];
    part[i * (D + 2) + c] = o;
  }
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    const int i = warp + 4 * u;
    if (i < n && lane == 0) {
      part[i * (D + 2) + D] = mrun[u];
      part[i * (D + 2) + D + 1] = lrun[u];
    }
  }
}

// Merge: per (head, query) the chunks' partials (O_s unnormalised, max m_s,
// sum l_s, all in log2 units) rescaled to the common maximum M:
// O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s, lse = (M + log2 l) ln 2.
// A query that saw no key is the empty sum (O = 0, lse = -inf).
template <int D>
__global__ void __launch_bounds__(128) attn_decode_merge_kernel(const DecParams p, long long rows) {
  const long long row = static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int n = p.n;
  const long long bh = row / n;
  const int i = static_cast<int>(row % n);
  const float* part = p.part + (static_cast<size_t>(bh) * p.splits * n + i) * (D + 2);
  const size_t stride = static_cast<size_t>(n) * (D + 2);
  float M = -INFINITY;
  for (int s = 0; s < p.splits; ++s) M = fmaxf(M, part[s * stride + D]);
  constexpr int PER = (D + 31) / 32;
  float o[PER];
#pragma unroll
  for (int u = 0; u < PER; ++u) o[u] = 0.f;
  float l = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < p.splits; ++s) {
      const float ms = part[s * stride + D];
      if (ms == -INFINITY) continue;  // a chunk without a visible key holds no O
      const float w = dec_ex2(ms - M);
      l += w * part[s * stride + D + 1];
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int c = lane + 32 * u;
        if (c < D) o[u] += w * part[s * stride + c];
      }
    }
  }
  const float inv = (l > 0.f) ? 1.f / l : 0.f;
  __nv_bfloat16* orow = p.o + static_cast<size_t>(row) * D;
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int c = lane + 32 * u;
    if (c < D) orow[c] = __float2bfloat16_rn(o[u] * inv);
  }
  if (lane == 0 && p.lse != nullptr) p.lse[row] = (l > 0.f) ? (M + log2f(l)) * kDecLn2 : -INFINITY;
}

template <int D, int NQ>
cudaError_t launch_decode_step(const CUtensorMap& tk, const CUtensorMap& tv, const DecParams& p, int BH,
                               cudaStream_t stream) {
  using C = Dec<D, NQ>;
  static std::once_flag once[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaError_t attr = cudaSuccess;
  std::call_once(once[dev & 63], [&] {
    attr = cudaFuncSetAttribute(attn_decode_kernel<D, NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(C::SMEM));
  });
  if (attr != cudaSuccess) return attr;
  prof_begin(kKindDecode, stream);
  attn_decode_kernel<D, NQ><<<dim3(static_cast<unsigned>(p.splits), static_cast<unsigned>(BH)), kDecThreads,
                              C::SMEM, stream>>>(tk, tv, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  prof_end(kKindDecode, stream);
  return cudaSuccess;
}

template <int D>
cudaError_t launch_decode_d(const CUtensorMap& tk, const CUtensorMap& tv, const DecParams& p, int BH,
                            cudaStream_t stream) {
  cudaError_t e;
  if (p.n <= 1) e = launch_decode_step<D, 1>(tk, tv, p, BH, stream);
  else if (p.n <= 2) e = launch_decode_step<D, 2>(tk, tv, p, BH, stream);
  else if (p.n <= 4) e = launch_decode_step<D, 4>(tk, tv, p, BH, stream);
  else if (p.n <= 8) e = launch_decode_step<D, 8>(tk, tv, p, BH, stream);
  else e = launch_decode_step<D, 16>(tk, tv, p, BH, stream);
  if (e != cudaSuccess) return e;
  const long long rows = static_cast<long long>(BH) * p.n;
  prof_begin(kKindDecodeMerge, stream);
  attn_decode_merge_kernel<D><<<static_cast<unsigned>((rows + 3) / 4), 128, 0, stream>>>(p, rows);
  e = cudaGetLastError();
  prof_end(kKindDecodeMerge, stream);
  return e;
}

}  // namespace

void decode_split(long long BH, int m, int* splits, int* chunk) {
  const int tiles = (m + kDecTK - 1) / kDecTK;
  // about 4096 CTAs over the whole batch (enough loads in flight per SM to
  // cover the HBM latency), each at least one tile
  long long want = (4096 + BH - 1) / (BH > 0 ? BH : 1);
  if (want < 1) want = 1;
  if (want > tiles) want = tiles;
  const int per = static_cast<int>((tiles + want - 1) / want);  // tiles per chunk
  *chunk = per * kDecTK;
  *splits = (m + *chunk - 1) / *chunk;
}

cudaError_t launch_decode(int d, const CUtensorMap& tk, const CUtensorMap& tv, const DecParams& p, int BH,
                          cudaStream_t stream) {
  switch (d) {
    case 32: return launch_decode_d<32>(tk, tv, p, BH, stream);
    case 64: return launch_decode_d<64>(tk, tv, p, BH, stream);
    case 128: return launch_decode_d<128>(tk, tv, p, BH, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attn
