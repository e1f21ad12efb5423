// Backward of the multi-head projections ("Attention Is All You Need" §3.2.2,
// MultiHead(Q, K, V) = Concat(head_1, ..., head_h) W^O with
// head_i = Attention(Q W_i^Q, K W_i^K, V W_i^V)), as tcgen05 GEMMs.
// For Y = X W and a loss gradient dY: dX = dY W^T and dW = X^T dY. Here
//   kind 0 (dX):  out[token][c] = sum_k A[token][k] W[c][k]       (M = tokens)
//                 A K-major: the [B, h, S, d] gradients of Q | K | V (the
//                 concatenation is the reduction loop, one head's 64 columns
//                 per step, up to three maps), or the rows of dY;
//                 W K-major: rows of W^{QKV} (columns k_base..) or of W^O;
//                 out bf16: rows [B, S, N] or, for dO, the [B, h, S, d] layout.
//   kind 1 (dW):  part[z][r][c] = sum_{tokens of split z} A[token][r] B[token][c]
//                 A MN-major: X rows, or O read from its [B, h, S, d] layout;
//                 B MN-major: the gradients of Q | K | V from their [B, h, S, d]
//                 layout, or dY rows; fp32 partial sums per token split, added
//                 in split order by attn_proj_reduce_kernel (deterministic).
// Tiles of 128 x 128 outputs; the reduction streams 64 at a time through a
// 5-stage TMA ring of 32 KB stages (seven stages, in the staging area that
// kind 1 does not use, measured slower). Warp 0 loads, warp 1 issues the MMAs
// into one of two TMEM accumulators, warps 4-7 move the other one out, so a
// tile's epilogue overlaps the next tile's products (as in attn_proj.cu).
#include "attn_kernels.cuh"

#include <mutex>

namespace attn {
namespace {

using namespace sm103;

constexpr int kBM = 128, kBN = 128, kBK = 64;
constexpr int kBStages = 5;
constexpr uint32_t kBHalf = 64 * 64 * 2;             // 8 KB: 64 x 64 bf16 box
constexpr uint32_t kBTile = 2 * kBHalf;              // 16 KB: one operand of a stage
constexpr uint32_t kBStage = 2 * kBTile;             // A and B
constexpr uint32_t kBOffOut = kBStages * kBStage;    // bf16 staging: 2 sets x 2 boxes [128 rows][64 columns]
constexpr uint32_t kBOutBox = kBM * 64 * 2;          // 16 KB
constexpr uint32_t kBSmem = kBOffOut + 4 * kBOutBox + 1024;
constexpr int kBThreads = 256;

struct ProjBwdShared {
  uint64_t full[kBStages], empty[kBStages];
  uint64_t acc_full[2], acc_free[2];
  uint64_t staged, stage_free[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void drain_wait_pb(uint64_t* bar, uint32_t parity, const Watchdog& wd) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > wd.budget_ns) {
      atomicCAS(wd.status, 0u, kDevTimeout | kSiteDrain);
      return;
    }
  }
}

// Work unit t -> output tile and, for kind 1, its token split and chunk range.
struct PbUnit {
  int b, s0;        // kind 0: sequence and first token of the tile
  int m0, n0;       // output rows (kind 1) / columns
  int z, c0, c1;    // kind 1: split and its 64-token chunks [c0, c1)
};

__device__ __forceinline__ PbUnit pb_unit(const ProjBwdParams& p, int t) {
  PbUnit u{};
  const int tiles_n = (p.N + kBN - 1) / kBN;
  if (p.kind == 0) {
    const int mt = t / tiles_n;
    u.n0 = (t - mt * tiles_n) * kBN;
    u.b = mt / p.tiles_s;
    u.s0 = (mt - u.b * p.tiles_s) * kBM;
    u.c0 = 0;
    u.c1 = p.K / kBK;
  } else {
    const int per_split = p.tiles_m * tiles_n;
    u.z = t / per_split;
    const int r = t - u.z * per_split;
    const int mt = r / tiles_n;
    u.m0 = mt * kBM;
    u.n0 = (r - mt * tiles_n) * kBN;
    u.c0 = min(u.z * p.cps, p.chunks);
    u.c1 = min(u.c0 + p.cps, p.chunks);
  }
  return u;
}

__global__ void __launch_bounds__(kBThreads, 1)
attn_proj_bwd_kernel(const __grid_constant__ CUtensorMap ta0, const __grid_constant__ CUtensorMap ta1,
                     const __grid_constant__ CUtensorMap ta2, const __grid_constant__ CUtensorMap tb0,
                     const __grid_constant__ CUtensorMap tb1, const __grid_constant__ CUtensorMap tb2,
                     const __grid_constant__ CUtensorMap to, const ProjBwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) ProjBwdShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &sh.abort_flag;
  const Watchdog wd = p.wd;
  const int hd = p.h * p.d;
  constexpr int NS = kBStages;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.acc_full[i], 1);
      mbar_init(&sh.acc_free[i], 128);
    }
    mbar_init(&sh.staged, 128);
    mbar_init(&sh.stage_free[0], 1);
    mbar_init(&sh.stage_free[1], 1);
    mbar_init(&sh.drain, 1);
    sh.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc<256>(&sh.tmem_base);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      long long g = 0;  // stages filled so far
      uint32_t filled = 0, last_ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_units; t += gridDim.x) {
        const PbUnit u = pb_unit(p, t);
        for (int kc = u.c0; ok && kc < u.c1; ++kc, ++g) {
          const int st = static_cast<int>(g % NS);
          if (g >= NS &&
              !(ok = guarded_wait(&sh.empty[st], static_cast<uint32_t>((g / NS - 1) & 1), abort_flag, wd,
                                  kSiteKEmpty)))
            break;
          uint8_t* sA = smem + st * kBStage;
          uint8_t* sB = sA + kBTile;
          mbar_arrive_expect_tx(&sh.full[st], kBStage);
          filled |= 1u << st;
          last_ph = (last_ph & ~(1u << st)) | (static_cast<uint32_t>((g / NS) & 1) << st);
          if (p.kind == 0) {
            const int k0 = kc * kBK;
            if (p.a_heads) {
              // column k0 of Concat(G_0 | G_1 | G_2): map k0 / hd, head and column within it
              const int which = k0 / hd, within = k0 - which * hd;
              const CUtensorMap* ma = which == 0 ? &ta0 : (which == 1 ? &ta1 : &ta2);
              tma_load_3d(sA, ma, &sh.full[st], within % p.d, u.s0, u.b * p.h + within / p.d);
            } else {
              tma_load_3d(sA, &ta0, &sh.full[st], k0, u.s0, u.b);
            }
            // W rows n0 .. n0 + 127, columns k_base + k0 .. + 63 (K-major)
            tma_load_3d(sB, &tb0, &sh.full[st], p.k_base + k0, u.n0, 0);
          } else {
            // 64 tokens of sequence b; both operands MN-major, two 64-column boxes each
            const int b = kc / p.chunks_s, t0 = (kc - b * p.chunks_s) * kBK;
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int r = u.m0 + 64 * i;  // A column (weight row)
              if (p.a_heads)
                tma_load_3d(sA + i * kBHalf, &ta0, &sh.full[st], r % p.d, t0, b * p.h + r / p.d);
              else
                tma_load_3d(sA + i * kBHalf, &ta0, &sh.full[st], r, t0, b);
              const int c = p.n_base + u.n0 + 64 * i;  // B column
              if (p.b_heads) {
                const int which = c / hd, within = c - which * hd;
                const CUtensorMap* mb = which == 0 ? &tb0 : (which == 1 ? &tb1 : &tb2);
                tma_load_3d(sB + i * kBHalf, mb, &sh.full[st], within % p.d, t0, b * p.h + within / p.d);
              } else {
                tma_load_3d(sB + i * kBHalf, &tb0, &sh.full[st], c, t0, b);
              }
            }
          }
        }
      }
      // Let every copy this thread started land before shared memory is released.
      for (int s = 0; s < NS; ++s)
        if ((filled >> s) & 1u) drain_wait_pb(&sh.full[s], (last_ph >> s) & 1u, wd);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // kind 0: A and W K-major; kind 1: A and B MN-major (64-column boxes 8 KB apart)
      const uint32_t idesc = p.kind == 0 ? idesc_bf16_f32(kBM, kBN, false, false) : idesc_bf16_f32(kBM, kBN, true, true);
      long long g = 0;
      int tc = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_units; t += gridDim.x, ++tc) {
        const PbUnit u = pb_unit(p, t);
        const int buf = tc & 1;
        // the epilogue must have read this accumulator's previous tile
        if (tc >= 2 &&
            !(ok = guarded_wait(&sh.acc_free[buf], static_cast<uint32_t>((tc / 2 - 1) & 1), abort_flag, wd,
                                kSiteOFull)))
          break;
        for (int kc = u.c0; ok && kc < u.c1; ++kc, ++g) {
          const int st = static_cast<int>(g % NS);
          if (!(ok = guarded_wait(&sh.full[st], static_cast<uint32_t>((g / NS) & 1), abort_flag, wd,
                                  kSiteKFull)))
            break;
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + st * kBStage), sB = sA + kBTile;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            uint64_t da, db;
            if (p.kind == 0) {
              da = smem_desc(sA + k * 32, 16, 1024, 2);
              db = smem_desc(sB + k * 32, 16, 1024, 2);
            } else {
              da = smem_desc(sA + k * 16 * 128, kBHalf, 1024, 2);
              db = smem_desc(sB + k * 16 * 128, kBHalf, 1024, 2);
            }
            mma_ss(tmem + buf * kBN, da, db, idesc, (kc > u.c0 || k > 0) ? 1u : 0u);
          }
          mma_commit(&sh.empty[st]);  // the stage may be refilled once these products read it
        }
        // (a unit without chunks issues no product: the epilogue writes zeros)
        if (ok) mma_commit(&sh.acc_full[buf]);
      }
      // Every MMA this thread issued must finish before TMEM is released.
      mma_commit(&sh.drain);
      drain_wait_pb(&sh.drain, 0, wd);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int r = tid - 128;  // output row of the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint8_t* stage = smem + kBOffOut;
    int tc = 0;
    for (int t = blockIdx.x; t < p.num_units; t += gridDim.x, ++tc) {
      const PbUnit u = pb_unit(p, t);
      const int buf = tc & 1;
      bool ok = __all_sync(0xffffffffu, guarded_wait(&sh.acc_full[buf], static_cast<uint32_t>((tc / 2) & 1),
                                                     abort_flag, wd, kSiteOFull));
      if (!ok) break;
      tc_fence_after();
      const bool have = u.c1 > u.c0;
      if (p.kind == 1) {
        // fp32 partial sums of split z: row m0 + r, columns n0 .. n0 + 127
        const int row = u.m0 + r;
#pragma unroll
        for (int q = 0; q < kBN / 32; ++q) {
          uint32_t v[32];
          if (have) {
            tmem_ld32(tmem + lane_base + buf * kBN + q * 32, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
          }
          if (q == kBN / 32 - 1) {
            tc_fence_before();
            mbar_arrive(&sh.acc_free[buf]);
          }
          if (row < p.M) {
            float* dst = p.ws + (static_cast<size_t>(u.z) * p.M + row) * p.ws_ld + p.n_base + u.n0 + q * 32;
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4)
              if (u.n0 + q * 32 + c4 * 4 < p.N)
                *reinterpret_cast<float4*>(dst + c4 * 4) =
                    make_float4(__uint_as_float(v[4 * c4]), __uint_as_float(v[4 * c4 + 1]),
                                __uint_as_float(v[4 * c4 + 2]), __uint_as_float(v[4 * c4 + 3]));
          }
        }
        continue;
      }
      // kind 0: bf16 through a swizzled staging set, one thread stores it
      const int sb = tc & 1;
      if (tc >= 2)
        ok = __all_sync(0xffffffffu, guarded_wait(&sh.stage_free[sb], static_cast<uint32_t>((tc / 2 - 1) & 1),
                                                  abort_flag, wd, kSiteOFull));
      if (!ok) break;
      uint8_t* tstage = stage + sb * 2 * kBOutBox;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t v[2][32];
        tmem_ld32(tmem + lane_base + buf * kBN + half * 64, v[0]);
        tmem_ld32(tmem + lane_base + buf * kBN + half * 64 + 32, v[1]);
        tmem_ld_wait();
        if (half == 1) {
          tc_fence_before();
          mbar_arrive(&sh.acc_free[buf]);  // the MMAs of a later tile may overwrite this accumulator
        }
        uint8_t* box = tstage + half * kBOutBox;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t* f = v[c >> 2] + (c & 3) * 8;
          const uint4 w4 = make_uint4(pack_bf16x2(__uint_as_float(f[0]), __uint_as_float(f[1])),
                                      pack_bf16x2(__uint_as_float(f[2]), __uint_as_float(f[3])),
                                      pack_bf16x2(__uint_as_float(f[4]), __uint_as_float(f[5])),
                                      pack_bf16x2(__uint_as_float(f[6]), __uint_as_float(f[7])));
          *reinterpret_cast<uint4*>(box + r * 128 + ((c ^ (r & 7)) << 4)) = w4;
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&sh.staged);
      if (r == 0) {
        if (guarded_wait(&sh.staged, static_cast<uint32_t>(tc & 1), abort_flag, wd, kSiteOFull)) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int c = u.n0 + half * 64;  // output column of this box
            if (c >= p.N) break;
            if (p.out_heads)
              tma_store_3d(&to, tstage + half * kBOutBox, c % p.d, u.s0, u.b * p.h + c / p.d);
            else
              tma_store_3d(&to, tstage + half * kBOutBox, c, u.s0, u.b);  // rows past S are clipped
          }
          tma_store_commit();
        }
        // the previous tile's stores (the other staging set) have read their source
        bulk_wait_read_but_last();
        if (tc >= 1) mbar_arrive(&sh.stage_free[sb ^ 1]);
      }
    }
    if (r == 0) tma_store_wait_all();  // stores must complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<256>(tmem);
  }
}

// out[i] = bf16(sum over splits z = 0, 1, ... of part[z][i]), 8 elements a thread.
__global__ void attn_proj_reduce_kernel(const float* __restrict__ part, __nv_bfloat16* __restrict__ out,
                                        long long count, int splits) {
  const long long i = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) * 8;
  if (i >= count) return;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int z = 0; z < splits; ++z) {
    const float4* src = reinterpret_cast<const float4*>(part + z * count + i);
    const float4 a = src[0], b = src[1];
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
  }
  uint4 w;
  w.x = pack_bf16x2(acc[0], acc[1]);
  w.y = pack_bf16x2(acc[2], acc[3]);
  w.z = pack_bf16x2(acc[4], acc[5]);
  w.w = pack_bf16x2(acc[6], acc[7]);
  *reinterpret_cast<uint4*>(out + i) = w;
}

int sm_count_cached() {
  static int count[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (count[dev & 63] == 0) {
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    count[dev & 63] = c > 0 ? c : 1;
  }
  return count[dev & 63];
}

}  // namespace

// About two work units per SM (measured faster on GB300 than one wave of
// longer units), up to 32 splits and at most one per 64-token chunk.
int proj_bwd_splits(int M, int N, int chunks) {
  const int sms = sm_count_cached();
  if (sms <= 0) return 0;
  const int tiles = ((M + kBM - 1) / kBM) * ((N + kBN - 1) / kBN);
  int z = (2 * sms + tiles - 1) / tiles;
  if (z > chunks) z = chunks;
  if (z > 32) z = 32;
  return z < 1 ? 1 : z;
}

cudaError_t launch_proj_bwd(const CUtensorMap& ta0, const CUtensorMap& ta1, const CUtensorMap& ta2,
                            const CUtensorMap& tb0, const CUtensorMap& tb1, const CUtensorMap& tb2,
                            const CUtensorMap& to, ProjBwdParams p, cudaStream_t stream) {
  static std::once_flag once[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaError_t attr = cudaSuccess;
  std::call_once(once[dev & 63], [&] {
    attr = cudaFuncSetAttribute(attn_proj_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kBSmem));
  });
  if (attr != cudaSuccess) return attr;
  const int sms = sm_count_cached();
  if (sms <= 0) return cudaErrorUnknown;
  const int tiles_n = (p.N + kBN - 1) / kBN;
  long long units;
  if (p.kind == 0) {
    p.tiles_s = (p.S + kBM - 1) / kBM;
    units = static_cast<long long>(p.B) * p.tiles_s * tiles_n;
  } else {
    p.tiles_m = (p.M + kBM - 1) / kBM;
    p.chunks_s = (p.S + kBK - 1) / kBK;
    p.chunks = p.B * p.chunks_s;
    p.cps = (p.chunks + p.splits - 1) / p.splits;
    units = static_cast<long long>(p.splits) * p.tiles_m * tiles_n;
  }
  if (units > 0x7fffffffLL) return cudaErrorInvalidValue;
  p.num_units = static_cast<int>(units);
  if (p.num_units == 0) return cudaSuccess;
  const int grid = p.num_units < sms ? p.num_units : sms;
  prof_begin(kKindProj, stream);
  attn_proj_bwd_kernel<<<grid, kBThreads, kBSmem, stream>>>(ta0, ta1, ta2, tb0, tb1, tb2, to, p);
  e = cudaGetLastError();
  prof_end(kKindProj, stream);
  return e;
}

cudaError_t launch_proj_reduce(const float* part, void* out, long long count, int splits, cudaStream_t stream) {
  if (count == 0) return cudaSuccess;
  const long long threads = (count + 7) / 8;
  const int block = 256;
  const long long grid = (threads + block - 1) / block;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  prof_begin(kKindProj, stream);
  attn_proj_reduce_kernel<<<static_cast<int>(grid), block, 0, stream>>>(
      part, reinterpret_cast<__nv_bfloat16*>(out), count, splits);
  const cudaError_t e = cudaGetLastError();
  prof_end(kKindProj, stream);
  return e;
}

}  // namespace attn
