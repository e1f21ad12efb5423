// The multi-head projections around eq. (1) ("Attention Is All You Need"
// §3.2.2) as tcgen05 GEMMs:
//   mode 0:  Q = x_q W^Q,  K = x_kv W^K,  V = x_kv W^V  (x [B, S, d_model] rows,
//            W [d_model, h d] per projection), written straight into the
//            [B, h, S, d] layout of the attention kernels: the head split is
//            the output tensor map;
//   mode 1:  Y = Concat(head_1, ..., head_h) W^O, reading O straight from its
//            [B, h, S, d] layout: the concatenation is the reduction loop, one
//            head's columns per 64-wide step.
// Tiles are 128 tokens of one sequence (TMEM lanes) x 128 output columns;
// the reduction streams 64-wide A tiles (K-major) and W tiles (N-major,
// two 64-column boxes) through a 5-stage TMA ring. Persistent CTAs: warp 0
// loads, warp 1 issues the MMAs into one of two TMEM accumulators, warps 4-7
// move the other accumulator out (bf16, swizzled staging, TMA store), so a
// tile's epilogue overlaps the next tile's products.
#include "attn_kernels.cuh"

#include <mutex>

namespace attn {
namespace {

using namespace sm103;

constexpr int kPM = 128;                            // tokens per tile
constexpr int kPN = 128;                            // output columns per tile
constexpr int kPK = 64;                             // reduction per stage (one swizzle atom)
constexpr int kPStages = 5;
constexpr uint32_t kPATile = kPM * kPK * 2;         // 16 KB
constexpr uint32_t kPBBox = kPK * 64 * 2;           // 8 KB: 64 reduction rows x 64 columns
constexpr uint32_t kPStage = kPATile + 2 * kPBBox;  // 32 KB
constexpr uint32_t kPOffOut = kPStages * kPStage;   // staging: 2 tiles x 2 x [128 rows x 64 columns] bf16
constexpr uint32_t kPOutBox = kPM * 64 * 2;         // 16 KB
constexpr uint32_t kPSmem = kPOffOut + 4 * kPOutBox + 1024;
constexpr int kPThreads = 256;

struct ProjShared {
  uint64_t full[kPStages], empty[kPStages];
  uint64_t acc_full[2], acc_free[2];
  uint64_t staged, stage_free[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void drain_wait_proj(uint64_t* bar, uint32_t parity, const Watchdog& wd) {
  if (mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > wd.budget_ns) {
      atomicCAS(wd.status, 0u, kDevTimeout | kSiteDrain);
      return;
    }
  }
}

__global__ void __launch_bounds__(kPThreads, 1)
attn_proj_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                 const __grid_constant__ CUtensorMap tm_o0, const __grid_constant__ CUtensorMap tm_o1,
                 const __grid_constant__ CUtensorMap tm_o2, const ProjParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) ProjShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &sh.abort_flag;
  const Watchdog wd = p.wd;
  const int kchunks = p.K / kPK;
  const int tiles_n = (p.N + kPN - 1) / kPN;
  // tile t: output columns n0 = (t % tiles_n) * 128 of tokens s0.. of sequence b
  auto tile_of = [&](int t, int& b, int& s0, int& n0) {
    const int mt = t / tiles_n;
    n0 = (t - mt * tiles_n) * kPN;
    b = mt / p.tiles_s;
    s0 = (mt - b * p.tiles_s) * kPM;
  };

  if (tid == 0) {
    for (int s = 0; s < kPStages; ++s) {
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
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_a);
    prefetch_tensormap(&tm_b);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      long long g = 0;  // stages filled so far
      uint32_t filled = 0, last_ph = 0;  // per stage: filled at least once, parity of its last fill
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
        int b, s0, n0;
        tile_of(t, b, s0, n0);
        for (int kc = 0; ok && kc < kchunks; ++kc, ++g) {
          const int st = static_cast<int>(g % kPStages);
          if (g >= kPStages &&
              !(ok = guarded_wait(&sh.empty[st], static_cast<uint32_t>((g / kPStages - 1) & 1), abort_flag, wd,
                                  kSiteKEmpty)))
            break;
          uint8_t* sA = smem + st * kPStage;
          uint8_t* sB = sA + kPATile;
          mbar_arrive_expect_tx(&sh.full[st], kPStage);
          filled |= 1u << st;
          last_ph = (last_ph & ~(1u << st)) | (static_cast<uint32_t>((g / kPStages) & 1) << st);
          if (p.mode == 0) {
            tma_load_3d(sA, &tm_a, &sh.full[st], kc * kPK, s0, b);
          } else {
            const int k0 = kc * kPK;  // columns c0.. of head hh
            tma_load_3d(sA, &tm_a, &sh.full[st], k0 % p.d, s0, b * p.h + k0 / p.d);
          }
          tma_load_3d(sB, &tm_b, &sh.full[st], p.n_base + n0, kc * kPK, 0);
          tma_load_3d(sB + kPBBox, &tm_b, &sh.full[st], p.n_base + n0 + 64, kc * kPK, 0);
        }
      }
      // Let every copy this thread started land before shared memory is released.
      for (int s = 0; s < kPStages; ++s)
        if ((filled >> s) & 1u) drain_wait_proj(&sh.full[s], (last_ph >> s) & 1u, wd);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kPM, kPN, false, true);  // A K-major, B N-major
      long long g = 0;
      int tc = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x, ++tc) {
        const int buf = tc & 1;
        // the epilogue must have read this accumulator's previous tile
        if (tc >= 2 &&
            !(ok = guarded_wait(&sh.acc_free[buf], static_cast<uint32_t>((tc / 2 - 1) & 1), abort_flag, wd,
                                kSiteOFull)))
          break;
        for (int kc = 0; ok && kc < kchunks; ++kc, ++g) {
          const int st = static_cast<int>(g % kPStages);
          if (!(ok = guarded_wait(&sh.full[st], static_cast<uint32_t>((g / kPStages) & 1), abort_flag, wd,
                                  kSiteKFull)))
            break;
          tc_fence_after();
          const uint32_t sA = smem_u32(smem + st * kPStage), sB = sA + kPATile;
#pragma unroll
          for (int k = 0; k < kPK / 16; ++k) {
            const uint64_t da = smem_desc(sA + k * 32, 16, 1024, 2);
            const uint64_t db = smem_desc(sB + k * 16 * 128, kPBBox, 1024, 2);
            mma_ss(tmem + buf * kPN, da, db, idesc, (kc > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(&sh.empty[st]);  // the stage may be refilled once these products read it
        }
        if (ok) mma_commit(&sh.acc_full[buf]);
      }
      // Every MMA this thread issued must finish before TMEM is released.
      mma_commit(&sh.drain);
      drain_wait_proj(&sh.drain, 0, wd);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue: TMEM -> bf16 -> TMA store
    const int r = tid - 128;  // token row of the tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint8_t* stage = smem + kPOffOut;
    int tc = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++tc) {
      int b, s0, n0;
      tile_of(t, b, s0, n0);
      const int buf = tc & 1;
      bool ok = __all_sync(0xffffffffu, guarded_wait(&sh.acc_full[buf], static_cast<uint32_t>((tc / 2) & 1),
                                                     abort_flag, wd, kSiteOFull));
      // staging set sb (of two) was last used by tile tc - 2: its stores must have read it
      const int sb = tc & 1;
      if (ok && tc >= 2)
        ok = __all_sync(0xffffffffu, guarded_wait(&sh.stage_free[sb], static_cast<uint32_t>((tc / 2 - 1) & 1),
                                                  abort_flag, wd, kSiteOFull));
      if (!ok) break;
      uint8_t* tstage = stage + sb * 2 * kPOutBox;
      tc_fence_after();
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t v[2][32];
        tmem_ld32(tmem + lane_base + buf * kPN + half * 64, v[0]);
        tmem_ld32(tmem + lane_base + buf * kPN + half * 64 + 32, v[1]);
        tmem_ld_wait();
        if (half == 1) {
          tc_fence_before();
          mbar_arrive(&sh.acc_free[buf]);  // the MMAs of a later tile may overwrite this accumulator
        }
        uint8_t* box = tstage + half * kPOutBox;
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
            const int c = n0 + half * 64;  // output column of this box
            if (c >= p.N) break;
            if (p.mode == 0) {
              // column p.n_base + c of Q | K | V: projection, head and column within the head
              const int gc = p.n_base + c, hd = p.h * p.d;
              const int which = gc / hd, within = gc - which * hd;
              const CUtensorMap* map = which == 0 ? &tm_o0 : (which == 1 ? &tm_o1 : &tm_o2);
              tma_store_3d(map, tstage + half * kPOutBox, within % p.d, s0, b * p.h + within / p.d);
            } else {
              tma_store_3d(&tm_o0, tstage + half * kPOutBox, c, s0, b);
            }
          }
          tma_store_commit();
        }
        // the previous tile's stores (the other staging set) have read their source
        // once every group but this tile's has: that set may be written again
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

}  // namespace

cudaError_t launch_proj(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& to0,
                        const CUtensorMap& to1, const CUtensorMap& to2, ProjParams p, cudaStream_t stream) {
  static std::once_flag once[64];
  static int sm_count[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaError_t attr = cudaSuccess;
  std::call_once(once[dev & 63], [&] {
    attr = cudaFuncSetAttribute(attn_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kPSmem));
  });
  if (attr != cudaSuccess) return attr;
  if (sm_count[dev & 63] == 0) {
    int c = 0;
    if ((e = cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    sm_count[dev & 63] = c > 0 ? c : 1;
  }
  p.tiles_s = (p.S + kPM - 1) / kPM;
  const long long tiles = static_cast<long long>(p.B) * p.tiles_s * ((p.N + kPN - 1) / kPN);
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  p.num_tiles = static_cast<int>(tiles);
  if (p.num_tiles == 0) return cudaSuccess;
  const int grid = p.num_tiles < sm_count[dev & 63] ? p.num_tiles : sm_count[dev & 63];
  prof_begin(kKindProj, stream);
  attn_proj_kernel<<<grid, kPThreads, kPSmem, stream>>>(ta, tb, to0, to1, to2, p);
  e = cudaGetLastError();
  prof_end(kKindProj, stream);
  return e;
}

}  // namespace attn
