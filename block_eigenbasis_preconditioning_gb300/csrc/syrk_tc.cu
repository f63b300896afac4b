// Block second moments on the tensor cores, bf16 activations:
//   A_b <- beta2 A_b + (1 - beta2) X_b^T X_b / N
// ("Dobb", Abstract: diagonal blocks of the input-activation second moment;
// Table 3 caption: n^2/B entries per matrix).
//
// D = X_b^T X_b is a contraction over tokens.  One TMA tile of X (64 tokens x
// 64 features per box, 128-byte swizzle) is both MMA operands: A = X_b^T
// (M = features of a 128-row slice, MN-major) and B = X_b (N = the block's
// features from the slice's first one on: only the upper triangle of D is
// needed, so later slices read fewer features), MN-major.  bf16 x bf16 products are exact in fp32; the
// tensor core accumulates them in fp32 in TMEM.
//
// Work unit: (matrix, block, 128-row slice of the block).  The epilogue
// warps read D row by row from TMEM and write the EMA of the upper triangle
// to both A[i][j] and A[j][i], so A stays exactly symmetric.  When every
// block of a launch spans at most 256 columns, two accumulators alternate in
// TMEM, so the next unit's products run while the epilogue drains the last.
//
// TMA needs a 16-byte aligned start column: a block starting at column b k
// is loaded from column x0 = (b k) & ~7 and all indices shift by
// d = b k - x0 (the extra columns belong to the neighbouring block and are
// never written).
#include <cuda.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace dobb {
namespace {

using namespace ptx;

constexpr int kThreads = 192;       // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kTok = 64;            // tokens per stage
constexpr int kBoxBytes = kTok * 128;  // 64 tokens x 64 bf16 features
constexpr uint32_t kTmemCols = 512;

constexpr int kMaxSyStages = 16;

struct SySmem {
  uint64_t full[kMaxSyStages], empty[kMaxSyStages];
  uint64_t d_full[2], d_free[2];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool sy_aborted(const SySmem* sh) {
  return *reinterpret_cast<const volatile int*>(&sh->abort) != 0;
}

struct SyTile {
  int64_t N, n;
  int k, delta, nbox, ext;  // ext = k + delta (features spanned)
  int x0, np;               // np: ext padded to 16
  int t0, t1;               // the unit's slices [t0, t1)
  int wbox, nboxw;          // the unit's feature window: first box, boxes
};

__device__ __forceinline__ SyTile sy_tile(const SyrkTcArgs& a, const Tile& tl) {
  SyTile s;
  const MatInfo mi = a.info[tl.mat];
  s.N = a.N[tl.mat - a.mat_base];
  s.n = mi.n;
  s.k = mi.k;
  const int64_t c0 = (int64_t)tl.blk * mi.k;
  s.x0 = (int)(c0 & ~int64_t(7));
  s.delta = (int)(c0 - s.x0);
  s.ext = s.k + s.delta;
  s.nbox = ((s.ext + 127) / 128) * 2;  // whole 128-feature slices
  s.np = (s.ext + 15) & ~15;
  // slice t holds rows [128 t, 128 t + 128) of the extended block and needs
  // only the columns at or right of them (the upper triangle); a unit of
  // slices [t0, t1) reads the window from its first slice's first feature
  s.t0 = tl.a;
  s.t1 = tl.b;
  s.wbox = 2 * tl.a;
  s.nboxw = s.nbox - s.wbox;
  return s;
}

__global__ void __launch_bounds__(kThreads, 1)
syrk_tc_kernel(const __grid_constant__ SyrkTcArgs a) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const int nst = a.stages;
  const int stage_bytes = a.stage_bytes;
  SySmem* sh = reinterpret_cast<SySmem*>(base + (size_t)nst * stage_bytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(&sh->full[i], 1);
      mbar_init(&sh->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh->d_full[i], 1);
      mbar_init(&sh->d_free[i], 4);
    }
    sh->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&sh->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t st = 0, ph = 0;
      for (int w = blockIdx.x; w < a.num_tiles && !sy_aborted(sh); w += gridDim.x) {
        const Tile tl = a.tiles[w];
        const SyTile s = sy_tile(a, tl);
        if (a.X[tl.mat - a.mat_base] == nullptr || s.N <= 0) continue;
        const CUtensorMap* map = &a.maps[tl.mat - a.mat_base];
        for (int64_t t0 = 0; t0 < s.N; t0 += kTok) {
          if (!mbar_wait(&sh->empty[st], ph ^ 1)) { sh->abort = 1; atomicOr(a.err, 16u); break; }
          mbar_arrive_expect_tx(&sh->full[st], (uint32_t)(s.nboxw * kBoxBytes));
          for (int q = 0; q < s.nboxw; ++q)
            tma_load_2d(base + (size_t)st * stage_bytes + q * kBoxBytes, map,
                        s.x0 + 64 * (s.wbox + q), (int)t0, &sh->full[st]);
          if (++st == (uint32_t)nst) { st = 0; ph ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    uint32_t st = 0, ph = 0, tile_i = 0;
    for (int w = blockIdx.x; w < a.num_tiles && !sy_aborted(sh); w += gridDim.x) {
      const Tile tl = a.tiles[w];
      const SyTile s = sy_tile(a, tl);
      if (a.X[tl.mat - a.mat_base] == nullptr || s.N <= 0) continue;
      // this unit's accumulator must have been drained by the epilogue
      const uint32_t b = a.dbuf ? (tile_i & 1) : 0u;       // accumulator
      const uint32_t use = a.dbuf ? (tile_i >> 1) : tile_i;  // earlier uses of it
      if (use > 0 && !warp_wait(&sh->d_free[b], (use - 1) & 1)) {
        sh->abort = 1;
        atomicOr(a.err, 32u);
        break;
      }
      tc_fence_after();
      const uint32_t dacc = tmem + 256 * b;
      bool ok = true;
      uint32_t first = 1;
      for (int64_t t0 = 0; t0 < s.N; t0 += kTok) {
        if (!warp_wait(&sh->full[st], ph)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t sb = smem_u32(base + (size_t)st * stage_bytes);
          const uint32_t lbo = kBoxBytes;  // next 64-feature box
          // slice t: A = its own 128 features, B = the features from them
          // on; accumulators side by side from column 0 of this unit's TMEM
          uint32_t col = 0;
          for (int t = s.t0; t < s.t1; ++t) {
            const int nt = s.np - 128 * t;
            const int n0 = min(256, nt), n1 = nt - n0;
            // MN-major operands: transpose bits for A and B
            const uint32_t id0 = instr_desc(1, 128, n0) | (1u << 15) | (1u << 16);
            const uint32_t id1 = n1 > 0 ? (instr_desc(1, 128, n1) | (1u << 15) | (1u << 16)) : 0u;
            const uint32_t sbt = sb + (uint32_t)(2 * (t - s.t0)) * kBoxBytes;
            for (int kk = 0; kk < kTok / 16; ++kk) {
              const uint32_t koff = kk * 2048;  // 16 tokens x 128 B
              const uint64_t da = smem_desc(sbt + koff, lbo, 1024, kSw128);
              const uint32_t acc = (first && kk == 0) ? 0u : 1u;  // the unit's first product
              mma_f16_ss(dacc + col, da, da, id0, acc);
              if (n1 > 0) {
                const uint64_t db1 = smem_desc(sbt + 4 * kBoxBytes + koff, lbo, 1024, kSw128);
                mma_f16_ss(dacc + col + 256, da, db1, id1, acc);
              }
            }
            col += (uint32_t)syrk_tc_slice_cols(s.np, t);
          }
          first = 0;
          tc_commit(&sh->empty[st]);
        }
        __syncwarp();
        if (++st == (uint32_t)nst) { st = 0; ph ^= 1; }
      }
      if (!ok) { sh->abort = 1; atomicOr(a.err, 64u); break; }
      if (lane == 0) tc_commit(&sh->d_full[b]);
      __syncwarp();
      ++tile_i;
    }
    // drain before TMEM is released: the last use of each accumulator
    for (uint32_t b = 0; b < 2; ++b) {
      const uint32_t uses = a.dbuf ? (tile_i + 1 - b) / 2 : (b == 0 ? tile_i : 0u);
      if (uses > 0) warp_wait(&sh->d_free[b], (uses - 1) & 1);
    }
  } else {
    const int g = warp & 3;
    const int r = 32 * g + lane;  // row of the 128-row slice
    const uint32_t trow = tmem + ((uint32_t)(32 * g) << 16);
    uint32_t tile_i = 0;
    for (int w = blockIdx.x; w < a.num_tiles && !sy_aborted(sh); w += gridDim.x) {
      const Tile tl = a.tiles[w];
      const SyTile s = sy_tile(a, tl);
      if (a.X[tl.mat - a.mat_base] == nullptr || s.N <= 0) continue;
      const MatInfo mi = a.info[tl.mat];
      const uint32_t b = a.dbuf ? (tile_i & 1) : 0u;
      const uint32_t use = a.dbuf ? (tile_i >> 1) : tile_i;
      if (!warp_wait(&sh->d_full[b], use & 1)) { sh->abort = 1; atomicOr(a.err, 128u); break; }
      tc_fence_after();
      float* Ab = a.A + mi.a_off + (int64_t)tl.blk * s.k * s.k;
      const float c1 = (1.f - a.beta2) / (float)s.N;
      int bad = 0;
      uint32_t col = 0;
      for (int t = s.t0; t < s.t1; ++t) {
        const int i = 128 * t + r - s.delta;  // row within the block
        const bool rvalid = i >= 0 && i < s.k;
        const int nt = s.np - 128 * t;
        for (int c0 = 0; c0 < nt; c0 += 32) {
          float v[32];
          tmem_ld32(trow + 256 * b + col + c0, v);
          tmem_wait_ld(v);
          if (rvalid) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int j = 128 * t + c0 + e - s.delta;
              if (j >= i && j < s.k) {
                bad |= !isfinite(v[e]);
                const float nv = fmaf(a.beta2, Ab[(int64_t)i * s.k + j], c1 * v[e]);
                Ab[(int64_t)i * s.k + j] = nv;
                if (j != i) Ab[(int64_t)j * s.k + i] = nv;
              }
            }
          }
        }
        col += (uint32_t)syrk_tc_slice_cols(s.np, t);
      }
      if (__any_sync(0xffffffffu, bad) && lane == 0)
        atomicOr(a.flags + mi.blk0 + tl.blk, (uint32_t)DOBB_FLAG_NONFINITE_X);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->d_free[b]);
      ++tile_i;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

size_t syrk_tc_stage_bytes(int max_k) {
  // every block may start up to 7 columns early; whole 128-feature slices
  const int ext = max_k + 7;
  return (size_t)((ext + 127) / 128) * 2 * kBoxBytes;
}

int syrk_tc_stages(int max_k, size_t smem_limit) {
  const size_t sb = syrk_tc_stage_bytes(max_k);
  int st = (int)((smem_limit - 2048) / sb);
  return std::max(2, std::min(kMaxSyStages, st));
}

size_t syrk_tc_smem(int max_k, int stages) {
  return 1024 + (size_t)stages * syrk_tc_stage_bytes(max_k) + sizeof(SySmem) + 64;
}

bool syrk_tc_double_buffer(int max_k) { return ((max_k + 7 + 15) & ~15) <= 256; }

bool syrk_tc_eligible(int64_t n, int k) { return n % 8 == 0 && k <= kMaxTcK && k >= 8; }

cudaError_t configure_syrk_tc(size_t smem_limit) {
  return cudaFuncSetAttribute(syrk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem_limit);
}

cudaError_t launch_syrk_tc(const SyrkTcArgs& a, int grid, size_t smem, cudaStream_t s) {
  if (a.num_tiles <= 0) return cudaSuccess;
  syrk_tc_kernel<<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dobb
