// Grouped update kernel on the 5th-generation tensor cores (tcgen05, TMEM).
//
// For one tile of 128 rows of one column block b (width k) of one matrix:
//   M <- beta1 M + G                        converter warps (fp32)
//   C_b = M_b Q_b                           tcgen05 kind::tf32, 3 passes
//   S_b = sign(C_b)                         epilogue warps, S kept in TMEM
//   U_b = S_b Q_b^T                         tcgen05 kind::f16, A = S from TMEM
//   W <- W - lr s U_b                       epilogue warps
// "Dobb", Abstract (project the momentum into the block bases, sign-normalise
// the coefficients, reconstruct the update) and Table 9 (update scale s).
//
// Precision.  sign(C) is decided near |C| ~ 0, so C is formed at fp32-level
// accuracy with the split-precision product M Q ~ Mh Qh + Mh Ql + Ml Qh
// (h = TF32 rounding, l = remainder), relative error ~2^-21.  S is exactly
// representable in bf16, so U needs only Q split into bf16 pieces: three
// (Q = Qh + Ql + Qll, 24 significant bits, representation error <= 2^-27 |Q|
// per entry, i.e. |dU_ij| <= 2^-27 sum_l |Q_jl| <= 2^-27 sqrt(k)) for the fp32
// basis, one (exact) for the bf16 basis.
//
// Warp roles (320 threads): warp 0 loads (TMA for M tiles, bulk copies for
// the pre-packed Q operand images), warp 1 allocates TMEM and issues the
// MMAs, warps 2-5 update the momentum and split it into the TF32 operand
// pair in shared memory, warps 6-9 (one per TMEM lane quarter) turn C into
// packed bf16 signs in TMEM and drain U into W.  Stages are handed over with
// mbarriers; every wait gives up after a timeout and raises an error flag.
//
// TMEM columns: C at [0, kpN) during the projection, S (bf16 pairs) at
// [0, kpN/2) afterwards, U chunks of 128 columns double-buffered at 256 and
// 384.  Blocks with kpN <= 128 alternate C between [0, 128) and [128, 256),
// which lets the MMA warp project tile t+1 before it reconstructs tile t.
#include <cuda.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace dobb {
namespace {

using namespace ptx;

constexpr int kThreads = 320;
constexpr int kTM = 128;
constexpr int kMaxAStages = 4;   // momentum stages: the launch picks 2 ... 4
constexpr int kMaxBStages = 16;  // the launch picks how many fit (small blocks: many)
constexpr int kAChunkBytes = kTM * 32 * 4;  // 32 fp32 columns, 128B swizzle
constexpr int kUCols = 128;
constexpr uint32_t kTmemCols = 512;

struct TcSmem {
  uint64_t a_full[kMaxAStages], a_conv[kMaxAStages], a_empty[kMaxAStages];
  uint64_t b_full[kMaxBStages], b_empty[kMaxBStages];
  uint64_t c_full[2], s_full;   // c_full per C region (tile parity)
  uint64_t u_full[2], u_empty[2];
  uint64_t r_done, fin;
  uint32_t tmem_base;
  int abort;
};

// Reconstruct K steps (16 wide) that one basis stage carries: as many
// sub-step images of sb bytes as fit the stage.
__device__ __forceinline__ int recon_per_stage(int bstage, uint32_t sb) {
  return max(1, bstage / (int)sb);
}

// mbarrier wait whose outcome is the same on every lane of the warp (the
// callers run warp-collective tcgen05 instructions right after it).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool aborted(const TcSmem* sh) {
  return *reinterpret_cast<const volatile int*>(&sh->abort) != 0;
}

// C / S columns of a tile: small blocks alternate between two regions so the
// next tile's projection never overwrites signs still being consumed.
__device__ __forceinline__ uint32_t c_base(int kpN, uint32_t tile_i) {
  return (kpN <= 128 && (tile_i & 1)) ? 128u : 0u;
}

__device__ __forceinline__ void raise(TcSmem* sh, uint32_t* err, uint32_t code) {
  sh->abort = 1;
  atomicOr(err, code);
}

template <typename PT>
__device__ __forceinline__ void load4(const PT* p, float (&v)[4]);
template <>
__device__ __forceinline__ void load4<float>(const float* p, float (&v)[4]) {
  const float4 t = *reinterpret_cast<const float4*>(p);
  v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
}
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 t = *reinterpret_cast<const uint2*>(p);
  v[0] = __uint_as_float(t.x << 16);
  v[1] = __uint_as_float(t.x & 0xFFFF0000u);
  v[2] = __uint_as_float(t.y << 16);
  v[3] = __uint_as_float(t.y & 0xFFFF0000u);
}

template <typename PT>
__device__ __forceinline__ void store4(PT* p, const float (&v)[4]);
template <>
__device__ __forceinline__ void store4<float>(float* p, const float (&v)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, const float (&v)[4]) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
  const __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
  uint2 t;
  t.x = *reinterpret_cast<const uint32_t*>(&a);
  t.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = t;
}

// Four consecutive columns of one row of a matrix whose caller's buffer is
// the transpose (output side): elements `stride` apart.
template <typename PT>
__device__ __forceinline__ void load4_t(const PT* p, int64_t stride, float (&v)[4]);
template <>
__device__ __forceinline__ void load4_t<float>(const float* p, int64_t stride, float (&v)[4]) {
#pragma unroll
  for (int z = 0; z < 4; ++z) v[z] = p[z * stride];
}
template <>
__device__ __forceinline__ void load4_t<__nv_bfloat16>(const __nv_bfloat16* p, int64_t stride,
                                                      float (&v)[4]) {
#pragma unroll
  for (int z = 0; z < 4; ++z) v[z] = __bfloat162float(p[z * stride]);
}
template <typename PT>
__device__ __forceinline__ void store4_t(PT* p, int64_t stride, const float (&v)[4]);
template <>
__device__ __forceinline__ void store4_t<float>(float* p, int64_t stride, const float (&v)[4]) {
#pragma unroll
  for (int z = 0; z < 4; ++z) p[z * stride] = v[z];
}
template <>
__device__ __forceinline__ void store4_t<__nv_bfloat16>(__nv_bfloat16* p, int64_t stride,
                                                       const float (&v)[4]) {
#pragma unroll
  for (int z = 0; z < 4; ++z) p[z * stride] = __float2bfloat16_rn(v[z]);
}

__device__ __forceinline__ uint32_t bf16_sign_bits(float x) {
  return x > 0.f ? 0x3F80u : (x < 0.f ? 0xBF80u : 0u);
}

// kMayT: the launch may hold output-side matrices (caller's buffers
// transposed); the instantiation without it carries none of that addressing.
template <typename PT, bool kMayT>
__global__ void __launch_bounds__(kThreads, 1)
step_tc_kernel(const __grid_constant__ StepArgs a, const __grid_constant__ TcArgs t) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  // 1024-byte aligned operand region
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  const int nas = t.nastage;                                     // momentum stages
  unsigned char* a_buf = base;                                   // [stage][hi|lo]
  unsigned char* b_buf = base + nas * 2 * kAChunkBytes;          // [stage] t.bstage bytes
  TcSmem* sh = reinterpret_cast<TcSmem*>(b_buf + t.nbstage * t.bstage);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t nbs = (uint32_t)t.nbstage;  // B stages of this launch
  const bool two = t.npieces == 2;           // fp32 basis: hi and lo operand pieces
  if (threadIdx.x == 0) {
    for (int i = 0; i < nas; ++i) {
      mbar_init(&sh->a_full[i], 1);
      mbar_init(&sh->a_conv[i], 4);
      mbar_init(&sh->a_empty[i], 1);
    }
    for (int i = 0; i < t.nbstage; ++i) {
      mbar_init(&sh->b_full[i], 1);
      mbar_init(&sh->b_empty[i], 1);
    }
    mbar_init(&sh->c_full[0], 1);
    mbar_init(&sh->c_full[1], 1);
    mbar_init(&sh->s_full, 4);
    mbar_init(&sh->r_done, 1);
    mbar_init(&sh->fin, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh->u_full[i], 1);
      mbar_init(&sh->u_empty[i], 4);
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

  // Narrow blocks (C of two tiles fits the two halves of TMEM columns
  // [0, 256)) defer each tile's reconstruct until the next tile's projection
  // has been issued: the MMA warp then projects while the epilogue signs.
  const bool defer = t.defer != 0;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // momentum chunks and basis images, the images in the order the MMA
    // warp consumes them
    if (lane == 0) {
      uint32_t as = 0, ap = 0, bs = 0, bp = 0;
      const unsigned char* pend_qr = nullptr;  // deferred reconstruct images
      int pend_kpN = 0;
      auto load_recon = [&](const unsigned char* qr, int kpN) {
        // reconstruct operands: chunks of 128 output columns, 16-wide K steps
        int64_t off = 0;
        for (int c0 = 0; c0 < kpN && !aborted(sh); c0 += kUCols) {
          const int nn = min(kUCols, kpN - c0);
          const uint32_t sb = (uint32_t)t.rpieces * nn * 32u;   // one K step's images
          const int per = recon_per_stage(t.bstage, sb), nsteps = kpN / 16;
          for (int s = 0; s < nsteps; s += per) {
            const uint32_t bytes = sb * (uint32_t)min(per, nsteps - s);
            if (!mbar_wait(&sh->b_empty[bs], bp ^ 1)) { raise(sh, t.err, 3); return; }
            mbar_arrive_expect_tx(&sh->b_full[bs], bytes);
            bulk_load(b_buf + bs * t.bstage, qr + off, bytes, &sh->b_full[bs]);
            off += bytes;
            if (++bs == nbs) { bs = 0; bp ^= 1; }
          }
        }
      };
      for (int w = blockIdx.x; w < a.num_tiles && !aborted(sh); w += gridDim.x) {
        const Tile tl = a.tiles[w];
        const MatInfo mi = a.info[tl.mat];
        const int k = mi.k, kpN = (k + 15) & ~15;
        const int nsub = (k + 7) / 8, nk32 = (k + 31) / 32;
        const unsigned char* qp = t.qpack + mi.qp_off + (int64_t)tl.blk * mi.qblk_bytes;
        const unsigned char* qr = qp + (int64_t)nsub * t.npieces * kpN * 32;
        const CUtensorMap* map = reinterpret_cast<const CUtensorMap*>(t.maps) + tl.mat;
        for (int kc = 0; kc < nk32; ++kc) {
          if (!mbar_wait(&sh->a_empty[as], ap ^ 1)) { raise(sh, t.err, 1); break; }
          mbar_arrive_expect_tx(&sh->a_full[as], kAChunkBytes);
          tma_load_2d(a_buf + as * 2 * kAChunkBytes, map, tl.blk * k + kc * 32, tl.a,
                      &sh->a_full[as]);
          if (++as == (uint32_t)nas) { as = 0; ap ^= 1; }
          for (int s4 = 0; s4 < 4; ++s4) {
            const int sub = kc * 4 + s4;
            if (sub >= nsub) break;
            if (!mbar_wait(&sh->b_empty[bs], bp ^ 1)) { raise(sh, t.err, 2); break; }
            const uint32_t bytes = (uint32_t)t.npieces * kpN * 32u;
            mbar_arrive_expect_tx(&sh->b_full[bs], bytes);
            bulk_load(b_buf + bs * t.bstage, qp + (int64_t)sub * bytes, bytes, &sh->b_full[bs]);
            if (++bs == nbs) { bs = 0; bp ^= 1; }
          }
        }
        if (defer) {
          if (pend_qr) load_recon(pend_qr, pend_kpN);
          pend_qr = qr;
          pend_kpN = kpN;
        } else {
          load_recon(qr, kpN);
        }
      }
      if (pend_qr && !aborted(sh)) load_recon(pend_qr, pend_kpN);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    uint32_t as = 0, ap = 0, bs = 0, bp = 0, tile_i = 0;
    uint32_t uses[2] = {0, 0}, waited[2] = {0, 0}, ucount = 0;
    uint32_t r_issued = 0, r_waited = 0;     // reconstruct completions
    uint32_t prev_lo = 0, prev_hi = 0;       // S columns of the last reconstructed tile
    // U = S Q^T for the tile whose signs are at columns [cb, cb + kpN / 2)
    auto reconstruct = [&](uint32_t ti, uint32_t cb, int kpN) -> bool {
      // wait for the signs in TMEM, then reconstruct U chunk by chunk
      if (!warp_wait(&sh->s_full, ti & 1)) { raise(sh, t.err, 6); return false; }
      tc_fence_after();
      for (int c0 = 0; c0 < kpN; c0 += kUCols) {
        const int nn = min(kUCols, kpN - c0);
        const int b = ucount & 1;
        while (waited[b] < uses[b]) {
          if (!warp_wait(&sh->u_empty[b], waited[b] & 1)) { raise(sh, t.err, 7); return false; }
          ++waited[b];
        }
        tc_fence_after();
        const uint32_t idr = instr_desc(1, kTM, nn);
        const uint32_t d = tmem + 256 + kUCols * b;
        const uint32_t sb = (uint32_t)t.rpieces * nn * 32u;
        const int per = recon_per_stage(t.bstage, sb), nsteps = kpN / 16;
        for (int s = 0; s < nsteps; s += per) {
          const int cnt = min(per, nsteps - s);
          if (!warp_wait(&sh->b_full[bs], bp)) { raise(sh, t.err, 7); return false; }
          tc_fence_after();
          if (lane == 0) {
            for (int u = 0; u < cnt; ++u) {
              const uint32_t b_hi = smem_u32(b_buf + bs * t.bstage) + (uint32_t)u * sb;
              for (int p = 0; p < t.rpieces; ++p)
                mma_f16_ts(d, tmem + cb + 8 * (s + u), smem_desc(b_hi + p * nn * 32, 16, 256, kSw32), idr,
                           (s + u == 0 && p == 0) ? 0u : 1u);
            }
            tc_commit(&sh->b_empty[bs]);
          }
          __syncwarp();
          if (++bs == nbs) { bs = 0; bp ^= 1; }
        }
        if (lane == 0) tc_commit(&sh->u_full[b]);
        __syncwarp();
        ++uses[b];
        ++ucount;
      }
      // completion of this tile's reconstruct MMAs (they read the signs).
      // At most one phase of r_done is ever pending: retire the previous one
      // before committing the next, so a parity wait cannot skip a phase.
      if (r_issued > r_waited) {
        if (!warp_wait(&sh->r_done, r_waited & 1)) { raise(sh, t.err, 12); return false; }
        ++r_waited;
      }
      if (lane == 0) tc_commit(&sh->r_done);
      __syncwarp();
      ++r_issued;
      prev_lo = cb;
      prev_hi = cb + (uint32_t)(kpN / 2);
      return true;
    };
    bool pending = false;                    // a projected tile awaits its reconstruct
    uint32_t pend_ti = 0, pend_cb = 0;
    int pend_kpN = 0;
    for (int w = blockIdx.x; w < a.num_tiles && !aborted(sh); w += gridDim.x, ++tile_i) {
      const Tile tl = a.tiles[w];
      const MatInfo mi = a.info[tl.mat];
      const int k = mi.k, kpN = (k + 15) & ~15;
      const int nsub = (k + 7) / 8, nk32 = (k + 31) / 32;
      bool ok = true;
      if (kpN > 256) {
        // C overlaps the U buffers: wait until the previous tile is drained
        for (int b = 0; b < 2 && ok; ++b)
          while (waited[b] < uses[b]) {
            if (!warp_wait(&sh->u_empty[b], waited[b] & 1)) { ok = false; break; }
            ++waited[b];
          }
        tc_fence_after();
      }
      if (!ok) { raise(sh, t.err, 4); break; }
      const uint32_t cb = c_base(kpN, tile_i);
      if (r_waited < r_issued && cb < prev_hi && prev_lo < cb + (uint32_t)kpN) {
        // this tile's C would overwrite signs the last reconstruct reads
        if (!warp_wait(&sh->r_done, r_waited & 1)) { raise(sh, t.err, 11); break; }
        ++r_waited;
        tc_fence_after();
      }
      const int n0a = min(256, kpN), n1a = kpN - n0a;
      const uint32_t id0 = instr_desc(2, kTM, n0a);
      const uint32_t id1 = n1a > 0 ? instr_desc(2, kTM, n1a) : 0;
      for (int kc = 0; kc < nk32 && ok; ++kc) {
        if (!warp_wait(&sh->a_conv[as], ap)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_hi = smem_u32(a_buf + as * 2 * kAChunkBytes);
        const uint32_t a_lo = a_hi + kAChunkBytes;
        for (int s4 = 0; s4 < 4; ++s4) {
          const int sub = kc * 4 + s4;
          if (sub >= nsub) break;
          if (!warp_wait(&sh->b_full[bs], bp)) { ok = false; break; }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t b_hi = smem_u32(b_buf + bs * t.bstage);
            const uint32_t b_lo = b_hi + kpN * 32;
            const uint64_t dah = smem_desc(a_hi + s4 * 32, 16, 1024, kSw128);
            const uint64_t dal = smem_desc(a_lo + s4 * 32, 16, 1024, kSw128);
            const uint32_t first = (sub == 0) ? 0u : 1u;
            // fp32 basis: Mh Qh + Mh Ql + Ml Qh; bf16 basis (exact in TF32): Mh Q + Ml Q
            {
              const uint64_t dbh = smem_desc(b_hi, 16, 256, kSw32);
              mma_tf32_ss(tmem + cb, dah, dbh, id0, first);
              if (two) mma_tf32_ss(tmem + cb, dah, smem_desc(b_lo, 16, 256, kSw32), id0, 1);
              mma_tf32_ss(tmem + cb, dal, dbh, id0, 1);
            }
            if (n1a > 0) {
              const uint64_t dbh = smem_desc(b_hi + 256 * 32, 16, 256, kSw32);
              mma_tf32_ss(tmem + cb + 256, dah, dbh, id1, first);
              if (two) mma_tf32_ss(tmem + cb + 256, dah, smem_desc(b_lo + 256 * 32, 16, 256, kSw32), id1, 1);
              mma_tf32_ss(tmem + cb + 256, dal, dbh, id1, 1);
            }
            tc_commit(&sh->b_empty[bs]);
          }
          __syncwarp();
          if (++bs == nbs) { bs = 0; bp ^= 1; }
        }
        if (lane == 0) tc_commit(&sh->a_empty[as]);
        __syncwarp();
        if (++as == (uint32_t)nas) { as = 0; ap ^= 1; }
      }
      if (!ok) { raise(sh, t.err, 5); break; }
      if (lane == 0) tc_commit(&sh->c_full[tile_i & 1]);
      __syncwarp();
      if (defer) {
        if (pending && !reconstruct(pend_ti, pend_cb, pend_kpN)) break;
        pending = true;
        pend_ti = tile_i;
        pend_cb = cb;
        pend_kpN = kpN;
      } else if (!reconstruct(tile_i, cb, kpN)) {
        break;
      }
    }
    if (pending && !aborted(sh)) reconstruct(pend_ti, pend_cb, pend_kpN);
    // let every issued MMA finish before TMEM is released
    if (lane == 0) tc_commit(&sh->fin);
    __syncwarp();
    warp_wait(&sh->fin, 0);
    for (int b = 0; b < 2; ++b)
      while (waited[b] < uses[b]) {
        if (!warp_wait(&sh->u_empty[b], waited[b] & 1)) break;
        ++waited[b];
      }
  } else if (warp < 6) {
    // ----------------------------------------------------------- converters
    const int ct = threadIdx.x - 64;  // 0..127
    const int cchunk = ct & 7, crow = ct >> 3;  // 16-byte chunk, row within 16-row pass
    uint32_t as = 0, ap = 0;
    for (int w = blockIdx.x; w < a.num_tiles && !aborted(sh); w += gridDim.x) {
      const Tile tl = a.tiles[w];
      const int slot = tl.mat - a.mat_base;
      const MatInfo mi = a.info[tl.mat];
      const int k = mi.k, nk32 = (k + 31) / 32;
      const int64_t n = mi.n;
      const int row0 = tl.a;
      const PT* G = static_cast<const PT*>(a.G[slot]);
      float* Mg = a.M + mi.m_off;
      int bad = 0;
      bool ok = true;
      for (int kc = 0; kc < nk32; ++kc) {
        const int col = kc * 32 + cchunk * 4;        // within the block
        const bool cvalid = col < k;                 // k % 4 == 0: all four or none
        float g[8][4];
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const int r = crow + 16 * p;
          if (cvalid && row0 + r < mi.m) {
            if (kMayT && mi.wt)   // caller's G is the transpose: element (i, j) at j m + i
              load4_t(G + ((int64_t)tl.blk * k + col) * mi.m + row0 + r, mi.m, g[p]);
            else
              load4(G + (int64_t)(row0 + r) * n + (int64_t)tl.blk * k + col, g[p]);
          } else {
            g[p][0] = g[p][1] = g[p][2] = g[p][3] = 0.f;
          }
        }
        if (!warp_wait(&sh->a_full[as], ap)) { ok = false; break; }
        unsigned char* hi = a_buf + as * 2 * kAChunkBytes;
        unsigned char* lo = hi + kAChunkBytes;
#pragma unroll
        for (int p = 0; p < 8; ++p) {
          const int r = crow + 16 * p;
          const uint32_t off = swz_offset((uint32_t)(r * 128 + cchunk * 16), 3);
          float4 mv = *reinterpret_cast<float4*>(hi + off);
          float4 h4 = make_float4(0.f, 0.f, 0.f, 0.f), l4 = h4;
          if (cvalid && row0 + r < mi.m) {
            float mn[4] = {fmaf(a.beta1, mv.x, g[p][0]), fmaf(a.beta1, mv.y, g[p][1]),
                           fmaf(a.beta1, mv.z, g[p][2]), fmaf(a.beta1, mv.w, g[p][3])};
            bad |= !(isfinite(mn[0]) && isfinite(mn[1]) && isfinite(mn[2]) && isfinite(mn[3]));
            *reinterpret_cast<float4*>(Mg + (int64_t)(row0 + r) * n + (int64_t)tl.blk * k + col) =
                make_float4(mn[0], mn[1], mn[2], mn[3]);
            float hv[4], lv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              hv[e] = tf32_rna(mn[e]);
              lv[e] = tf32_rna(mn[e] - hv[e]);
            }
            h4 = make_float4(hv[0], hv[1], hv[2], hv[3]);
            l4 = make_float4(lv[0], lv[1], lv[2], lv[3]);
          }
          *reinterpret_cast<float4*>(hi + off) = h4;
          *reinterpret_cast<float4*>(lo + off) = l4;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->a_conv[as]);
        if (++as == (uint32_t)nas) { as = 0; ap ^= 1; }
      }
      if (!ok) { raise(sh, t.err, 8); break; }
      if (__any_sync(0xffffffffu, bad) && lane == 0)
        atomicOr(a.flags + mi.blk0 + tl.blk, (uint32_t)DOBB_FLAG_NONFINITE_G);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int g = warp & 3;             // TMEM lane quarter
    const int r = 32 * g + lane;        // row within the tile
    const uint32_t trow = tmem + ((uint32_t)(32 * g) << 16);
    uint32_t tile_i = 0, ucount = 0, uphase[2] = {0, 0};
    for (int w = blockIdx.x; w < a.num_tiles && !aborted(sh); w += gridDim.x, ++tile_i) {
      const Tile tl = a.tiles[w];
      const int slot = tl.mat - a.mat_base;
      const MatInfo mi = a.info[tl.mat];
      const int k = mi.k, kpN = (k + 15) & ~15;
      const int64_t n = mi.n;
      const bool rvalid = tl.a + r < mi.m;
      const int64_t rowoff = (int64_t)(tl.a + r) * n + (int64_t)tl.blk * k;
      // output side: the caller's W, G and signs are the transpose, element
      // (i, j) at j m + i; this row's column 0 of the block is at colbase
      const bool wt = kMayT && mi.wt != 0;
      const int64_t colbase = (int64_t)tl.blk * k * mi.m + tl.a + r;
      PT* W = static_cast<PT*>(a.W[slot]);
      int8_t* Sout = a.S[slot];
      float c2 = 0.f, u2 = 0.f;
      if (!warp_wait(&sh->c_full[tile_i & 1], (tile_i >> 1) & 1)) { raise(sh, t.err, 9); break; }
      tc_fence_after();
      const uint32_t tc_row = trow + c_base(kpN, tile_i);
      for (int cc = 0; cc * 32 < kpN; ++cc) {
        float v[32];
        tmem_ld32(tc_row + 32 * cc, v);
        tmem_wait_ld(v);
        uint32_t pk[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int j0 = 32 * cc + 2 * q;
          const uint32_t s0 = j0 < kpN ? bf16_sign_bits(v[2 * q]) : 0u;
          const uint32_t s1 = j0 + 1 < kpN ? bf16_sign_bits(v[2 * q + 1]) : 0u;
          pk[q] = s0 | (s1 << 16);
        }
        if (rvalid) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * cc + i < k) c2 = fmaf(v[i], v[i], c2);
          if (Sout) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (32 * cc + i < k)
                Sout[wt ? colbase + (int64_t)(32 * cc + i) * mi.m : rowoff + 32 * cc + i] =
                    (int8_t)sign_of(v[i]);
          }
        }
        tmem_st16(tc_row + 16 * cc, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->s_full);
      // drain U piece by piece; the parameters of the next 32-column piece
      // load while this one is applied
      bool ok = true;
      float wn[32];
      auto loadw = [&](int l0, float (&dst)[32]) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          float t4[4];
          if (rvalid && l0 + 4 * e < k) {
            if (wt) load4_t(W + colbase + (int64_t)(l0 + 4 * e) * mi.m, mi.m, t4);
            else load4(W + rowoff + l0 + 4 * e, t4);
          } else {
            t4[0] = t4[1] = t4[2] = t4[3] = 0.f;
          }
          dst[4 * e] = t4[0]; dst[4 * e + 1] = t4[1]; dst[4 * e + 2] = t4[2]; dst[4 * e + 3] = t4[3];
        }
      };
      loadw(0, wn);
      for (int c0 = 0; c0 < kpN; c0 += kUCols) {
        const int nn = min(kUCols, kpN - c0);
        const int b = ucount & 1;
        if (!warp_wait(&sh->u_full[b], uphase[b])) { ok = false; break; }
        uphase[b] ^= 1;
        tc_fence_after();
        for (int q = 0; q * 32 < nn; ++q) {
          const int l0 = c0 + 32 * q;
          float wv[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) wv[i] = wn[i];
          if (l0 + 32 < kpN) loadw(l0 + 32, wn);
          const bool any = rvalid && l0 < k;
          float u[32];
          tmem_ld32(trow + 256 + kUCols * b + 32 * q, u);
          tmem_wait_ld(u);
          if (any) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              if (l0 + 4 * e < k) {
                float o[4];
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                  const float uu = u[4 * e + z];
                  u2 = fmaf(uu, uu, u2);
                  o[z] = fmaf(-a.lr_s, uu, wv[4 * e + z]);
                }
                if (wt) store4_t(W + colbase + (int64_t)(l0 + 4 * e) * mi.m, mi.m, o);
                else store4(W + rowoff + l0 + 4 * e, o);
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->u_empty[b]);
        ++ucount;
      }
      if (!ok) { raise(sh, t.err, 10); break; }
      c2 = warp_sum(c2);
      u2 = warp_sum(u2);
      if (lane == 0) {
        float* st = a.stats + 4 * (int64_t)(mi.blk0 + tl.blk);
        atomicAdd(st + 0, u2);
        atomicAdd(st + 1, c2);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- packing
// Q (row-major, column j = eigenvector j) -> the two operand images, with
// npieces = 2 (fp32 basis: hi and lo pieces) or 1 (bf16 basis, "Dobb",
// Table 18: Q rounded once to bf16, exact in both TF32 and bf16).
//   project, K = l, N = j: per 8-wide K step s and piece (TF32 hi[, lo]),
//     kpN rows of 32 bytes (row n holds Q[8s .. 8s+7][n]), 32-byte swizzle;
//   reconstruct, K = j, N = l: per 128-wide output chunk, per 16-wide K step
//     and piece (bf16 hi[, lo, lo2]), nn rows of 32 bytes (row n holds
//     Q[c0 + n][16s .. 16s+15]), 32-byte swizzle.
__global__ void __launch_bounds__(256)
pack_bases_kernel(const float* Q, unsigned char* qpack, const MatInfo* info, const Tile* items,
                  int num_items, int npieces, int rpieces) {
  for (int w = blockIdx.x; w < num_items; w += gridDim.x) {
    const Tile tl = items[w];
    const MatInfo mi = info[tl.mat];
    if (!mi.tc) continue;
    const int k = mi.k, kpN = (k + 15) & ~15, nsub = (k + 7) / 8;
    const float* Qb = Q + mi.a_off + (int64_t)tl.blk * k * k;
    unsigned char* img = qpack + mi.qp_off + (int64_t)tl.blk * mi.qblk_bytes;
    // project image
    const int np = nsub * kpN * 8;
    for (int e = threadIdx.x; e < np; e += blockDim.x) {
      const int kk = e & 7, n = (e >> 3) % kpN, s = (e >> 3) / kpN;
      const int l = 8 * s + kk;
      float q = (l < k && n < k) ? Qb[(int64_t)l * k + n] : 0.f;
      if (npieces == 1) q = __bfloat162float(__float2bfloat16_rn(q));
      const float h = ptx::tf32_rna(q);
      const uint32_t off = ptx::swz_offset((uint32_t)(n * 32 + kk * 4), 1);
      unsigned char* sub = img + (int64_t)s * npieces * kpN * 32;
      *reinterpret_cast<float*>(sub + off) = h;
      if (npieces == 2) *reinterpret_cast<float*>(sub + kpN * 32 + off) = ptx::tf32_rna(q - h);
    }
    // reconstruct image
    unsigned char* rimg = img + (int64_t)nsub * npieces * kpN * 32;
    const int nr = kpN * kpN;  // (l, j) over the padded square
    for (int e = threadIdx.x; e < nr; e += blockDim.x) {
      const int l = e / kpN, j = e % kpN;
      const int c0 = (l / kUCols) * kUCols, nn = min(kUCols, kpN - c0), nrow = l - c0;
      const int s = j / 16, jj = j % 16;
      const float q = (l < k && j < k) ? Qb[(int64_t)l * k + j] : 0.f;
      const __nv_bfloat16 h = __float2bfloat16_rn(q);
      const int64_t cbase = (int64_t)c0 * (kpN / 16) * rpieces * 32;  // chunks before: 128 rows each
      unsigned char* sub = rimg + cbase + (int64_t)s * rpieces * nn * 32;
      const uint32_t off = ptx::swz_offset((uint32_t)(nrow * 32 + jj * 2), 1);
      *reinterpret_cast<__nv_bfloat16*>(sub + off) = h;
      if (rpieces == 3) {
        // q - h and q - h - l are exact in fp32 (bf16 pieces of an fp32 value)
        const float r1 = q - __bfloat162float(h);
        const __nv_bfloat16 l = __float2bfloat16_rn(r1);
        *reinterpret_cast<__nv_bfloat16*>(sub + nn * 32 + off) = l;
        *reinterpret_cast<__nv_bfloat16*>(sub + 2 * nn * 32 + off) =
            __float2bfloat16_rn(r1 - __bfloat162float(l));
      }
    }
  }
}

}  // namespace

size_t step_tc_bstage(int max_k) {
  const int kpN = (max_k + 15) & ~15;
  return (size_t)std::max(2 * kpN * 32, 3 * kUCols * 32);
}

size_t step_tc_smem(int max_k, int nastage, int nbstage) {
  return 1024 + (size_t)nastage * 2 * kAChunkBytes + nbstage * step_tc_bstage(max_k) + sizeof(TcSmem) + 64;
}

// Momentum stages of a launch.
int step_tc_astages(int max_k) { (void)max_k; return 2; }

// Basis stages a launch uses at most.  Shared memory left unused stays L1
// cache, which the per-row gradient and parameter accesses of the converter
// and epilogue warps rely on.
static int step_tc_bstage_cap(int max_k) { return max_k <= 128 ? 8 : 6; }

int step_tc_bstages(int max_k, int nastage, size_t smem_limit) {
  const size_t fixed = step_tc_smem(max_k, nastage, 0);
  const size_t per = step_tc_bstage(max_k);
  const int nb = smem_limit > fixed ? (int)((smem_limit - fixed) / per) : 0;
  return std::min(std::min(kMaxBStages, step_tc_bstage_cap(max_k)), nb);
}

int64_t tc_block_image_bytes(int k) {
  const int kpN = (k + 15) & ~15, nsub = (k + 7) / 8;
  // project: up to two TF32 pieces; reconstruct: up to three bf16 pieces
  int64_t bytes = (int64_t)nsub * 2 * kpN * 32 + (int64_t)kpN * kpN * 6;
  return (bytes + 1023) / 1024 * 1024;
}

bool tc_eligible(int64_t m, int64_t n, int k) {
  (void)m;
  return k % 4 == 0 && n % 4 == 0 && k <= kMaxTcK && k >= 4;
}

cudaError_t configure_step_tc(size_t smem_limit) {
  const int lim = (int)smem_limit;
  const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(step_tc_kernel<float, false>, attr, lim);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(step_tc_kernel<float, true>, attr, lim);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(step_tc_kernel<__nv_bfloat16, false>, attr, lim);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(step_tc_kernel<__nv_bfloat16, true>, attr, lim);
  return e;
}

cudaError_t launch_step_tc(const StepArgs& a, const TcArgs& t, int param_dtype, bool may_t,
                           int grid, size_t smem, cudaStream_t s) {
  if (a.num_tiles <= 0) return cudaSuccess;
  if (param_dtype == kBF16) {
    if (may_t) step_tc_kernel<__nv_bfloat16, true><<<grid, kThreads, smem, s>>>(a, t);
    else step_tc_kernel<__nv_bfloat16, false><<<grid, kThreads, smem, s>>>(a, t);
  } else {
    if (may_t) step_tc_kernel<float, true><<<grid, kThreads, smem, s>>>(a, t);
    else step_tc_kernel<float, false><<<grid, kThreads, smem, s>>>(a, t);
  }
  return cudaGetLastError();
}

cudaError_t launch_pack_bases(const float* Q, unsigned char* qpack, const MatInfo* info,
                              const Tile* items, int num_items, int npieces, int grid, cudaStream_t s) {
  if (num_items <= 0) return cudaSuccess;
  pack_bases_kernel<<<grid, 256, 0, s>>>(Q, qpack, info, items, num_items, npieces,
                                         npieces == 2 ? 3 : 1);
  return cudaGetLastError();
}

}  // namespace dobb
