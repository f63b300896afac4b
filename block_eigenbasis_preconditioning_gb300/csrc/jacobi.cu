// Batched symmetric eigensolver for the k x k block moments
// ("Dobb", Abstract: a complete basis within each block; Table 15: exact
// eigendecomposition refresh).
//
// Method: cyclic two-sided Jacobi (Golub & Van Loan's 2x2 symmetric Schur
// rotation, applied as B <- J^T B J, V <- V J) inside a Rayleigh-Ritz
// restart loop:
//
//   V = current basis (the identity before the first refresh)
//   B = V^T (A V)
//   repeat
//     one sweep on B, rotating V along; off = ||off(B)||_F / ||B||_F after it
//     stop when B was freshly formed before this sweep and off <= tol (2e-6
//       by default), or the sweep rotated nothing, or off <= 1e-5 has
//       stopped shrinking (the fp32 floor): after a sweep on a fresh B, off
//       is the residual that the result will have
//     while off > 3e-4 keep sweeping the same B (far from diagonal the
//       rotations are large and a restart buys nothing); otherwise restart:
//       V <- V + V (I - V^T V) / 2 (Newton-Schulz), B = V^T (A V); a B
//       that has been swept twice is never trusted to end the iteration,
//       since its entries carry the rounding of every rotation so far
//   Lambda = diag(B), V <- V + V (I - V^T V) / 2, columns sorted by
//   descending eigenvalue, written as row-major Q (column j = eigenvector j).
//
// The restart is what keeps fp32 results at the level of a Householder
// solver: every sweep adds rounding to B and to the column norms of V (each
// column takes ~k rotations per sweep), and recomputing B from A and a
// re-orthogonalised V removes that before the final, small sweep.  A warm
// start from the previous basis usually needs two or three restarts.
//
// A sweep is blocked so that all O(k^3) work is small dense products.  The
// k columns form nG = 2 ceil(k / 64) groups of g <= 32; the groups play a
// round-robin tournament (nG - 1 rounds of nG / 2 tables).  In a round each
// table (two groups, index set P_t of 2g columns) loads its diagonal tile
// S_t = B[P_t, P_t] into shared memory and rotates every pair of its columns
// once (in the first round also the pairs inside each group), accumulating
// R_t.  The round then updates the rest of B tile pair by tile pair,
// B[P_s, P_t] <- R_s^T B[P_s, P_t] R_t, and V panel by panel,
// V[:, P_t] <- V[:, P_t] R_t.  Every column pair is rotated once per sweep.
// A pair is rotated when |b_pq| exceeds 1e-3 eps ||A||_F.
//
// One CTA of 256 threads per block; B, V and a third k x k work matrix live
// in a global scratch area of the state buffer (L2-resident), staged through
// shared memory by the products.
#include <algorithm>

#include "common.cuh"

namespace dobb {
namespace {

constexpr int kThreads = 256;

#include "fp32_tiles.cuh"
#include "jacobi_common.cuh"
static_assert(kThreads == kTileThreads, "the tile products assume 256 threads");
constexpr int kApplyFloats = 4 * kT * kLd;      // R_s, R_t, X, Y^T of the tile updates
constexpr int kMaxTables = kThreads / 32;       // tables solved together (a team of warps each)
static_assert(kGemmFloats <= kApplyFloats, "product stages live in the tile-update area");

// eigenvalues and permutation of the sort, rounded to 16 bytes
__host__ __device__ __forceinline__ int sort_floats(int k) { return (2 * pow2_ceil(k) + 3) & ~3; }
__host__ __device__ __forceinline__ int fixed_floats(int k) { return sort_floats(k); }

// Tables solved together for a given shared-memory size (floats); 0 when it
// does not fit.
__host__ __device__ __forceinline__ int tables_per_chunk(int k, int smem_floats) {
  const Geo G = geo_for(k);
  const int per_table = 2 * G.n2 * G.n2;
  const int avail = smem_floats - fixed_floats(k);
  if (G.nT == 1) return avail >= kApplyFloats + per_table ? 1 : 0;
  if (avail < kApplyFloats) return 0;
  const int tc = avail / per_table;
  return tc < G.nT ? (tc < kMaxTables ? tc : kMaxTables) : (G.nT < kMaxTables ? G.nT : kMaxTables);
}

// T = A V, B = V^T T (A symmetric; V, T column-major; B symmetric)
__device__ void rayleigh_ritz(const float* A, const float* V, float* T, float* B, int k, float* gs) {
  block_gemm<false>(A, V, T, nullptr, 1.f, false, false, k, gs);
  block_gemm<true>(V, T, B, nullptr, 1.f, false, true, k, gs);
}

// Vout = V + V (I - V^T V) / 2, with E = I - V^T V in Ebuf
__device__ void newton_schulz(const float* V, float* Vout, float* Ebuf, int k, float* gs) {
  block_gemm<true>(V, V, Ebuf, nullptr, -1.f, true, true, k, gs);
  block_gemm<false>(V, Ebuf, Vout, V, 0.5f, false, false, k, gs);
}

// ||off(B)||_F / ||B||_F, the off-diagonal part summed directly (a
// difference of the two squares would cancel).
__device__ float off_rel(const float* B, int k, float* red) {
  float tot = 0.f, off = 0.f;
  for (int e = threadIdx.x; e < k * k; e += blockDim.x) {
    const float v = B[e];
    tot = fmaf(v, v, tot);
    const int i = e / k;
    if (e - i * k != i) off = fmaf(v, v, off);
  }
  tot = block_sum(tot, red);
  off = block_sum(off, red);
  return tot > 0.f ? sqrtf(off / tot) : 0.f;
}

constexpr int kPre = kT * kT / kThreads;  // elements of a 64 x 64 tile per thread

// One blocked sweep on B (row-major = column-major, symmetric) rotating the
// columns of V (column-major).  Rbuf: nT n2^2 floats of global scratch for the
// tables' rotations (unused when there is a single table).  Returns the
// number of rotations (the same value in every thread).
__device__ int blocked_sweep(float* B, float* V, float* Rbuf, int k, const Geo& G, int tc,
                             float bfloor, float* work, int* s_cnt) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int n2 = G.n2, nn = n2 * n2;
  float* Rs = work;
  float* Rt = work + kT * kLd;
  float* Xt = work + 2 * kT * kLd;
  float* Yt = work + 3 * kT * kLd;
  // tables' S and R (2 nn floats per table): after the tile buffers when a
  // single table keeps R in shared memory, else over them
  float* solve = G.nT == 1 ? work + kApplyFloats : work;
  const int nI = (k + kT - 1) / kT;
  int rots = 0;
  for (int br = 0; br < G.nG - 1; ++br) {
    // ---- diagonal tiles of the round's tables, tc at a time
    for (int t0 = 0; t0 < G.nT; t0 += tc) {
      const int tcn = min(tc, G.nT - t0);
      // rows of the tables' tiles: a warp per row, lanes along it
      for (int row = warp; row < tcn * n2; row += nw) {
        const int tt = row / n2, a = row - tt * n2;
        int gI, gJ;
        rr_pair(br, t0 + tt, G.nG, gI, gJ);
        const int ca = table_col(a, gI, gJ, G.g, k);
        float* Srow = solve + tt * 2 * nn + a * n2;
        for (int b = lane; b < n2; b += 32) {
          const int cb = table_col(b, gI, gJ, G.g, k);
          Srow[b] = (ca < k && cb < k) ? B[ca * k + cb] : 0.f;
          Srow[nn + b] = a == b ? 1.f : 0.f;
        }
      }
      __syncthreads();
      {
        // a team of wpt warps per table (named barriers 1 ... tcn)
        int wpt = nw / tcn;
        wpt = wpt >= 4 ? 4 : (wpt >= 2 ? 2 : 1);
        const int tt = warp / wpt;
        if (tt < tcn)
          rots += solve_table(solve + tt * 2 * nn, solve + tt * 2 * nn + nn, br, t0 + tt, G, k, bfloor,
                              warp - tt * wpt, wpt, 1 + tt);
      }
      __syncthreads();
      for (int row = warp; row < tcn * n2; row += nw) {
        const int tt = row / n2, a = row - tt * n2;
        int gI, gJ;
        rr_pair(br, t0 + tt, G.nG, gI, gJ);
        const int ca = table_col(a, gI, gJ, G.g, k);
        const float* Srow = solve + tt * 2 * nn + a * n2;
        for (int b = lane; b < n2; b += 32) {
          const int cb = table_col(b, gI, gJ, G.g, k);
          if (ca < k && cb < k) B[ca * k + cb] = Srow[b];
          if (G.nT > 1) Rbuf[(t0 + tt) * nn + a * n2 + b] = Srow[nn + b];
        }
      }
      __syncthreads();
    }
    // ---- off-diagonal tile pairs (s < t): B[P_s, P_t] <- R_s^T B[P_s, P_t] R_t
    // and its transpose; the next pair's tile and R_t are fetched into
    // registers while the current pair is multiplied
    const int npair = G.nT * (G.nT - 1) / 2;
    if (npair > 0) {
      float preX[kPre], preR[kPre];
      auto fetch_pair = [&](int s, int t) {
        int sI, sJ, tI, tJ;
        rr_pair(br, s, G.nG, sI, sJ);
        rr_pair(br, t, G.nG, tI, tJ);
#pragma unroll
        for (int r = 0; r < kPre; ++r) {
          const int e = tid + r * kThreads;
          const int a = e / kT, b = e - a * kT;
          const int ca = a < n2 ? table_col(a, sI, sJ, G.g, k) : k;
          const int cb = b < n2 ? table_col(b, tI, tJ, G.g, k) : k;
          preX[r] = (ca < k && cb < k) ? B[ca * k + cb] : 0.f;
          preR[r] = (a < n2 && b < n2) ? Rbuf[t * nn + a * n2 + b] : 0.f;
        }
      };
      int s = 0, t = 1, cur_s = -1;
      fetch_pair(0, 1);
      for (int idx = 0; idx < npair; ++idx) {
        if (s != cur_s) {
          load_rot(Rs, Rbuf + s * nn, n2);
          cur_s = s;
        }
#pragma unroll
        for (int r = 0; r < kPre; ++r) {
          const int e = tid + r * kThreads;
          const int a = e / kT, b = e - a * kT;
          Xt[a * kLd + b] = preX[r];
          Rt[a * kLd + b] = preR[r];
        }
        __syncthreads();
        int sn = s, tn = t + 1;
        if (tn == G.nT) {
          ++sn;
          tn = sn + 1;
        }
        if (idx + 1 < npair) fetch_pair(sn, tn);
        float acc[4][4];
        zero_acc(acc);
        micro_tn(Rs, Xt, kLd, n2, acc);  // Y = R_s^T X
        store_acc_t(Yt, kLd, acc);       // Y^T
        __syncthreads();
        zero_acc(acc);
        micro_tn(Yt, Rt, kLd, n2, acc);  // Z = Y R_t
        __syncthreads();
        store_acc(Xt, kLd, acc);         // Z
        store_acc_t(Yt, kLd, acc);       // Z^T
        __syncthreads();
        int sI, sJ, tI, tJ;
        rr_pair(br, s, G.nG, sI, sJ);
        rr_pair(br, t, G.nG, tI, tJ);
        // Z to rows P_s and Z^T to rows P_t, a warp per row, lanes along it
        for (int a = warp; a < n2; a += nw) {
          const int ca = table_col(a, sI, sJ, G.g, k), ct = table_col(a, tI, tJ, G.g, k);
          for (int b = lane; b < n2; b += 32) {
            const int cb = table_col(b, tI, tJ, G.g, k), cs = table_col(b, sI, sJ, G.g, k);
            if (ca < k && cb < k) B[ca * k + cb] = Xt[a * kLd + b];
            if (ct < k && cs < k) B[ct * k + cs] = Yt[a * kLd + b];
          }
        }
        __syncthreads();
        s = sn;
        t = tn;
      }
    }
    // ---- panels of V: V[i0:i0+64, P_t] <- V[i0:i0+64, P_t] R_t, the next
    // panel fetched into registers while the current one is multiplied
    {
      float pre[kPre];
      auto fetch_panel = [&](int task) {
        const int t = task / nI, i0 = (task - t * nI) * kT;
        int tI, tJ;
        rr_pair(br, t, G.nG, tI, tJ);
#pragma unroll
        for (int r = 0; r < kPre; ++r) {
          const int e = tid + r * kThreads;
          const int a = e / kT, i = e - a * kT;
          const int ca = a < n2 ? table_col(a, tI, tJ, G.g, k) : k;
          pre[r] = (ca < k && i0 + i < k) ? V[ca * k + i0 + i] : 0.f;
        }
      };
      const int ntask = G.nT * nI;
      int cur_t = -1;
      fetch_panel(0);
      for (int task = 0; task < ntask; ++task) {
        const int t = task / nI, i0 = (task - t * nI) * kT;
        if (t != cur_t) {
          load_rot(Rt, G.nT > 1 ? Rbuf + t * nn : solve + nn, n2);
          cur_t = t;
        }
#pragma unroll
        for (int r = 0; r < kPre; ++r) {
          const int e = tid + r * kThreads;
          const int a = e / kT, i = e - a * kT;
          Xt[a * kLd + i] = pre[r];
        }
        __syncthreads();
        if (task + 1 < ntask) fetch_panel(task + 1);
        float acc[4][4];
        zero_acc(acc);
        micro_tn(Xt, Rt, kLd, n2, acc);  // rows i of V times R_t
        store_acc_t(Yt, kLd, acc);
        __syncthreads();
        int tI, tJ;
        rr_pair(br, t, G.nG, tI, tJ);
        for (int b = warp; b < n2; b += nw) {
          const int cb = table_col(b, tI, tJ, G.g, k);
          if (cb >= k) continue;
          for (int i = lane; i < kT; i += 32)
            if (i0 + i < k) V[cb * k + i0 + i] = Yt[b * kLd + i];
        }
        __syncthreads();
      }
    }
  }
  if (tid == 0) *s_cnt = 0;
  __syncthreads();
  if (rots) atomicAdd(s_cnt, rots);
  __syncthreads();
  const int total = *s_cnt;
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kThreads, 2)
jacobi_kernel(const __grid_constant__ EigArgs a, int smem_floats) {
  extern __shared__ __align__(16) float sm[];
  __shared__ float red[32];
  __shared__ int s_cnt;
  const int tid = threadIdx.x;
  for (int w = blockIdx.x; w < a.num_tiles; w += gridDim.x) {
    const Tile t = a.tiles[w];
    const MatInfo mi = a.info[t.mat];
    const int k = mi.k;
    const int kp2 = pow2_ceil(k);
    const int64_t kk2 = (int64_t)k * k;
    const int64_t boff = mi.a_off + (int64_t)t.blk * kk2;
    const float* Ab = a.A + boff;
    float* Qb = a.Q + boff;
    uint32_t* flag = a.flags + mi.blk0 + t.blk;
    const Geo G = geo_for(k);
    const int tc = tables_per_chunk(k, smem_floats);
    if (tc < 1) {  // launch configured with too little shared memory for this k
      if (tid == 0) atomicOr(flag, (uint32_t)DOBB_FLAG_NOT_CONVERGED);
      continue;
    }
    float* lamv = sm;
    int* perm = reinterpret_cast<int*>(sm + kp2);
    float* work = sm + sort_floats(k);
    float* Bm = a.scratch + 3 * boff;
    float* V = Bm + kk2;
    float* T = V + kk2;

    // V = current basis (column j of V = column j of the row-major Q); the
    // finiteness of A and ||A||_F^2 on the way
    float ss = 0.f;
    int bad = 0;
    for (int e = tid; e < k * k; e += blockDim.x) {
      const float v = Ab[e];
      bad |= !isfinite(v);
      ss = fmaf(v, v, ss);
      const int c = e / k, i = e - c * k;
      V[e] = Qb[i * k + c];
    }
    if (__syncthreads_or(bad)) {
      if (tid == 0) atomicOr(flag, (uint32_t)DOBB_FLAG_NONFINITE_A);
      continue;  // keep the previous basis
    }
    const float fro2 = block_sum(ss, red);
    const float bfloor = 1e-3f * kEps * sqrtf(fro2);
    const float stop = a.tol > 0.f ? a.tol : kStopOff;
    __syncthreads();
    rayleigh_ritz(Ab, V, T, Bm, k, work);
    // fresh: B was formed from A and an orthonormal V and swept once; only
    // such a sweep may be the last one.  After it, off(B) measures what the
    // sweep left undone, i.e. the residual of the result.
    int sweeps = 0, last_rot = 0;
    bool conv = false, fresh = true;
    float prev = INFINITY;  // off(B) after the previous sweep on a fresh B
    for (;;) {
      last_rot = blocked_sweep(Bm, V, T, k, G, tc, bfloor, work, &s_cnt);
      ++sweeps;
      const float off = off_rel(Bm, k, red);
      if (fresh) {
        // converged, or at the fp32 floor: small and no longer shrinking
        if (off <= stop || last_rot == 0 || (off <= kStallOff && off > 0.7f * prev)) {
          conv = true;
          break;
        }
        prev = off;
      }
      if (sweeps >= a.max_sweeps) break;
      fresh = false;
      if (off > kColdOff) continue;  // far from diagonal: sweep the same B again
      newton_schulz(V, T, Bm, k, work);
      float* tmp = V;
      V = T;
      T = tmp;
      rayleigh_ritz(Ab, V, T, Bm, k, work);
      fresh = true;
    }
    for (int p = tid; p < kp2; p += blockDim.x) {
      lamv[p] = p < k ? Bm[p * k + p] : -INFINITY;
      perm[p] = p;
    }
    __syncthreads();
    newton_schulz(V, T, Bm, k, work);
    V = T;
    // sort descending by eigenvalue
    for (int size = 2; size <= kp2; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < kp2; i += blockDim.x) {
          const int j = i ^ stride;
          if (j > i) {
            const bool desc = (i & size) == 0;
            const float li = lamv[i], lj = lamv[j];
            if (desc ? (li < lj) : (li > lj)) {
              lamv[i] = lj;
              lamv[j] = li;
              const int pt = perm[i];
              perm[i] = perm[j];
              perm[j] = pt;
            }
          }
        }
        __syncthreads();
      }
    }
    for (int e = tid; e < k * k; e += blockDim.x) {
      const int i = e / k, j = e - i * k;
      int p = perm[j];
      if (p < 0 || p >= k) p = j;  // only reachable with a NaN eigenvalue
      Qb[e] = V[p * k + i];
    }
    for (int j = tid; j < k; j += blockDim.x) a.lam[mi.lam_off + (int64_t)t.blk * k + j] = lamv[j];
    if (tid == 0) {
      float* st = a.stats + 4 * (int64_t)(mi.blk0 + t.blk);
      st[2] = (float)sweeps;
      st[3] = (float)last_rot;
      if (!conv) atomicOr(flag, (uint32_t)DOBB_FLAG_NOT_CONVERGED);
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_jacobi(const EigArgs& a, int grid, size_t smem_bytes, cudaStream_t s) {
  if (a.num_tiles <= 0) return cudaSuccess;
  jacobi_kernel<<<grid, kThreads, smem_bytes, s>>>(a, (int)(smem_bytes / 4));
  return cudaGetLastError();
}

size_t jacobi_smem_for(int k, size_t budget) {
  const Geo G = geo_for(k);
  const size_t per_table = 2 * (size_t)G.n2 * G.n2;
  const size_t fixed = fixed_floats(k);
  size_t work;
  if (G.nT == 1) {
    work = kApplyFloats + per_table;
  } else {
    const int tc = tables_per_chunk(k, (int)std::min<size_t>(budget / 4, (size_t)1 << 28));
    if (tc < 1) return 0;
    work = std::max<size_t>(kApplyFloats, (size_t)tc * per_table);
  }
  const size_t bytes = 4 * (fixed + work);
  return bytes <= budget ? bytes : 0;
}

int jacobi_ctas_per_sm() { return 2048 / kThreads; }

cudaError_t configure_jacobi(size_t smem_limit) {
  return cudaFuncSetAttribute(jacobi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem_limit);
}

}  // namespace dobb
