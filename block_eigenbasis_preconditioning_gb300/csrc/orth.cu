// Orthogonal-iteration refresh of the block bases ("Dobb", Table 15: one
// orthogonal-iteration step per refresh is the principal setting; Table 16:
// the Cholesky QR routine).
//
// Per block, `steps` times, starting from the current basis V:
//   T = A V;  V = T R^{-1} with R^T R = T^T T  (the QR factor of T whose R has
//   a positive diagonal)
// then Lambda_j = v_j^T A v_j (Rayleigh quotients; the update uses only V).
//
// In fp32 the Cholesky QR of T loses orthogonality like eps kappa(T)^2, so it
// is applied twice (CholeskyQR2: the second pass factors the nearly
// orthonormal result again and leaves ||V^T V - I|| at the unit-roundoff
// level for kappa(T) up to ~1e3).  While the Gram matrix is not numerically
// positive definite, a pass with a shift s I is taken first (shifted
// CholeskyQR, Fukaya et al., SIAM J. Sci. Comput. 2020); s = 10 k eps
// tr(X^T X), ten times larger while the shifted factorisation still fails
// (their bound 11 (k^2 + k (k + 1)) eps ||X||^2 would lower kappa by only
// ~0.9 per pass at k = 400 in fp32).  Each shifted pass lowers kappa by about
// sqrt(s / ||X||^2); the R factors of all passes multiply to the R of T.
//
// Blocked, one CTA of 256 threads per block; V, T and the Gram matrix G live
// in the eigensolver's scratch area (3 k^2 floats per block).
//   Cholesky (lower, in place on G, 32-wide panels, right-looking): the
//   diagonal tile is factored in shared memory, the panel below is solved one
//   row per thread, the trailing lower triangle is updated with the 64 x 64
//   micro-kernel.
//   V = X L^{-T} (row-wise forward substitution, 32-wide column panels): the
//   panel is first reduced by the finished panels with the micro-kernel, then
//   solved one row per thread against the diagonal tile in shared memory.
#include <algorithm>

#include "common.cuh"

namespace dobb {
namespace {

constexpr int kThreads = 256;

#include "fp32_tiles.cuh"
static_assert(kThreads == kTileThreads, "the tile products assume 256 threads");

#include "cholqr.cuh"

constexpr float kEps = 5.9604645e-8f;  // 2^-24
constexpr int kMaxShifted = 8;         // shifted passes before a block gives up
// shared memory: diagonal tile (64 x kLd) + two staging tiles / product stages
constexpr int kOrthSmemFloats = kT * kLd + std::max(2 * kT * kLd, kGemmFloats);

// Y = X L^{-T} (X, Y k x k column-major; Y may alias X): row r of Y solves
// L y_r^T = x_r^T.  L lower in G (column-major).
__device__ void trsm_right_lt(const float* X, float* Y, const float* G, int k, float* sm) {
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float* D = sm;
  float* Ps = sm + kT * kLd;   // Y[i0 .. i0+64, q0 .. q0+64]^T staged as [q][i]
  float* Ls = Ps + kT * kLd;   // L[j0 .. j0+64, q0 .. q0+64]^T staged as [q][j]
  for (int j0 = 0; j0 < k; j0 += kPW) {
    const int jb = min(kPW, k - j0);
    // reduce the panel by the finished panels: Y[:, j0:j0+jb] = X[:, ...] - Y[:, :j0] L[j0:, :j0]^T
    if (j0 > 0) {
      for (int i0 = 0; i0 < k; i0 += kT) {
        float acc[4][4];
        zero_acc(acc);
        for (int q0 = 0; q0 < j0; q0 += kT) {
          const int nq = min(kT, j0 - q0);
          __syncthreads();
          for (int e = tid; e < kT * kT; e += blockDim.x) {
            const int q = e / kT, i = e - q * kT;
            Ps[q * kLd + i] = (q < nq && i0 + i < k) ? Y[(int64_t)(q0 + q) * k + i0 + i] : 0.f;
            Ls[q * kLd + i] = (q < nq && i < jb) ? G[(int64_t)(q0 + q) * k + j0 + i] : 0.f;
          }
          __syncthreads();
          micro_tn(Ps, Ls, kLd, nq, acc);
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const int r = i0 + 4 * ty + a, c = 4 * tx + b;
            if (r < k && c < jb) Y[(int64_t)(j0 + c) * k + r] = X[(int64_t)(j0 + c) * k + r] - acc[a][b];
          }
      }
    } else if (X != Y) {
      for (int e = tid; e < k * jb; e += blockDim.x) {
        const int c = e / k, r = e - c * k;
        Y[(int64_t)c * k + r] = X[(int64_t)c * k + r];
      }
    }
    __syncthreads();
    load_diag(D, G, k, j0, jb);
    __syncthreads();
    // in-panel forward substitution, one row per thread
    for (int r = tid; r < k; r += blockDim.x) {
      float w[kPW];
#pragma unroll
      for (int c = 0; c < kPW; ++c) w[c] = c < jb ? Y[(int64_t)(j0 + c) * k + r] : 0.f;
      row_forward_solve(w, D);
#pragma unroll
      for (int c = 0; c < kPW; ++c)
        if (c < jb) Y[(int64_t)(j0 + c) * k + r] = w[c];
    }
    __syncthreads();
  }
}

// One Cholesky QR pass: G = X^T X (+ shift I), L = chol(G), Y = X L^{-T}.
__device__ bool cholqr_pass(const float* X, float* Y, float* G, int k, float shift, float* sm,
                            int* s_ok) {
  block_gemm<true>(X, X, G, nullptr, 1.f, false, true, k, sm + kT * kLd);
  if (shift > 0.f) {
    for (int i = threadIdx.x; i < k; i += blockDim.x) G[(int64_t)i * k + i] += shift;
    __syncthreads();
  }
  if (!chol_lower(G, k, sm, s_ok)) return false;
  trsm_right_lt(X, Y, G, k, sm);
  return true;
}

__global__ void __launch_bounds__(kThreads, 1)
orth_kernel(const __grid_constant__ EigArgs a, int steps) {
  extern __shared__ __align__(16) float sm[];
  __shared__ float red[32];
  __shared__ int s_ok;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  for (int w = blockIdx.x; w < a.num_tiles; w += gridDim.x) {
    // after a grid pass: only the blocks whose Gram matrix was not
    // numerically positive definite there (their basis is still the old one)
    if (a.ctl && (a.ctl[w].skip || a.ctl[w].conv)) continue;
    const Tile t = a.tiles[w];
    const MatInfo mi = a.info[t.mat];
    const int k = mi.k;
    const int64_t kk2 = (int64_t)k * k;
    const int64_t boff = mi.a_off + (int64_t)t.blk * kk2;
    const float* Ab = a.A + boff;
    float* Qb = a.Q + boff;
    uint32_t* flag = a.flags + mi.blk0 + t.blk;
    float* V = a.scratch + 3 * boff;
    float* T = V + kk2;
    float* G = T + kk2;
    int bad = 0;
    for (int e = tid; e < k * k; e += blockDim.x) {
      bad |= !isfinite(Ab[e]);
      const int c = e / k, i = e - c * k;
      V[e] = Qb[(int64_t)i * k + c];
    }
    if (__syncthreads_or(bad)) {
      if (tid == 0) atomicOr(flag, (uint32_t)DOBB_FLAG_NONFINITE_A);
      continue;  // keep the previous basis
    }
    bool ok = true;
    int shifted = 0;
    for (int s = 0; s < steps && ok; ++s) {
      block_gemm<false>(Ab, V, T, nullptr, 1.f, false, false, k, sm + kT * kLd);  // T = A V
      // plain Cholesky QR; while the Gram matrix is not numerically positive
      // definite, a shifted pass first (each lowers kappa by about
      // sqrt(shift / ||X||^2)), then the plain pass again
      const float* X = T;
      ok = false;
      for (int attempt = 0; attempt <= kMaxShifted; ++attempt) {
        if (cholqr_pass(X, V, G, k, 0.f, sm, &s_ok)) {
          ok = true;
          break;
        }
        if (attempt == kMaxShifted) break;
        block_gemm<true>(X, X, G, nullptr, 1.f, false, true, k, sm + kT * kLd);
        float tr = 0.f;
        for (int i = tid; i < k; i += blockDim.x) tr += G[(int64_t)i * k + i];
        tr = block_sum(tr, red);
        // shift: 10 k eps tr(X^T X), ten times larger while it is not enough
        float shift = 10.f * (float)k * kEps * tr;
        bool done = false;
        for (int grow = 0; grow < 4 && !done; ++grow, shift *= 10.f)
          done = cholqr_pass(X, V, G, k, shift, sm, &s_ok);
        if (!done) break;
        X = V;
        ++shifted;
      }
      ok = ok && cholqr_pass(V, V, G, k, 0.f, sm, &s_ok);  // CholeskyQR2
    }
    if (!ok) {
      if (tid == 0) atomicOr(flag, (uint32_t)DOBB_FLAG_NOT_CONVERGED);
      __syncthreads();
      continue;  // keep the previous basis
    }
    // Rayleigh quotients: T = A V, lambda_j = v_j . t_j (a warp per column)
    block_gemm<false>(Ab, V, T, nullptr, 1.f, false, false, k, sm + kT * kLd);
    for (int j = warp; j < k; j += nw) {
      float d = 0.f;
      for (int i = lane; i < k; i += 32) d = fmaf(V[(int64_t)j * k + i], T[(int64_t)j * k + i], d);
      d = warp_sum(d);
      if (lane == 0) a.lam[mi.lam_off + (int64_t)t.blk * k + j] = d;
    }
    for (int e = tid; e < k * k; e += blockDim.x) {
      const int i = e / k, j = e - i * k;
      Qb[e] = V[(int64_t)j * k + i];
    }
    if (tid == 0) {
      float* st = a.stats + 4 * (int64_t)(mi.blk0 + t.blk);
      st[2] = (float)steps;
      st[3] = (float)shifted;  // shifted Cholesky QR passes taken
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_orth(const EigArgs& a, int steps, int grid, cudaStream_t s) {
  if (a.num_tiles <= 0) return cudaSuccess;
  orth_kernel<<<grid, kThreads, orth_smem_bytes(), s>>>(a, steps);
  return cudaGetLastError();
}

size_t orth_smem_bytes() { return (size_t)kOrthSmemFloats * sizeof(float); }

cudaError_t configure_orth() {
  return cudaFuncSetAttribute(orth_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)orth_smem_bytes());
}

}  // namespace dobb
