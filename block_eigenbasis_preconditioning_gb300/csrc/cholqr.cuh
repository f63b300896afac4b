// Cholesky pieces of the Cholesky QR refresh ("Dobb", Table 16: the
// Cholesky QR routine), shared by the one-CTA-per-block orthogonal iteration
// (orth.cu) and its grid form (jacobi_grid.cu).  Included inside an
// anonymous namespace after fp32_tiles.cuh (256 threads per CTA; shared
// memory: three 64 x kLd tiles).  Matrices are k x k, column-major.
#pragma once

constexpr int kPW = 32;  // panel width of the Cholesky and the triangular solve

// In-panel forward substitution for one row held in registers:
// w <- w L^{-T}, L = the kPW x kPW lower diagonal tile D (row stride kLd,
// identity beyond the panel width), i.e. solve L y = w.
__device__ __forceinline__ void row_forward_solve(float (&w)[kPW], const float* D) {
#pragma unroll
  for (int c = 0; c < kPW; ++c) {
    const float y = w[c] / D[c * kLd + c];
    w[c] = y;
#pragma unroll
    for (int q = c + 1; q < kPW; ++q) w[q] = fmaf(-y, D[q * kLd + c], w[q]);
  }
}

// Load the lower triangle of the diagonal tile G[j0 : j0+jb, j0 : j0+jb]
// (column-major lower storage) into D, identity beyond jb.
__device__ void load_diag(float* D, const float* G, int k, int j0, int jb) {
  for (int e = threadIdx.x; e < kPW * kPW; e += blockDim.x) {
    const int r = e / kPW, c = e - r * kPW;
    float v = 0.f;
    if (r < jb && c < jb) {
      if (c <= r) v = G[(int64_t)(j0 + c) * k + j0 + r];
    } else if (r == c) {
      v = 1.f;
    }
    D[r * kLd + c] = v;
  }
}

// Cholesky G = L L^T in place (L lower, column-major: L(i, j) at G[j k + i]).
// Only the lower triangle of G is read.  Returns false (uniformly) when a
// pivot is not positive or not finite.
__device__ bool chol_lower(float* G, int k, float* sm, int* s_ok) {
  const int tid = threadIdx.x;
  float* D = sm;
  float* Pa = sm + kT * kLd;
  float* Pb = Pa + kT * kLd;
  if (tid == 0) *s_ok = 1;
  for (int j0 = 0; j0 < k; j0 += kPW) {
    const int jb = min(kPW, k - j0);
    __syncthreads();
    load_diag(D, G, k, j0, jb);
    __syncthreads();
    // (1) unblocked factor of the diagonal tile by the first warp (lane r
    // holds row r; jb <= 32): the same operations, column by column, as a
    // CTA-wide loop, without its three barriers per column
    if (tid < 32) {
      const int r = tid;
      const bool row = r < jb;
      for (int c = 0; c < jb; ++c) {
        const float d = D[c * kLd + c];          // the same value on every lane
        if (!(d > 0.f) || !isfinite(d)) {
          if (r == 0) *s_ok = 0;
          break;
        }
        const float dc = sqrtf(d);
        const float l = (row && r > c) ? D[r * kLd + c] / dc : 0.f;
        __syncwarp();
        if (r == c) D[c * kLd + c] = dc;
        if (row && r > c) D[r * kLd + c] = l;
        __syncwarp();
        if (row && r > c)
          for (int q = c + 1; q <= r; ++q) D[r * kLd + q] = fmaf(-l, D[q * kLd + c], D[r * kLd + q]);
        __syncwarp();
      }
    }
    __syncthreads();
    if (!*s_ok) return false;
    for (int e = tid; e < jb * jb; e += blockDim.x) {
      const int r = e / jb, c = e - r * jb;
      if (c <= r) G[(int64_t)(j0 + c) * k + j0 + r] = D[r * kLd + c];
    }
    // (2) the panel below: row r solves x L_jj^T = g_r
    for (int r = j0 + jb + tid; r < k; r += blockDim.x) {
      float w[kPW];
#pragma unroll
      for (int c = 0; c < kPW; ++c) w[c] = c < jb ? G[(int64_t)(j0 + c) * k + r] : 0.f;
      row_forward_solve(w, D);
#pragma unroll
      for (int c = 0; c < kPW; ++c)
        if (c < jb) G[(int64_t)(j0 + c) * k + r] = w[c];
    }
    __syncthreads();
    // (3) trailing lower triangle: G[r, q] -= sum_c L[r, j0 + c] L[q, j0 + c]
    const int t0 = j0 + jb;
    const int nt = (k - t0 + kT - 1) / kT;
    for (int tile = 0; tile < nt * nt; ++tile) {
      const int ti = tile % nt, tj = tile / nt;
      if (ti < tj) continue;
      const int i0 = t0 + ti * kT, q0 = t0 + tj * kT;
      for (int e = tid; e < kT * kT; e += blockDim.x) {
        const int c = e / kT, i = e - c * kT;
        Pa[c * kLd + i] = (c < jb && i0 + i < k) ? G[(int64_t)(j0 + c) * k + i0 + i] : 0.f;
        Pb[c * kLd + i] = (c < jb && q0 + i < k) ? G[(int64_t)(j0 + c) * k + q0 + i] : 0.f;
      }
      __syncthreads();
      float acc[4][4];
      zero_acc(acc);
      micro_tn(Pa, Pb, kLd, jb, acc);
      const int tx = tid & 15, ty = tid >> 4;
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int r = i0 + 4 * ty + a, q = q0 + 4 * tx + b;
          if (r < k && q < k && q <= r) G[(int64_t)q * k + r] -= acc[a][b];
        }
      __syncthreads();
    }
  }
  __syncthreads();
  return true;
}

// Rows [i0, i0 + 64) of Y = X L^{-T} (X, Y k x k column-major; Y may alias
// X): row r of Y solves L y_r^T = x_r^T, L lower in G (column-major).  The
// rows of one call depend on no other rows, so a grid of CTAs can split Y by
// 64-row panels.  Column panels of kPW: the panel is first reduced by the
// finished ones with the micro-kernel, then solved row by row against the
// diagonal tile in shared memory.
__device__ void trsm_rows(const float* X, float* Y, const float* G, int k, int i0, float* sm) {
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  float* D = sm;
  float* Ps = sm + kT * kLd;   // Y[i0 .. i0+64, q0 .. q0+64]^T staged as [q][i]
  float* Ls = Ps + kT * kLd;   // L[j0 .. j0+64, q0 .. q0+64]^T staged as [q][j]
  const int i1 = min(k, i0 + kT);
  for (int j0 = 0; j0 < k; j0 += kPW) {
    const int jb = min(kPW, k - j0);
    if (j0 > 0) {
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
    } else if (X != Y) {
      for (int e = tid; e < kT * jb; e += blockDim.x) {
        const int c = e / kT, r = i0 + (e - c * kT);
        if (r < k) Y[(int64_t)c * k + r] = X[(int64_t)c * k + r];
      }
    }
    __syncthreads();
    load_diag(D, G, k, j0, jb);
    __syncthreads();
    for (int r = i0 + tid; r < i1; r += blockDim.x) {
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
