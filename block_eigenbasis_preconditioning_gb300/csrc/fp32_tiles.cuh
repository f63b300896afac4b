// FP32 tile products shared by the eigensolvers (one CTA of 256 threads per
// k x k block): a 64 x 64 register-blocked micro-kernel and a tiled product
// over whole k x k operands.  Included inside an anonymous namespace of the
// kernel file that uses them.
#pragma once

constexpr int kTileThreads = 256;          // CTA size the products are written for
constexpr int kT = 64;                     // tile edge of every product
constexpr int kLd = kT + 4;                // padded row of a staged 64-wide tile
constexpr int kGK = 32;                    // reduction depth of one stage of the k x k product
constexpr int kGemmFloats = 2 * 2 * kGK * kLd;  // two stages of the X and Y tiles

// ---------------------------------------------------------------------------
// 64 x 64 register-blocked product: acc[i][j] += sum_{c < n} P[c][4ty+i] Q[c][4tx+j]
// (rows of P and Q at stride ld, 16-byte aligned); 4 x 4 outputs per thread.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void micro_tn(const float* P, const float* Q, int ld, int n,
                                         float acc[4][4]) {
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const float* pp = P + 4 * ty;
  const float* qq = Q + 4 * tx;
#pragma unroll 4
  for (int c = 0; c < n; ++c) {
    const float4 a = *reinterpret_cast<const float4*>(pp + c * ld);
    const float4 b = *reinterpret_cast<const float4*>(qq + c * ld);
    const float av[4] = {a.x, a.y, a.z, a.w};
    const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
  }
}

__device__ __forceinline__ void zero_acc(float acc[4][4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
}

// out[4ty+i][4tx+j] = acc[i][j] (rows of stride ld)
__device__ __forceinline__ void store_acc(float* out, int ld, const float acc[4][4]) {
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<float4*>(out + (4 * ty + i) * ld + 4 * tx) =
        make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
}

// out[4tx+j][4ty+i] = acc[i][j]
__device__ __forceinline__ void store_acc_t(float* out, int ld, const float acc[4][4]) {
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<float4*>(out + (4 * tx + j) * ld + 4 * ty) =
        make_float4(acc[0][j], acc[1][j], acc[2][j], acc[3][j]);
}

// ---------------------------------------------------------------------------
// Product over the k x k operands of one block, FP32 (one 64 x 64 output tile
// (ti, tj) per call of gemm_tile; block_gemm runs them all):
//   C(i, j) = alpha * sum_l X(i, l) Y(l, j) + D(i, j) + (eye ? delta_ij : 0)
// with Y(l, j) = Y[j k + l], X(i, l) = X[l k + i] (XT = false) or X[i k + l]
// (XT = true); C and D at [j k + i].  sym: the result is symmetric by
// construction, so only tiles on or above the diagonal are computed and each
// value is written to both (i, j) and (j, i) (on diagonal tiles the i <= j
// triangle is kept, so C is exactly symmetric).  64 x 64 output tiles; the
// reduction is staged 32 deep through shared memory, the next stage loaded
// into registers while the current one is multiplied.
// ---------------------------------------------------------------------------
template <bool XT>
__device__ void gemm_tile(const float* X, const float* Y, float* C, const float* D, float alpha,
                          bool eye, bool sym, int k, int ti, int tj, float* gs) {
  float* xs[2] = {gs, gs + 2 * kGK * kLd};
  float* ys[2] = {gs + kGK * kLd, gs + 3 * kGK * kLd};
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int nch = (k + kGK - 1) / kGK;
  constexpr int kPer4 = kGK * kT / (4 * kTileThreads);  // float4 groups of each operand per thread and stage
  const int i0 = ti * kT, j0 = tj * kT;
  float acc[4][4];
  zero_acc(acc);
  // each thread moves groups of four: four rows (X^T, Y) or four
  // consecutive elements (X) of one reduction index, stored as one float4
  float4 rx[kPer4], ry[kPer4];
  auto gload = [&](int l0) {
#pragma unroll
    for (int r = 0; r < kPer4; ++r) {
      const int e = tid + r * kTileThreads;
      float v[4];
      if (XT) {
        const int l = e % kGK, iq = e / kGK;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = 4 * iq + u;
          v[u] = (i0 + i < k && l0 + l < k) ? X[(int64_t)(i0 + i) * k + l0 + l] : 0.f;
        }
      } else {
        const int iq = e % (kT / 4), l = e / (kT / 4);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = 4 * iq + u;
          v[u] = (i0 + i < k && l0 + l < k) ? X[(int64_t)(l0 + l) * k + i0 + i] : 0.f;
        }
      }
      rx[r] = make_float4(v[0], v[1], v[2], v[3]);
      const int l = e % kGK, jq = e / kGK;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int j = 4 * jq + u;
        v[u] = (j0 + j < k && l0 + l < k) ? Y[(int64_t)(j0 + j) * k + l0 + l] : 0.f;
      }
      ry[r] = make_float4(v[0], v[1], v[2], v[3]);
    }
  };
  auto sstore = [&](float* xd, float* yd) {
#pragma unroll
    for (int r = 0; r < kPer4; ++r) {
      const int e = tid + r * kTileThreads;
      const int lx = XT ? e % kGK : e / (kT / 4), iq = XT ? e / kGK : e % (kT / 4);
      *reinterpret_cast<float4*>(xd + lx * kLd + 4 * iq) = rx[r];
      const int l = e % kGK, jq = e / kGK;
      *reinterpret_cast<float4*>(yd + l * kLd + 4 * jq) = ry[r];
    }
  };
  gload(0);
  sstore(xs[0], ys[0]);
  __syncthreads();
  for (int c = 0; c < nch; ++c) {
    if (c + 1 < nch) gload((c + 1) * kGK);
    micro_tn(xs[c & 1], ys[c & 1], kLd, min(kGK, k - c * kGK), acc);
    if (c + 1 < nch) sstore(xs[(c + 1) & 1], ys[(c + 1) & 1]);
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gi = i0 + 4 * ty + i, gj = j0 + 4 * tx + j;
      if (gi < k && gj < k) {
        float v = alpha * acc[i][j];
        if (D) v += D[(int64_t)gj * k + gi];
        if (eye && gi == gj) v += 1.f;
        if (!sym) {
          C[(int64_t)gj * k + gi] = v;
        } else if (ti < tj || gi <= gj) {
          C[(int64_t)gj * k + gi] = v;
          C[(int64_t)gi * k + gj] = v;
        }
      }
    }
  }
}

// The whole k x k product by one CTA, tile after tile.
template <bool XT>
__device__ void block_gemm(const float* X, const float* Y, float* C, const float* D, float alpha,
                           bool eye, bool sym, int k, float* gs) {
  const int nt = (k + kT - 1) / kT;
  for (int tile = 0; tile < nt * nt; ++tile) {
    const int ti = tile % nt, tj = tile / nt;
    if (sym && ti > tj) continue;
    gemm_tile<XT>(X, Y, C, D, alpha, eye, sym, k, ti, tj, gs);
  }
  __syncthreads();
}
