// Batched symmetric eigensolver for the k x k block moments
// ("Dobb", Abstract: a complete basis within each block; Table 15: exact
// eigendecomposition refresh).
//
// One-sided (Hestenes) Jacobi with V accumulated: V starts as the current
// basis Q (the identity before the first refresh) and U as A V; each
// rotation of a column pair (p, q) makes u_p and u_q orthogonal and applies
// the same rotation to v_p, v_q, so A V = U is kept.  Pairs are visited in
// round-robin (circle) order: each round holds k/2 disjoint pairs that the
// warps of one CTA rotate in parallel; k - 1 rounds form a sweep.  A pair is
// rotated only when its columns are measurably non-orthogonal both relative
// to their own norms (|u_p.u_q| > tol |u_p||u_q|) and relative to the block
// (|u_p.u_q| > tau ||A||_F max(|u_p|, |u_q|), tau = eps / 4): below that the
// residual the rotation would remove is under fp32 rounding of A, and
// rotating there only adds rounding noise to V.  Sweeps stop when one sweep
// rotates nothing, or at the sweep cap.
//
// Finish (a polish that brings the backward error to the fp32 floor of a
// Householder-based solver instead of the ~sqrt(rotations) eps that the
// accumulated rotations leave):
//   V1 = V + V (I - V^T V) / 2          (Newton-Schulz re-orthogonalisation)
//   B  = V1^T A V1                      (nearly diagonal)
//   one two-sided cyclic Jacobi sweep on B (rotations J, Golub & Van Loan's
//   2x2 symmetric Schur step), accumulating W = J_1 J_2 ...
//   V2 = V1 W, Q = V2 + V2 (I - V2^T V2) / 2, Lambda = diag(B)
// then eigenpairs are sorted by descending eigenvalue and written as
// row-major Q (column j = j-th eigenvector) and Lambda.
//
// One CTA per block.  U and V live in shared memory when 8 k^2 bytes fit,
// otherwise in a global scratch area of the state buffer.
#include "common.cuh"

namespace dobb {
namespace {

constexpr int kThreads = 512;
constexpr float kEps = 5.9604645e-8f;  // 2^-24, fp32 unit roundoff

__host__ __device__ __forceinline__ int pow2_ceil(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

// Pair i of round r in the circle schedule over kk (even) players.
__device__ __forceinline__ void rr_pair(int r, int i, int kk, int& p, int& q) {
  if (i == 0) {
    p = kk - 1;
    q = r;
  } else {
    p = (r + i) % (kk - 1);
    q = (r - i + kk - 1) % (kk - 1);
  }
}

// E = I - V^T V (symmetric), column q of E at E + q k; one warp per column.
__device__ __forceinline__ void newton_schulz_cols(const float* V, float* E, int k, int warp, int nw,
                                                   int lane) {
  for (int q = warp; q < k; q += nw) {
    const float* vq = V + (int64_t)q * k;
    for (int p = 0; p < k; ++p) {
      const float* vp = V + (int64_t)p * k;
      float d = 0.f;
      for (int i = lane; i < k; i += 32) d = fmaf(vp[i], vq[i], d);
      d = warp_sum(d);
      if (lane == 0) E[(int64_t)q * k + p] = (p == q ? 1.f : 0.f) - d;
    }
  }
}

// One rotation of the column pair (p, q) with the four columns held in
// registers (k <= 32 kRegCols): all loads are issued at once, the dot products
// and the rotation use the registers, results are stored once.  Same
// arithmetic, in the same order, as the streaming loop.
template <int kRegCols>
__device__ __forceinline__ void rotate_pair_regs(float* up, float* uq, float* vp, float* vq, int k,
                                                 int lane, float tol, float tau, int& rots) {
  float xu[kRegCols], yu[kRegCols], xv[kRegCols], yv[kRegCols];
#pragma unroll
  for (int e = 0; e < kRegCols; ++e) {
    const int i = lane + 32 * e;
    const bool ok = i < k;
    xu[e] = ok ? up[i] : 0.f;
    yu[e] = ok ? uq[i] : 0.f;
    xv[e] = ok ? vp[i] : 0.f;
    yv[e] = ok ? vq[i] : 0.f;
  }
  float al = 0.f, be = 0.f, ga = 0.f;
#pragma unroll
  for (int e = 0; e < kRegCols; ++e) {
    al = fmaf(xu[e], xu[e], al);
    be = fmaf(yu[e], yu[e], be);
    ga = fmaf(xu[e], yu[e], ga);
  }
  al = warp_sum(al);
  be = warp_sum(be);
  ga = warp_sum(ga);
  if (fabsf(ga) > tol * sqrtf(al) * sqrtf(be) && fabsf(ga) > tau * sqrtf(fmaxf(al, be))) {
    const float zeta = (be - al) / (2.f * ga);
    const float tt = copysignf(1.f, zeta) / (fabsf(zeta) + sqrtf(1.f + zeta * zeta));
    const float c = 1.f / sqrtf(1.f + tt * tt);
    const float sn = c * tt;
#pragma unroll
    for (int e = 0; e < kRegCols; ++e) {
      const int i = lane + 32 * e;
      if (i < k) {
        up[i] = c * xu[e] - sn * yu[e];
        uq[i] = sn * xu[e] + c * yu[e];
        vp[i] = c * xv[e] - sn * yv[e];
        vq[i] = sn * xv[e] + c * yv[e];
      }
    }
    ++rots;
  }
}

// Shared-memory tiled product over the k x k operands of one block, FP32:
//   C(i, j) = alpha * sum_l X(i, l) Y(l, j) + D(i, j) + (eye ? delta_ij : 0)
// with Y(l, j) = Y[j k + l], X(i, l) = X[l k + i] (XT = false) or X[i k + l]
// (XT = true); C(i, j) and D(i, j) are stored at [j k + i].  64 x 64 output
// tiles, 32-deep reduction chunks, the CTA's 512 threads own 2 x 4 outputs.
constexpr int kGT = 64, kGK = 32, kGP = kGT + 4;
constexpr size_t kGemmSmemFloats = 2 * kGK * kGP;

template <bool XT>
__device__ void block_gemm(const float* X, const float* Y, float* C, const float* D, float alpha,
                           bool eye, int k, float* gs) {
  float* Xs = gs;
  float* Ys = gs + kGK * kGP;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;  // ty < 32 for 512 threads
  const int nt = (k + kGT - 1) / kGT;
  for (int tile = 0; tile < nt * nt; ++tile) {
    const int i0 = (tile % nt) * kGT, j0 = (tile / nt) * kGT;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    for (int l0 = 0; l0 < k; l0 += kGK) {
      for (int e = tid; e < kGK * kGT; e += blockDim.x) {
        // X tile: rows i0.., reduction l0..; coalesced along the contiguous index
        int l, i;
        if (XT) { l = e % kGK; i = e / kGK; } else { i = e % kGT; l = e / kGT; }
        float xv = 0.f;
        if (i0 + i < k && l0 + l < k)
          xv = XT ? X[(int64_t)(i0 + i) * k + l0 + l] : X[(int64_t)(l0 + l) * k + i0 + i];
        Xs[l * kGP + i] = xv;
        const int ly = e % kGK, j = e / kGK;
        float yv = 0.f;
        if (j0 + j < k && l0 + ly < k) yv = Y[(int64_t)(j0 + j) * k + l0 + ly];
        Ys[ly * kGP + j] = yv;
      }
      __syncthreads();
#pragma unroll 8
      for (int l = 0; l < kGK; ++l) {
        const float a0 = Xs[l * kGP + ty * 2], a1 = Xs[l * kGP + ty * 2 + 1];
        float b[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) b[q] = Ys[l * kGP + tx * 4 + q];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[0][q] = fmaf(a0, b[q], acc[0][q]);
          acc[1][q] = fmaf(a1, b[q], acc[1][q]);
        }
      }
      __syncthreads();
    }
#pragma unroll
    for (int p = 0; p < 2; ++p) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = i0 + ty * 2 + p, j = j0 + tx * 4 + q;
        if (i < k && j < k) {
          float v = alpha * acc[p][q];
          if (D) v += D[(int64_t)j * k + i];
          if (eye && i == j) v += 1.f;
          C[(int64_t)j * k + i] = v;
        }
      }
    }
  }
  __syncthreads();
}

__host__ __device__ __forceinline__ size_t smem_bytes_for(int k) {
  return (size_t)8 * k * k + (size_t)8 * pow2_ceil(k);
}

// Polish of a block whose U, V live in global scratch, with the tiled
// products above (same steps as the in-shared-memory polish of the kernel):
// E = I - V^T V; V1 = V + V E / 2; T = A V1; B = sym(V1^T T); one two-sided
// Jacobi sweep on B accumulating W; V2 = V1 W; E2 = I - V2^T V2;
// Q = (V2 + V2 E2 / 2) with columns sorted by descending diag(B).
__device__ void polish_global(const float* Ab, float* U, float* V, float* Bm, float* Qb,
                              float* lamv, int* perm, int k, int kp2, float fro2, float* gs) {
  const int tid = threadIdx.x;
  block_gemm<true>(V, V, Bm, nullptr, -1.f, true, k, gs);        // E
  block_gemm<false>(V, Bm, U, V, 0.5f, false, k, gs);            // V1 (in U)
  block_gemm<false>(Ab, U, V, nullptr, 1.f, false, k, gs);       // T = A V1 (A symmetric)
  block_gemm<true>(U, V, Bm, nullptr, 1.f, false, k, gs);        // B = V1^T T
  for (int64_t e = tid; e < (int64_t)k * k; e += blockDim.x) {
    const int i = (int)(e % k), j = (int)(e / k);
    if (i < j) {
      const float v = 0.5f * (Bm[(int64_t)j * k + i] + Bm[(int64_t)i * k + j]);
      Bm[(int64_t)j * k + i] = v;
      Bm[(int64_t)i * k + j] = v;
    }
  }
  for (int64_t e = tid; e < (int64_t)k * k; e += blockDim.x) V[e] = ((e / k) == (e % k)) ? 1.f : 0.f;
  __syncthreads();
  const int kk = k + (k & 1);
  float* cs = lamv;
  float* sn = lamv + (kp2 >> 1);
  const float bfloor = 1e-3f * kEps * sqrtf(fro2);
  for (int r = 0; r < kk - 1; ++r) {
    for (int i = tid; i < kk / 2; i += blockDim.x) {
      int p, q;
      rr_pair(r, i, kk, p, q);
      float c = 1.f, sv = 0.f;
      if (p < k && q < k) {
        if (p > q) { const int tt = p; p = q; q = tt; }
        const float bpq = Bm[(int64_t)p * k + q];
        if (fabsf(bpq) > bfloor) {
          const float ta = (Bm[(int64_t)q * k + q] - Bm[(int64_t)p * k + p]) / (2.f * bpq);
          const float tt = ta >= 0.f ? 1.f / (ta + sqrtf(1.f + ta * ta)) : -1.f / (-ta + sqrtf(1.f + ta * ta));
          c = 1.f / sqrtf(1.f + tt * tt);
          sv = tt * c;
        }
      }
      cs[i] = c;
      sn[i] = sv;
    }
    __syncthreads();
    for (int64_t e = tid; e < (int64_t)(kk / 2) * k; e += blockDim.x) {
      const int i = (int)(e / k), j = (int)(e % k);
      if (sn[i] == 0.f) continue;
      int p, q;
      rr_pair(r, i, kk, p, q);
      if (p > q) { const int tt = p; p = q; q = tt; }
      const float x = Bm[(int64_t)p * k + j], y = Bm[(int64_t)q * k + j];
      Bm[(int64_t)p * k + j] = cs[i] * x - sn[i] * y;
      Bm[(int64_t)q * k + j] = sn[i] * x + cs[i] * y;
    }
    __syncthreads();
    for (int64_t e = tid; e < (int64_t)(kk / 2) * k; e += blockDim.x) {
      const int i = (int)(e / k), j = (int)(e % k);
      if (sn[i] == 0.f) continue;
      int p, q;
      rr_pair(r, i, kk, p, q);
      if (p > q) { const int tt = p; p = q; q = tt; }
      float x = Bm[(int64_t)j * k + p], y = Bm[(int64_t)j * k + q];
      Bm[(int64_t)j * k + p] = cs[i] * x - sn[i] * y;
      Bm[(int64_t)j * k + q] = sn[i] * x + cs[i] * y;
      x = V[(int64_t)p * k + j];
      y = V[(int64_t)q * k + j];
      V[(int64_t)p * k + j] = cs[i] * x - sn[i] * y;
      V[(int64_t)q * k + j] = sn[i] * x + cs[i] * y;
    }
    __syncthreads();
  }
  block_gemm<false>(U, V, Qb, nullptr, 1.f, false, k, gs);       // V2 = V1 W (in Qb)
  for (int p = tid; p < kp2; p += blockDim.x) {
    lamv[p] = p < k ? Bm[(int64_t)p * k + p] : -INFINITY;
    perm[p] = p;
  }
  __syncthreads();
  block_gemm<true>(Qb, Qb, Bm, nullptr, -1.f, true, k, gs);      // E2
  block_gemm<false>(Qb, Bm, U, Qb, 0.5f, false, k, gs);          // R = V2 + V2 E2 / 2 (in U)
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
  for (int64_t e = tid; e < (int64_t)k * k; e += blockDim.x) {
    const int j = (int)(e / k), i = (int)(e % k);
    int p = perm[j];
    if (p < 0 || p >= k) p = j;  // only reachable with a NaN eigenvalue
    Qb[(int64_t)i * k + j] = U[(int64_t)p * k + i];
  }
  __syncthreads();
}

template <int kRegCols>
__global__ void __launch_bounds__(kThreads)
jacobi_kernel(const __grid_constant__ EigArgs a, int smem_floats) {
  extern __shared__ __align__(16) float sm[];
  __shared__ float red[32];
  __shared__ int s_rot;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  for (int w = blockIdx.x; w < a.num_tiles; w += gridDim.x) {
    const Tile t = a.tiles[w];
    const MatInfo mi = a.info[t.mat];
    const int k = mi.k;
    const int kp2 = pow2_ceil(k);
    const int64_t kk2 = (int64_t)k * k;
    const int64_t boff = mi.a_off + (int64_t)t.blk * kk2;
    const float* Ab = a.A + boff;
    uint32_t* flag = a.flags + mi.blk0 + t.blk;
    const bool in_smem = smem_bytes_for(k) <= (size_t)smem_floats * 4;
    float* U;
    float* V;
    float* lamv;
    float* Bm = a.scratch + 3 * boff + 2 * kk2;  // polish matrix, global
    if (in_smem) {
      U = sm;
      V = sm + kk2;
      lamv = sm + 2 * kk2;
    } else {
      U = a.scratch + 3 * boff;
      V = U + kk2;
      lamv = sm;
    }
    int* perm = reinterpret_cast<int*>(lamv + kp2);

    // Warm start from the current basis: V = Q (column j of V is column j of
    // the row-major Q), U = A V.  With Q = I (no refresh yet) this is the
    // plain start U = A, V = I.  ||A||_F^2 and a finiteness check on the way.
    float ss = 0.f;
    int bad = 0;
    const float* Qold = a.Q + boff;
    for (int64_t e = tid; e < kk2; e += blockDim.x) {
      const float v = Ab[e];
      bad |= !isfinite(v);
      ss = fmaf(v, v, ss);
      const int j = (int)(e / k), l = (int)(e % k);
      V[e] = Qold[(int64_t)l * k + j];
    }
    if (__syncthreads_or(bad)) {
      if (tid == 0) atomicOr(flag, (uint32_t)DOBB_FLAG_NONFINITE_A);
      continue;  // keep the previous basis
    }
    const float fro2 = block_sum(ss, red);
    for (int p = warp; p < k; p += nw) {
      const float* vp = V + (int64_t)p * k;
      for (int i = lane; i < k; i += 32) {
        float acc = 0.f;
        for (int l = 0; l < k; ++l) acc = fmaf(Ab[(int64_t)l * k + i], vp[l], acc);  // A symmetric
        U[(int64_t)p * k + i] = acc;
      }
    }
    __syncthreads();
    const float tol = a.tol > 0.f ? a.tol : 4.f * sqrtf((float)k) * kEps;
    const float tau = 0.25f * kEps * sqrtf(fro2);
    const int kk = k + (k & 1);
    int sweep = 0, last_rot = 0;
    for (; sweep < a.max_sweeps; ++sweep) {
      if (tid == 0) s_rot = 0;
      __syncthreads();
      int my_rot = 0;
      for (int r = 0; r < kk - 1; ++r) {
        for (int pi = warp; pi < kk / 2; pi += nw) {
          int p, q;
          rr_pair(r, pi, kk, p, q);
          if (p >= k || q >= k) continue;
          float* up = U + (int64_t)p * k;
          float* uq = U + (int64_t)q * k;
          if (kRegCols > 0 && k <= 32 * kRegCols) {
            rotate_pair_regs<(kRegCols > 0 ? kRegCols : 1)>(up, uq, V + (int64_t)p * k,
                                                            V + (int64_t)q * k, k, lane, tol, tau,
                                                            my_rot);
            continue;
          }
          float al = 0.f, be = 0.f, ga = 0.f;
          for (int i = lane; i < k; i += 32) {
            const float x = up[i], y = uq[i];
            al = fmaf(x, x, al);
            be = fmaf(y, y, be);
            ga = fmaf(x, y, ga);
          }
          al = warp_sum(al);
          be = warp_sum(be);
          ga = warp_sum(ga);
          if (fabsf(ga) > tol * sqrtf(al) * sqrtf(be) && fabsf(ga) > tau * sqrtf(fmaxf(al, be))) {
            const float zeta = (be - al) / (2.f * ga);
            const float tt = copysignf(1.f, zeta) / (fabsf(zeta) + sqrtf(1.f + zeta * zeta));
            const float c = 1.f / sqrtf(1.f + tt * tt);
            const float s = c * tt;
            for (int i = lane; i < k; i += 32) {
              const float x = up[i], y = uq[i];
              up[i] = c * x - s * y;
              uq[i] = s * x + c * y;
            }
            float* vp = V + (int64_t)p * k;
            float* vq = V + (int64_t)q * k;
            for (int i = lane; i < k; i += 32) {
              const float x = vp[i], y = vq[i];
              vp[i] = c * x - s * y;
              vq[i] = s * x + c * y;
            }
            ++my_rot;
          }
        }
        __syncthreads();
      }
      if (lane == 0 && my_rot) atomicAdd(&s_rot, my_rot);
      __syncthreads();
      last_rot = s_rot;
      __syncthreads();
      if (last_rot == 0) break;
    }

    if (!in_smem) {
      polish_global(Ab, U, V, Bm, a.Q + boff, lamv, perm, k, kp2, fro2, sm + 2 * kp2);
      for (int j = tid; j < k; j += blockDim.x) a.lam[mi.lam_off + (int64_t)t.blk * k + j] = lamv[j];
      if (tid == 0) {
        float* st = a.stats + 4 * (int64_t)(mi.blk0 + t.blk);
        st[2] = (float)sweep;
        st[3] = (float)last_rot;
        if (sweep >= a.max_sweeps && last_rot > 0) atomicOr(flag, (uint32_t)DOBB_FLAG_NOT_CONVERGED);
      }
      __syncthreads();
      continue;
    }
    float* Qb = a.Q + boff;  // holds V1 (column-major) until the final write
    // (1) E = I - V^T V into U (column q at U + q k), then V1 = V + V E / 2
    newton_schulz_cols(V, U, k, warp, nw, lane);
    __syncthreads();
    for (int j = warp; j < k; j += nw) {
      const float* ej = U + (int64_t)j * k;
      for (int i = lane; i < k; i += 32) {
        float acc = 0.f;
        for (int q = 0; q < k; ++q) acc = fmaf(V[(int64_t)q * k + i], ej[q], acc);
        Qb[(int64_t)j * k + i] = fmaf(0.5f, acc, V[(int64_t)j * k + i]);
      }
    }
    __syncthreads();
    // (2) T = A V1 into U; B = V1^T T (symmetrised) into Bm; W = I into V
    for (int p = warp; p < k; p += nw) {
      const float* v1 = Qb + (int64_t)p * k;
      for (int i = lane; i < k; i += 32) {
        float acc = 0.f;
        for (int l = 0; l < k; ++l) acc = fmaf(Ab[(int64_t)l * k + i], v1[l], acc);  // A symmetric
        U[(int64_t)p * k + i] = acc;
      }
    }
    __syncthreads();
    for (int p = warp; p < k; p += nw) {
      const float* v1p = Qb + (int64_t)p * k;
      const float* tp = U + (int64_t)p * k;
      for (int q = p; q < k; ++q) {
        const float* v1q = Qb + (int64_t)q * k;
        const float* tq = U + (int64_t)q * k;
        float d = 0.f;
        for (int i = lane; i < k; i += 32) d = fmaf(v1p[i], tq[i], fmaf(v1q[i], tp[i], d));
        d = 0.5f * warp_sum(d);
        if (lane == 0) {
          Bm[(int64_t)p * k + q] = d;
          Bm[(int64_t)q * k + p] = d;
        }
      }
    }
    for (int64_t e = tid; e < kk2; e += blockDim.x) V[e] = ((e / k) == (e % k)) ? 1.f : 0.f;
    __syncthreads();
    // (3) one two-sided sweep on B, W accumulated (column-major in V)
    float* cs = lamv;                         // kk/2 cosines
    float* sn = lamv + (kp2 >> 1);            // kk/2 sines
    const float bfloor = 1e-3f * kEps * sqrtf(fro2);
    for (int r = 0; r < kk - 1; ++r) {
      for (int i = tid; i < kk / 2; i += blockDim.x) {
        int p, q;
        rr_pair(r, i, kk, p, q);
        float c = 1.f, sv = 0.f;
        if (p < k && q < k) {
          if (p > q) { const int tt = p; p = q; q = tt; }
          const float bpq = Bm[(int64_t)p * k + q];
          if (fabsf(bpq) > bfloor) {
            const float tau = (Bm[(int64_t)q * k + q] - Bm[(int64_t)p * k + p]) / (2.f * bpq);
            const float tt = tau >= 0.f ? 1.f / (tau + sqrtf(1.f + tau * tau))
                                        : -1.f / (-tau + sqrtf(1.f + tau * tau));
            c = 1.f / sqrtf(1.f + tt * tt);
            sv = tt * c;
          }
        }
        cs[i] = c;
        sn[i] = sv;
      }
      __syncthreads();
      // rows p, q of B <- J^T B
      for (int64_t e = tid; e < (int64_t)(kk / 2) * k; e += blockDim.x) {
        const int i = (int)(e / k), j = (int)(e % k);
        if (sn[i] == 0.f) continue;
        int p, q;
        rr_pair(r, i, kk, p, q);
        if (p > q) { const int tt = p; p = q; q = tt; }
        const float x = Bm[(int64_t)p * k + j], y = Bm[(int64_t)q * k + j];
        Bm[(int64_t)p * k + j] = cs[i] * x - sn[i] * y;
        Bm[(int64_t)q * k + j] = sn[i] * x + cs[i] * y;
      }
      __syncthreads();
      // columns p, q of B <- B J, and of W <- W J
      for (int64_t e = tid; e < (int64_t)(kk / 2) * k; e += blockDim.x) {
        const int i = (int)(e / k), j = (int)(e % k);
        if (sn[i] == 0.f) continue;
        int p, q;
        rr_pair(r, i, kk, p, q);
        if (p > q) { const int tt = p; p = q; q = tt; }
        float x = Bm[(int64_t)j * k + p], y = Bm[(int64_t)j * k + q];
        Bm[(int64_t)j * k + p] = cs[i] * x - sn[i] * y;
        Bm[(int64_t)j * k + q] = sn[i] * x + cs[i] * y;
        x = V[(int64_t)p * k + j];
        y = V[(int64_t)q * k + j];
        V[(int64_t)p * k + j] = cs[i] * x - sn[i] * y;
        V[(int64_t)q * k + j] = sn[i] * x + cs[i] * y;
      }
      __syncthreads();
    }
    // (4) V2 = V1 W into U; eigenvalues = diag(B)
    for (int j = warp; j < k; j += nw) {
      const float* wj = V + (int64_t)j * k;
      for (int i = lane; i < k; i += 32) {
        float acc = 0.f;
        for (int q = 0; q < k; ++q) acc = fmaf(Qb[(int64_t)q * k + i], wj[q], acc);
        U[(int64_t)j * k + i] = acc;
      }
    }
    __syncthreads();
    for (int p = tid; p < kp2; p += blockDim.x) {
      lamv[p] = p < k ? Bm[(int64_t)p * k + p] : -INFINITY;
      perm[p] = p;
    }
    __syncthreads();
    // (5) E2 = I - V2^T V2 into Bm (column q at Bm + q k)
    newton_schulz_cols(U, Bm, k, warp, nw, lane);
    // sort descending by eigenvalue
    for (int size = 2; size <= kp2; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        __syncthreads();
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
      }
    }
    __syncthreads();
    // (6) Q[:, j] = v2_p + (1/2) V2 e2_p with p = perm[j]
    for (int j = warp; j < k; j += nw) {
      int p = perm[j];
      if (p < 0 || p >= k) p = j;  // only reachable with a NaN eigenvalue
      const float* vp = U + (int64_t)p * k;
      const float* ep = Bm + (int64_t)p * k;
      for (int i = lane; i < k; i += 32) {
        float acc = 0.f;
        for (int q = 0; q < k; ++q) acc = fmaf(U[(int64_t)q * k + i], ep[q], acc);
        Qb[(int64_t)i * k + j] = fmaf(0.5f, acc, vp[i]);
      }
    }
    for (int j = tid; j < k; j += blockDim.x) a.lam[mi.lam_off + (int64_t)t.blk * k + j] = lamv[j];
    if (tid == 0) {
      float* st = a.stats + 4 * (int64_t)(mi.blk0 + t.blk);
      st[2] = (float)sweep;
      st[3] = (float)last_rot;
      if (sweep >= a.max_sweeps && last_rot > 0) atomicOr(flag, (uint32_t)DOBB_FLAG_NOT_CONVERGED);
    }
    __syncthreads();
  }
}

}  // namespace

int jacobi_smem_max_k(size_t smem_limit) {
  int k = 1;
  while (smem_bytes_for(k + 1) <= smem_limit) ++k;
  return k;
}

// wide = blocks whose U, V live in global scratch: those rotate column pairs
// held in registers (k <= 512) and polish with the tiled products.
cudaError_t launch_jacobi(const EigArgs& a, int grid, size_t smem_bytes, cudaStream_t s, bool wide) {
  if (a.num_tiles <= 0) return cudaSuccess;
  if (wide)
    jacobi_kernel<16><<<grid, kThreads, smem_bytes, s>>>(a, (int)(smem_bytes / 4));
  else
    jacobi_kernel<0><<<grid, kThreads, smem_bytes, s>>>(a, (int)(smem_bytes / 4));
  return cudaGetLastError();
}

size_t jacobi_smem_for(int k) { return smem_bytes_for(k); }
size_t jacobi_sort_smem_for(int k) { return (size_t)8 * pow2_ceil(k) + 4 * kGemmSmemFloats; }
int jacobi_ctas_per_sm() { return 2048 / kThreads; }

cudaError_t configure_jacobi(size_t smem_limit) {
  cudaError_t e = cudaFuncSetAttribute(jacobi_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_limit);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(jacobi_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem_limit);
}

}  // namespace dobb
