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

__host__ __device__ __forceinline__ size_t smem_bytes_for(int k) {
  return (size_t)8 * k * k + (size_t)8 * pow2_ceil(k);
}

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

cudaError_t launch_jacobi(const EigArgs& a, int grid, size_t smem_bytes, cudaStream_t s) {
  if (a.num_tiles <= 0) return cudaSuccess;
  jacobi_kernel<<<grid, kThreads, smem_bytes, s>>>(a, (int)(smem_bytes / 4));
  return cudaGetLastError();
}

size_t jacobi_smem_for(int k) { return smem_bytes_for(k); }
size_t jacobi_sort_smem_for(int k) { return (size_t)8 * pow2_ceil(k); }
int jacobi_ctas_per_sm() { return 2048 / kThreads; }

cudaError_t configure_jacobi(size_t smem_limit) {
  return cudaFuncSetAttribute(jacobi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem_limit);
}

}  // namespace dobb

// ===========================================================================
// Cluster variant for blocks too wide for one CTA's shared memory (k <= 448).
//
// The same one-sided Jacobi and polish, spread over a cluster of kCl CTAs.
// Columns are split into 2 kCl groups of g = ceil(k / (2 kCl)) columns; the
// groups play a round-robin tournament (2 kCl - 1 block rounds per sweep).
// In each block round CTA c loads its two groups (U and V columns) from the
// L2-resident scratch into shared memory, rotates every cross pair (g rounds
// of g disjoint pairs, one warp per pair; in the first block round of a sweep
// also every pair inside each group), writes them back, and the cluster
// synchronises.  Every pair of columns is thus rotated once per sweep.  The
// polish phases split their columns (or pairs) over the cluster's CTAs, with
// a cluster barrier between phases.
// ===========================================================================
#include <cooperative_groups.h>

namespace dobb {
namespace {

namespace cg = cooperative_groups;
constexpr int kCl = 8;           // CTAs per cluster
constexpr int kClThreads = 1024;

__device__ __forceinline__ void rotate_pair(float* up, float* uq, float* vp, float* vq, int k,
                                            int lane, float tol, float tau, int& rots) {
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
    for (int i = lane; i < k; i += 32) {
      const float x = vp[i], y = vq[i];
      vp[i] = c * x - s * y;
      vq[i] = s * x + c * y;
    }
    ++rots;
  }
}

__global__ void __launch_bounds__(kClThreads, 1)
jacobi_cluster_kernel(const __grid_constant__ EigArgs a, int num_clusters) {
  extern __shared__ __align__(16) float sm[];
  __shared__ float red[32];
  __shared__ int s_rot;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = (int)cl.block_rank();
  const int cid = blockIdx.x / kCl;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  for (int w = cid; w < a.num_tiles; w += num_clusters) {
    const Tile t = a.tiles[w];
    const MatInfo mi = a.info[t.mat];
    const int k = mi.k;
    const int kp2 = pow2_ceil(k);
    const int64_t kk2 = (int64_t)k * k;
    const int64_t boff = mi.a_off + (int64_t)t.blk * kk2;
    const float* Ab = a.A + boff;
    uint32_t* flag = a.flags + mi.blk0 + t.blk;
    float* U = a.scratch + 3 * boff;
    float* V = U + kk2;
    float* Bm = U + 2 * kk2;
    float* Qb = a.Q + boff;
    // per-block rotation counters (two, alternating by sweep) after the moments
    int* counters = reinterpret_cast<int*>(a.lam + mi.lam_off + (int64_t)t.blk * k);
    const int g = (k + 2 * kCl - 1) / (2 * kCl);
    float* sU = sm;                     // [2g][k]
    float* sV = sm + 2 * g * k;         // [2g][k]
    float* lamv = sm + 4 * g * k;       // kp2
    int* perm = reinterpret_cast<int*>(lamv + kp2);
    // columns of phase-split work: [c0, c1)
    const int per = (k + kCl - 1) / kCl;
    const int c0 = min(k, rank * per), c1 = min(k, c0 + per);

    // ||A||_F and finiteness (every CTA, identical result)
    float ss = 0.f;
    int bad = 0;
    for (int64_t e = tid; e < kk2; e += blockDim.x) {
      const float v = Ab[e];
      bad |= !isfinite(v);
      ss = fmaf(v, v, ss);
    }
    bad = __syncthreads_or(bad);
    if (bad) {
      if (rank == 0 && tid == 0) atomicOr(flag, (uint32_t)DOBB_FLAG_NONFINITE_A);
      cl.sync();
      continue;
    }
    const float fro2 = block_sum(ss, red);
    const float tol = a.tol > 0.f ? a.tol : 4.f * sqrtf((float)k) * kEps;
    const float tau = 0.25f * kEps * sqrtf(fro2);
    // warm start: V = Q (columns), U = A V, for this CTA's columns
    for (int64_t e = tid; e < (int64_t)(c1 - c0) * k; e += blockDim.x) {
      const int j = c0 + (int)(e / k), l = (int)(e % k);
      V[(int64_t)j * k + l] = Qb[(int64_t)l * k + j];
    }
    __syncthreads();
    for (int p = c0 + warp; p < c1; p += nw) {
      const float* vp = V + (int64_t)p * k;
      for (int i = lane; i < k; i += 32) {
        float acc = 0.f;
        for (int l = 0; l < k; ++l) acc = fmaf(Ab[(int64_t)l * k + i], vp[l], acc);
        U[(int64_t)p * k + i] = acc;
      }
    }
    if (rank == 0 && tid < 2) counters[tid] = 0;
    cl.sync();

    int sweep = 0, last_rot = 0;
    const int G2 = 2 * kCl;
    for (; sweep < a.max_sweeps; ++sweep) {
      if (tid == 0) s_rot = 0;
      int my_rot = 0;
      for (int br = 0; br < G2 - 1; ++br) {
        int gI, gJ;
        rr_pair(br, rank, G2, gI, gJ);
        const int nI = max(0, min(g, k - gI * g)), nJ = max(0, min(g, k - gJ * g));
        // load both groups (local columns 0..g-1 = I, g..2g-1 = J)
        for (int64_t e = tid; e < (int64_t)2 * g * k; e += blockDim.x) {
          const int lc = (int)(e / k), i = (int)(e % k);
          const int gc = lc < g ? gI * g + lc : gJ * g + (lc - g);
          const bool ok = lc < g ? lc < nI : (lc - g) < nJ;
          sU[e] = ok ? U[(int64_t)gc * k + i] : 0.f;
          sV[e] = ok ? V[(int64_t)gc * k + i] : 0.f;
        }
        __syncthreads();
        if (br == 0) {
          // pairs inside each group: round robin over gg players
          const int gg = g + (g & 1);
          for (int r = 0; r < gg - 1; ++r) {
            for (int pw = warp; pw < gg; pw += nw) {  // gg/2 pairs per group, two groups
              const int grp = pw / (gg / 2), i = pw % (gg / 2);
              int p, q;
              rr_pair(r, i, gg, p, q);
              const int n = grp == 0 ? nI : nJ;
              if (p >= n || q >= n) continue;
              const int lp = grp * g + p, lq = grp * g + q;
              rotate_pair(sU + (int64_t)lp * k, sU + (int64_t)lq * k, sV + (int64_t)lp * k,
                          sV + (int64_t)lq * k, k, lane, tol, tau, my_rot);
            }
            __syncthreads();
          }
        }
        // cross pairs: round rho pairs I-column i with J-column (i + rho) mod g
        for (int rho = 0; rho < g; ++rho) {
          for (int i = warp; i < g; i += nw) {
            const int j = (i + rho) % g;
            if (i >= nI || j >= nJ) continue;
            rotate_pair(sU + (int64_t)i * k, sU + (int64_t)(g + j) * k, sV + (int64_t)i * k,
                        sV + (int64_t)(g + j) * k, k, lane, tol, tau, my_rot);
          }
          __syncthreads();
        }
        // write back
        for (int64_t e = tid; e < (int64_t)2 * g * k; e += blockDim.x) {
          const int lc = (int)(e / k), i = (int)(e % k);
          const int gc = lc < g ? gI * g + lc : gJ * g + (lc - g);
          const bool ok = lc < g ? lc < nI : (lc - g) < nJ;
          if (ok) {
            U[(int64_t)gc * k + i] = sU[e];
            V[(int64_t)gc * k + i] = sV[e];
          }
        }
        cl.sync();
      }
      if (lane == 0 && my_rot) atomicAdd(&s_rot, my_rot);
      __syncthreads();
      if (tid == 0 && s_rot) atomicAdd(&counters[sweep & 1], s_rot);
      cl.sync();
      last_rot = *reinterpret_cast<volatile int*>(&counters[sweep & 1]);
      cl.sync();
      if (rank == 0 && tid == 0) counters[sweep & 1] = 0;
      if (last_rot == 0) break;
    }
    cl.sync();

    // ---- polish (columns / pairs split over the cluster) ----
    // (1) E = I - V^T V (columns c0..c1) into U; then V1 = V + V E / 2 into Q
    for (int q = c0 + warp; q < c1; q += nw) {
      const float* vq = V + (int64_t)q * k;
      for (int p = 0; p < k; ++p) {
        const float* vp = V + (int64_t)p * k;
        float d = 0.f;
        for (int i = lane; i < k; i += 32) d = fmaf(vp[i], vq[i], d);
        d = warp_sum(d);
        if (lane == 0) U[(int64_t)q * k + p] = (p == q ? 1.f : 0.f) - d;
      }
    }
    cl.sync();
    for (int j = c0 + warp; j < c1; j += nw) {
      const float* ej = U + (int64_t)j * k;
      for (int i = lane; i < k; i += 32) {
        float acc = 0.f;
        for (int q = 0; q < k; ++q) acc = fmaf(V[(int64_t)q * k + i], ej[q], acc);
        Qb[(int64_t)j * k + i] = fmaf(0.5f, acc, V[(int64_t)j * k + i]);
      }
    }
    cl.sync();
    // (2) T = A V1 into U; B = V1^T T into Bm; W = I into V
    for (int p = c0 + warp; p < c1; p += nw) {
      const float* v1 = Qb + (int64_t)p * k;
      for (int i = lane; i < k; i += 32) {
        float acc = 0.f;
        for (int l = 0; l < k; ++l) acc = fmaf(Ab[(int64_t)l * k + i], v1[l], acc);
        U[(int64_t)p * k + i] = acc;
      }
    }
    cl.sync();
    for (int p = c0 + warp; p < c1; p += nw) {
      const float* v1p = Qb + (int64_t)p * k;
      const float* tp = U + (int64_t)p * k;
      for (int q = 0; q < k; ++q) {
        const float* v1q = Qb + (int64_t)q * k;
        const float* tq = U + (int64_t)q * k;
        float d = 0.f;
        for (int i = lane; i < k; i += 32) d = fmaf(v1p[i], tq[i], fmaf(v1q[i], tp[i], d));
        d = 0.5f * warp_sum(d);
        if (lane == 0) Bm[(int64_t)p * k + q] = d;  // row p; symmetric by construction
      }
    }
    for (int64_t e = (int64_t)c0 * k + tid; e < (int64_t)c1 * k; e += blockDim.x)
      V[e] = ((e / k) == (e % k)) ? 1.f : 0.f;
    cl.sync();
    // (3) one two-sided sweep on B; pairs of a round split over the cluster
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
            const float tau2 = (Bm[(int64_t)q * k + q] - Bm[(int64_t)p * k + p]) / (2.f * bpq);
            const float tt = tau2 >= 0.f ? 1.f / (tau2 + sqrtf(1.f + tau2 * tau2))
                                         : -1.f / (-tau2 + sqrtf(1.f + tau2 * tau2));
            c = 1.f / sqrtf(1.f + tt * tt);
            sv = tt * c;
          }
        }
        cs[i] = c;
        sn[i] = sv;
      }
      __syncthreads();
      // rows p, q of B (pairs i with i % kCl == rank)
      for (int64_t e = tid; e < (int64_t)(kk / 2) * k; e += blockDim.x) {
        const int i = (int)(e / k), j = (int)(e % k);
        if (i % kCl != rank || sn[i] == 0.f) continue;
        int p, q;
        rr_pair(r, i, kk, p, q);
        if (p > q) { const int tt = p; p = q; q = tt; }
        const float x = Bm[(int64_t)p * k + j], y = Bm[(int64_t)q * k + j];
        Bm[(int64_t)p * k + j] = cs[i] * x - sn[i] * y;
        Bm[(int64_t)q * k + j] = sn[i] * x + cs[i] * y;
      }
      cl.sync();
      // columns p, q of B and W
      for (int64_t e = tid; e < (int64_t)(kk / 2) * k; e += blockDim.x) {
        const int i = (int)(e / k), j = (int)(e % k);
        if (i % kCl != rank || sn[i] == 0.f) continue;
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
      cl.sync();
    }
    // (4) V2 = V1 W into U; eigenvalues = diag(B), sorted in every CTA
    for (int j = c0 + warp; j < c1; j += nw) {
      const float* wj = V + (int64_t)j * k;
      for (int i = lane; i < k; i += 32) {
        float acc = 0.f;
        for (int q = 0; q < k; ++q) acc = fmaf(Qb[(int64_t)q * k + i], wj[q], acc);
        U[(int64_t)j * k + i] = acc;
      }
    }
    for (int p = tid; p < kp2; p += blockDim.x) {
      lamv[p] = p < k ? Bm[(int64_t)p * k + p] : -INFINITY;
      perm[p] = p;
    }
    cl.sync();
    // (5) E2 = I - V2^T V2 into Bm (columns c0..c1)
    for (int q = c0 + warp; q < c1; q += nw) {
      const float* vq = U + (int64_t)q * k;
      for (int p = 0; p < k; ++p) {
        const float* vp = U + (int64_t)p * k;
        float d = 0.f;
        for (int i = lane; i < k; i += 32) d = fmaf(vp[i], vq[i], d);
        d = warp_sum(d);
        if (lane == 0) Bm[(int64_t)q * k + p] = (p == q ? 1.f : 0.f) - d;
      }
    }
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
    cl.sync();
    // (6) Q columns c0..c1 (row-major)
    for (int j = c0 + warp; j < c1; j += nw) {
      int p = perm[j];
      if (p < 0 || p >= k) p = j;
      const float* vp = U + (int64_t)p * k;
      const float* ep = Bm + (int64_t)p * k;
      for (int i = lane; i < k; i += 32) {
        float acc = 0.f;
        for (int q = 0; q < k; ++q) acc = fmaf(U[(int64_t)q * k + i], ep[q], acc);
        Qb[(int64_t)i * k + j] = fmaf(0.5f, acc, vp[i]);
      }
    }
    if (rank == 0) {
      for (int j = tid; j < k; j += blockDim.x) a.lam[mi.lam_off + (int64_t)t.blk * k + j] = lamv[j];
      if (tid == 0) {
        float* st = a.stats + 4 * (int64_t)(mi.blk0 + t.blk);
        st[2] = (float)sweep;
        st[3] = (float)last_rot;
        if (sweep >= a.max_sweeps && last_rot > 0) atomicOr(flag, (uint32_t)DOBB_FLAG_NOT_CONVERGED);
      }
    }
    cl.sync();
  }
}

}  // namespace

size_t jacobi_cluster_smem(int k) {
  const int g = (k + 2 * kCl - 1) / (2 * kCl);
  return (size_t)16 * g * k + (size_t)8 * pow2_ceil(k);
}

bool jacobi_cluster_fits(int k, size_t smem_limit) {
  const int g = (k + 2 * kCl - 1) / (2 * kCl);
  return g <= 32 && jacobi_cluster_smem(k) <= smem_limit;
}

cudaError_t configure_jacobi_cluster(size_t smem_limit) {
  return cudaFuncSetAttribute(jacobi_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem_limit);
}

int jacobi_cluster_max_active(size_t smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCl * 64);
  cfg.blockDim = dim3(kClThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, jacobi_cluster_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_jacobi_cluster(const EigArgs& a, int clusters, size_t smem, cudaStream_t s) {
  if (a.num_tiles <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCl * clusters);
  cfg.blockDim = dim3(kClThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, jacobi_cluster_kernel, a, clusters);
}

}  // namespace dobb
