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
// Finish: lambda_p = (v_p . u_p) / (v_p . v_p); one Newton-Schulz step
// V <- V + V (I - V^T V) / 2 removes the norm and orthogonality drift that
// thousands of fp32 rotations leave in V; eigenpairs are sorted by
// descending eigenvalue and written as row-major Q (column j = j-th
// eigenvector) and Lambda.
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
    if (in_smem) {
      U = sm;
      V = sm + kk2;
      lamv = sm + 2 * kk2;
    } else {
      U = a.scratch + 2 * boff;
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

    // eigenvalues lambda_p = (v_p . u_p) / (v_p . v_p)
    for (int p = warp; p < k; p += nw) {
      const float* up = U + (int64_t)p * k;
      const float* vp = V + (int64_t)p * k;
      float d = 0.f, nv = 0.f;
      for (int i = lane; i < k; i += 32) {
        d = fmaf(vp[i], up[i], d);
        nv = fmaf(vp[i], vp[i], nv);
      }
      d = warp_sum(d);
      nv = warp_sum(nv);
      if (lane == 0) lamv[p] = d / nv;
    }
    for (int p = k + tid; p < kp2; p += blockDim.x) lamv[p] = -INFINITY;
    for (int p = tid; p < kp2; p += blockDim.x) perm[p] = p;
    __syncthreads();
    // E = I - V^T V (symmetric) into U's storage, column q at U + q k
    for (int q = warp; q < k; q += nw) {
      const float* vq = V + (int64_t)q * k;
      for (int p = 0; p < k; ++p) {
        const float* vp = V + (int64_t)p * k;
        float d = 0.f;
        for (int i = lane; i < k; i += 32) d = fmaf(vp[i], vq[i], d);
        d = warp_sum(d);
        if (lane == 0) U[(int64_t)q * k + p] = (p == q ? 1.f : 0.f) - d;
      }
    }
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
    // Q[:, j] = v_p + (1/2) V e_p with p = perm[j] (Newton-Schulz step)
    float* Qb = a.Q + boff;
    for (int j = warp; j < k; j += nw) {
      int p = perm[j];
      if (p < 0 || p >= k) p = j;  // only reachable with a NaN eigenvalue
      const float* vp = V + (int64_t)p * k;
      const float* ep = U + (int64_t)p * k;
      for (int i = lane; i < k; i += 32) {
        float acc = 0.f;
        for (int q = 0; q < k; ++q) acc = fmaf(V[(int64_t)q * k + i], ep[q], acc);
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
