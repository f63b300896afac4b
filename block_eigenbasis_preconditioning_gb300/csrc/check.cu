// Invariant checks of the block eigenbases, and basis initialisation.
//
// For every block: ||A Q - Q Lambda||_F / ||A||_F, ||Q^T Q - I||_F and
// ||Q Lambda Q^T - A||_F / ||A||_F, with fp32 products summed in fp64 so the
// check is accurate well below the fp32 residuals it measures ("Dobb",
// Abstract: a complete orthonormal basis of each block's second moment).
#include "common.cuh"

namespace dobb {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) check_bases_kernel(const __grid_constant__ CheckArgs a) {
  __shared__ double red[32];
  for (int w = blockIdx.x; w < a.num_tiles; w += gridDim.x) {
    const Tile t = a.tiles[w];
    const MatInfo mi = a.info[t.mat];
    const int k = mi.k;
    const int64_t boff = mi.a_off + (int64_t)t.blk * k * k;
    const float* A = a.A + boff;
    const float* Q = a.Q + boff;
    const float* L = a.lam + mi.lam_off + (int64_t)t.blk * k;
    double r1 = 0.0, r2 = 0.0, r3 = 0.0, a2 = 0.0;
    for (int64_t e = threadIdx.x; e < (int64_t)k * k; e += kThreads) {
      const int i = (int)(e / k), j = (int)(e % k);
      double aq = 0.0, qq = 0.0, rc = 0.0;
      for (int l = 0; l < k; ++l) {
        aq += (double)A[(int64_t)i * k + l] * (double)Q[(int64_t)l * k + j];
        qq += (double)Q[(int64_t)l * k + i] * (double)Q[(int64_t)l * k + j];
        rc += (double)Q[(int64_t)i * k + l] * (double)L[l] * (double)Q[(int64_t)j * k + l];
      }
      const double aij = A[e];
      const double d1 = aq - (double)L[j] * (double)Q[e];
      const double d2 = qq - (i == j ? 1.0 : 0.0);
      const double d3 = rc - aij;
      r1 += d1 * d1;
      r2 += d2 * d2;
      r3 += d3 * d3;
      a2 += aij * aij;
    }
    r1 = block_sum_d(r1, red);
    r2 = block_sum_d(r2, red);
    r3 = block_sum_d(r3, red);
    a2 = block_sum_d(a2, red);
    if (threadIdx.x == 0) {
      const double fa = a2 > 0.0 ? sqrt(a2) : 1.0;
      float* o = a.out + 3 * (int64_t)(mi.blk0 + t.blk);
      o[0] = (float)(sqrt(r1) / fa);
      o[1] = (float)sqrt(r2);
      o[2] = (float)(sqrt(r3) / fa);
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kThreads)
init_bases_kernel(float* Q, float* lam, const MatInfo* info, const Tile* items, int num_items) {
  for (int w = blockIdx.x; w < num_items; w += gridDim.x) {
    const Tile t = items[w];
    const MatInfo mi = info[t.mat];
    const int k = mi.k;
    float* Qb = Q + mi.a_off + (int64_t)t.blk * k * k;
    for (int64_t e = threadIdx.x; e < (int64_t)k * k; e += kThreads)
      Qb[e] = ((e / k) == (e % k)) ? 1.f : 0.f;
    for (int j = threadIdx.x; j < k; j += kThreads) lam[mi.lam_off + (int64_t)t.blk * k + j] = 0.f;
  }
}

}  // namespace

cudaError_t launch_check(const CheckArgs& a, int grid, cudaStream_t s) {
  if (a.num_tiles <= 0) return cudaSuccess;
  check_bases_kernel<<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_init_bases(float* Q, float* lam, const MatInfo* info, const Tile* items,
                              int num_items, int grid, cudaStream_t s) {
  if (num_items <= 0) return cudaSuccess;
  init_bases_kernel<<<grid, kThreads, 0, s>>>(Q, lam, info, items, num_items);
  return cudaGetLastError();
}

}  // namespace dobb
