// Block second-moment accumulation with fused EMA:
//   A_b <- beta2 A_b + (1 - beta2) X_b^T X_b / N
// ("Dobb", Abstract: diagonal blocks of the input-activation second moment;
// Table 3 caption: n^2/B entries per matrix).  One grouped launch covers
// every (matrix, block, 64 x 64 output tile) of the upper triangle; the tile
// writes both (i, j) and (j, i) so A stays exactly symmetric.
#include "common.cuh"

namespace dobb {
namespace {

constexpr int kT = 64;       // output tile edge
constexpr int kKT = 32;      // tokens per smem stage
constexpr int kThreads = 256;

template <typename XT>
__global__ void __launch_bounds__(kThreads)
syrk_ema_kernel(const __grid_constant__ AccArgs a) {
  __shared__ float xi[kKT][kT + 4];
  __shared__ float xj[kKT][kT + 4];
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  for (int w = blockIdx.x; w < a.num_tiles; w += gridDim.x) {
    const Tile t = a.tiles[w];
    const int slot = t.mat - a.mat_base;
    const XT* X = static_cast<const XT*>(a.X[slot]);
    const int64_t N = a.N[slot];
    if (X == nullptr || N <= 0) continue;  // uniform over the CTA
    const MatInfo mi = a.info[t.mat];
    const int k = mi.k;
    const int64_t n = mi.n;
    const int i0 = t.a * kT, j0 = t.b * kT;
    const int64_t ci = (int64_t)t.blk * k + i0, cj = (int64_t)t.blk * k + j0;
    float acc[4][4];
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[p][q] = 0.f;
    int bad = 0;
    for (int64_t t0 = 0; t0 < N; t0 += kKT) {
      for (int e = tid; e < kKT * kT; e += kThreads) {
        const int r = e / kT, c = e % kT;
        const int64_t tok = t0 + r;
        float vi = 0.f, vj = 0.f;
        if (tok < N) {
          const XT* row = X + tok * n;
          if (i0 + c < k) vi = load_f32(row + ci + c);
          if (j0 + c < k) vj = load_f32(row + cj + c);
        }
        bad |= !(isfinite(vi) && isfinite(vj));
        xi[r][c] = vi;
        xj[r][c] = vj;
      }
      __syncthreads();
      // two-level sum: the stage's 32 products, then the running total
      float part[4][4];
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) part[p][q] = 0.f;
#pragma unroll 8
      for (int r = 0; r < kKT; ++r) {
        float av[4], bv[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          av[q] = xi[r][ty * 4 + q];
          bv[q] = xj[r][tx * 4 + q];
        }
#pragma unroll
        for (int p = 0; p < 4; ++p)
#pragma unroll
          for (int q = 0; q < 4; ++q) part[p][q] = fmaf(av[p], bv[q], part[p][q]);
      }
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[p][q] += part[p][q];
      __syncthreads();
    }
    if (__syncthreads_or(bad) && tid == 0) atomicOr(a.flags + mi.blk0 + t.blk, 1u);
    const float c1 = (1.f - a.beta2) / (float)N;
    float* Ab = a.A + mi.a_off + (int64_t)t.blk * k * k;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = i0 + ty * 4 + p, j = j0 + tx * 4 + q;
        if (i < k && j < k) {
          const float v = fmaf(a.beta2, Ab[(int64_t)i * k + j], c1 * acc[p][q]);
          Ab[(int64_t)i * k + j] = v;
          if (t.a != t.b) Ab[(int64_t)j * k + i] = v;
        }
      }
    }
  }
}

}  // namespace

int syrk_tile() { return kT; }

cudaError_t launch_syrk_ema(const AccArgs& a, int act_dtype, int grid, cudaStream_t s) {
  if (a.num_tiles <= 0) return cudaSuccess;
  if (act_dtype == kBF16)
    syrk_ema_kernel<__nv_bfloat16><<<grid, kThreads, 0, s>>>(a);
  else
    syrk_ema_kernel<float><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dobb
