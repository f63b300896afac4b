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

// Four consecutive activations of one token (the caller checks alignment).
template <typename XT>
__device__ __forceinline__ void load4x(const XT* p, float (&v)[4]);
template <>
__device__ __forceinline__ void load4x<float>(const float* p, float (&v)[4]) {
  const float4 t = *reinterpret_cast<const float4*>(p);
  v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
}
template <>
__device__ __forceinline__ void load4x<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[4]) {
  const uint2 t = *reinterpret_cast<const uint2*>(p);
  v[0] = __uint_as_float(t.x << 16);
  v[1] = __uint_as_float(t.x & 0xFFFF0000u);
  v[2] = __uint_as_float(t.y << 16);
  v[3] = __uint_as_float(t.y & 0xFFFF0000u);
}

// One 64 x 64 output tile per CTA iteration.  Tokens are staged 32 at a time
// through shared memory; the next stage is loaded into registers (four
// consecutive activations per load where the rows allow it) while the
// current one is multiplied.
template <typename XT>
__global__ void __launch_bounds__(kThreads)
syrk_ema_kernel(const __grid_constant__ AccArgs a) {
  __shared__ __align__(16) float xs[2][kKT][kT + 4];
  __shared__ __align__(16) float ys[2][kKT][kT + 4];
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  // each thread moves two groups of four of each operand per stage:
  // token r = e / 16, columns 4 (e % 16) ... + 3, e = tid + 256 u
  constexpr int kGroups = kKT * kT / (4 * kThreads);
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
    const bool diag = t.a == t.b;
    const int64_t ci = (int64_t)t.blk * k + i0, cj = (int64_t)t.blk * k + j0;
    const bool vec = (n % 4 == 0) && (k % 4 == 0) &&
                     (reinterpret_cast<uintptr_t>(X) % (4 * sizeof(XT)) == 0);
    float acc[4][4];
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[p][q] = 0.f;
    int bad = 0;
    float rx[kGroups][4], ry[kGroups][4];
    auto gload = [&](int64_t t0) {
#pragma unroll
      for (int u = 0; u < kGroups; ++u) {
        const int e = tid + u * kThreads;
        const int r = e / (kT / 4), c = 4 * (e % (kT / 4));
        const int64_t tok = t0 + r;
#pragma unroll
        for (int z = 0; z < 4; ++z) rx[u][z] = ry[u][z] = 0.f;
        if (tok < N) {
          const XT* row = X + tok * n;
          if (vec && i0 + c + 3 < k) {
            load4x(row + ci + c, rx[u]);
          } else {
#pragma unroll
            for (int z = 0; z < 4; ++z)
              if (i0 + c + z < k) rx[u][z] = load_f32(row + ci + c + z);
          }
          if (!diag) {
            if (vec && j0 + c + 3 < k) {
              load4x(row + cj + c, ry[u]);
            } else {
#pragma unroll
              for (int z = 0; z < 4; ++z)
                if (j0 + c + z < k) ry[u][z] = load_f32(row + cj + c + z);
            }
          }
        }
      }
    };
    auto sstore = [&](int buf) {
#pragma unroll
      for (int u = 0; u < kGroups; ++u) {
        const int e = tid + u * kThreads;
        const int r = e / (kT / 4), c = 4 * (e % (kT / 4));
#pragma unroll
        for (int z = 0; z < 4; ++z) bad |= !isfinite(rx[u][z]) || !isfinite(ry[u][z]);
        *reinterpret_cast<float4*>(&xs[buf][r][c]) = make_float4(rx[u][0], rx[u][1], rx[u][2], rx[u][3]);
        if (!diag)
          *reinterpret_cast<float4*>(&ys[buf][r][c]) = make_float4(ry[u][0], ry[u][1], ry[u][2], ry[u][3]);
      }
    };
    const int64_t nst = (N + kKT - 1) / kKT;
    gload(0);
    sstore(0);
    __syncthreads();
    for (int64_t st = 0; st < nst; ++st) {
      const int buf = (int)(st & 1);
      if (st + 1 < nst) gload((st + 1) * kKT);
      const float(*xa)[kT + 4] = xs[buf];
      const float(*xb)[kT + 4] = diag ? xs[buf] : ys[buf];
      // two-level sum: the stage's 32 products, then the running total
      float part[4][4];
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) part[p][q] = 0.f;
#pragma unroll 8
      for (int r = 0; r < kKT; ++r) {
        const float4 av = *reinterpret_cast<const float4*>(&xa[r][ty * 4]);
        const float4 bv = *reinterpret_cast<const float4*>(&xb[r][tx * 4]);
        const float a4[4] = {av.x, av.y, av.z, av.w};
        const float b4[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
        for (int p = 0; p < 4; ++p)
#pragma unroll
          for (int q = 0; q < 4; ++q) part[p][q] = fmaf(a4[p], b4[q], part[p][q]);
      }
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[p][q] += part[p][q];
      if (st + 1 < nst) sstore(buf ^ 1);
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
