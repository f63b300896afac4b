// Grouped update kernel, FP32 FFMA version (reference-precision path for
// every block width, and the path for widths the tensor-core kernel does not
// cover).  For one tile of TM rows of one column block b of one matrix:
//
//   M <- beta1 M + G                      (momentum, written back to HBM)
//   C_b = M_b Q_b ; S_b = sign(C_b)       (project, sign: S kept in smem)
//   U_b = S_b Q_b^T ; W <- W - lr s U_b   (reconstruct, apply)
//
// "Dobb", Abstract (project momentum into the block bases, sign-normalise the
// coefficients, reconstruct the update) and Table 9 (update scale s).
#include "common.cuh"

namespace dobb {
namespace {

constexpr int kTM = 16;         // rows per tile
constexpr int kThreads = 256;
constexpr int kRG = kTM / 4;    // row groups (4 rows per thread)
constexpr int kCG = kThreads / kRG;
constexpr int kNC = kCG * 4;    // output columns per pass (256)
constexpr int kKC = 32;         // reduction chunk
constexpr int kQS = kNC + 4;    // padded row of the Q stage

__host__ __device__ __forceinline__ int pad16(int k) { return (k + 15) & ~15; }

__host__ __device__ __forceinline__ size_t smem_bytes(int k) {
  return (size_t)kTM * pad16(k)                      // S (int8)
         + (size_t)4 * (kKC * kQS + kTM * (kKC + 1));  // Q stage + M / S chunk
}

template <typename PT>
__global__ void __launch_bounds__(kThreads)
step_ffma_kernel(const __grid_constant__ StepArgs a) {
  extern __shared__ __align__(16) unsigned char smraw[];
  __shared__ float red[32];
  const int tid = threadIdx.x, rg = tid / kCG, cg = tid % kCG;
  for (int w = blockIdx.x; w < a.num_tiles; w += gridDim.x) {
    const Tile t = a.tiles[w];
    const int slot = t.mat - a.mat_base;
    const MatInfo mi = a.info[t.mat];
    const int k = mi.k, kp = pad16(k);
    const int64_t n = mi.n;
    const int row0 = t.a;
    const int rows = (int)((mi.m - row0) < kTM ? (mi.m - row0) : kTM);
    const float* Qb = a.Q + mi.a_off + (int64_t)t.blk * k * k;
    PT* W = static_cast<PT*>(a.W[slot]);
    const PT* G = static_cast<const PT*>(a.G[slot]);
    int8_t* Sout = a.S[slot];
    float* Mg = a.M + mi.m_off;
    const int64_t col0 = (int64_t)t.blk * k;
    int8_t* Ss = reinterpret_cast<int8_t*>(smraw);
    float* Qs = reinterpret_cast<float*>(smraw + (size_t)kTM * kp);
    float* Mc = Qs + kKC * kQS;

    // momentum
    int bad = 0;
    for (int e = tid; e < rows * k; e += kThreads) {
      const int r = e / k, c = e % k;
      const int64_t idx = (int64_t)(row0 + r) * n + col0 + c;
      const float mn = fmaf(a.beta1, Mg[idx], load_f32(G + idx));
      bad |= !isfinite(mn);
      Mg[idx] = mn;
    }
    __syncthreads();

    // project + sign
    float c2 = 0.f;
    for (int jc = 0; jc < k; jc += kNC) {
      float acc[4][4];
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[p][q] = 0.f;
      for (int l0 = 0; l0 < k; l0 += kKC) {
        for (int e = tid; e < kKC * kNC; e += kThreads) {
          const int ll = e / kNC, cc = e % kNC;
          float v = 0.f;
          if (l0 + ll < k && jc + cc < k) v = Qb[(int64_t)(l0 + ll) * k + jc + cc];
          if (a.basis_bf16) v = __bfloat162float(__float2bfloat16_rn(v));
          Qs[ll * kQS + cc] = v;
        }
        for (int e = tid; e < kTM * kKC; e += kThreads) {
          const int r = e / kKC, ll = e % kKC;
          float v = 0.f;
          if (r < rows && l0 + ll < k) v = Mg[(int64_t)(row0 + r) * n + col0 + l0 + ll];
          Mc[r * (kKC + 1) + ll] = v;
        }
        __syncthreads();
        const int lmax = min(kKC, k - l0);
        for (int ll = 0; ll < lmax; ++ll) {
          float av[4], bv[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) av[p] = Mc[(rg * 4 + p) * (kKC + 1) + ll];
#pragma unroll
          for (int q = 0; q < 4; ++q) bv[q] = Qs[ll * kQS + cg * 4 + q];
#pragma unroll
          for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[p][q] = fmaf(av[p], bv[q], acc[p][q]);
        }
        __syncthreads();
      }
#pragma unroll
      for (int p = 0; p < 4; ++p) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int r = rg * 4 + p, j = jc + cg * 4 + q;
          if (j < k) {
            const float sg = sign_of(acc[p][q]);
            Ss[r * kp + j] = (int8_t)sg;
            if (r < rows) {
              c2 = fmaf(acc[p][q], acc[p][q], c2);
              if (Sout) Sout[(int64_t)(row0 + r) * n + col0 + j] = (int8_t)sg;
            }
          }
        }
      }
    }
    __syncthreads();

    // reconstruct + apply
    float u2 = 0.f;
    for (int lc = 0; lc < k; lc += kNC) {
      float acc[4][4];
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[p][q] = 0.f;
      for (int j0 = 0; j0 < k; j0 += kKC) {
        for (int e = tid; e < kKC * kNC; e += kThreads) {
          const int cc = e / kKC, jj = e % kKC;
          float v = 0.f;
          if (lc + cc < k && j0 + jj < k) v = Qb[(int64_t)(lc + cc) * k + j0 + jj];
          if (a.basis_bf16) v = __bfloat162float(__float2bfloat16_rn(v));
          Qs[jj * kQS + cc] = v;
        }
        for (int e = tid; e < kTM * kKC; e += kThreads) {
          const int r = e / kKC, jj = e % kKC;
          Mc[r * (kKC + 1) + jj] = (j0 + jj < k) ? (float)Ss[r * kp + j0 + jj] : 0.f;
        }
        __syncthreads();
        const int jmax = min(kKC, k - j0);
        for (int jj = 0; jj < jmax; ++jj) {
          float av[4], bv[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) av[p] = Mc[(rg * 4 + p) * (kKC + 1) + jj];
#pragma unroll
          for (int q = 0; q < 4; ++q) bv[q] = Qs[jj * kQS + cg * 4 + q];
#pragma unroll
          for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[p][q] = fmaf(av[p], bv[q], acc[p][q]);
        }
        __syncthreads();
      }
#pragma unroll
      for (int p = 0; p < 4; ++p) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int r = rg * 4 + p, l = lc + cg * 4 + q;
          if (r < rows && l < k) {
            const int64_t idx = (int64_t)(row0 + r) * n + col0 + l;
            store_f32(W + idx, fmaf(-a.lr_s, acc[p][q], load_f32(W + idx)));
            u2 = fmaf(acc[p][q], acc[p][q], u2);
          }
        }
      }
    }
    const float tu = block_sum(u2, red);
    const float tc = block_sum(c2, red);
    const int any_bad = __syncthreads_or(bad);
    if (tid == 0) {
      float* st = a.stats + 4 * (int64_t)(mi.blk0 + t.blk);
      atomicAdd(st + 0, tu);
      atomicAdd(st + 1, tc);
      if (any_bad) atomicOr(a.flags + mi.blk0 + t.blk, (uint32_t)DOBB_FLAG_NONFINITE_G);
    }
    __syncthreads();
  }
}

}  // namespace

int step_rows_per_tile() { return kTM; }
size_t step_smem_for(int k) { return smem_bytes(k); }

cudaError_t configure_step(size_t smem_limit) {
  cudaError_t e = cudaFuncSetAttribute(step_ffma_kernel<float>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_limit);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(step_ffma_kernel<__nv_bfloat16>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_limit);
}

cudaError_t launch_step_ffma(const StepArgs& a, int param_dtype, int grid, size_t smem,
                             cudaStream_t s) {
  if (a.num_tiles <= 0) return cudaSuccess;
  if (param_dtype == kBF16)
    step_ffma_kernel<__nv_bfloat16><<<grid, kThreads, smem, s>>>(a);
  else
    step_ffma_kernel<float><<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dobb
