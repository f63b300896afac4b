// Grouped update kernel, FP32 FFMA version (reference-precision path for
// every block width, the path for widths the tensor-core kernel does not
// cover, and the path of the column-l2 normalisation).  For one tile of TM
// rows of one column block b of one matrix:
//
//   M <- beta1 M + G                      (momentum, written back to HBM)
//   C_b = M_b Q_b ; S_b = N(C_b)          (project, normalise: S in smem)
//   U_b = S_b Q_b^T ; W <- W - lr s U_b   (reconstruct, apply)
//
// "Dobb", Abstract (project momentum into the block bases, sign-normalise the
// coefficients, reconstruct the update) and Table 9 (update scale s).
// N is the sign (kModeSign), or for "Dobb-l2" (Table 11) the column l2
// normalisation S[:, j] = sqrt(m) C[:, j] / ||C[:, j]||, whose column norms run
// over all m rows: l2_norms_kernel first walks every row chunk of every
// (matrix, block), updating M and summing C^2 per column, and the update
// kernel then runs with kModeL2Apply (no momentum update, scaled coefficients).
#include "common.cuh"

namespace dobb {
namespace {

constexpr int kTM = 32;         // rows per tile (the basis is staged once per tile and pass)
constexpr int kThreads = 256;
constexpr int kRG = kTM / 4;    // row groups (4 rows per thread)
constexpr int kCG = kThreads / kRG;
constexpr int kNC = kCG * 4;    // output columns per pass (128)
constexpr int kKC = 32;         // reduction chunk
constexpr int kQS = kNC + 4;    // padded row of the Q stage
constexpr int kMS = kTM + 4;    // padded row of the M / S chunk, stored [reduction index][row]
constexpr int kL2MaxPass = 8;   // column passes of the l2 norm kernel

__host__ __device__ __forceinline__ int pad16(int k) { return (k + 15) & ~15; }

__host__ __device__ __forceinline__ size_t smem_bytes(int k) {
  return (size_t)4 * kTM * pad16(k)              // S (fp32)
         + (size_t)4 * (kKC * kQS + kKC * kMS);    // Q stage + M / S chunk
}

// One basis element as the update multiplies with it (bf16 basis storage:
// rounded once to bf16, "Dobb", Table 18).
__device__ __forceinline__ float basis_at(const float* Qb, int64_t idx, int basis_bf16) {
  const float v = Qb[idx];
  return basis_bf16 ? __bfloat162float(__float2bfloat16_rn(v)) : v;
}

// acc += A B over `len` reduction indices of one staged chunk: A = the M / S
// chunk ([index][row], rows rg 4 .. rg 4 + 3), B = the Q stage ([index][col],
// columns cg 4 .. cg 4 + 3): two 16-byte shared loads per 16 FMAs (the A
// load is a broadcast: a warp is one row group).
__device__ __forceinline__ void chunk_product(const float* Ac, const float* Bs, int len, int rg, int cg,
                                              float (&acc)[4][4]) {
  for (int ll = 0; ll < len; ++ll) {
    const float4 a4 = *reinterpret_cast<const float4*>(Ac + ll * kMS + rg * 4);
    const float4 b4 = *reinterpret_cast<const float4*>(Bs + ll * kQS + cg * 4);
    const float av[4] = {a4.x, a4.y, a4.z, a4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[p][q] = fmaf(av[p], bv[q], acc[p][q]);
  }
}

// acc[p][q] = C(rg 4 + p, jc + cg 4 + q) = sum_l M(row0 + rg 4 + p, l) Q(l, jc + cg 4 + q)
// for the rows of the tile (zero beyond `rows`).  Reads M from HBM.
__device__ __forceinline__ void project_pass(const float* Mg, const float* Qb, int64_t n,
                                             int64_t col0, int row0, int rows, int k, int jc,
                                             int basis_bf16, float* Qs, float* Mc,
                                             float (&acc)[4][4]) {
  const int tid = threadIdx.x, rg = tid / kCG, cg = tid % kCG;
#pragma unroll
  for (int p = 0; p < 4; ++p)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[p][q] = 0.f;
  for (int l0 = 0; l0 < k; l0 += kKC) {
    for (int e = tid; e < kKC * kNC; e += kThreads) {
      const int ll = e / kNC, cc = e % kNC;
      Qs[ll * kQS + cc] = (l0 + ll < k && jc + cc < k)
                              ? basis_at(Qb, (int64_t)(l0 + ll) * k + jc + cc, basis_bf16)
                              : 0.f;
    }
    for (int e = tid; e < kTM * kKC; e += kThreads) {
      const int r = e / kKC, ll = e % kKC;
      float v = 0.f;
      if (r < rows && l0 + ll < k) v = Mg[(int64_t)(row0 + r) * n + col0 + l0 + ll];
      Mc[ll * kMS + r] = v;
    }
    __syncthreads();
    chunk_product(Mc, Qs, min(kKC, k - l0), rg, cg, acc);
    __syncthreads();
  }
}

// Offset of element (r, c) of the problem in the caller's W / G / sign
// buffers: row-major m x n, or for an output-side ("Dobb-G") matrix the
// caller's n x m buffer seen transposed.
__device__ __forceinline__ int64_t pidx(const MatInfo& mi, int64_t r, int64_t c) {
  return mi.wt ? c * mi.m + r : r * mi.n + c;
}

// M <- beta1 M + G on the rows of one tile; returns this thread's non-finite flag.
template <typename PT>
__device__ __forceinline__ int momentum_tile(float* Mg, const PT* G, float beta1, const MatInfo& mi,
                                             int64_t col0, int row0, int rows, int k) {
  int bad = 0;
  for (int e = threadIdx.x; e < rows * k; e += kThreads) {
    const int r = e / k, c = e % k;
    const int64_t idx = (int64_t)(row0 + r) * mi.n + col0 + c;
    const float mn = fmaf(beta1, Mg[idx], load_f32(G + pidx(mi, row0 + r, col0 + c)));
    bad |= !isfinite(mn);
    Mg[idx] = mn;
  }
  return bad;
}

template <typename PT>
__global__ void __launch_bounds__(kThreads)
step_ffma_kernel(const __grid_constant__ StepArgs a) {
  extern __shared__ __align__(16) unsigned char smraw[];
  __shared__ float red[32];
  const int tid = threadIdx.x, rg = tid / kCG, cg = tid % kCG;
  const bool l2 = a.mode == kModeL2Apply;
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
    float* Ss = reinterpret_cast<float*>(smraw);
    float* Qs = Ss + kTM * kp;
    float* Mc = Qs + kKC * kQS;

    // momentum (the l2 apply pass finds it updated by the norm pass)
    const int bad = l2 ? 0 : momentum_tile(Mg, G, a.beta1, mi, col0, row0, rows, k);
    __syncthreads();

    // project + normalise
    const float* colsq = l2 ? a.colsq + mi.lam_off + (int64_t)t.blk * k : nullptr;
    const float sqm = sqrtf((float)mi.m);
    float c2 = 0.f;
    for (int jc = 0; jc < k; jc += kNC) {
      float acc[4][4];
      project_pass(Mg, Qb, n, col0, row0, rows, k, jc, a.basis_bf16, Qs, Mc, acc);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = jc + cg * 4 + q;
        if (j >= k) continue;
        float f = 0.f;
        if (l2) {
          const float cn = colsq[j];
          f = cn > 0.f ? sqm / sqrtf(cn) : 0.f;
        }
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int r = rg * 4 + p;
          const float sv = l2 ? acc[p][q] * f : sign_of(acc[p][q]);
          Ss[r * kp + j] = r < rows ? sv : 0.f;
          if (r < rows) {
            c2 = fmaf(acc[p][q], acc[p][q], c2);
            if (Sout) Sout[pidx(mi, row0 + r, col0 + j)] = (int8_t)sign_of(acc[p][q]);
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
          Qs[jj * kQS + cc] = (lc + cc < k && j0 + jj < k)
                                  ? basis_at(Qb, (int64_t)(lc + cc) * k + j0 + jj, a.basis_bf16)
                                  : 0.f;
        }
        for (int e = tid; e < kTM * kKC; e += kThreads) {
          const int r = e / kKC, jj = e % kKC;
          Mc[jj * kMS + r] = (j0 + jj < k) ? Ss[r * kp + j0 + jj] : 0.f;
        }
        __syncthreads();
        chunk_product(Mc, Qs, min(kKC, k - j0), rg, cg, acc);
        __syncthreads();
      }
#pragma unroll
      for (int p = 0; p < 4; ++p) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int r = rg * 4 + p, l = lc + cg * 4 + q;
          if (r < rows && l < k) {
            const int64_t idx = pidx(mi, row0 + r, col0 + l);
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

// First pass of the column-l2 normalisation: one (matrix, block, row chunk)
// per item (Tile::a = first row, Tile::b = rows), over its rows in tiles of
// kTM: M <- beta1 M + G, C = M Q, and the sum of C^2 per column, kept per
// thread and added once per column and chunk into colsq (the eigenvalue
// region's layout: lam_off + blk k + j; zeroed before the launch).
template <typename PT>
__global__ void __launch_bounds__(kThreads)
l2_norms_kernel(const __grid_constant__ StepArgs a) {
  extern __shared__ __align__(16) unsigned char smraw[];
  const int tid = threadIdx.x, cg = tid % kCG;
  constexpr int kMaxPass = kL2MaxPass;  // k <= kMaxPass kNC = 1024 (the widest block in this mode)
  for (int w = blockIdx.x; w < a.num_tiles; w += gridDim.x) {
    const Tile t = a.tiles[w];
    const int slot = t.mat - a.mat_base;
    const MatInfo mi = a.info[t.mat];
    const int k = mi.k, kp = pad16(k);
    const int64_t n = mi.n;
    const float* Qb = a.Q + mi.a_off + (int64_t)t.blk * k * k;
    const PT* G = static_cast<const PT*>(a.G[slot]);
    float* Mg = a.M + mi.m_off;
    const int64_t col0 = (int64_t)t.blk * k;
    float* Ss = reinterpret_cast<float*>(smraw);
    float* Qs = Ss + kTM * kp;
    float* Mc = Qs + kKC * kQS;
    float sq[kMaxPass][4];
#pragma unroll
    for (int p = 0; p < kMaxPass; ++p)
#pragma unroll
      for (int q = 0; q < 4; ++q) sq[p][q] = 0.f;
    int bad = 0;
    const int rend = (int)min((int64_t)t.a + t.b, mi.m);
    for (int row0 = t.a; row0 < rend; row0 += kTM) {
      const int rows = rend - row0 < kTM ? rend - row0 : kTM;
      bad |= momentum_tile(Mg, G, a.beta1, mi, col0, row0, rows, k);
      __syncthreads();
#pragma unroll
      for (int pass = 0; pass < kMaxPass; ++pass) {
        const int jc = pass * kNC;
        if (jc >= k) break;
        float acc[4][4];
        project_pass(Mg, Qb, n, col0, row0, rows, k, jc, a.basis_bf16, Qs, Mc, acc);
#pragma unroll
        for (int p = 0; p < 4; ++p)
#pragma unroll
          for (int q = 0; q < 4; ++q) sq[pass][q] = fmaf(acc[p][q], acc[p][q], sq[pass][q]);
      }
    }
    // column totals over the row groups, then one store per column
    float* colbuf = Ss;  // kRG x k partial sums
    __syncthreads();
#pragma unroll
    for (int pass = 0; pass < kMaxPass; ++pass)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = pass * kNC + cg * 4 + q;
        if (j < k) colbuf[(tid / kCG) * kp + j] = sq[pass][q];
      }
    __syncthreads();
    for (int j = tid; j < k; j += kThreads) {
      float s = 0.f;
#pragma unroll
      for (int r = 0; r < kRG; ++r) s += colbuf[r * kp + j];
      atomicAdd(a.colsq + mi.lam_off + (int64_t)t.blk * k + j, s);
    }
    const int any_bad = __syncthreads_or(bad);
    if (tid == 0 && any_bad) atomicOr(a.flags + mi.blk0 + t.blk, (uint32_t)DOBB_FLAG_NONFINITE_G);
    __syncthreads();
  }
}

}  // namespace

int step_rows_per_tile() { return kTM; }
size_t step_smem_for(int k) { return smem_bytes(k); }
int l2_max_k() { return kL2MaxPass * kNC; }

cudaError_t configure_step(size_t smem_limit) {
  cudaError_t e = cudaFuncSetAttribute(step_ffma_kernel<float>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_limit);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(step_ffma_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_limit);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(l2_norms_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_limit);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(l2_norms_kernel<__nv_bfloat16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_limit);
  return e;
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

cudaError_t launch_l2_norms(const StepArgs& a, int param_dtype, int grid, size_t smem,
                            cudaStream_t s) {
  if (a.num_tiles <= 0) return cudaSuccess;
  if (param_dtype == kBF16)
    l2_norms_kernel<__nv_bfloat16><<<grid, kThreads, smem, s>>>(a);
  else
    l2_norms_kernel<float><<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dobb
