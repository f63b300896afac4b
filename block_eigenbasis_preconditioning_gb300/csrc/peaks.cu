// Throughput probes that give the roofline denominators of the kernels in
// this library, measured on the GPU that runs them: FP32 FFMA (the
// eigensolvers' products and rotations), TF32 and BF16 on the tcgen05
// tensor cores (the update's projection and reconstruction, the moments),
// and TF32 on the warp-level mma.sync path.  Each probe is one launch of one
// CTA per SM running long independent chains of the instruction; the flop
// count is exact (2 per multiply-add), the time comes from CUDA events around
// the launch.  Every value a probe computes is written to the caller's buffer
// so that no work can be elided; the values themselves are meaningless.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace dobb {
namespace {

using namespace ptx;

// ------------------------------------------------------------------- FFMA
constexpr int kFfmaThreads = 512;
constexpr int kFfmaChains = 8;

__global__ void __launch_bounds__(kFfmaThreads) ffma_probe(float* out, int iters, float seed) {
  float v[kFfmaChains];
#pragma unroll
  for (int c = 0; c < kFfmaChains; ++c) v[c] = seed + 1e-3f * (threadIdx.x + c);
  const float a = 0.999f, b = 1e-4f;
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int u = 0; u < 16; ++u)
#pragma unroll
      for (int c = 0; c < kFfmaChains; ++c) v[c] = fmaf(v[c], a, b);
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kFfmaChains; ++c) s += v[c];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// ------------------------------------------------------- mma.sync (TF32)
constexpr int kMmaThreads = 256;
constexpr int kMmaChains = 4;

__global__ void __launch_bounds__(kMmaThreads) mma_sync_tf32_probe(float* out, int iters) {
  uint32_t a[4], b[2];
  const uint32_t lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = __float_as_uint(tf32_rna(1e-3f * (lane + i)));
#pragma unroll
  for (int i = 0; i < 2; ++i) b[i] = __float_as_uint(tf32_rna(1e-3f * (lane + 2 * i)));
  float d[kMmaChains][4];
#pragma unroll
  for (int c = 0; c < kMmaChains; ++c)
#pragma unroll
    for (int i = 0; i < 4; ++i) d[c][i] = 0.f;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int c = 0; c < kMmaChains; ++c)
      asm volatile(
          "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
          "{%8,%9}, {%0,%1,%2,%3};"
          : "+f"(d[c][0]), "+f"(d[c][1]), "+f"(d[c][2]), "+f"(d[c][3])
          : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  }
  float s = 0.f;
#pragma unroll
  for (int c = 0; c < kMmaChains; ++c) s += d[c][0] + d[c][1] + d[c][2] + d[c][3];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

// ---------------------------------------------------- tcgen05 (TF32, BF16)
// One elected thread issues back-to-back 128 x 256 MMAs from one A tile
// (128 rows of 128 bytes, 128-byte swizzle) and one B tile (256 rows of 32
// bytes, 32-byte swizzle) into a TMEM accumulator of 256 columns; the other
// threads wait on the commit barrier (bounded) and read the accumulator out.
constexpr int kTcThreads = 128;
constexpr int kTcABytes = 128 * 128;
constexpr int kTcBBytes = 256 * 32;

struct ProbeSmem {
  uint64_t done;
  uint32_t tmem;
  int ok;
};

template <int kFmt>  // 2: kind::tf32 (K = 8), 1: kind::f16 with bf16 inputs (K = 16)
__global__ void __launch_bounds__(kTcThreads, 1) tc_probe(float* out, int iters, uint32_t* err) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  unsigned char* a_tile = base;
  unsigned char* b_tile = base + kTcABytes;
  ProbeSmem* sh = reinterpret_cast<ProbeSmem*>(b_tile + kTcBBytes);
  const int warp = threadIdx.x >> 5;
  // operands: small finite values in either format
  for (int i = threadIdx.x; i < (kTcABytes + kTcBBytes) / 4; i += blockDim.x) {
    const float f = tf32_rna(1e-3f * (float)(i % 97));
    uint32_t w = __float_as_uint(f);
    if (kFmt == 1) w = (w & 0xFFFF0000u) | (w >> 16);
    reinterpret_cast<uint32_t*>(base)[i] = w;
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(&sh->done, 1);
    sh->ok = 1;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&sh->tmem, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem;
  if (threadIdx.x == 0) {
    const uint32_t id = instr_desc(kFmt, 128, 256);
    const uint32_t a0 = smem_u32(a_tile), b0 = smem_u32(b_tile);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint64_t da = smem_desc(a0 + 32 * s, 16, 1024, kSw128);
        const uint64_t db = smem_desc(b0, 16, 256, kSw32);
        if (kFmt == 2)
          mma_tf32_ss(tmem, da, db, id, (it | s) ? 1u : 0u);
        else
          mma_f16_ss(tmem, da, db, id, (it | s) ? 1u : 0u);
      }
    }
    tc_commit(&sh->done);
  }
  __syncwarp();
  bool ok = mbar_wait(&sh->done, 0, 4000000000ull);
  if (!__all_sync(0xffffffffu, ok)) {
    if ((threadIdx.x & 31) == 0) atomicOr(err, 1u);
    sh->ok = 0;
    // give the issued MMAs a second bounded wait before TMEM is released
    ok = mbar_wait(&sh->done, 0, 4000000000ull);
  }
  tc_fence_after();
  __syncthreads();
  if (sh->ok) {
    float v[32];
    tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16), v);
    tmem_wait_ld(v);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) s += v[i];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace
}  // namespace dobb

using namespace dobb;

extern "C" dobb_status dobb_peak_probe(int which, void* scratch_dev, size_t scratch_bytes, int iters,
                                       float* ms_out, double* flops_out, void* stream) {
  if (!scratch_dev || !ms_out || !flops_out || iters < 1 || which < 0 || which > 3)
    return DOBB_ERR_INVALID_ARG;
  int dev = 0, sms = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return DOBB_ERR_CUDA;
  const int threads = which == 0 ? kFfmaThreads : (which == 1 ? kMmaThreads : kTcThreads);
  // FFMA and mma.sync: 4 CTAs per SM; tcgen05: one per SM
  const int grid = which >= 2 ? sms : 4 * sms;
  // output floats + one error word
  const size_t need = sizeof(float) * (size_t)grid * threads + 256;
  if (scratch_bytes < need) return DOBB_ERR_INVALID_ARG;
  float* out = static_cast<float*>(scratch_dev);
  uint32_t* err = reinterpret_cast<uint32_t*>(static_cast<char*>(scratch_dev) + need - 256);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t tc_smem = 1024 + kTcABytes + kTcBBytes + sizeof(ProbeSmem);
  if (which >= 2) {
    if ((int)tc_smem > optin) return DOBB_ERR_UNSUPPORTED;
    cudaError_t e = cudaFuncSetAttribute(which == 2 ? tc_probe<2> : tc_probe<1>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem);
    if (e != cudaSuccess) return DOBB_ERR_CUDA;
  }
  if (cudaMemsetAsync(err, 0, 4, s) != cudaSuccess) return DOBB_ERR_CUDA;
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess) return DOBB_ERR_CUDA;
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaEventDestroy(e0);
    return DOBB_ERR_CUDA;
  }
  cudaEventRecord(e0, s);
  double flops = 0.0;
  switch (which) {
    case 0:
      ffma_probe<<<grid, threads, 0, s>>>(out, iters, 0.5f);
      flops = 2.0 * grid * threads * (double)iters * 16 * kFfmaChains;
      break;
    case 1:
      mma_sync_tf32_probe<<<grid, threads, 0, s>>>(out, iters);
      flops = 2.0 * 16 * 8 * 8 * (double)(grid * threads / 32) * iters * kMmaChains;
      break;
    case 2:
      tc_probe<2><<<grid, threads, tc_smem, s>>>(out, iters, err);
      flops = 2.0 * 128 * 256 * 8 * 4 * (double)iters * grid;
      break;
    default:
      tc_probe<1><<<grid, threads, tc_smem, s>>>(out, iters, err);
      flops = 2.0 * 128 * 256 * 16 * 4 * (double)iters * grid;
      break;
  }
  cudaEventRecord(e1, s);
  cudaError_t e = cudaEventSynchronize(e1);
  float ms = 0.f;
  if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
  uint32_t herr = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&herr, err, 4, cudaMemcpyDeviceToHost);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (e != cudaSuccess) return DOBB_ERR_CUDA;
  if (herr) return DOBB_ERR_CUDA;
  *ms_out = ms;
  *flops_out = flops;
  return DOBB_OK;
}

// ------------------------------------------------------------------
// Failure-detection self-test: the bounded mbarrier wait every tensor-core
// kernel of this library uses, on a barrier that nothing arrives on.  The
// wait gives up after `timeout_ns`, the kernel records DOBB error code 0x100
// in `err_dev` and returns; the context stays usable.
namespace dobb {
namespace {
__global__ void wait_timeout_kernel(uint32_t* err, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  const bool ok = ptx::mbar_wait(&bar, 0, timeout_ns);
  if (!ok && threadIdx.x == 0) atomicOr(err, 0x100u);
}
}  // namespace
}  // namespace dobb

extern "C" dobb_status dobb_selftest_wait_timeout(uint32_t* err_dev, uint64_t timeout_ns, void* stream) {
  if (!err_dev || timeout_ns == 0 || timeout_ns > 5000000000ull) return DOBB_ERR_INVALID_ARG;
  dobb::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(err_dev, timeout_ns);
  return cudaGetLastError() == cudaSuccess ? DOBB_OK : DOBB_ERR_CUDA;
}
