// Block eigendecomposition for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc at all: inference or
// embedded runtimes whose memory is fully reserved up front by an arena they
// do not control, and plugins hosted by frameworks that forbid allocations
// outside their own allocator.  They still want the exact block
// eigendecomposition the optimizer refresh computes.  dobb_eigh_noalloc runs
// the same eigensolver kernel (restarted Rayleigh-Ritz two-sided Jacobi,
// started from the identity) on caller-provided inputs and outputs and keeps
// its working memory in file-scope __device__ arrays of a fixed maximum size,
// which every GPU that loads the library holds until the process exits.
//
// The arrays are shared by every call: calls whose work overlaps on the GPU
// (different streams, or different host threads) race.  Set-up per device
// (cudaGetSymbolAddress of each array, kernel attributes) happens on the
// first call on that device, under a lock.
#include <algorithm>
#include <mutex>
#include <string>

#include "dobb_internal.cuh"

namespace dobb {
namespace {

// fp32 scratch: three k x k matrices per block (the rotated moment, the
// basis and a work matrix), 16 MiB in total.
constexpr size_t kNoAllocScratchFloats = (size_t)4 << 20;
constexpr int kNoAllocMaxBlocks = 4096;
constexpr int kNoAllocMaxK = 1024;
constexpr int kMaxDevices = 64;

__device__ __align__(256) float g_scratch[kNoAllocScratchFloats];
__device__ __align__(256) MatInfo g_info[1];
__device__ __align__(256) Tile g_items[kNoAllocMaxBlocks];
__device__ __align__(256) uint32_t g_flags[kNoAllocMaxBlocks];
__device__ __align__(256) float g_stats[4 * kNoAllocMaxBlocks];

struct DevPtrs {
  bool ready = false;
  float* scratch = nullptr;
  MatInfo* info = nullptr;
  Tile* items = nullptr;
  uint32_t* flags = nullptr;
  float* stats = nullptr;
  int sm_count = 1;
  size_t smem_limit = 0, smem_per_sm = 0;
};

std::mutex g_mu;
DevPtrs g_dev[kMaxDevices];

thread_local std::string g_noalloc_err;

dobb_status noalloc_fail(dobb_status st, const char* msg, cudaError_t e = cudaSuccess) {
  g_noalloc_err = msg;
  if (e != cudaSuccess) {
    g_noalloc_err += ": ";
    g_noalloc_err += cudaGetErrorString(e);
  }
  return st;
}

// Device addresses of the file-scope arrays for the current device.  The
// host-side names of __device__ arrays are stand-ins, not device addresses,
// so every pointer handed to a kernel comes from cudaGetSymbolAddress.
dobb_status setup_device(int dev, DevPtrs** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  DevPtrs& d = g_dev[dev];
  if (!d.ready) {
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.scratch), g_scratch);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.info), g_info);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.items), g_items);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.flags), g_flags);
    if (e == cudaSuccess) e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.stats), g_stats);
    if (e != cudaSuccess) return noalloc_fail(DOBB_ERR_CUDA, "cudaGetSymbolAddress failed", e);
    int optin = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess)
      e = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (e != cudaSuccess) return noalloc_fail(DOBB_ERR_CUDA, "device query failed", e);
    d.smem_limit = (size_t)optin - 2048;
    d.smem_per_sm = (size_t)per_sm;
    e = configure_jacobi(d.smem_limit);
    if (e != cudaSuccess) return noalloc_fail(DOBB_ERR_CUDA, "kernel configuration failed", e);
    d.ready = true;
  }
  *out = &d;
  return DOBB_OK;
}

}  // namespace

const char* noalloc_last_error() { return g_noalloc_err.c_str(); }

}  // namespace dobb

using namespace dobb;

extern "C" dobb_status dobb_eigh_noalloc(const float* A_dev, float* Q_dev, float* lam_dev, int k,
                                         int count, int max_sweeps, uint32_t* flags_host,
                                         void* stream) {
  g_noalloc_err.clear();
  if (!A_dev || !Q_dev || !lam_dev) return noalloc_fail(DOBB_ERR_INVALID_ARG, "NULL pointer argument");
  if (k < 1 || k > kNoAllocMaxK) return noalloc_fail(DOBB_ERR_INVALID_ARG, "k must lie in [1, 1024]");
  if (count < 0) return noalloc_fail(DOBB_ERR_INVALID_ARG, "count must be >= 0");
  if (count > kNoAllocMaxBlocks)
    return noalloc_fail(DOBB_ERR_INVALID_ARG, "count exceeds the 4096 blocks the fixed work list holds");
  if ((size_t)count * 3 * (size_t)k * k > kNoAllocScratchFloats)
    return noalloc_fail(DOBB_ERR_INVALID_ARG,
                        "count * 3 * k * k exceeds the 4 Mi-float (16 MiB) fixed scratch array");
  if (max_sweeps < 1) return noalloc_fail(DOBB_ERR_INVALID_ARG, "max_sweeps must be >= 1");
  {
    // the basis is set to the identity before the solver reads A: outputs
    // that overlap the input would corrupt it
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(A_dev);
    const uintptr_t a1 = a0 + sizeof(float) * (size_t)count * k * k;
    const uintptr_t q0 = reinterpret_cast<uintptr_t>(Q_dev);
    const uintptr_t q1 = q0 + sizeof(float) * (size_t)count * k * k;
    const uintptr_t l0 = reinterpret_cast<uintptr_t>(lam_dev);
    const uintptr_t l1 = l0 + sizeof(float) * (size_t)count * k;
    if (count > 0 && ((q0 < a1 && a0 < q1) || (l0 < a1 && a0 < l1)))
      return noalloc_fail(DOBB_ERR_INVALID_ARG, "Q_dev and lam_dev must not overlap A_dev");
  }
  if (count == 0) return DOBB_OK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return noalloc_fail(DOBB_ERR_CUDA, "cudaGetDevice failed", e);
  if (dev < 0 || dev >= kMaxDevices) return noalloc_fail(DOBB_ERR_UNSUPPORTED, "device index too large");
  DevPtrs* d = nullptr;
  dobb_status st = setup_device(dev, &d);
  if (st != DOBB_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // one matrix descriptor covering `count` blocks of width k laid out back to back
  MatInfo mi{};
  mi.m = 1;
  mi.n = (int64_t)k * count;
  mi.k = k;
  mi.B = count;
  mi.blk0 = 0;
  Tile items[256];
  e = cudaMemcpyAsync(d->info, &mi, sizeof(MatInfo), cudaMemcpyHostToDevice, s);
  for (int b0 = 0; b0 < count && e == cudaSuccess; b0 += 256) {
    const int nb = std::min(256, count - b0);
    for (int i = 0; i < nb; ++i) items[i] = Tile{0, b0 + i, 0, 0};
    // pageable source: the copy is staged before cudaMemcpyAsync returns
    e = cudaMemcpyAsync(d->items + b0, items, sizeof(Tile) * nb, cudaMemcpyHostToDevice, s);
  }
  // the arrays keep the previous call's contents: clear the flags
  if (e == cudaSuccess) e = cudaMemsetAsync(d->flags, 0, sizeof(uint32_t) * count, s);
  if (e != cudaSuccess) return noalloc_fail(DOBB_ERR_CUDA, "staging the work list failed", e);

  // cold start: Q = I, Lambda = 0
  const int gi = std::max(1, std::min(count, d->sm_count * 4));
  e = launch_init_bases(Q_dev, lam_dev, d->info, d->items, count, gi, s);
  if (e != cudaSuccess) return noalloc_fail(DOBB_ERR_CUDA, "basis initialisation launch failed", e);

  EigArgs a{};
  a.info = d->info;
  a.tiles = d->items;
  a.num_tiles = count;
  a.max_sweeps = max_sweeps;
  a.A = A_dev;
  a.Q = Q_dev;
  a.lam = lam_dev;
  a.scratch = d->scratch;
  a.flags = d->flags;
  a.stats = d->stats;
  a.tol = 0.f;
  const size_t half = d->smem_per_sm / 2 > 2048 ? d->smem_per_sm / 2 - 2048 : 0;
  size_t smem = jacobi_smem_for(k, half);
  if (smem == 0) smem = jacobi_smem_for(k, d->smem_limit);
  if (smem == 0) return noalloc_fail(DOBB_ERR_UNSUPPORTED, "block width exceeds the eigensolver's shared memory");
  const int by_smem = std::max(1, (int)(d->smem_per_sm / (smem + 1024)));
  const int g = std::max(1, std::min(count, d->sm_count * std::min(jacobi_ctas_per_sm(), by_smem)));
  e = launch_jacobi(a, g, smem, s);
  if (e != cudaSuccess) return noalloc_fail(DOBB_ERR_CUDA, "eigensolver launch failed", e);
  if (flags_host) {
    e = cudaMemcpyAsync(flags_host, d->flags, sizeof(uint32_t) * count, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return noalloc_fail(DOBB_ERR_CUDA, "reading the flags failed", e);
  }
  return DOBB_OK;
}

extern "C" const char* dobb_eigh_noalloc_last_error(void) { return dobb::noalloc_last_error(); }
