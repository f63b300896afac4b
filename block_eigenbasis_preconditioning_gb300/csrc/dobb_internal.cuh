// Internal declarations shared by the host API and the kernels of the Dobb
// optimizer step ("Dobb: Shard-Local Preconditioning in Block-Diagonal
// Eigenbases", arXiv 2610.39412).  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "dobb.h"

namespace dobb {

// Matrices addressed by one grouped launch; larger sets are split into
// several launches of at most this many matrices (pointer tables travel in
// the kernel parameter block).
constexpr int kMaxMatPerLaunch = 512;

// Largest block width k the library accepts.
constexpr int kMaxK = 8192;
// Largest block width of the tensor-core update kernel (TMEM holds C).
constexpr int kMaxTcK = 448;

// Per-matrix metadata, resident in device memory (built at dobb_create).
struct MatInfo {
  int64_t m, n;      // W is m x n
  int32_t k, B;      // block width, blocks per matrix
  int32_t blk0;      // global index of this matrix's block 0
  int32_t pad0;
  int64_t a_off;     // float offset of block 0 in the A (and Q) regions
  int64_t lam_off;   // float offset of block 0 in the Lambda region
  int64_t m_off;     // float offset of the matrix in the M region (16-float aligned)
  int64_t qp_off;    // byte offset of block 0's packed operand images
  int64_t qblk_bytes;  // bytes of one block's packed images
  int32_t tc;        // 1 if the tensor-core update kernel handles this matrix
  int32_t wt;        // 1: the caller's W, G (and signs) are stored transposed
                     //    (m_orig x n_orig row-major = this n x m problem's transpose)
};

// Extra arguments of the tensor-core update kernel.
struct TcArgs {
  const void* maps;        // one CUtensorMap (128 B) per matrix, for M
  const unsigned char* qpack;
  uint32_t* err;           // device error word (timeouts)
  int32_t bstage;          // bytes of one B stage
  int32_t nbstage;         // B stages (2 ... 16)
  int32_t npieces;         // basis operand pieces: 2 (fp32 basis: hi, lo) or 1 (bf16 basis)
  int32_t defer;           // 1: every block of the launch has kpN <= 128 (reconstructs deferred)
  int32_t nastage;         // momentum (A operand) stages (2 ... 4)
  int32_t rpieces;         // reconstruct basis pieces: 3 (fp32 basis: bf16 hi, lo, lo2) or 1
};

// One unit of grouped work: matrix, block and two phase-specific indices.
struct Tile {
  int32_t mat, blk, a, b;
};

enum DType : int { kF32 = 0, kBF16 = 1 };

struct AccArgs {
  const MatInfo* info;
  const Tile* tiles;
  int32_t num_tiles;
  int32_t mat_base;       // matrix index of pointer-table slot 0
  float* A;
  uint32_t* flags;
  float beta2;
  const void* X[kMaxMatPerLaunch];
  int64_t N[kMaxMatPerLaunch];
};

// Matrices per tensor-core accumulate launch (their X tensor maps travel in
// the kernel parameter block).
constexpr int kMaxSyrkTcMat = 200;

struct SyrkTcArgs {
  const MatInfo* info;
  const Tile* tiles;      // (matrix, block, first slice, end slice) of 128 rows
  int32_t num_tiles;
  int32_t mat_base;       // slot i of X / N / maps is matrix mat_base + i
  float* A;
  uint32_t* flags;
  uint32_t* err;
  float beta2;
  int32_t stages;
  int32_t stage_bytes;
  int32_t dbuf;           // 1: every block fits 256 TMEM columns, two accumulators alternate
  int32_t pad;
  const void* X[kMaxSyrkTcMat];
  int64_t N[kMaxSyrkTcMat];
  CUtensorMap maps[kMaxSyrkTcMat];
};

struct GjCtl;

struct EigArgs {
  const MatInfo* info;
  const Tile* tiles;
  int32_t num_tiles;
  int32_t max_sweeps;
  const float* A;
  float* Q;
  float* lam;
  float* scratch;         // 3 * (floats of the A region): B, V and a work matrix of each block
  uint32_t* flags;
  float* stats;
  float tol;              // relative off-diagonal norm of the last sweep's B (0 = default)
  const GjCtl* ctl;       // orthogonal iteration: only the items a grid pass left (see orth.cu)
};

// Grid eigensolver (jacobi_grid.cu): control record of one block, 64 bytes.
struct GjCtl {
  int32_t active;    // 1 while the block iterates
  int32_t fresh;     // B was formed by Rayleigh-Ritz before the current sweep
  int32_t restart;   // Newton-Schulz + Rayleigh-Ritz due after this sweep
  int32_t sweeps;
  int32_t conv;      // Jacobi: converged; orthogonal iteration: the grid pass holds
  int32_t rot;       // rotations of the current sweep
  int32_t last_rot;
  int32_t skip;      // A non-finite: basis kept
  int32_t vsel;      // which of the two basis buffers holds V
  float prev;        // off(B) after the previous sweep on a fresh B
  float bfloor;      // rotation threshold
  float pad;
  double off2, tot2; // sums of the current off(B) evaluation
};
static_assert(sizeof(GjCtl) == 64, "GjCtl is 64 bytes");

// One batch of the grid eigensolver: items of one width k.
struct GjArgs {
  const MatInfo* info;
  const Tile* items;
  int32_t nitems;
  int32_t k;
  const float* A;
  float* Q;
  float* lam;
  float* scratch;       // 3 k^2 floats per block at 3 x the block's A offset
  float* rbuf;          // per item rstride floats: the tables' rotations
  int64_t rstride;
  GjCtl* ctl;           // per item
  int32_t* active_count;
  uint32_t* flags;
  float* stats;
  int32_t max_sweeps;
  float tol;
};

// batches of the grid eigensolver that run at once (interleaved, on their own streams)
constexpr int kGjMaxBatches = 16;
// streams the grid eigensolver uses besides the caller's
constexpr int kGjStreams = 2;

int64_t gj_rbuf_floats(int k);
size_t gj_finish_smem(int k);
cudaError_t configure_jacobi_grid(size_t smem_limit);
// the whole refresh of nb batches (batch b on streams[b]); synchronises the
// streams once per sweep
cudaError_t run_jacobi_grid(const GjArgs* batches, int nb, const cudaStream_t* streams,
                            int* host_counts, int64_t* launches);
// the orthogonal-iteration refresh of nb batches on the grid (batch b on
// streams[b]), blocks whose Gram matrix is not numerically positive definite
// redone by orth.cu; no host synchronisation
cudaError_t run_orth_grid(const GjArgs* batches, int nb, const cudaStream_t* streams, int steps,
                          int sm_count, int64_t* launches);

// Coefficient normalisation of the FP32 update kernel.
constexpr int32_t kModeSign = 0;
constexpr int32_t kModeL2Apply = 2;

struct StepArgs {
  const MatInfo* info;
  const Tile* tiles;
  int32_t num_tiles;
  int32_t mat_base;
  const float* Q;
  float* M;
  uint32_t* flags;
  float* stats;
  float beta1;
  float lr_s;             // lr * s
  int32_t basis_bf16;     // multiply with bf16(Q) (bf16 basis storage)
  int32_t mode;           // kModeSign, or kModeL2Apply (column-l2 pass 2)
  float* colsq;           // column sums of C^2 (column-l2), eigenvalue-region layout
  void* W[kMaxMatPerLaunch];
  const void* G[kMaxMatPerLaunch];
  int8_t* S[kMaxMatPerLaunch];
};

struct CheckArgs {
  const MatInfo* info;
  const Tile* tiles;
  int32_t num_tiles;
  const float* A;
  const float* Q;
  const float* lam;
  float* out;             // 3 floats per block
};

// Launchers (return cudaGetLastError() of the launch).
cudaError_t launch_syrk_ema(const AccArgs& a, int act_dtype, int grid, cudaStream_t s);
cudaError_t launch_jacobi(const EigArgs& a, int grid, size_t smem_bytes, cudaStream_t s);
cudaError_t launch_step_ffma(const StepArgs& a, int param_dtype, int grid, size_t smem,
                             cudaStream_t s);
// column-l2 pass 1 over (matrix, block) items; writes StepArgs::colsq
cudaError_t launch_l2_norms(const StepArgs& a, int param_dtype, int grid, size_t smem,
                            cudaStream_t s);
int l2_max_k();
cudaError_t launch_check(const CheckArgs& a, int grid, cudaStream_t s);

// Kernel resource queries used by the scheduler at create time.
int step_rows_per_tile();
int syrk_tile();
// shared memory of the eigensolver for a block of width k within `budget`
// bytes (0 when it does not fit)
size_t jacobi_smem_for(int k, size_t budget);
int jacobi_ctas_per_sm();
size_t step_smem_for(int k);
cudaError_t configure_jacobi(size_t smem_limit);
// orthogonal-iteration refresh (steps Cholesky-QR iterations per block)
cudaError_t launch_orth(const EigArgs& a, int steps, int grid, cudaStream_t s);
size_t orth_smem_bytes();
cudaError_t configure_orth();
cudaError_t configure_step(size_t smem_limit);
size_t step_tc_smem(int max_k, int nastage, int nbstage);
size_t step_tc_bstage(int max_k);
int step_tc_astages(int max_k);                                  // momentum stages for a launch
int step_tc_bstages(int max_k, int nastage, size_t smem_limit);  // B stages that fit (0: none)
int64_t tc_block_image_bytes(int k);
bool tc_eligible(int64_t m, int64_t n, int k);
cudaError_t configure_step_tc(size_t smem_limit);
// may_t: some matrix of the launch has its W / G stored transposed (output side)
cudaError_t launch_step_tc(const StepArgs& a, const TcArgs& t, int param_dtype, bool may_t,
                           int grid, size_t smem, cudaStream_t s);
cudaError_t launch_pack_bases(const float* Q, unsigned char* qpack, const MatInfo* info,
                              const Tile* items, int num_items, int npieces, int grid,
                              cudaStream_t s);
size_t syrk_tc_stage_bytes(int max_k);
int syrk_tc_stages(int max_k, size_t smem_limit);
size_t syrk_tc_smem(int max_k, int stages);
bool syrk_tc_eligible(int64_t n, int k);
cudaError_t configure_syrk_tc(size_t smem_limit);
cudaError_t launch_syrk_tc(const SyrkTcArgs& a, int grid, size_t smem, cudaStream_t s);
bool syrk_tc_double_buffer(int max_k);  // two accumulators fit TMEM
// TMEM columns of slice t's accumulator (np: padded extended block width)
__host__ __device__ inline int syrk_tc_slice_cols(int np, int t) { return (np - 128 * t + 31) & ~31; }
cudaError_t launch_init_bases(float* Q, float* lam, const MatInfo* info, const Tile* items,
                              int num_items, int grid, cudaStream_t s);

}  // namespace dobb
