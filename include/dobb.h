/*
 * dobb.h -- C ABI of the Dobb optimizer step on one GPU (sm_103a).
 *
 * Dobb ("Dobb: Shard-Local Preconditioning in Block-Diagonal Eigenbases",
 * arXiv 2610.39412, Abstract) keeps, for every weight matrix W (m x n, y = W x,
 * Table 6 notation), the input-activation second moment as B diagonal k x k
 * blocks (k = n / B, Table 3 caption: n^2/B entries per matrix), a complete
 * orthonormal eigenbasis of every block, and a momentum buffer.  One
 * optimizer step projects the momentum into the block bases, takes the sign
 * of the coefficients (the l_inf normalisation of Table 13), reconstructs the
 * update and applies it:
 *
 *     A_b <- beta2 A_b + (1 - beta2) X_b^T X_b / N     dobb_accumulate_moments
 *     Q_b, Lambda_b : A_b = Q_b Lambda_b Q_b^T          dobb_refresh_bases
 *     M <- beta1 M + G ; C_b = M_b Q_b ; S_b = sign(C_b) ;
 *     U_b = S_b Q_b^T ; W <- W - lr * s * U              dobb_step
 *
 * The refresh is the exact eigendecomposition of Table 15; it runs inside the
 * step call every `refresh_period` steps (Table 21 footnote a: the moment
 * reduction runs behind the backward pass, the refresh inside the optimizer
 * call).
 *
 * Conventions shared by every call
 *  - All pointers named *_dev or documented as device pointers are CUDA
 *    device memory of the device that was current at dobb_create; pointer
 *    arrays themselves (const void* const* ...) are host arrays.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call is asynchronous on that stream unless stated.
 *  - Matrices are row-major.  X for matrix i is N_i x n_i (one row per token).
 *    W and G are m_i x n_i in the parameter dtype; M is fp32 library state.
 *  - The library never allocates device memory after dobb_create: the state
 *    lives in a caller-provided device buffer of dobb_state_bytes() bytes,
 *    which the caller owns and must keep alive until dobb_destroy.
 *  - Errors: every call returns a dobb_status; on failure dobb_last_error()
 *    (thread-local, valid until the next call on the same thread) gives a
 *    message.  Device-side conditions (non-finite input, non-convergence)
 *    never trap: they set per-block flag bits read by dobb_get_block_flags.
 */
#ifndef DOBB_H
#define DOBB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dobb_ctx* dobb_handle;

typedef enum {
  DOBB_OK = 0,
  DOBB_ERR_INVALID_ARG = 1,   /* bad shape, pointer, size or value          */
  DOBB_ERR_CUDA = 2,          /* a CUDA runtime call failed                  */
  DOBB_ERR_NONFINITE = 3,     /* reserved for callers mapping flag bits      */
  DOBB_ERR_NOT_CONVERGED = 4, /* reserved for callers mapping flag bits      */
  DOBB_ERR_STATE = 5,         /* wrong device, buffer too small, bad handle  */
  DOBB_ERR_UNSUPPORTED = 6    /* shape outside what the kernels support      */
} dobb_status;

typedef enum { DOBB_F32 = 0, DOBB_BF16 = 1 } dobb_dtype;

/* Per-block flag bits, OR-ed on the device, cleared by dobb_clear_block_flags. */
#define DOBB_FLAG_NONFINITE_X 1u     /* accumulate saw a non-finite activation      */
#define DOBB_FLAG_NONFINITE_G 2u     /* step saw a non-finite gradient / momentum   */
#define DOBB_FLAG_NONFINITE_A 4u     /* refresh skipped (A non-finite); basis kept  */
#define DOBB_FLAG_NOT_CONVERGED 8u   /* eigensolver hit its sweep cap; basis written */

/* Which state tensor dobb_state_tensor() returns. */
typedef enum {
  DOBB_T_MOMENTS = 0,  /* A: per matrix B blocks of k x k fp32, row-major, full symmetric */
  DOBB_T_BASES = 1,    /* Q: per matrix B blocks of k x k fp32, row-major; column j is the
                          eigenvector of the j-th largest eigenvalue                         */
  DOBB_T_EIGVALS = 2,  /* Lambda: per matrix B x k fp32, descending within a block         */
  DOBB_T_MOMENTUM = 3, /* M: per matrix m x n fp32, row-major                              */
  DOBB_T_FLAGS = 4,    /* per block uint32 flag bits (all blocks of all matrices)          */
  DOBB_T_STATS = 5,    /* per block 4 fp32: ||U_b||_F^2, ||C_b||_F^2 of the last step,
                          Jacobi sweeps and rotations of the last sweep of the last refresh */
  DOBB_T_ERROR = 6     /* one uint32: nonzero if a device-side wait timed out (the step
                          that set it must be treated as failed); cleared by the caller    */
} dobb_tensor;

/* Bytes of device state for the given matrix set (m[i] x n[i], n[i] % B == 0).
 * Returns 0 if the arguments are invalid (see dobb_last_error). */
size_t dobb_state_bytes(int num_matrices, const int64_t* m, const int64_t* n, int B);

/* Create an optimizer over `num_matrices` matrices.
 *   m, n            host arrays of the matrix shapes; n[i] % B == 0, k = n/B in [1, 8192]
 *   B               blocks per matrix (same for all matrices)
 *   beta1, beta2    momentum and second-moment EMA coefficients, in [0, 1)
 *   refresh_period  T: dobb_step refreshes the bases when t % T == 0; 0 = never
 *   scale_s         update scale s (Table 9), W <- W - lr * s * U
 *   param_dtype     dtype of W and G; act_dtype dtype of X
 *   state_mem       caller-owned device buffer of at least dobb_state_bytes()
 *                   bytes, 256-byte aligned
 * Initialises A = 0, Q = I, Lambda = 0, M = 0, flags = 0, t = 0 on `stream`.
 * The handle is bound to the current CUDA device. */
dobb_status dobb_create(dobb_handle* out, int num_matrices, const int64_t* m,
                        const int64_t* n, int B, float beta1, float beta2,
                        int refresh_period, float scale_s, dobb_dtype param_dtype,
                        dobb_dtype act_dtype, void* state_mem, size_t state_bytes,
                        void* stream);

dobb_status dobb_destroy(dobb_handle h);

/* Thread-local message of the last failed call on this thread ("" if none). */
const char* dobb_last_error(void);

/* Accumulate block second moments (one grouped launch over all matrices):
 * A_b <- beta2 A_b + (1 - beta2) X_b^T X_b / N_i for every block of matrix i.
 *   X   host array of num_matrices device pointers (X[i] may be NULL to skip i)
 *   N   host array of token counts (N[i] == 0 skips matrix i) */
dobb_status dobb_accumulate_moments(dobb_handle h, const void* const* X,
                                    const int64_t* N, void* stream);

/* Recompute Q_b, Lambda_b of every block from the current A_b now (one
 * grouped launch).  Blocks whose A is non-finite keep their basis and get
 * DOBB_FLAG_NONFINITE_A. */
dobb_status dobb_refresh_bases(dobb_handle h, void* stream);

/* One optimizer step over all matrices (one grouped launch, plus the refresh
 * first when refresh_period > 0 and t % refresh_period == 0); then t += 1.
 *   W   host array of device pointers, updated in place (param_dtype)
 *   G   host array of device pointers (param_dtype) */
dobb_status dobb_step(dobb_handle h, void* const* W, const void* const* G,
                      float lr, void* stream);

/* dobb_step that also writes S = sign(C) as int8 (m_i x n_i, row-major) to
 * S_out[i] (device pointers; an entry may be NULL).  Test hook. */
dobb_status dobb_step_with_signs(dobb_handle h, void* const* W, const void* const* G,
                                 float lr, int8_t* const* S_out, void* stream);

/* Host-side step counter. */
dobb_status dobb_get_step(dobb_handle h, int64_t* t);
dobb_status dobb_set_step(dobb_handle h, int64_t t);

/* Coefficient normalisation of the update.
 * DOBB_NORM_SIGN (default): S_b = sign(C_b) ("Dobb", Abstract; l_inf).
 * DOBB_NORM_L2: "Dobb-l2" (Table 11), each column of C_b over all m rows
 *   scaled to l2 norm sqrt(m): S_b[:, j] = sqrt(m) C_b[:, j] / ||C_b[:, j]||
 *   (0 for a zero column), so U / sqrt(m) has Table 9's ||O||_F^2 = n as the
 *   sign update does.  Runs on the FP32 kernels in two passes (momentum and
 *   column norms over all rows, then the update); blocks up to 1024 wide.
 *   dobb_step's optional sign output receives sign(C_b).
 * DOBB_ERR_INVALID_ARG for another value, DOBB_ERR_UNSUPPORTED for wider
 * blocks. */
enum { DOBB_NORM_SIGN = 0, DOBB_NORM_L2 = 1 };
dobb_status dobb_set_normalization(dobb_handle h, int norm);

/* Which axis of a weight the blocks and moments cover ("Dobb", Tables
 * 12-13).  `matrix` is an index, or -1 for every matrix.
 * DOBB_SIDE_INPUT (default): Dobb.  The matrix registered as (m, n) is the
 *   caller's W (m x n, row-major); blocks split its n input columns and
 *   dobb_accumulate_moments takes input activations X (N x n).
 * DOBB_SIDE_OUTPUT: "Dobb-G".  The matrix registered as (m, n) is the
 *   TRANSPOSE of the caller's weight: W, G (and the optional sign output)
 *   are n x m row-major buffers, i.e. a weight with n output rows and m
 *   input columns; blocks split its n output rows, dobb_accumulate_moments
 *   takes output gradients (N x n), and the update is C_b = Q_b^T M_b,
 *   U_b = S_b' Q_b applied from the left (S_b' the normalised C_b, a sign
 *   or, with DOBB_NORM_L2, each ROW of C_b scaled to l2 norm sqrt(m)).  The
 *   momentum buffer (dobb_state_tensor) keeps the registered m x n layout,
 *   i.e. the transpose of the caller's momentum.  The update kernels read
 *   and write the caller's buffers through the transposed index.
 * Copies the per-matrix table on `stream` and waits for it.  The side is
 * configuration, like the normalisation and the refresh method: the state
 * that dobb_get_state / dobb_set_state carry does not include it.
 * DOBB_ERR_INVALID_ARG for another side or a matrix out of range;
 * DOBB_ERR_UNSUPPORTED for a block too wide for the FP32 update kernel. */
enum { DOBB_SIDE_INPUT = 0, DOBB_SIDE_OUTPUT = 1 };
dobb_status dobb_set_side(dobb_handle h, int matrix, int side, void* stream);

/* Refresh method ("Dobb", Table 15).
 * DOBB_REFRESH_EIGH (default): complete eigendecomposition of every block,
 *   Q_b with A_b = Q_b Lambda_b Q_b^T (two-sided Jacobi), columns by
 *   descending eigenvalue.
 * DOBB_REFRESH_ORTH: `steps` orthogonal-iteration steps from the current
 *   basis (one step is the pages' principal setting): Q_b <- T R^{-1} with
 *   T = A_b Q_b and R = chol(T^T T) (Table 16: Cholesky QR; computed as
 *   CholeskyQR2 in fp32, with a shifted first pass when T^T T is not
 *   numerically positive definite); Lambda_b holds the Rayleigh quotients
 *   diag(Q_b^T A_b Q_b).  Blocks at least as wide as dobb_set_eig_grid's
 *   min_k run on the grid (batched products, a Cholesky factorisation per
 *   block, the triangular solve by 64-row panels); a block whose Gram
 *   matrix is not numerically positive definite there is redone from its
 *   old basis with the shifted passes, one CTA per block, like the narrower
 *   blocks.  A block whose QR fails keeps its basis and gets
 *   DOBB_FLAG_NOT_CONVERGED.
 * DOBB_ERR_INVALID_ARG for another method or steps < 1.  Takes effect at the
 * next refresh. */
enum { DOBB_REFRESH_EIGH = 0, DOBB_REFRESH_ORTH = 1 };
dobb_status dobb_set_refresh(dobb_handle h, int method, int steps);

/* Precision of the basis the update multiplies with ("Dobb", Table 18:
 * fp32 moment accumulation with a bf16 basis is the principal setting).
 * DOBB_F32 (default): C_b = M_b Q_b and U_b = S_b Q_b^T with the fp32 basis.
 * DOBB_BF16: every entry of Q_b is rounded once to bf16 (nearest, ties to
 * even) and the products use that basis at fp32 accuracy.  The eigensolver
 * keeps the fp32 basis as its warm start either way.  Re-packs the
 * tensor-core operand images on `stream`; DOBB_ERR_INVALID_ARG for another
 * dtype. */
dobb_status dobb_set_basis_dtype(dobb_handle h, dobb_dtype basis_dtype, void* stream);

/* Change the refresh period T of dobb_step (0 = never); the step counter is
 * kept.  DOBB_ERR_INVALID_ARG for T < 0. */
dobb_status dobb_set_refresh_period(dobb_handle h, int refresh_period);

/* Which eigensolver refreshes a block: blocks at least `min_k` wide use the
 * grid solver (every table, tile pair and panel of a sweep its own CTA, a
 * launch per phase over a batch of blocks of one width; the call then
 * synchronises `stream` once per sweep), narrower ones one CTA per block.
 * Both run the same restarted Rayleigh-Ritz two-sided Jacobi.  The same
 * threshold and batches apply to the orthogonal-iteration refresh (no
 * synchronisation there).  0 = never the grid solver; otherwise min_k >= 64.  A batch holds the blocks of one width
 * whose scratch (12 k^2 bytes each) fits `batch_bytes` (at least one block;
 * 0 = all blocks of that width).  Defaults: 64, 0.  DOBB_ERR_INVALID_ARG for
 * other values. */
dobb_status dobb_set_eig_grid(dobb_handle h, int min_k, int64_t batch_bytes);

/* Eigensolver controls: sweep cap (default 40) and the convergence
 * threshold, the relative off-diagonal norm ||off(B)||_F / ||B||_F that the
 * last sweep of B = V^T A V may leave (0 = default 2e-6). */
dobb_status dobb_set_jacobi(dobb_handle h, int max_sweeps, float tol);

/* Device pointer and byte size of a state tensor of one matrix
 * (matrix >= 0) or of the whole region over all matrices (matrix == -1). */
dobb_status dobb_state_tensor(dobb_handle h, dobb_tensor which, int matrix,
                              void** dev_ptr, size_t* bytes);

/* Number of blocks over all matrices and the index of matrix i's first block
 * (blocks are numbered matrix by matrix). */
int64_t dobb_num_blocks(dobb_handle h);
int64_t dobb_block_offset(dobb_handle h, int matrix);

/* Copy the per-block flags / stats to host memory (num_blocks entries of
 * uint32, or 4 * num_blocks floats).  Synchronises `stream`. */
dobb_status dobb_get_block_flags(dobb_handle h, uint32_t* host_out, void* stream);
dobb_status dobb_clear_block_flags(dobb_handle h, void* stream);
dobb_status dobb_get_block_stats(dobb_handle h, float* host_out, void* stream);

/* Invariant check of the current bases (one grouped launch, fp64 sums):
 * per block 3 floats ||A Q - Q Lambda||_F / ||A||_F, ||Q^T Q - I||_F,
 * ||Q Lambda Q^T - A||_F / ||A||_F written to host_out (3 * num_blocks).
 * Synchronises `stream`. */
dobb_status dobb_check_bases(dobb_handle h, float* host_out, void* stream);

/* Checkpoint: bytes of the persistent state (A, Q, Lambda, M, flags), copy
 * it to / from a caller device buffer, together with the step counter. */
size_t dobb_checkpoint_bytes(dobb_handle h);
dobb_status dobb_get_state(dobb_handle h, void* dst_dev, size_t dst_bytes,
                           int64_t* t_out, void* stream);
dobb_status dobb_set_state(dobb_handle h, const void* src_dev, size_t src_bytes,
                           int64_t t, void* stream);

/* Number of kernel launches issued by this handle since creation (host count). */
int64_t dobb_launch_count(dobb_handle h);

/* Host-side view of the grouped work lists (the scheduler) of a handle over
 * this matrix set; needs no device.  phase 0: the update tiles of a step on
 * the default path (tensor-core launches, then the FFMA rest); 1: the moment
 * units of an accumulate with bf16 activations; 2: the eigen items of a
 * refresh.  Writes min(count, cap) entries of 7 int64 to `out` (may be NULL):
 *   (launch, kind, mat_base, matrix, block, a, b)
 * launch = index of the launch in the phase's sequence, kind = 0 for the
 * tensor-core kernel (phase 0, 1) or the eigensolver (2) and 1 for the FFMA
 * kernel, mat_base = the matrix in slot 0 of that launch's pointer table;
 * (a, b) = (first row, rows) for update tiles, (first, end) 128-row slice of
 * a tensor-core moment unit, (row, column) 64-tile of an FFMA moment tile,
 * (0, 0) for eigen items.  Returns the number of entries, -1 on bad
 * arguments (see dobb_last_error). */
int64_t dobb_describe_work(int num_matrices, const int64_t* m, const int64_t* n, int B,
                           int phase, int64_t* out, int64_t cap);

/* Update-kernel selection: 0 (default) runs the tcgen05 tensor-core kernel for
 * every matrix with k % 4 == 0 and k <= 448 (and 16-byte aligned W, G) and the
 * FP32 FFMA kernel for the rest; 1 runs the FFMA kernel for all matrices.
 * Both compute the same update within the documented tolerance. */
dobb_status dobb_set_step_path(dobb_handle h, int path);

/* Re-derive the tensor-core operand images of the bases after the caller
 * wrote Q directly through dobb_state_tensor(DOBB_T_BASES).  Refresh, create
 * and dobb_set_state do this themselves. */
dobb_status dobb_sync_bases(dobb_handle h, void* stream);

/* Throughput probe for the roofline denominators (the pages have no
 * counterpart): one launch of one instruction stream on every SM,
 *   which 0: FP32 FFMA, 1: TF32 mma.sync (m16n8k8), 2: TF32 tcgen05.mma
 *   (128 x 256 x 8), 3: BF16 tcgen05.mma (128 x 256 x 16);
 * `iters` scales the work.  scratch_dev: caller device memory of at least
 * 4 * (sms * 2048) + 256 bytes for the results (which mean nothing).
 * Synchronises `stream`; returns the launch's event time in ms and its exact
 * flop count (2 per multiply-add). */
dobb_status dobb_peak_probe(int which, void* scratch_dev, size_t scratch_bytes, int iters,
                            float* ms_out, double* flops_out, void* stream);

/* Failure-detection self-test (the pages have no counterpart): one launch of
 * the bounded mbarrier wait the tensor-core kernels use, on a barrier that
 * nothing arrives on.  After timeout_ns (1 ns ... 5 s) the wait gives up, the
 * kernel ORs 0x100 into *err_dev (device memory) and returns; asynchronous on
 * `stream`.  DOBB_ERR_INVALID_ARG for a NULL pointer or a timeout out of
 * range. */
dobb_status dobb_selftest_wait_timeout(uint32_t* err_dev, uint64_t timeout_ns, void* stream);

/* ------------------------------------------------------------------------
 * Allocation-free block eigendecomposition.
 *
 * The pages have no counterpart of this call.  It exists for callers of
 * this library that cannot call cudaMalloc: runtimes whose device memory is
 * reserved up front by an arena they do not control, and plugins of
 * frameworks that forbid allocations outside their own allocator.  It runs
 * the refresh eigensolver (the restarted Rayleigh-Ritz two-sided Jacobi of
 * dobb_refresh_bases, started from the identity) on caller buffers and
 * allocates nothing: its working memory is a file-scope device array of
 * DOBB_NOALLOC_SCRATCH_FLOATS floats (16 MiB) plus small fixed work-list
 * arrays, which every GPU that loads the library holds until the process
 * exits.
 *
 *   A_dev    count symmetric k x k fp32 matrices, row-major, back to back (in)
 *   Q_dev    count k x k fp32 outputs, row-major, column j = eigenvector of
 *            the j-th largest eigenvalue (out; its contents are overwritten)
 *   lam_dev  count x k fp32 eigenvalues, descending (out)
 *            Q_dev and lam_dev must not overlap A_dev (the basis is set to
 *            the identity before A is read): DOBB_ERR_INVALID_ARG otherwise
 *   k        1 <= k <= 1024;  count 0 <= count <= 4096 and
 *            count * 3 * k * k <= DOBB_NOALLOC_SCRATCH_FLOATS, otherwise the
 *            call returns DOBB_ERR_INVALID_ARG without touching the device
 *   max_sweeps  sweep cap of the Jacobi iteration (e.g. 40)
 *   flags_host  optional host array of count uint32 (DOBB_FLAG_* bits); when
 *               non-NULL the call synchronises `stream` and fills it
 * Asynchronous on `stream` otherwise.  The first call on a device resolves
 * the device addresses of the arrays (cudaGetSymbolAddress) and configures
 * the kernel; later calls only enqueue work.  All calls share the arrays,
 * which keep the last call's contents (the call clears what must start at
 * zero): calls that overlap on the GPU race.  Errors are reported by
 * dobb_eigh_noalloc_last_error() (thread-local). */
#define DOBB_NOALLOC_SCRATCH_FLOATS (4u << 20)
dobb_status dobb_eigh_noalloc(const float* A_dev, float* Q_dev, float* lam_dev, int k, int count,
                              int max_sweeps, uint32_t* flags_host, void* stream);
const char* dobb_eigh_noalloc_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* DOBB_H */
