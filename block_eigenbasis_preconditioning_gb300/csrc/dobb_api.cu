// Host side of the C ABI declared in include/dobb.h: argument checks, the
// state layout inside the caller's device buffer, the grouped work lists
// (one list per phase, cost-sorted, consumed by persistent CTAs) and the
// per-phase launches.
//
// "Dobb: Shard-Local Preconditioning in Block-Diagonal Eigenbases": the
// per-matrix state is the block second moments (Table 3 caption: n^2/B
// entries), the block bases (Table 18: fp32 accumulation and basis storage,
// 8 n^2/B bytes with both), and the momentum; the refresh runs inside the
// optimizer call every T steps (Table 5 caption, Table 21 footnote a).
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "dobb_internal.cuh"

using namespace dobb;

namespace {

thread_local std::string g_err;

dobb_status fail(dobb_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

#define CUDA_TRY(expr)                                                                   \
  do {                                                                                   \
    cudaError_t e_ = (expr);                                                             \
    if (e_ != cudaSuccess) return fail(DOBB_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(e_)); \
  } while (0)

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

struct Layout {
  size_t a_floats = 0, lam_floats = 0, m_floats = 0, pack_bytes = 0;
  int64_t nblocks = 0;
  size_t off_colsq = 0;  // column sums of squares (column-l2 normalisation), eigenvalue layout
  size_t off_A = 0, off_Q = 0, off_lam = 0, off_M = 0, off_flags = 0, off_stats = 0,
         off_check = 0, off_err = 0, off_info = 0, off_maps = 0, off_tiles = 0, off_pack = 0,
         off_scratch = 0, off_gj_rbuf = 0, off_gj_ctl = 0, off_gj_count = 0, total = 0;
  size_t gj_rbuf_floats = 0, gj_ctl_items = 0;
  size_t n_tiles = 0;
};

constexpr int kTcRows = 128;
// tensor-core tiles of blocks up to this width get their own launch, whose
// small operand stages leave room for many in flight
constexpr int kTcSmallK = 128;

int64_t pad16f(int64_t v) { return (v + 15) / 16 * 16; }

// Grid eigensolver: blocks at least this wide use it by default (narrower
// ones run one CTA per block), it is never used below kGjMinK, and a batch
// holds as many blocks of one width as keep their scratch (3 k^2 floats)
// within kGjL2Budget bytes of L2.
constexpr int kGjDefaultMinK = 64;
constexpr int kGjMinK = 64;
constexpr int64_t kGjDefaultBatchBytes = 0;   // 0: every block of one width in one batch

// blocks of width k in one batch whose scratch (3 k^2 floats each) stays
// within batch_bytes (0: no limit)
int gj_batch_items(int k, int64_t batch_bytes) {
  if (batch_bytes <= 0) return 1 << 30;
  const int64_t per = 12 * (int64_t)k * k;
  return (int)std::max<int64_t>(1, std::min<int64_t>(1 << 30, batch_bytes / per));
}

struct Chunk {
  int mat_base = 0, mat_end = 0;
  int step_off = 0, step_n = 0;     // FFMA tiles of every matrix
  int tc_off = 0, tc_n = 0;         // tensor-core tiles (eligible matrices), widest first
  int tc_small = 0;                 // index (within them) of the first tile with k <= 128
  int rest_off = 0, rest_n = 0;     // FFMA tiles of the other matrices
  int max_k_tc = 0, max_k_rest = 1;
  int syrk_off = 0, syrk_n = 0;
  int syrk_rest_off = 0, syrk_rest_n = 0;  // FFMA moment tiles of matrices the tensor-core kernel skips
  int eig_off = 0, eig_n = 0;
  int l2_off = 0, l2_n = 0;         // column-l2 norm items: (matrix, block, row chunk)
  int max_k = 1;
};

// rows per item of the column-l2 norm pass (one chunk's partial column sums
// are added with one atomic per column)
constexpr int64_t kL2Rows = 1024;

struct SyrkChunk {
  int mat_base = 0, mat_end = 0, off = 0, n = 0, max_k = 8;
  int small = 0;  // index (within the chunk) of the first tile with k <= kTcSmallK
};

// Work lists of all phases, in the order they are stored on the device.
struct WorkLists {
  std::vector<Tile> tiles;
  std::vector<Chunk> chunks;
  std::vector<SyrkChunk> syrk_tc;
  int syrk_rest_total = 0;  // FFMA moment tiles over all chunks
  int blocks_off = 0, blocks_n = 0;  // every (matrix, block) once, by matrix
};

bool validate_shapes(int num, const int64_t* m, const int64_t* n, int B) {
  if (num <= 0 || !m || !n) {
    fail(DOBB_ERR_INVALID_ARG, "num_matrices must be > 0 and shape arrays non-NULL");
    return false;
  }
  if (B <= 0) {
    fail(DOBB_ERR_INVALID_ARG, "B must be > 0 (got %d)", B);
    return false;
  }
  for (int i = 0; i < num; ++i) {
    if (m[i] <= 0 || n[i] <= 0) {
      fail(DOBB_ERR_INVALID_ARG, "matrix %d has shape %lld x %lld", i, (long long)m[i], (long long)n[i]);
      return false;
    }
    if (n[i] % B != 0) {
      fail(DOBB_ERR_INVALID_ARG, "matrix %d: n=%lld is not divisible by B=%d", i, (long long)n[i], B);
      return false;
    }
    const int64_t k = n[i] / B;
    if (k > kMaxK) {
      fail(DOBB_ERR_UNSUPPORTED, "matrix %d: block width k=%lld exceeds %d", i, (long long)k, kMaxK);
      return false;
    }
    if (m[i] > (int64_t)1 << 31) {
      fail(DOBB_ERR_UNSUPPORTED, "matrix %d: m=%lld too large", i, (long long)m[i]);
      return false;
    }
  }
  return true;
}

WorkLists build_work(int num, const int64_t* m, const int64_t* n, int B) {
  WorkLists wl;
  const int TM = step_rows_per_tile();
  const int ST = syrk_tile();
  for (int c0 = 0; c0 < num; c0 += kMaxMatPerLaunch) {
    Chunk ch;
    ch.mat_base = c0;
    ch.mat_end = std::min(num, c0 + kMaxMatPerLaunch);
    std::vector<std::pair<int64_t, Tile>> v;
    // step tiles: (matrix, block, row0); cost ~ rows * k
    for (int i = ch.mat_base; i < ch.mat_end; ++i) {
      const int k = (int)(n[i] / B);
      ch.max_k = std::max(ch.max_k, k);
      for (int b = 0; b < B; ++b)
        for (int64_t r = 0; r < m[i]; r += TM) v.push_back({(int64_t)k, Tile{i, b, (int)r, 0}});
    }
    std::stable_sort(v.begin(), v.end(), [](auto& x, auto& y) { return x.first > y.first; });
    ch.step_off = (int)wl.tiles.size();
    ch.step_n = (int)v.size();
    for (auto& e : v) wl.tiles.push_back(e.second);
    // tensor-core tiles of 128 rows, and FFMA tiles of the ineligible rest
    v.clear();
    std::vector<std::pair<int64_t, Tile>> rest;
    for (int i = ch.mat_base; i < ch.mat_end; ++i) {
      const int k = (int)(n[i] / B);
      if (tc_eligible(m[i], n[i], k)) {
        ch.max_k_tc = std::max(ch.max_k_tc, k);
        for (int b = 0; b < B; ++b)
          for (int64_t r = 0; r < m[i]; r += kTcRows) v.push_back({(int64_t)k, Tile{i, b, (int)r, 0}});
      } else {
        ch.max_k_rest = std::max(ch.max_k_rest, k);
        for (int b = 0; b < B; ++b)
          for (int64_t r = 0; r < m[i]; r += TM) rest.push_back({(int64_t)k, Tile{i, b, (int)r, 0}});
      }
    }
    std::stable_sort(v.begin(), v.end(), [](auto& x, auto& y) { return x.first > y.first; });
    std::stable_sort(rest.begin(), rest.end(), [](auto& x, auto& y) { return x.first > y.first; });
    ch.tc_off = (int)wl.tiles.size();
    ch.tc_n = (int)v.size();
    ch.tc_small = ch.tc_n;
    for (int j = 0; j < ch.tc_n; ++j)
      if (v[j].first <= kTcSmallK) { ch.tc_small = j; break; }
    for (auto& e : v) wl.tiles.push_back(e.second);
    ch.rest_off = (int)wl.tiles.size();
    ch.rest_n = (int)rest.size();
    for (auto& e : rest) wl.tiles.push_back(e.second);
    // syrk tiles: upper triangle of ceil(k / ST)^2 output tiles per block
    v.clear();
    for (int i = ch.mat_base; i < ch.mat_end; ++i) {
      const int k = (int)(n[i] / B);
      const int nt = (k + ST - 1) / ST;
      for (int b = 0; b < B; ++b)
        for (int ti = 0; ti < nt; ++ti)
          for (int tj = ti; tj < nt; ++tj) v.push_back({(int64_t)k, Tile{i, b, ti, tj}});
    }
    std::stable_sort(v.begin(), v.end(), [](auto& x, auto& y) { return x.first > y.first; });
    ch.syrk_off = (int)wl.tiles.size();
    ch.syrk_n = (int)v.size();
    for (auto& e : v) wl.tiles.push_back(e.second);
    // column-l2 norm items: row chunks of every block, in matrix order
    ch.l2_off = (int)wl.tiles.size();
    for (int i = ch.mat_base; i < ch.mat_end; ++i)
      for (int b = 0; b < B; ++b)
        for (int64_t r = 0; r < m[i]; r += kL2Rows)
          wl.tiles.push_back(Tile{i, b, (int)r, (int)std::min<int64_t>(kL2Rows, m[i] - r)});
    ch.l2_n = (int)wl.tiles.size() - ch.l2_off;
    // eigen items: one per block, largest k first (cost ~ k^3)
    v.clear();
    for (int i = ch.mat_base; i < ch.mat_end; ++i) {
      const int k = (int)(n[i] / B);
      for (int b = 0; b < B; ++b) v.push_back({(int64_t)k, Tile{i, b, 0, 0}});
    }
    std::stable_sort(v.begin(), v.end(), [](auto& x, auto& y) { return x.first > y.first; });
    ch.eig_off = (int)wl.tiles.size();
    ch.eig_n = (int)v.size();
    for (auto& e : v) wl.tiles.push_back(e.second);
    wl.chunks.push_back(ch);
  }
  // tensor-core accumulate: chunks of eligible matrices; a unit is a run of
  // 128-row slices [a, b) of one block whose accumulators share TMEM (the
  // slice count depends on each block's misalignment to 8 columns)
  {
    std::vector<int> elig;
    for (int i = 0; i < num; ++i)
      if (syrk_tc_eligible(n[i], (int)(n[i] / B))) elig.push_back(i);
    for (size_t c0 = 0; c0 < elig.size();) {
      SyrkChunk sc;
      sc.mat_base = elig[c0];
      std::vector<std::pair<int64_t, Tile>> v;
      size_t c1 = c0;
      int kmax_wide = 0;
      while (c1 < elig.size() && elig[c1] - sc.mat_base < kMaxSyrkTcMat) {
        const int k = (int)(n[elig[c1]] / B);
        if (k > kTcSmallK) kmax_wide = std::max(kmax_wide, k);
        ++c1;
      }
      for (size_t c = c0; c < c1; ++c) {
        const int i = elig[c];
        const int k = (int)(n[i] / B);
        sc.max_k = std::max(sc.max_k, k);
        // TMEM columns a unit may use: one of two alternating accumulators,
        // or all of TMEM (as in the kernel's launch of these blocks)
        const int budget = syrk_tc_double_buffer(k > kTcSmallK ? kmax_wide : kTcSmallK) ? 256 : 512;
        for (int b = 0; b < B; ++b) {
          const int d = (int)(((int64_t)b * k) & 7);
          const int np = (k + d + 15) & ~15, ns = (k + d + 127) / 128;
          for (int t0 = 0; t0 < ns;) {
            int t1 = t0, cols = 0;
            while (t1 < ns && cols + syrk_tc_slice_cols(np, t1) <= budget) cols += syrk_tc_slice_cols(np, t1++);
            if (t1 == t0) t1 = t0 + 1;  // a first slice always fits its launch
            v.push_back({(int64_t)k, Tile{i, b, t0, t1}});
            t0 = t1;
          }
        }
      }
      sc.mat_end = elig[c1 - 1] + 1;
      std::stable_sort(v.begin(), v.end(), [](auto& x, auto& y) { return x.first > y.first; });
      sc.off = (int)wl.tiles.size();
      sc.n = (int)v.size();
      sc.small = sc.n;
      for (int j = 0; j < sc.n; ++j)
        if (v[j].first <= kTcSmallK) { sc.small = j; break; }
      for (auto& e : v) wl.tiles.push_back(e.second);
      wl.syrk_tc.push_back(sc);
      c0 = c1;
    }
    // FFMA accumulate tiles of the matrices the tensor-core kernel skips, per
    // launch chunk (the pointer table of a launch holds kMaxMatPerLaunch)
    for (Chunk& ch : wl.chunks) {
      std::vector<std::pair<int64_t, Tile>> v;
      for (int i = ch.mat_base; i < ch.mat_end; ++i) {
        const int k = (int)(n[i] / B);
        if (syrk_tc_eligible(n[i], k)) continue;
        const int nt = (k + ST - 1) / ST;
        for (int b = 0; b < B; ++b)
          for (int ti = 0; ti < nt; ++ti)
            for (int tj = ti; tj < nt; ++tj) v.push_back({(int64_t)k, Tile{i, b, ti, tj}});
      }
      std::stable_sort(v.begin(), v.end(), [](auto& x, auto& y) { return x.first > y.first; });
      ch.syrk_rest_off = (int)wl.tiles.size();
      ch.syrk_rest_n = (int)v.size();
      wl.syrk_rest_total += ch.syrk_rest_n;
      for (auto& e : v) wl.tiles.push_back(e.second);
    }
  }
  wl.blocks_off = (int)wl.tiles.size();
  for (int i = 0; i < num; ++i)
    for (int b = 0; b < B; ++b) wl.tiles.push_back(Tile{i, b, 0, 0});
  wl.blocks_n = (int)wl.tiles.size() - wl.blocks_off;
  return wl;
}

Layout compute_layout(int num, const int64_t* m, const int64_t* n, int B, size_t n_tiles) {
  Layout L;
  for (int i = 0; i < num; ++i) {
    const int64_t k = n[i] / B;
    L.a_floats += (size_t)B * k * k;
    L.lam_floats += (size_t)B * k;
    L.m_floats += (size_t)pad16f(m[i] * n[i]);
    L.nblocks += B;
    if (tc_eligible(m[i], n[i], (int)k)) L.pack_bytes += (size_t)B * tc_block_image_bytes((int)k);
  }
  size_t off = 0;
  L.off_A = off;      off = align_up(off + 4 * L.a_floats);
  L.off_Q = off;      off = align_up(off + 4 * L.a_floats);
  L.off_lam = off;    off = align_up(off + 4 * L.lam_floats);
  L.off_M = off;      off = align_up(off + 4 * L.m_floats);
  L.off_flags = off;  off = align_up(off + 4 * (size_t)L.nblocks);
  L.off_stats = off;  off = align_up(off + 16 * (size_t)L.nblocks);
  L.off_check = off;  off = align_up(off + 12 * (size_t)L.nblocks);
  L.off_colsq = off;  off = align_up(off + 4 * L.lam_floats);
  L.off_err = off;    off = align_up(off + 4);
  L.off_info = off;   off = align_up(off + sizeof(MatInfo) * (size_t)num);
  L.off_maps = off;   off = align_up(off + sizeof(CUtensorMap) * (size_t)num);
  L.off_tiles = off;  off = align_up(off + sizeof(Tile) * n_tiles);
  L.off_pack = off;   off = align_up(off + L.pack_bytes);
  L.off_scratch = off; off = align_up(off + 12 * L.a_floats);  // 3 k^2 floats per block
  // grid eigensolver: rotations and control records of the largest batch of
  // any width it may be used for
  {
    std::vector<std::pair<int, size_t>> count;  // (width, blocks of that width)
    for (int i = 0; i < num; ++i) {
      const int k = (int)(n[i] / B);
      if (k < kGjMinK) continue;
      auto it = std::find_if(count.begin(), count.end(), [&](auto& c) { return c.first == k; });
      if (it == count.end()) count.push_back({k, (size_t)B});
      else it->second += B;
    }
    // every width's blocks may be in flight at once (concurrent batches)
    for (auto& c : count) {
      L.gj_rbuf_floats += c.second * (size_t)gj_rbuf_floats(c.first);
      L.gj_ctl_items += c.second;
    }
  }
  L.off_gj_rbuf = off;  off = align_up(off + 4 * L.gj_rbuf_floats);
  L.off_gj_ctl = off;   off = align_up(off + sizeof(GjCtl) * L.gj_ctl_items);
  L.off_gj_count = off; off = align_up(off + 4 * kGjMaxBatches);
  L.total = off;
  L.n_tiles = n_tiles;
  return L;
}

}  // namespace

struct dobb_ctx {
  int device = 0;
  int num = 0, B = 1, T = 0;
  float beta1 = 0.95f, beta2 = 0.99f, scale_s = 1.f;
  dobb_dtype pdt = DOBB_F32, adt = DOBB_F32;
  std::vector<int64_t> m, n;
  std::vector<MatInfo> info;
  WorkLists wl;
  Layout L;
  char* base = nullptr;
  size_t bytes = 0;
  int64_t t = 0;
  int max_sweeps = 40;
  float tol = 0.f;
  bool basis_bf16 = false;  // the update multiplies with bf16(Q)
  int refresh_method = DOBB_REFRESH_EIGH;
  int norm = DOBB_NORM_SIGN;
  int orth_steps = 1;
  int sm_count = 1;
  size_t smem_limit = 0;
  size_t smem_per_sm = 0;
  int64_t launches = 0;
  int path = 0;            // 0: tensor-core kernel where eligible, 1: FFMA only
  int gj_min_k = kGjDefaultMinK;  // blocks at least this wide use the grid eigensolver
  int64_t gj_batch_bytes = kGjDefaultBatchBytes;
  int gj_host_counts[kGjMaxBatches] = {};
  cudaStream_t gj_streams[kGjStreams] = {};   // the grid eigensolver's own streams
  cudaEvent_t gj_events[kGjStreams + 1] = {};
  ~dobb_ctx() {
    for (int i = 0; i < kGjStreams; ++i)
      if (gj_streams[i]) cudaStreamDestroy(gj_streams[i]);
    for (int i = 0; i <= kGjStreams; ++i)
      if (gj_events[i]) cudaEventDestroy(gj_events[i]);
  }
  // cached X tensor maps (pointer and token count they were encoded for)
  std::vector<CUtensorMap> xmaps;
  std::vector<const void*> xmap_ptr;
  std::vector<int64_t> xmap_N;
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  bool any_tc = false;
  std::vector<float> check_host;
  std::vector<CUtensorMap> maps;

  float* A() const { return reinterpret_cast<float*>(base + L.off_A); }
  float* Q() const { return reinterpret_cast<float*>(base + L.off_Q); }
  float* lam() const { return reinterpret_cast<float*>(base + L.off_lam); }
  float* M() const { return reinterpret_cast<float*>(base + L.off_M); }
  uint32_t* flags() const { return reinterpret_cast<uint32_t*>(base + L.off_flags); }
  float* stats() const { return reinterpret_cast<float*>(base + L.off_stats); }
  float* check() const { return reinterpret_cast<float*>(base + L.off_check); }
  float* colsq() const { return reinterpret_cast<float*>(base + L.off_colsq); }
  MatInfo* dinfo() const { return reinterpret_cast<MatInfo*>(base + L.off_info); }
  Tile* dtiles() const { return reinterpret_cast<Tile*>(base + L.off_tiles); }
  float* scratch() const { return reinterpret_cast<float*>(base + L.off_scratch); }
  uint32_t* err() const { return reinterpret_cast<uint32_t*>(base + L.off_err); }
  void* dmaps() const { return base + L.off_maps; }
  float* gj_rbuf() const { return reinterpret_cast<float*>(base + L.off_gj_rbuf); }
  GjCtl* gj_ctl() const { return reinterpret_cast<GjCtl*>(base + L.off_gj_ctl); }
  int32_t* gj_count() const { return reinterpret_cast<int32_t*>(base + L.off_gj_count); }
  unsigned char* pack() const { return reinterpret_cast<unsigned char*>(base + L.off_pack); }
};

namespace {

dobb_status check_handle(dobb_handle h) {
  if (!h) return fail(DOBB_ERR_STATE, "NULL handle");
  int dev = -1;
  CUDA_TRY(cudaGetDevice(&dev));
  if (dev != h->device)
    return fail(DOBB_ERR_STATE, "current device %d differs from the handle's device %d", dev, h->device);
  return DOBB_OK;
}

dobb_status do_pack(dobb_handle h, cudaStream_t s) {
  if (!h->any_tc) return DOBB_OK;
  const int g = std::max(1, std::min(h->wl.blocks_n, h->sm_count * 8));
  cudaError_t e = launch_pack_bases(h->Q(), h->pack(), h->dinfo(), h->dtiles() + h->wl.blocks_off,
                                    h->wl.blocks_n, h->basis_bf16 ? 1 : 2, g, s);
  if (e != cudaSuccess) return fail(DOBB_ERR_CUDA, "pack launch: %s", cudaGetErrorString(e));
  ++h->launches;
  return DOBB_OK;
}

// Run grid batches (the eigensolver, or the orthogonal iteration when
// orth_steps > 0): batch i on the caller's stream (i % 3 == 0) or one of the
// handle's two streams, joined back into the caller's stream.
cudaError_t run_grid_batches(dobb_handle h, const GjArgs* batches, int nb, cudaStream_t s,
                             int orth_steps) {
  if (nb <= 0) return cudaSuccess;
  cudaStream_t streams[kGjMaxBatches];
  const int nstreams = std::min(nb, kGjStreams + 1);
  for (int b = 0; b < nb; ++b) streams[b] = (b % nstreams) == 0 ? s : h->gj_streams[b % nstreams - 1];
  cudaError_t e = cudaSuccess;
  if (nstreams > 1) {
    e = cudaEventRecord(h->gj_events[0], s);
    for (int i = 1; i < nstreams && e == cudaSuccess; ++i)
      e = cudaStreamWaitEvent(h->gj_streams[i - 1], h->gj_events[0], 0);
    if (e != cudaSuccess) return e;
  }
  e = orth_steps > 0 ? run_orth_grid(batches, nb, streams, orth_steps, h->sm_count, &h->launches)
                     : run_jacobi_grid(batches, nb, streams, h->gj_host_counts, &h->launches);
  for (int i = 1; i < nstreams; ++i) {
    cudaError_t e2 = cudaEventRecord(h->gj_events[i], h->gj_streams[i - 1]);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(s, h->gj_events[i], 0);
    if (e == cudaSuccess) e = e2;
  }
  return e;
}

// The blocks of chunk ch at least gj_min_k wide (the front of its list,
// sorted by decreasing k) on the grid, with the eigensolver (orth_steps = 0)
// or the orthogonal iteration.  Batches are runs of one width, split by the
// byte budget, or in two when no budget is set and the width has many blocks
// (two batches of one width interleave their latency-bound and
// bandwidth-bound launches).  Sets *g_end to the first block left for the
// one-CTA kernels.
dobb_status grid_refresh(dobb_handle h, const Chunk& ch, cudaStream_t s, int orth_steps, int* g_end) {
  const Tile* items = h->wl.tiles.data() + ch.eig_off;
  auto kof = [&](int idx) { return (int)(h->n[items[idx].mat] / h->B); };
  const char* what = orth_steps > 0 ? "grid orthogonal iteration" : "grid eigensolver";
  int g0 = 0;
  if (h->gj_min_k > 0) {
    GjArgs batches[kGjMaxBatches];
    int nb = 0;
    int64_t ctl_off = 0, rbuf_off = 0;
    while (g0 < ch.eig_n && kof(g0) >= h->gj_min_k) {
      const int k = kof(g0);
      int g1 = g0;
      while (g1 < ch.eig_n && kof(g1) == k) ++g1;
      const int count = g1 - g0;
      int per = std::min(count, gj_batch_items(k, h->gj_batch_bytes));
      if (h->gj_batch_bytes == 0 && count >= 64) per = (count + 1) / 2;
      for (int b0 = g0; b0 < g1; b0 += per) {
        const int nitems = std::min(per, g1 - b0);
        if (nb == kGjMaxBatches) {
          cudaError_t e = run_grid_batches(h, batches, nb, s, orth_steps);
          if (e != cudaSuccess) return fail(DOBB_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
          nb = 0;
          ctl_off = rbuf_off = 0;
        }
        if ((size_t)(ctl_off + nitems) > h->L.gj_ctl_items ||
            (size_t)(rbuf_off + (int64_t)nitems * gj_rbuf_floats(k)) > h->L.gj_rbuf_floats)
          return fail(DOBB_ERR_STATE, "grid eigensolver buffers too small for width %d", k);
        GjArgs& ga = batches[nb];
        ga = GjArgs{};
        ga.info = h->dinfo();
        ga.items = h->dtiles() + ch.eig_off + b0;
        ga.nitems = nitems;
        ga.k = k;
        ga.A = h->A();
        ga.Q = h->Q();
        ga.lam = h->lam();
        ga.scratch = h->scratch();
        ga.rbuf = h->gj_rbuf() + rbuf_off;
        ga.rstride = gj_rbuf_floats(k);
        ga.ctl = h->gj_ctl() + ctl_off;
        ga.active_count = h->gj_count() + nb;
        ga.flags = h->flags();
        ga.stats = h->stats();
        ga.max_sweeps = h->max_sweeps;
        ga.tol = h->tol;
        ctl_off += nitems;
        rbuf_off += (int64_t)nitems * gj_rbuf_floats(k);
        ++nb;
      }
      g0 = g1;
    }
    cudaError_t e = run_grid_batches(h, batches, nb, s, orth_steps);
    if (e != cudaSuccess) return fail(DOBB_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  }
  *g_end = g0;
  return DOBB_OK;
}

// Orthogonal iteration: blocks at least gj_min_k wide on the grid, the rest
// one CTA per block.
dobb_status do_refresh_orth(dobb_handle h, cudaStream_t s) {
  for (const Chunk& ch : h->wl.chunks) {
    if (ch.eig_n == 0) continue;
    int g0 = 0;
    dobb_status st = grid_refresh(h, ch, s, h->orth_steps, &g0);
    if (st != DOBB_OK) return st;
    if (g0 >= ch.eig_n) continue;
    EigArgs a{};
    a.info = h->dinfo();
    a.tiles = h->dtiles() + ch.eig_off + g0;
    a.num_tiles = ch.eig_n - g0;
    a.A = h->A();
    a.Q = h->Q();
    a.lam = h->lam();
    a.scratch = h->scratch();
    a.flags = h->flags();
    a.stats = h->stats();
    const int g = std::max(1, std::min(a.num_tiles, h->sm_count));
    cudaError_t e = launch_orth(a, h->orth_steps, g, s);
    if (e != cudaSuccess) return fail(DOBB_ERR_CUDA, "orthogonal-iteration launch: %s", cudaGetErrorString(e));
    ++h->launches;
  }
  return do_pack(h, s);
}

dobb_status do_refresh(dobb_handle h, cudaStream_t s) {
  if (h->refresh_method == DOBB_REFRESH_ORTH) return do_refresh_orth(h, s);
  // blocks whose solver fits in half of an SM's shared memory run two CTAs per SM
  const size_t half = h->smem_per_sm / 2 > 2048 ? h->smem_per_sm / 2 - 2048 : 0;
  for (const Chunk& ch : h->wl.chunks) {
    if (ch.eig_n == 0) continue;
    // the list is sorted by decreasing k: [grid solver | one CTA per SM | two or more]
    const Tile* items = h->wl.tiles.data() + ch.eig_off;
    auto kof = [&](int idx) { return (int)(h->n[items[idx].mat] / h->B); };
    int g0 = 0;
    dobb_status st = grid_refresh(h, ch, s, 0, &g0);
    if (st != DOBB_OK) return st;
    int b = g0;
    while (b < ch.eig_n && jacobi_smem_for(kof(b), half) == 0) ++b;
    EigArgs a{};
    a.info = h->dinfo();
    a.max_sweeps = h->max_sweeps;
    a.A = h->A();
    a.Q = h->Q();
    a.lam = h->lam();
    a.scratch = h->scratch();
    a.flags = h->flags();
    a.stats = h->stats();
    a.tol = h->tol;
    for (int part = 0; part < 2; ++part) {
      const int lo = part == 0 ? g0 : b, hi = part == 0 ? b : ch.eig_n;
      if (hi <= lo) continue;
      size_t smem = 0;
      for (int idx = lo; idx < hi; ++idx) {
        const size_t need = jacobi_smem_for(kof(idx), part == 0 ? h->smem_limit : half);
        if (need == 0) return fail(DOBB_ERR_UNSUPPORTED, "block width %d exceeds the eigensolver's shared memory", kof(idx));
        smem = std::max(smem, need);
      }
      a.tiles = h->dtiles() + ch.eig_off + lo;
      a.num_tiles = hi - lo;
      const int by_smem = std::max(1, (int)(h->smem_per_sm / (smem + 1024)));
      const int per_sm = std::min(jacobi_ctas_per_sm(), by_smem);
      const int g = std::max(1, std::min(a.num_tiles, h->sm_count * per_sm));
      cudaError_t e = launch_jacobi(a, g, smem, s);
      if (e != cudaSuccess) return fail(DOBB_ERR_CUDA, "eigen launch: %s", cudaGetErrorString(e));
      ++h->launches;
    }
  }
  return do_pack(h, s);
}

dobb_status do_step(dobb_handle h, void* const* W, const void* const* G, float lr,
                    int8_t* const* S_out, cudaStream_t s) {
  if (!W || !G) return fail(DOBB_ERR_INVALID_ARG, "W and G arrays must be non-NULL");
  for (int i = 0; i < h->num; ++i)
    if (!W[i] || !G[i]) return fail(DOBB_ERR_INVALID_ARG, "W[%d] or G[%d] is NULL", i, i);
  if (!(lr == lr)) return fail(DOBB_ERR_INVALID_ARG, "lr is NaN");
  if (h->T > 0 && h->t % h->T == 0) {
    dobb_status st = do_refresh(h, s);
    if (st != DOBB_OK) return st;
  }
  // zero the per-step sums (slots 0 and 1 of each block's 4 stats)
  CUDA_TRY(cudaMemset2DAsync(h->stats(), 16, 0, 8, (size_t)h->L.nblocks, s));
  bool aligned = true;
  for (int i = 0; i < h->num; ++i)
    if ((reinterpret_cast<uintptr_t>(W[i]) | reinterpret_cast<uintptr_t>(G[i])) % 16 != 0) aligned = false;
  const bool l2 = h->norm == DOBB_NORM_L2;
  const bool use_tc = h->path == 0 && aligned && !l2;
  for (const Chunk& ch : h->wl.chunks) {
    if (ch.step_n == 0) continue;
    StepArgs a{};
    a.info = h->dinfo();
    a.tiles = h->dtiles() + ch.step_off;
    a.num_tiles = ch.step_n;
    a.mat_base = ch.mat_base;
    a.Q = h->Q();
    a.M = h->M();
    a.flags = h->flags();
    a.stats = h->stats();
    a.beta1 = h->beta1;
    a.lr_s = lr * h->scale_s;
    a.basis_bf16 = h->basis_bf16 ? 1 : 0;
    a.mode = kModeSign;
    a.colsq = h->colsq();
    for (int i = ch.mat_base; i < ch.mat_end; ++i) {
      a.W[i - ch.mat_base] = W[i];
      a.G[i - ch.mat_base] = G[i];
      a.S[i - ch.mat_base] = S_out ? S_out[i] : nullptr;
    }
    if (use_tc && ch.tc_n > 0) {
      // two launches: blocks wider than kTcSmallK, then the narrow ones
      for (int part = 0; part < 2; ++part) {
        const int lo = part == 0 ? 0 : ch.tc_small, hi = part == 0 ? ch.tc_small : ch.tc_n;
        if (hi <= lo) continue;
        int kmax = 4;
        for (int j = lo; j < hi; ++j) {
          const Tile& tl = h->wl.tiles[ch.tc_off + j];
          kmax = std::max(kmax, (int)(h->n[tl.mat] / h->B));
        }
        StepArgs at = a;
        at.tiles = h->dtiles() + ch.tc_off + lo;
        at.num_tiles = hi - lo;
        TcArgs t{};
        t.maps = h->dmaps();
        t.qpack = h->pack();
        t.err = h->err();
        t.bstage = (int32_t)step_tc_bstage(kmax);
        t.nastage = step_tc_astages(kmax);
        t.nbstage = step_tc_bstages(kmax, t.nastage, h->smem_limit);
        t.npieces = h->basis_bf16 ? 1 : 2;
        t.rpieces = h->basis_bf16 ? 1 : 3;
        t.defer = ((kmax + 15) & ~15) <= 128 ? 1 : 0;
        if (t.nbstage < 2)
          return fail(DOBB_ERR_UNSUPPORTED, "block width %d leaves no room for operand stages", kmax);
        const size_t smem = step_tc_smem(kmax, t.nastage, t.nbstage);
        const int g = std::max(1, std::min(hi - lo, h->sm_count));
        bool may_t = false;
        for (int i = ch.mat_base; i < ch.mat_end; ++i) may_t = may_t || h->info[i].wt;
        cudaError_t e = launch_step_tc(at, t, h->pdt, may_t, g, smem, s);
        if (e != cudaSuccess) return fail(DOBB_ERR_CUDA, "tensor-core step launch: %s", cudaGetErrorString(e));
        ++h->launches;
      }
    }
    if (l2) {
      // column l2: pass 1 over every (matrix, block) of the chunk (momentum
      // update and column sums of C^2), then the update with scaled coefficients
      StepArgs an = a;
      an.tiles = h->dtiles() + ch.l2_off;
      an.num_tiles = ch.l2_n;
      const MatInfo& m0 = h->info[ch.mat_base];
      const MatInfo& m1 = h->info[ch.mat_end - 1];
      CUDA_TRY(cudaMemsetAsync(h->colsq() + m0.lam_off, 0,
                               4 * (size_t)(m1.lam_off + (int64_t)m1.B * m1.k - m0.lam_off), s));
      const size_t smem = step_smem_for(ch.max_k);
      const int by_smem = std::max(1, (int)(h->smem_per_sm / (smem + 1024)));
      const int g = std::max(1, std::min(an.num_tiles, h->sm_count * std::min(4, by_smem)));
      cudaError_t e = launch_l2_norms(an, h->pdt, g, smem, s);
      if (e != cudaSuccess) return fail(DOBB_ERR_CUDA, "column-norm launch: %s", cudaGetErrorString(e));
      ++h->launches;
      a.mode = kModeL2Apply;
    }
    const bool rest_only = use_tc && ch.tc_n > 0;
    const int n_ffma = rest_only ? ch.rest_n : ch.step_n;
    if (n_ffma == 0) continue;
    a.tiles = h->dtiles() + (rest_only ? ch.rest_off : ch.step_off);
    a.num_tiles = n_ffma;
    const int kmax = rest_only ? ch.max_k_rest : ch.max_k;
    const size_t smem = step_smem_for(kmax);
    if (smem > h->smem_limit)
      return fail(DOBB_ERR_UNSUPPORTED, "block width %d needs %zu bytes of shared memory", kmax, smem);
    const int by_smem = std::max(1, (int)(h->smem_per_sm / (smem + 1024)));
    const int g = std::max(1, std::min(n_ffma, h->sm_count * std::min(4, by_smem)));
    cudaError_t e = launch_step_ffma(a, h->pdt, g, smem, s);
    if (e != cudaSuccess) return fail(DOBB_ERR_CUDA, "step launch: %s", cudaGetErrorString(e));
    ++h->launches;
  }
  h->t += 1;
  return DOBB_OK;
}

}  // namespace

extern "C" {

const char* dobb_last_error(void) { return g_err.c_str(); }

size_t dobb_state_bytes(int num_matrices, const int64_t* m, const int64_t* n, int B) {
  if (!validate_shapes(num_matrices, m, n, B)) return 0;
  WorkLists wl = build_work(num_matrices, m, n, B);
  return compute_layout(num_matrices, m, n, B, wl.tiles.size()).total;
}

dobb_status dobb_create(dobb_handle* out, int num_matrices, const int64_t* m, const int64_t* n,
                        int B, float beta1, float beta2, int refresh_period, float scale_s,
                        dobb_dtype param_dtype, dobb_dtype act_dtype, void* state_mem,
                        size_t state_bytes, void* stream) {
  g_err.clear();
  if (!out) return fail(DOBB_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!validate_shapes(num_matrices, m, n, B)) return DOBB_ERR_INVALID_ARG;
  if (!(beta1 >= 0.f && beta1 < 1.f) || !(beta2 >= 0.f && beta2 < 1.f))
    return fail(DOBB_ERR_INVALID_ARG, "beta1=%g beta2=%g must lie in [0, 1)", beta1, beta2);
  if (refresh_period < 0) return fail(DOBB_ERR_INVALID_ARG, "refresh_period must be >= 0");
  if (!(scale_s == scale_s)) return fail(DOBB_ERR_INVALID_ARG, "scale_s is NaN");
  if ((param_dtype != DOBB_F32 && param_dtype != DOBB_BF16) ||
      (act_dtype != DOBB_F32 && act_dtype != DOBB_BF16))
    return fail(DOBB_ERR_INVALID_ARG, "unknown dtype");
  if (!state_mem) return fail(DOBB_ERR_INVALID_ARG, "state_mem is NULL");
  if (reinterpret_cast<uintptr_t>(state_mem) % kAlign != 0)
    return fail(DOBB_ERR_INVALID_ARG, "state_mem must be %zu-byte aligned", kAlign);

  dobb_ctx* h = new dobb_ctx();
  h->num = num_matrices;
  h->B = B;
  h->beta1 = beta1;
  h->beta2 = beta2;
  h->T = refresh_period;
  h->scale_s = scale_s;
  h->pdt = param_dtype;
  h->adt = act_dtype;
  h->m.assign(m, m + num_matrices);
  h->n.assign(n, n + num_matrices);
  h->wl = build_work(num_matrices, m, n, B);
  h->L = compute_layout(num_matrices, m, n, B, h->wl.tiles.size());
  if (state_bytes < h->L.total) {
    size_t need = h->L.total;
    delete h;
    return fail(DOBB_ERR_STATE, "state buffer of %zu bytes is smaller than the %zu required",
                state_bytes, need);
  }
  h->base = static_cast<char*>(state_mem);
  h->bytes = state_bytes;

  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->sm_count, cudaDevAttrMultiProcessorCount, h->device);
  int optin = 0, per_sm = 0;
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, h->device);
  h->smem_per_sm = (size_t)per_sm;
  if (e != cudaSuccess) {
    delete h;
    return fail(DOBB_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
  }
  h->smem_limit = (size_t)optin - 2048;  // room for static shared memory
  if ((e = configure_jacobi(h->smem_limit)) != cudaSuccess || (e = configure_orth()) != cudaSuccess ||
      (e = configure_jacobi_grid(h->smem_limit)) != cudaSuccess ||
      (e = configure_step(h->smem_limit)) != cudaSuccess ||
      (e = configure_step_tc(h->smem_limit)) != cudaSuccess ||
      (e = configure_syrk_tc(h->smem_limit)) != cudaSuccess) {
    delete h;
    return fail(DOBB_ERR_CUDA, "kernel configuration: %s", cudaGetErrorString(e));
  }

  for (int i = 0; i < kGjStreams && e == cudaSuccess; ++i)
    e = cudaStreamCreateWithFlags(&h->gj_streams[i], cudaStreamNonBlocking);
  for (int i = 0; i <= kGjStreams && e == cudaSuccess; ++i)
    e = cudaEventCreateWithFlags(&h->gj_events[i], cudaEventDisableTiming);
  if (e != cudaSuccess) {
    delete h;
    return fail(DOBB_ERR_CUDA, "stream creation: %s", cudaGetErrorString(e));
  }

  // per-matrix metadata
  int64_t aoff = 0, loff = 0, moff = 0, poff = 0;
  int32_t blk = 0;
  for (int i = 0; i < num_matrices; ++i) {
    MatInfo mi{};
    mi.m = m[i];
    mi.n = n[i];
    mi.k = (int32_t)(n[i] / B);
    mi.B = B;
    mi.blk0 = blk;
    mi.a_off = aoff;
    mi.lam_off = loff;
    mi.m_off = moff;
    mi.tc = tc_eligible(m[i], n[i], mi.k) ? 1 : 0;
    mi.qblk_bytes = mi.tc ? tc_block_image_bytes(mi.k) : 0;
    mi.qp_off = poff;
    h->info.push_back(mi);
    aoff += (int64_t)B * mi.k * mi.k;
    loff += (int64_t)B * mi.k;
    moff += pad16f(m[i] * n[i]);
    poff += (int64_t)B * mi.qblk_bytes;
    blk += B;
    h->any_tc = h->any_tc || mi.tc;
  }
  // one TMA descriptor per matrix for its momentum (fp32, box 32 x 128, 128B swizzle)
  h->maps.assign(num_matrices, CUtensorMap{});
  h->xmaps.assign(num_matrices, CUtensorMap{});
  h->xmap_ptr.assign(num_matrices, nullptr);
  h->xmap_N.assign(num_matrices, -1);
  if (h->any_tc || (act_dtype == DOBB_BF16 && !h->wl.syrk_tc.empty())) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || fn == nullptr || q != cudaDriverEntryPointSuccess) {
      delete h;
      return fail(DOBB_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
    }
    auto encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    h->encode = encode;
    for (int i = 0; i < num_matrices; ++i) {
      const MatInfo& mi = h->info[i];
      if (!mi.tc) continue;
      cuuint64_t dims[2] = {(cuuint64_t)mi.n, (cuuint64_t)mi.m};
      cuuint64_t strides[1] = {(cuuint64_t)mi.n * 4};
      cuuint32_t box[2] = {32, 128};
      cuuint32_t estr[2] = {1, 1};
      CUresult r = encode(&h->maps[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, h->M() + mi.m_off, dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) {
        delete h;
        return fail(DOBB_ERR_CUDA, "tensor map encode failed for matrix %d (code %d)", i, (int)r);
      }
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Layout& L = h->L;
  e = cudaMemcpyAsync(h->dinfo(), h->info.data(), sizeof(MatInfo) * h->info.size(),
                      cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(h->dtiles(), h->wl.tiles.data(), sizeof(Tile) * h->wl.tiles.size(),
                        cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->base + L.off_A, 0, 4 * L.a_floats, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->base + L.off_M, 0, 4 * L.m_floats, s);
  if (e == cudaSuccess && h->any_tc)
    e = cudaMemcpyAsync(h->dmaps(), h->maps.data(), sizeof(CUtensorMap) * h->maps.size(),
                        cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(h->base + L.off_flags, 0, L.off_info - L.off_flags, s);
  if (e == cudaSuccess) {
    const int g = std::max(1, std::min(h->wl.blocks_n, h->sm_count * 4));
    e = launch_init_bases(h->Q(), h->lam(), h->dinfo(), h->dtiles() + h->wl.blocks_off,
                          h->wl.blocks_n, g, s);
    ++h->launches;
  }
  if (e == cudaSuccess && do_pack(h, s) != DOBB_OK) e = cudaErrorUnknown;
  // the host arrays above must outlive the asynchronous copies: they belong
  // to the handle; make the copies complete before returning anyway so the
  // caller may reuse its shape arrays and the first call sees a ready state.
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    delete h;
    return fail(DOBB_ERR_CUDA, "state initialisation: %s", cudaGetErrorString(e));
  }
  *out = h;
  return DOBB_OK;
}

dobb_status dobb_destroy(dobb_handle h) {
  if (!h) return fail(DOBB_ERR_STATE, "NULL handle");
  delete h;
  return DOBB_OK;
}

dobb_status dobb_accumulate_moments(dobb_handle h, const void* const* X, const int64_t* N,
                                    void* stream) {
  dobb_status st = check_handle(h);
  if (st != DOBB_OK) return st;
  if (!X || !N) return fail(DOBB_ERR_INVALID_ARG, "X and N arrays must be non-NULL");
  for (int i = 0; i < h->num; ++i)
    if (N[i] < 0) return fail(DOBB_ERR_INVALID_ARG, "N[%d] < 0", i);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool x_aligned = true;
  for (int i = 0; i < h->num; ++i)
    if (X[i] && reinterpret_cast<uintptr_t>(X[i]) % 16 != 0) x_aligned = false;
  const bool use_tc = h->path == 0 && h->adt == DOBB_BF16 && h->encode && x_aligned &&
                      !h->wl.syrk_tc.empty();
  if (use_tc) {
    SyrkTcArgs* a = new SyrkTcArgs();
    for (const SyrkChunk& sc : h->wl.syrk_tc) {
      std::memset(a, 0, sizeof(SyrkTcArgs));
      a->info = h->dinfo();
      a->tiles = h->dtiles() + sc.off;
      a->num_tiles = sc.n;
      a->mat_base = sc.mat_base;
      a->A = h->A();
      a->flags = h->flags();
      a->err = h->err();
      a->beta2 = h->beta2;
      for (int i = sc.mat_base; i < sc.mat_end; ++i) {
        const int slot = i - sc.mat_base;
        a->X[slot] = X[i];
        a->N[slot] = X[i] ? N[i] : 0;
        if (!X[i] || N[i] <= 0 || !syrk_tc_eligible(h->n[i], (int)(h->n[i] / h->B))) continue;
        if (h->xmap_ptr[i] != X[i] || h->xmap_N[i] != N[i]) {
          cuuint64_t dims[2] = {(cuuint64_t)h->n[i], (cuuint64_t)N[i]};
          cuuint64_t strides[1] = {(cuuint64_t)h->n[i] * 2};
          cuuint32_t box[2] = {64, 64};
          cuuint32_t estr[2] = {1, 1};
          CUresult r = h->encode(&h->xmaps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                 const_cast<void*>(X[i]), dims, strides, box, estr,
                                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
          if (r != CUDA_SUCCESS) {
            delete a;
            return fail(DOBB_ERR_CUDA, "X tensor map encode failed for matrix %d (code %d)", i, (int)r);
          }
          h->xmap_ptr[i] = X[i];
          h->xmap_N[i] = N[i];
        }
        a->maps[slot] = h->xmaps[i];
      }
      // two launches: blocks wider than kTcSmallK, then the narrow ones with
      // stages sized for them (more tokens in flight)
      for (int part = 0; part < 2; ++part) {
        const int lo = part == 0 ? 0 : sc.small, hi = part == 0 ? sc.small : sc.n;
        if (hi <= lo) continue;
        int kmax = 8;
        for (int j = lo; j < hi; ++j) {
          const Tile& tl = h->wl.tiles[sc.off + j];
          kmax = std::max(kmax, (int)(h->n[tl.mat] / h->B));
        }
        a->tiles = h->dtiles() + sc.off + lo;
        a->num_tiles = hi - lo;
        a->stages = syrk_tc_stages(kmax, h->smem_limit - 1024);
        a->stage_bytes = (int32_t)syrk_tc_stage_bytes(kmax);
        a->dbuf = syrk_tc_double_buffer(kmax) ? 1 : 0;
        const size_t smem = syrk_tc_smem(kmax, a->stages);
        const int g = std::max(1, std::min(hi - lo, h->sm_count));
        cudaError_t e = launch_syrk_tc(*a, g, smem, s);
        if (e != cudaSuccess) {
          delete a;
          return fail(DOBB_ERR_CUDA, "tensor-core accumulate launch: %s", cudaGetErrorString(e));
        }
        ++h->launches;
      }
    }
    delete a;
    // the matrices the tensor-core kernel does not cover: one FFMA launch per
    // chunk that has any
    for (const Chunk& ch : h->wl.chunks) {
      if (ch.syrk_rest_n == 0) continue;
      AccArgs r{};
      r.info = h->dinfo();
      r.tiles = h->dtiles() + ch.syrk_rest_off;
      r.num_tiles = ch.syrk_rest_n;
      r.mat_base = ch.mat_base;
      r.A = h->A();
      r.flags = h->flags();
      r.beta2 = h->beta2;
      for (int i = ch.mat_base; i < ch.mat_end; ++i) {
        r.X[i - ch.mat_base] = X[i];
        r.N[i - ch.mat_base] = X[i] ? N[i] : 0;
      }
      const int g = std::max(1, std::min(r.num_tiles, h->sm_count * 4));
      cudaError_t e = launch_syrk_ema(r, h->adt, g, s);
      if (e != cudaSuccess) return fail(DOBB_ERR_CUDA, "accumulate launch: %s", cudaGetErrorString(e));
      ++h->launches;
    }
    return DOBB_OK;
  }
  for (const Chunk& ch : h->wl.chunks) {
    if (ch.syrk_n == 0) continue;
    AccArgs a{};
    a.info = h->dinfo();
    a.tiles = h->dtiles() + ch.syrk_off;
    a.num_tiles = ch.syrk_n;
    a.mat_base = ch.mat_base;
    a.A = h->A();
    a.flags = h->flags();
    a.beta2 = h->beta2;
    for (int i = ch.mat_base; i < ch.mat_end; ++i) {
      a.X[i - ch.mat_base] = X[i];
      a.N[i - ch.mat_base] = X[i] ? N[i] : 0;
    }
    const int g = std::max(1, std::min(ch.syrk_n, h->sm_count * 4));
    cudaError_t e = launch_syrk_ema(a, h->adt, g, s);
    if (e != cudaSuccess) return fail(DOBB_ERR_CUDA, "accumulate launch: %s", cudaGetErrorString(e));
    ++h->launches;
  }
  return DOBB_OK;
}

dobb_status dobb_refresh_bases(dobb_handle h, void* stream) {
  dobb_status st = check_handle(h);
  if (st != DOBB_OK) return st;
  return do_refresh(h, static_cast<cudaStream_t>(stream));
}

dobb_status dobb_step(dobb_handle h, void* const* W, const void* const* G, float lr, void* stream) {
  dobb_status st = check_handle(h);
  if (st != DOBB_OK) return st;
  return do_step(h, W, G, lr, nullptr, static_cast<cudaStream_t>(stream));
}

dobb_status dobb_step_with_signs(dobb_handle h, void* const* W, const void* const* G, float lr,
                                 int8_t* const* S_out, void* stream) {
  dobb_status st = check_handle(h);
  if (st != DOBB_OK) return st;
  if (!S_out) return fail(DOBB_ERR_INVALID_ARG, "S_out is NULL");
  return do_step(h, W, G, lr, S_out, static_cast<cudaStream_t>(stream));
}

dobb_status dobb_get_step(dobb_handle h, int64_t* t) {
  if (!h || !t) return fail(DOBB_ERR_INVALID_ARG, "NULL argument");
  *t = h->t;
  return DOBB_OK;
}

dobb_status dobb_set_step(dobb_handle h, int64_t t) {
  if (!h || t < 0) return fail(DOBB_ERR_INVALID_ARG, "bad handle or negative step");
  h->t = t;
  return DOBB_OK;
}

dobb_status dobb_set_basis_dtype(dobb_handle h, dobb_dtype basis_dtype, void* stream) {
  if (!h) return fail(DOBB_ERR_INVALID_ARG, "NULL handle");
  if (basis_dtype != DOBB_F32 && basis_dtype != DOBB_BF16)
    return fail(DOBB_ERR_INVALID_ARG, "basis dtype must be DOBB_F32 or DOBB_BF16");
  h->basis_bf16 = basis_dtype == DOBB_BF16;
  // the tensor-core operand images hold the basis in the chosen precision
  return do_pack(h, static_cast<cudaStream_t>(stream));
}

dobb_status dobb_set_normalization(dobb_handle h, int norm) {
  if (!h) return fail(DOBB_ERR_INVALID_ARG, "NULL handle");
  if (norm != DOBB_NORM_SIGN && norm != DOBB_NORM_L2)
    return fail(DOBB_ERR_INVALID_ARG, "normalisation must be DOBB_NORM_SIGN or DOBB_NORM_L2");
  if (norm == DOBB_NORM_L2) {
    for (int i = 0; i < h->num; ++i)
      if (h->n[i] / h->B > l2_max_k())
        return fail(DOBB_ERR_UNSUPPORTED, "column-l2 normalisation supports blocks up to %d wide", l2_max_k());
    if (step_smem_for((int)(h->n[0] / h->B)) > h->smem_limit)
      return fail(DOBB_ERR_UNSUPPORTED, "block too wide for the FP32 update kernel");
  }
  h->norm = norm;
  return DOBB_OK;
}

dobb_status dobb_set_side(dobb_handle h, int matrix, int side, void* stream) {
  if (!h) return fail(DOBB_ERR_INVALID_ARG, "NULL handle");
  if (matrix < -1 || matrix >= h->num) return fail(DOBB_ERR_INVALID_ARG, "matrix %d out of range", matrix);
  if (side != DOBB_SIDE_INPUT && side != DOBB_SIDE_OUTPUT)
    return fail(DOBB_ERR_INVALID_ARG, "side must be DOBB_SIDE_INPUT or DOBB_SIDE_OUTPUT");
  const int lo = matrix < 0 ? 0 : matrix, hi = matrix < 0 ? h->num : matrix + 1;
  for (int i = lo; i < hi; ++i) {
    if (side == DOBB_SIDE_OUTPUT && step_smem_for(h->info[i].k) > h->smem_limit)
      return fail(DOBB_ERR_UNSUPPORTED, "block too wide for the FP32 update kernel");
  }
  for (int i = lo; i < hi; ++i) h->info[i].wt = side == DOBB_SIDE_OUTPUT ? 1 : 0;
  CUDA_TRY(cudaMemcpyAsync(h->dinfo() + lo, h->info.data() + lo, sizeof(MatInfo) * (size_t)(hi - lo),
                           cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream)));
  // the host copy is the source of an asynchronous transfer: finish it here
  CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  return DOBB_OK;
}

dobb_status dobb_set_refresh(dobb_handle h, int method, int steps) {
  if (!h) return fail(DOBB_ERR_INVALID_ARG, "NULL handle");
  if (method != DOBB_REFRESH_EIGH && method != DOBB_REFRESH_ORTH)
    return fail(DOBB_ERR_INVALID_ARG, "refresh method must be DOBB_REFRESH_EIGH or DOBB_REFRESH_ORTH");
  if (steps < 1) return fail(DOBB_ERR_INVALID_ARG, "orthogonal-iteration steps must be >= 1");
  h->refresh_method = method;
  h->orth_steps = steps;
  return DOBB_OK;
}

dobb_status dobb_set_refresh_period(dobb_handle h, int refresh_period) {
  if (!h) return fail(DOBB_ERR_INVALID_ARG, "NULL handle");
  if (refresh_period < 0) return fail(DOBB_ERR_INVALID_ARG, "refresh_period must be >= 0");
  h->T = refresh_period;
  return DOBB_OK;
}

dobb_status dobb_set_eig_grid(dobb_handle h, int min_k, int64_t batch_bytes) {
  if (!h) return fail(DOBB_ERR_INVALID_ARG, "NULL handle");
  if (min_k != 0 && min_k < kGjMinK)
    return fail(DOBB_ERR_INVALID_ARG, "grid eigensolver width threshold must be 0 or >= %d", kGjMinK);
  if (batch_bytes < 0) return fail(DOBB_ERR_INVALID_ARG, "batch_bytes must be >= 0");
  h->gj_min_k = min_k;
  h->gj_batch_bytes = batch_bytes;
  return DOBB_OK;
}

dobb_status dobb_set_jacobi(dobb_handle h, int max_sweeps, float tol) {
  if (!h || max_sweeps < 1 || !(tol >= 0.f)) return fail(DOBB_ERR_INVALID_ARG, "bad eigensolver settings");
  h->max_sweeps = max_sweeps;
  h->tol = tol;
  return DOBB_OK;
}

dobb_status dobb_state_tensor(dobb_handle h, dobb_tensor which, int matrix, void** dev_ptr,
                              size_t* bytes) {
  if (!h || !dev_ptr || !bytes) return fail(DOBB_ERR_INVALID_ARG, "NULL argument");
  if (matrix < -1 || matrix >= h->num) return fail(DOBB_ERR_INVALID_ARG, "matrix %d out of range", matrix);
  const MatInfo* mi = matrix >= 0 ? &h->info[matrix] : nullptr;
  switch (which) {
    case DOBB_T_MOMENTS:
    case DOBB_T_BASES: {
      float* base = which == DOBB_T_MOMENTS ? h->A() : h->Q();
      if (mi) {
        *dev_ptr = base + mi->a_off;
        *bytes = 4 * (size_t)mi->B * mi->k * mi->k;
      } else {
        *dev_ptr = base;
        *bytes = 4 * h->L.a_floats;
      }
      return DOBB_OK;
    }
    case DOBB_T_EIGVALS:
      *dev_ptr = mi ? h->lam() + mi->lam_off : h->lam();
      *bytes = mi ? 4 * (size_t)mi->B * mi->k : 4 * h->L.lam_floats;
      return DOBB_OK;
    case DOBB_T_MOMENTUM:
      *dev_ptr = mi ? h->M() + mi->m_off : h->M();
      *bytes = mi ? 4 * (size_t)(mi->m * mi->n) : 4 * h->L.m_floats;
      return DOBB_OK;
    case DOBB_T_FLAGS:
      *dev_ptr = mi ? h->flags() + mi->blk0 : h->flags();
      *bytes = 4 * (mi ? (size_t)mi->B : (size_t)h->L.nblocks);
      return DOBB_OK;
    case DOBB_T_STATS:
      *dev_ptr = mi ? h->stats() + 4 * (size_t)mi->blk0 : h->stats();
      *bytes = 16 * (mi ? (size_t)mi->B : (size_t)h->L.nblocks);
      return DOBB_OK;
    case DOBB_T_ERROR:
      *dev_ptr = h->err();
      *bytes = 4;
      return DOBB_OK;
  }
  return fail(DOBB_ERR_INVALID_ARG, "unknown tensor %d", (int)which);
}

int64_t dobb_num_blocks(dobb_handle h) { return h ? h->L.nblocks : -1; }

int64_t dobb_block_offset(dobb_handle h, int matrix) {
  if (!h || matrix < 0 || matrix >= h->num) return -1;
  return h->info[matrix].blk0;
}

dobb_status dobb_get_block_flags(dobb_handle h, uint32_t* host_out, void* stream) {
  dobb_status st = check_handle(h);
  if (st != DOBB_OK) return st;
  if (!host_out) return fail(DOBB_ERR_INVALID_ARG, "host_out is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUDA_TRY(cudaMemcpyAsync(host_out, h->flags(), 4 * (size_t)h->L.nblocks, cudaMemcpyDeviceToHost, s));
  CUDA_TRY(cudaStreamSynchronize(s));
  return DOBB_OK;
}

dobb_status dobb_clear_block_flags(dobb_handle h, void* stream) {
  dobb_status st = check_handle(h);
  if (st != DOBB_OK) return st;
  CUDA_TRY(cudaMemsetAsync(h->flags(), 0, 4 * (size_t)h->L.nblocks, static_cast<cudaStream_t>(stream)));
  return DOBB_OK;
}

dobb_status dobb_get_block_stats(dobb_handle h, float* host_out, void* stream) {
  dobb_status st = check_handle(h);
  if (st != DOBB_OK) return st;
  if (!host_out) return fail(DOBB_ERR_INVALID_ARG, "host_out is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUDA_TRY(cudaMemcpyAsync(host_out, h->stats(), 16 * (size_t)h->L.nblocks, cudaMemcpyDeviceToHost, s));
  CUDA_TRY(cudaStreamSynchronize(s));
  return DOBB_OK;
}

dobb_status dobb_check_bases(dobb_handle h, float* host_out, void* stream) {
  dobb_status st = check_handle(h);
  if (st != DOBB_OK) return st;
  if (!host_out) return fail(DOBB_ERR_INVALID_ARG, "host_out is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CheckArgs a{};
  a.info = h->dinfo();
  a.tiles = h->dtiles() + h->wl.blocks_off;
  a.num_tiles = h->wl.blocks_n;
  a.A = h->A();
  a.Q = h->Q();
  a.lam = h->lam();
  a.out = h->check();
  const int g = std::max(1, std::min(a.num_tiles, h->sm_count * 8));
  cudaError_t e = launch_check(a, g, s);
  if (e != cudaSuccess) return fail(DOBB_ERR_CUDA, "check launch: %s", cudaGetErrorString(e));
  ++h->launches;
  CUDA_TRY(cudaMemcpyAsync(host_out, h->check(), 12 * (size_t)h->L.nblocks, cudaMemcpyDeviceToHost, s));
  CUDA_TRY(cudaStreamSynchronize(s));
  return DOBB_OK;
}

size_t dobb_checkpoint_bytes(dobb_handle h) { return h ? h->L.off_stats - h->L.off_A : 0; }

dobb_status dobb_get_state(dobb_handle h, void* dst_dev, size_t dst_bytes, int64_t* t_out,
                           void* stream) {
  dobb_status st = check_handle(h);
  if (st != DOBB_OK) return st;
  const size_t need = dobb_checkpoint_bytes(h);
  if (!dst_dev || dst_bytes < need)
    return fail(DOBB_ERR_INVALID_ARG, "checkpoint buffer needs %zu bytes", need);
  CUDA_TRY(cudaMemcpyAsync(dst_dev, h->base + h->L.off_A, need, cudaMemcpyDeviceToDevice,
                           static_cast<cudaStream_t>(stream)));
  if (t_out) *t_out = h->t;
  return DOBB_OK;
}

dobb_status dobb_set_state(dobb_handle h, const void* src_dev, size_t src_bytes, int64_t t,
                           void* stream) {
  dobb_status st = check_handle(h);
  if (st != DOBB_OK) return st;
  const size_t need = dobb_checkpoint_bytes(h);
  if (!src_dev || src_bytes < need || t < 0)
    return fail(DOBB_ERR_INVALID_ARG, "checkpoint needs %zu bytes and t >= 0", need);
  CUDA_TRY(cudaMemcpyAsync(h->base + h->L.off_A, src_dev, need, cudaMemcpyDeviceToDevice,
                           static_cast<cudaStream_t>(stream)));
  h->t = t;
  return do_pack(h, static_cast<cudaStream_t>(stream));
}

int64_t dobb_launch_count(dobb_handle h) { return h ? h->launches : -1; }

int64_t dobb_describe_work(int num_matrices, const int64_t* m, const int64_t* n, int B, int phase,
                           int64_t* out, int64_t cap) {
  if (!validate_shapes(num_matrices, m, n, B)) return -1;
  if (phase < 0 || phase > 2) {
    fail(DOBB_ERR_INVALID_ARG, "phase must be 0 (update), 1 (moments) or 2 (refresh)");
    return -1;
  }
  const WorkLists wl = build_work(num_matrices, m, n, B);
  const int TM = step_rows_per_tile();
  int64_t cnt = 0;
  int64_t launch = 0;
  auto emit = [&](int64_t kind, int64_t base, const Tile& t, int64_t a, int64_t b) {
    if (out && cnt < cap) {
      int64_t* e = out + 7 * cnt;
      e[0] = launch; e[1] = kind; e[2] = base; e[3] = t.mat; e[4] = t.blk; e[5] = a; e[6] = b;
    }
    ++cnt;
  };
  if (phase == 0) {
    for (const Chunk& ch : wl.chunks) {
      // the default path: tensor-core launches (wide, narrow), then the FFMA rest
      for (int part = 0; part < 2; ++part) {
        const int lo = part == 0 ? 0 : ch.tc_small, hi = part == 0 ? ch.tc_small : ch.tc_n;
        if (hi <= lo) continue;
        for (int j = lo; j < hi; ++j) {
          const Tile& t = wl.tiles[ch.tc_off + j];
          emit(0, ch.mat_base, t, t.a, std::min<int64_t>(kTcRows, m[t.mat] - t.a));
        }
        ++launch;
      }
      if (ch.tc_n > 0 ? ch.rest_n > 0 : ch.step_n > 0) {
        const int off = ch.tc_n > 0 ? ch.rest_off : ch.step_off;
        const int num = ch.tc_n > 0 ? ch.rest_n : ch.step_n;
        for (int j = 0; j < num; ++j) {
          const Tile& t = wl.tiles[off + j];
          emit(1, ch.mat_base, t, t.a, std::min<int64_t>(TM, m[t.mat] - t.a));
        }
        ++launch;
      }
    }
  } else if (phase == 1) {
    // bf16 activations: tensor-core launches per chunk (wide, narrow), then one
    // FFMA launch over the matrices the tensor-core kernel does not take
    for (const SyrkChunk& sc : wl.syrk_tc) {
      for (int part = 0; part < 2; ++part) {
        const int lo = part == 0 ? 0 : sc.small, hi = part == 0 ? sc.small : sc.n;
        if (hi <= lo) continue;
        for (int j = lo; j < hi; ++j) {
          const Tile& t = wl.tiles[sc.off + j];
          emit(0, sc.mat_base, t, t.a, t.b);
        }
        ++launch;
      }
    }
    for (const Chunk& ch : wl.chunks) {
      if (ch.syrk_rest_n == 0) continue;
      for (int j = 0; j < ch.syrk_rest_n; ++j) {
        const Tile& t = wl.tiles[ch.syrk_rest_off + j];
        emit(1, ch.mat_base, t, t.a, t.b);
      }
      ++launch;
    }
  } else {
    for (const Chunk& ch : wl.chunks) {
      for (int j = 0; j < ch.eig_n; ++j) emit(0, ch.mat_base, wl.tiles[ch.eig_off + j], 0, 0);
      if (ch.eig_n > 0) ++launch;
    }
  }
  return cnt;
}

dobb_status dobb_set_step_path(dobb_handle h, int path) {
  if (!h || path < 0 || path > 1) return fail(DOBB_ERR_INVALID_ARG, "path must be 0 or 1");
  h->path = path;
  return DOBB_OK;
}

dobb_status dobb_sync_bases(dobb_handle h, void* stream) {
  dobb_status st = check_handle(h);
  if (st != DOBB_OK) return st;
  return do_pack(h, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
