// Grid eigensolver for wide blocks ("Dobb", Abstract: a complete basis
// within each block; Table 15: exact eigendecomposition refresh).
//
// The same method as the one-CTA-per-block solver of jacobi.cu -- cyclic
// two-sided Jacobi in a Rayleigh-Ritz restart loop, sweeps blocked into a
// round-robin tournament of column groups -- with the work of one block
// spread over the whole GPU: every phase is one launch over a batch of
// blocks of the same width, and within a launch every table, tile pair,
// panel or product tile of every block is its own CTA.
//
//   init      V = current basis, ||A||_F, finiteness of A
//   RR        T = A V, B = V^T T                        (64 x 64 product tiles)
//   sweep     per round: tables (one CTA each: diagonal tile rotated, R_t
//             kept), then every tile pair B[P_s, P_t] <- R_s^T B[P_s, P_t] R_t
//             and every panel V[i0:i0+64, P_t] <- V[i0:i0+64, P_t] R_t
//   control   off(B) = ||off(B)||_F / ||B||_F, the stopping and restart rules
//             of jacobi.cu, per block, on the device
//   restart   V <- V + V (I - V^T V) / 2 (Newton-Schulz), RR again
//   finish    Lambda = diag(B), one more Newton-Schulz step, columns sorted by
//             descending eigenvalue, Q written row-major
//
// Every launch reads a per-block control record and does nothing for blocks
// that have finished, so the host issues a fixed sequence per sweep and only
// reads the number of active blocks once per sweep to stop early.
//
// Per block state lives in the eigensolver scratch of the state buffer
// (B, V and a work matrix: 3 k^2 floats) plus a rotation buffer and the
// control record, both reused by every batch.
#include <algorithm>

#include "common.cuh"

namespace dobb {
namespace {

constexpr int kThreads = 256;
#include "fp32_tiles.cuh"
#include "jacobi_common.cuh"
#include "mma_tf32.cuh"
#include "cholqr.cuh"
static_assert(kThreads == kTileThreads, "the tile products assume 256 threads");

constexpr int kTableThreads = 128;   // a table: one team of four warps

// Scratch of item i: B, V0, V1 (the basis and the work matrix swap roles at
// every Newton-Schulz step; ctl.vsel names the one holding the basis).
struct ItemBufs {
  float* B;
  float* V;
  float* W;
  const float* A;
  float* Q;
  int64_t boff;
  const MatInfo* mi;
};

__device__ __forceinline__ ItemBufs bufs_of(const GjArgs& a, int item) {
  const Tile t = a.items[item];
  const MatInfo* mi = a.info + t.mat;
  const int64_t kk2 = (int64_t)a.k * a.k;
  ItemBufs b;
  b.boff = mi->a_off + (int64_t)t.blk * kk2;
  b.B = a.scratch + 3 * b.boff;
  float* v0 = b.B + kk2;
  float* v1 = v0 + kk2;
  const int vsel = a.ctl[item].vsel;
  b.V = vsel ? v1 : v0;
  b.W = vsel ? v0 : v1;
  b.A = a.A + b.boff;
  b.Q = a.Q + b.boff;
  b.mi = mi;
  return b;
}

// ------------------------------------------------------------------- init
// V = Q^T-layout copy of the current basis (column j of V = column j of the
// row-major Q, moved through a 32 x 32 shared tile per warp so both sides
// are coalesced), ||A||_F^2 and the finiteness of A over this CTA's rows
// (per-thread fp32 partial sums of at most a few hundred terms, combined in
// fp64).
__global__ void __launch_bounds__(kThreads) gj_init_kernel(const __grid_constant__ GjArgs a) {
  __shared__ double red[32];
  __shared__ float tile[kThreads / 32][32][33];
  const int item = blockIdx.y;
  const ItemBufs b = bufs_of(a, item);
  const int k = a.k;
  const int rows = (k + gridDim.x - 1) / gridDim.x;
  const int r0 = min(k, (int)blockIdx.x * rows), r1 = min(k, r0 + rows);
  float ss = 0.f;
  int bad = 0;
  for (int i = r0; i < r1; ++i) {
    const float* row = b.A + (int64_t)i * k;
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
      const float v = row[j];
      bad |= !isfinite(v);
      ss = fmaf(v, v, ss);
    }
  }
  // the transpose: one 32 x 32 tile per warp at a time
  const int nt = (k + 31) / 32, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  float (*tw)[33] = tile[w];
  for (int tl = blockIdx.x * (kThreads / 32) + w; tl < nt * nt; tl += gridDim.x * (kThreads / 32)) {
    const int bi = tl / nt, bc = tl - bi * nt;   // Q rows 32 bi.., columns 32 bc..
    const int c = 32 * bc + lane;
#pragma unroll 8
    for (int rr = 0; rr < 32; ++rr) {
      const int i = 32 * bi + rr;
      tw[rr][lane] = (i < k && c < k) ? b.Q[(int64_t)i * k + c] : 0.f;
    }
    __syncwarp();
    const int i = 32 * bi + lane;
#pragma unroll 8
    for (int rr = 0; rr < 32; ++rr) {
      const int cc = 32 * bc + rr;
      if (cc < k && i < k) b.V[(int64_t)cc * k + i] = tw[lane][rr];
    }
    __syncwarp();
  }
  const double tot = block_sum_d((double)ss, red);
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) {
    atomicAdd(&a.ctl[item].tot2, tot);
    if (bad) atomicOr(&a.ctl[item].skip, 1);
  }
}

// One thread per item: start the iteration (or skip a non-finite block).
__global__ void gj_start_kernel(const __grid_constant__ GjArgs a) {
  const int item = blockIdx.x * blockDim.x + threadIdx.x;
  if (item >= a.nitems) return;
  GjCtl& c = a.ctl[item];
  const Tile t = a.items[item];
  const MatInfo mi = a.info[t.mat];
  if (c.skip) {
    atomicOr(a.flags + mi.blk0 + t.blk, (uint32_t)DOBB_FLAG_NONFINITE_A);
    c.active = 0;
  } else {
    c.active = 1;
  }
  c.fresh = 1;
  c.restart = 0;
  c.sweeps = 0;
  c.conv = 0;
  c.rot = 0;
  c.last_rot = 0;
  c.prev = INFINITY;
  c.bfloor = 1e-3f * kEps * (float)sqrt(c.tot2);
  c.tot2 = 0.0;
  c.off2 = 0.0;
}

// --------------------------------------------------------------- products
// One 64 x 64 output tile of a k x k product per CTA (blockIdx.x = tile,
// blockIdx.y = item).  Predicates: kAlways (every block not skipped),
// kActive (blocks still iterating), kRestart (blocks that restart now).
enum Pred : int { kAlways = 0, kActive = 1, kRestart = 2 };
// Products: T = A V (RR1), B = V^T T (RR2, symmetric), E = I - V^T V (NS1,
// symmetric, into B), V' = V + E V / 2 ... written as V + 0.5 V E (NS2, into W).
enum Prod : int { kRR1 = 0, kRR2 = 1, kNS1 = 2, kNS2 = 3 };

__device__ __forceinline__ bool pred_ok(const GjCtl& c, int pred) {
  if (c.skip) return false;
  if (pred == kActive) return c.active != 0;
  if (pred == kRestart) return c.active != 0 && c.restart != 0;
  return true;
}

__global__ void __launch_bounds__(kThreads) gj_gemm_kernel(const __grid_constant__ GjArgs a, int prod,
                                                           int pred) {
  extern __shared__ __align__(16) float gs[];
  const int item = blockIdx.y;
  if (!pred_ok(a.ctl[item], pred)) return;
  const int k = a.k;
  const int nt = (k + kT - 1) / kT;
  const int ti = blockIdx.x % nt, tj = blockIdx.x / nt;
  const bool sym = prod == kRR2 || prod == kNS1;
  if (sym && ti > tj) return;
  const ItemBufs b = bufs_of(a, item);
  switch (prod) {
    case kRR1:   // T (in W) = A V
      gemm_tile<false>(b.A, b.V, b.W, nullptr, 1.f, false, false, k, ti, tj, gs);
      break;
    case kRR2:   // B = V^T T
      gemm_tile<true>(b.V, b.W, b.B, nullptr, 1.f, false, true, k, ti, tj, gs);
      break;
    case kNS1:   // E (in B) = I - V^T V
      gemm_tile<true>(b.V, b.V, b.B, nullptr, -1.f, true, true, k, ti, tj, gs);
      break;
    default:     // W = V + 0.5 V E
      gemm_tile<false>(b.V, b.B, b.W, b.V, 0.5f, false, false, k, ti, tj, gs);
      break;
  }
}

// The basis moves to the other buffer after a Newton-Schulz step.
__global__ void gj_flip_kernel(const __grid_constant__ GjArgs a, int pred) {
  const int item = blockIdx.x * blockDim.x + threadIdx.x;
  if (item >= a.nitems) return;
  GjCtl& c = a.ctl[item];
  if (pred_ok(c, pred)) c.vsel ^= 1;
}

// ----------------------------------------------------------------- sweeps
// Tables of round br: one CTA of four warps per (table, item).  The table's
// diagonal tile S (2g x 2g, zero-padded to 64 x 64) and its rotation R (kept
// transposed, R^T) live in shared memory.  Each inner step rotates a set of
// disjoint column pairs ("slots", at most 32).  In the first round's steps
// inside each group, a slot has a single member when g is odd; that member
// is paired with the padding row kPadRow, which holds zeros.  The first warp
// computes the slots' rotations (lane = slot) into one 16-byte record each
// (two record buffers, one per step parity); every thread then works
// through a fixed list of items:
//  * S <- J^T S J, block by block.  For each unordered slot pair {X, Y}, the
//    2 x 2 block of S on their members becomes G_X S_XY G_Y^T (G = [[c, -s],
//    [s, c]]).  It is written to (X, Y) and mirrored to (Y, X), so every entry
//    is read and written once and S stays exactly symmetric.  The pairs are
//    dealt to the threads in circulant order (Y = X + d mod slots, d = 0, 1,
//    ...), so all lanes are busy.  With row stride 64 the lanes of a warp
//    (consecutive X, one d) address distinct columns, hence distinct banks,
//    on both the block and its mirror.
//  * R <- R J: for each (slot, column pair), rows p and q of R^T, two entries
//    per item (float2).
// Identity rotations (pairs past the block, single members, entries at the
// floor) leave their entries bit-for-bit unchanged, and the padding row
// stays zero.  Two barriers per step; between them the first warp computes
// the next step's rotations while the other warps update R.
constexpr int kLS = 64;        // row stride of S in shared memory
constexpr int kLR = 66;        // row stride of R^T (even for float2 rows; the transposed read-out is 2-way)
constexpr int kMaxSlots = 32;
constexpr int kPadRow = 63;    // partner of a single-member slot (odd g: 2g <= 62)
constexpr int kBlkPer = (32 * 33 / 2 + kTableThreads - 1) / kTableThreads;  // slot pairs per thread
constexpr int kRotThreads = kTableThreads - 32;                              // warps 1.. update R
constexpr int kRotPer = (32 * 32 + kRotThreads - 1) / kRotThreads;          // R items per thread

struct __align__(16) SlotRec {
  float c, s;
  int p, q;
};

// This thread's slot pairs among ns slots, in circulant order, packed as
// X | Y << 8 (-1 past the end): pair l is (X, X + d mod ns) with d = l / ns.
// d = 0 .. (ns - 1) / 2 lists every unordered pair once, plus, for even ns,
// the first ns / 2 pairs of d = ns / 2.
__device__ __forceinline__ void deal_pairs(int ns, int (&out)[kBlkPer]) {
  const int nb = ns * (ns + 1) / 2;
#pragma unroll
  for (int i = 0; i < kBlkPer; ++i) {
    const int l = threadIdx.x + i * kTableThreads;
    out[i] = -1;
    if (l < nb) {
      const int d = l / ns, X = l - d * ns;
      const int Y = X + d < ns ? X + d : X + d - ns;
      out[i] = X | (Y << 8);
    }
  }
}

// R items of thread rt (0 .. kRotThreads - 1) among ns slots x nh column
// pairs, packed X | jj << 8.
__device__ __forceinline__ void deal_rot(int ns, int nh, int rt, int (&out)[kRotPer]) {
#pragma unroll
  for (int i = 0; i < kRotPer; ++i) {
    const int l = rt + i * kRotThreads;
    out[i] = -1;
    if (rt >= 0 && l < ns * nh) {
      const int X = l / nh;
      out[i] = X | ((l - X * nh) << 8);
    }
  }
}

__global__ void __launch_bounds__(kTableThreads, 6) gj_table_kernel(const __grid_constant__ GjArgs a,
                                                                    int br) {
  __shared__ __align__(16) float S[64 * kLS];
  __shared__ __align__(16) float Rt[64 * kLR];
  __shared__ SlotRec sl[2][kMaxSlots];
  const int item = blockIdx.y, tt = blockIdx.x;
  GjCtl* c = a.ctl + item;
  if (!pred_ok(*c, kActive)) return;
  const int k = a.k;
  const Geo G = geo_for(k);
  if (br >= G.nG - 1 || tt >= G.nT) return;
  const ItemBufs b = bufs_of(a, item);
  const int n2 = G.n2, g = G.g, nn = n2 * n2;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int gI, gJ;
  rr_pair(br, tt, G.nG, gI, gJ);
  // S = the table's tile of B, R^T = I; zero outside the table
  for (int r = warp; r < 64; r += kTableThreads / 32) {
    const int cr = r < n2 ? table_col(r, gI, gJ, g, k) : k;
    for (int q = lane; q < 64; q += 32) {
      const int cq = q < n2 ? table_col(q, gI, gJ, g, k) : k;
      S[r * kLS + q] = (cr < k && cq < k) ? b.B[(int64_t)cr * k + cq] : 0.f;
      Rt[r * kLR + q] = (r == q && r < n2) ? 1.f : 0.f;
    }
  }
  const float bfloor = c->bfloor;
  const int gp = g + (g & 1);
  const int n_intra = br == 0 ? gp - 1 : 0;
  const int nsteps = n_intra + g;
  int rots = 0;
  // rotations of step `step` into out[lane] (warp 0)
  auto make_slots = [&](int step, SlotRec* out) {
    const bool intra = step < n_intra;
    const int r = intra ? step : step - n_intra;
    if (lane >= (intra ? gp : g)) return;
    int p, q;
    bool single = false;
    if (intra) {
      // group grp's round-robin pair; player g is the odd group's dummy
      const int half = gp >> 1, grp = lane / half, ii = lane - grp * half;
      int pp, qq;
      rr_pair(r, ii, gp, pp, qq);
      if (pp >= g) {
        pp = qq;
        single = true;
      } else if (qq >= g) {
        single = true;
      }
      if (!single && qq < pp) {
        const int t = pp; pp = qq; qq = t;
      }
      p = pp + grp * g;
      q = single ? kPadRow : qq + grp * g;
    } else {
      p = lane;
      q = g + (lane + r) % g;
    }
    float cs = 1.f, sn = 0.f;
    if (!single && table_col(p, gI, gJ, g, k) < k && table_col(q, gI, gJ, g, k) < k) {
      const float bpq = S[p * kLS + q];
      if (fabsf(bpq) > bfloor) {
        const float ta = (S[q * kLS + q] - S[p * kLS + p]) / (2.f * bpq);
        const float tn = ta >= 0.f ? 1.f / (ta + sqrtf(1.f + ta * ta)) : -1.f / (-ta + sqrtf(1.f + ta * ta));
        cs = 1.f / sqrtf(1.f + tn * tn);
        sn = tn * cs;
        ++rots;
      }
    }
    out[lane] = SlotRec{cs, sn, p, q};
  };
  int blk[kBlkPer], rit[kRotPer];
  deal_pairs(n_intra ? gp : g, blk);
  deal_rot(n_intra ? gp : g, g, tid - 32, rit);
  __syncthreads();   // S and R^T loaded
  if (warp == 0) make_slots(0, sl[0]);
  __syncthreads();
  // per step: S update by all warps on the step's rotations; then warp 0
  // computes the next step's rotations (into the other record buffer) while
  // warps 1.. apply this step's to R
  for (int step = 0; step < nsteps; ++step) {
    const SlotRec* cur = sl[step & 1];
    if (step == n_intra && n_intra) {
      deal_pairs(g, blk);
      deal_rot(g, g, tid - 32, rit);
    }
    // S blocks: the thread's pairs are disjoint from every other thread's
    // (only the zero padding entries are shared, and stay zero)
#pragma unroll
    for (int i = 0; i < kBlkPer; ++i) {
      const int xy = blk[i];
      if (xy < 0) continue;
      const SlotRec x = cur[xy & 255], y = cur[xy >> 8];
      const float m00 = S[x.p * kLS + y.p], m01 = S[x.p * kLS + y.q];
      const float m10 = S[x.q * kLS + y.p], m11 = S[x.q * kLS + y.q];
      // rows: G_X M
      const float t00 = x.c * m00 - x.s * m10, t01 = x.c * m01 - x.s * m11;
      const float t10 = x.s * m00 + x.c * m10, t11 = x.s * m01 + x.c * m11;
      // columns: (G_X M) G_Y^T; for X = Y the mirrored writes of the
      // off-diagonal pair both end as n10
      const float n00 = y.c * t00 - y.s * t01, n01 = y.s * t00 + y.c * t01;
      const float n10 = y.c * t10 - y.s * t11, n11 = y.s * t10 + y.c * t11;
      S[x.p * kLS + y.p] = n00;
      S[y.p * kLS + x.p] = n00;
      S[x.p * kLS + y.q] = n01;
      S[y.q * kLS + x.p] = n01;
      S[x.q * kLS + y.p] = n10;
      S[y.p * kLS + x.q] = n10;
      S[x.q * kLS + y.q] = n11;
      S[y.q * kLS + x.q] = n11;
    }
    __syncthreads();
    if (warp == 0) {
      if (step + 1 < nsteps) make_slots(step + 1, sl[(step + 1) & 1]);
    } else {
      // R^T rows p, q of each slot, two columns per item
#pragma unroll
      for (int i = 0; i < kRotPer; ++i) {
        const int xj = rit[i];
        if (xj < 0) continue;
        const SlotRec x = cur[xj & 255];
        float2* ra = reinterpret_cast<float2*>(Rt + x.p * kLR) + (xj >> 8);
        float2* rb = reinterpret_cast<float2*>(Rt + x.q * kLR) + (xj >> 8);
        const float2 u = *ra, v = *rb;
        *ra = make_float2(x.c * u.x - x.s * v.x, x.c * u.y - x.s * v.y);
        *rb = make_float2(x.s * u.x + x.c * v.x, x.s * u.y + x.c * v.y);
      }
    }
    __syncthreads();
  }
  float* Rg = a.rbuf + (int64_t)item * a.rstride + (int64_t)tt * nn;
  for (int r = warp; r < n2; r += kTableThreads / 32) {
    const int cr = table_col(r, gI, gJ, g, k);
    for (int q = lane; q < n2; q += 32) {
      const int cq = table_col(q, gI, gJ, g, k);
      if (cr < k && cq < k) b.B[(int64_t)cr * k + cq] = S[r * kLS + q];
      Rg[r * n2 + q] = Rt[q * kLR + r];   // R[r][q]
    }
  }
  int tot = rots;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
  if (tid == 0 && tot) atomicAdd(&c->rot, tot);
}

// E = R - I of table t into a zero-padded 64 x kLdM tile (warp rows, lanes
// along the row: coalesced loads, conflict-free stores).
constexpr int kRowsPerWarp = kT / (kThreads / 32);

__device__ __forceinline__ void load_corr(float* dst, const float* src, int n2) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float v[kRowsPerWarp][2];
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const int r = warp + (kThreads / 32) * i;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int q = lane + 32 * h;
      v[i][h] = (r < n2 && q < n2) ? src[r * n2 + q] - (r == q ? 1.f : 0.f) : 0.f;
    }
  }
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const int r = warp + (kThreads / 32) * i;
    dst[r * kLdM + lane] = v[i][0];
    dst[r * kLdM + lane + 32] = v[i][1];
  }
}

template <int kPasses>
__device__ __forceinline__ void corr_product(const float* P, const float* Q, int n, float (&acc)[4][4]) {
  mma_tn_64<kPasses>(P, Q, n, acc);
}

// Tile pairs and panels of round br.  Unit u < npair is the tile pair (s, t),
// s < t, in row order; the rest are panel runs (t, c0): the 64-row panels
// c0 .. c0 + kPanelRun - 1 of V's columns P_t, one after another on one
// E_t.  The products run on the warp-level tensor cores in correction form:
// with E = R - I,
//   Y = X + E_s^T X,  Z = Y + Y E_t       (B[P_s, P_t] <- R_s^T X R_t)
//   V' = V + V E_t                         (V[i0:i0+64, P_t] <- V R_t)
// the TF32-rounded products added onto fp32 X, Y, V.  A sweep on a freshly
// formed B (the only kind that can end the iteration) multiplies in split
// precision (~2^-21 |E| |X|); the other sweeps, whose B is re-formed from A
// before the iteration can stop and whose basis only seeds that re-forming,
// in plain TF32.  The columns of B (or V) that a table's local indices
// stand for are looked up once per CTA.
constexpr int kPanelRun = 4;

__host__ __device__ __forceinline__ int apply_units(int k) {
  const Geo G = geo_for(k);
  const int nI = (k + kT - 1) / kT;
  return G.nT * (G.nT - 1) / 2 + G.nT * ((nI + kPanelRun - 1) / kPanelRun);
}

__global__ void __launch_bounds__(kThreads, 4) gj_apply_kernel(const __grid_constant__ GjArgs a, int br) {
  extern __shared__ __align__(16) float sm[];
  __shared__ int colS[kT], colT[kT];
  const int item = blockIdx.y;
  const GjCtl& cref = a.ctl[item];
  if (!pred_ok(cref, kActive)) return;
  const bool precise = cref.fresh != 0;
  const int k = a.k;
  const Geo G = geo_for(k);
  if (br >= G.nG - 1) return;
  const int nI = (k + kT - 1) / kT;
  const int nPR = (nI + kPanelRun - 1) / kPanelRun;
  const int npair = G.nT * (G.nT - 1) / 2;
  const int u = blockIdx.x;
  if (u >= npair + G.nT * nPR) return;
  const ItemBufs b = bufs_of(a, item);
  const int n2 = G.n2, nn = n2 * n2;
  const float* Rb = a.rbuf + (int64_t)item * a.rstride;
  // three tiles: E_s (then Y^T and Z^T, or the panel output), E_t, X
  float* Es = sm;
  float* Et = sm + kT * kLdM;
  float* Xs = sm + 2 * kT * kLdM;
  float* Ys = Es;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool pair = u < npair;
  int s = 0, t = 0, c0 = 0;
  if (pair) {
    // (s, t) from the linear index of the strict upper triangle
    int rem = u;
    while (rem >= G.nT - 1 - s) {
      rem -= G.nT - 1 - s;
      ++s;
    }
    t = s + 1 + rem;
  } else {
    const int v = u - npair;
    t = v / nPR;
    c0 = (v - t * nPR) * kPanelRun;
  }
  if (tid < 2 * kT) {
    const int r = tid & (kT - 1);
    int gI, gJ;
    rr_pair(br, tid < kT ? s : t, G.nG, gI, gJ);
    (tid < kT ? colS : colT)[r] = r < n2 ? table_col(r, gI, gJ, G.g, k) : k;
  }
  __syncthreads();
  float acc[4][4];
  if (pair) {
    const int cq0 = colT[lane], cq1 = colT[lane + 32];
    {
      float v[kRowsPerWarp][2];
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        const int cr = colS[warp + (kThreads / 32) * i];
        const float* row = b.B + (int64_t)cr * k;
        v[i][0] = (cr < k && cq0 < k) ? row[cq0] : 0.f;
        v[i][1] = (cr < k && cq1 < k) ? row[cq1] : 0.f;
      }
      load_corr(Es, Rb + (int64_t)s * nn, n2);
      load_corr(Et, Rb + (int64_t)t * nn, n2);
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        const int r = warp + (kThreads / 32) * i;
        Xs[r * kLdM + lane] = v[i][0];
        Xs[r * kLdM + lane + 32] = v[i][1];
      }
    }
    __syncthreads();
    mma_load_acc<false>(Xs, acc);                     // X
    if (precise) corr_product<3>(Es, Xs, n2, acc);    // Y = X + E_s^T X
    else corr_product<1>(Es, Xs, n2, acc);
    __syncthreads();                                  // E_s read by every warp
    mma_store_acc<true>(Ys, acc);                     // Y^T over E_s
    __syncthreads();
    if (precise) corr_product<3>(Ys, Et, n2, acc);    // Z = Y + Y E_t
    else corr_product<1>(Ys, Et, n2, acc);
    __syncthreads();
    mma_store_acc<false>(Xs, acc);                    // Z
    mma_store_acc<true>(Ys, acc);                     // Z^T
    __syncthreads();
    const int cs0 = colS[lane], cs1 = colS[lane + 32];
#pragma unroll 2
    for (int i = 0; i < kRowsPerWarp; ++i) {
      const int r = warp + (kThreads / 32) * i;
      const int crS = colS[r], crT = colT[r];
      if (crS < k) {
        float* row = b.B + (int64_t)crS * k;
        if (cq0 < k) row[cq0] = Xs[r * kLdM + lane];
        if (cq1 < k) row[cq1] = Xs[r * kLdM + lane + 32];
      }
      if (crT < k) {
        float* row = b.B + (int64_t)crT * k;
        if (cs0 < k) row[cs0] = Ys[r * kLdM + lane];
        if (cs1 < k) row[cs1] = Ys[r * kLdM + lane + 32];
      }
    }
  } else {
    const int c1 = min(nI, c0 + kPanelRun);
    // the next panel's V tile loads into registers while this one is
    // multiplied (panels are disjoint row ranges of V)
    float v[kRowsPerWarp][2];
    auto load_panel = [&](int c) {
      const int i0 = c * kT;
      const bool ok0 = i0 + lane < k, ok1 = i0 + lane + 32 < k;
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        const int cr = colT[warp + (kThreads / 32) * i];
        const float* row = b.V + (int64_t)cr * k + i0;
        v[i][0] = (cr < k && ok0) ? row[lane] : 0.f;
        v[i][1] = (cr < k && ok1) ? row[lane + 32] : 0.f;
      }
    };
    load_panel(c0);
    load_corr(Et, Rb + (int64_t)t * nn, n2);
    for (int c = c0; c < c1; ++c) {
      const int i0 = c * kT;
      const bool ok0 = i0 + lane < k, ok1 = i0 + lane + 32 < k;
      // Xs is free: the previous panel's product ended before the barrier
      // that preceded its write-back
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        const int r = warp + (kThreads / 32) * i;
        Xs[r * kLdM + lane] = v[i][0];
        Xs[r * kLdM + lane + 32] = v[i][1];
      }
      if (c + 1 < c1) load_panel(c + 1);
      __syncthreads();
      mma_load_acc<true>(Xs, acc);                      // V rows i, table columns q
      if (precise) corr_product<3>(Xs, Et, n2, acc);    // V + V E_t
      else corr_product<1>(Xs, Et, n2, acc);
      mma_store_acc<true>(Ys, acc);
      __syncthreads();
      for (int q = warp; q < n2; q += kThreads / 32) {
        const int cq = colT[q];
        if (cq >= k) continue;
        float* row = b.V + (int64_t)cq * k + i0;
        if (ok0) row[lane] = Ys[q * kLdM + lane];
        if (ok1) row[lane + 32] = Ys[q * kLdM + lane + 32];
      }
    }
  }
}

// ---------------------------------------------------------------- control
// ||off(B)||_F^2 and ||B||_F^2 over this CTA's rows (per-thread fp32
// partial sums, combined in fp64; the two are summed separately, so off(B)
// keeps its relative accuracy however small it is).
__global__ void __launch_bounds__(kThreads) gj_off_kernel(const __grid_constant__ GjArgs a) {
  __shared__ double red[32];
  const int item = blockIdx.y;
  if (!pred_ok(a.ctl[item], kActive)) return;
  const ItemBufs b = bufs_of(a, item);
  const int k = a.k;
  const int rows = (k + gridDim.x - 1) / gridDim.x;
  const int r0 = min(k, (int)blockIdx.x * rows), r1 = min(k, r0 + rows);
  float tot = 0.f, off = 0.f;
  for (int i = r0; i < r1; ++i) {
    const float* row = b.B + (int64_t)i * k;
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
      const float v = row[j];
      tot = fmaf(v, v, tot);
      if (j != i) off = fmaf(v, v, off);
    }
  }
  const double dt = block_sum_d((double)tot, red);
  __syncthreads();
  const double doff = block_sum_d((double)off, red);
  if (threadIdx.x == 0) {
    atomicAdd(&a.ctl[item].tot2, dt);
    atomicAdd(&a.ctl[item].off2, doff);
  }
}

// One thread per item: the rules of jacobi.cu after a sweep.  Writes the
// number of blocks still iterating to a.active_count.
__global__ void gj_control_kernel(const __grid_constant__ GjArgs a) {
  const int item = blockIdx.x * blockDim.x + threadIdx.x;
  int still = 0;
  if (item < a.nitems) {
    GjCtl& c = a.ctl[item];
    if (!c.skip && c.active) {
      const float off = c.tot2 > 0.0 ? (float)sqrt(c.off2 / c.tot2) : 0.f;
      const float stop = a.tol > 0.f ? a.tol : kStopOff;
      c.sweeps += 1;
      c.last_rot = c.rot;
      c.restart = 0;
      bool done = false;
      if (c.fresh) {
        if (off <= stop || c.rot == 0 || (off <= kStallOff && off > 0.7f * c.prev)) {
          c.conv = 1;
          done = true;
        } else {
          c.prev = off;
        }
      }
      if (!done && c.sweeps >= a.max_sweeps) done = true;
      if (done) {
        c.active = 0;
      } else {
        c.fresh = 0;
        if (off <= kColdOff) {  // close to diagonal: restart from a fresh B
          c.restart = 1;
          c.fresh = 1;
        }
      }
      c.rot = 0;
      c.off2 = 0.0;
      c.tot2 = 0.0;
      still = c.active;
    }
  }
  still = __syncthreads_count(still);
  if (threadIdx.x == 0 && still) atomicAdd(a.active_count, still);
}

// ----------------------------------------------------------------- finish
// Lambda (unsorted) = diag(B) into the eigenvalue slots, before the last
// Newton-Schulz step reuses B's buffer.
__global__ void gj_diag_kernel(const __grid_constant__ GjArgs a) {
  const int item = blockIdx.y;
  if (a.ctl[item].skip) return;
  const ItemBufs b = bufs_of(a, item);
  const Tile t = a.items[item];
  const int k = a.k;
  float* lam = a.lam + b.mi->lam_off + (int64_t)t.blk * k;
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < k; j += gridDim.x * blockDim.x)
    lam[j] = b.B[(int64_t)j * k + j];
}

// One CTA per item: sort by descending eigenvalue (bitonic, in shared
// memory), write Q row-major with the columns permuted, stats and flags.
__global__ void __launch_bounds__(kThreads) gj_finish_kernel(const __grid_constant__ GjArgs a) {
  extern __shared__ __align__(16) float sm[];
  const int item = blockIdx.x;
  const GjCtl c = a.ctl[item];
  const Tile t = a.items[item];
  const MatInfo mi = a.info[t.mat];
  if (c.skip) return;
  const ItemBufs b = bufs_of(a, item);
  const int k = a.k, kp2 = pow2_ceil(k);
  float* lamv = sm;
  int* perm = reinterpret_cast<int*>(sm + kp2);
  float* lam = a.lam + mi.lam_off + (int64_t)t.blk * k;
  for (int p = threadIdx.x; p < kp2; p += blockDim.x) {
    lamv[p] = p < k ? lam[p] : -INFINITY;
    perm[p] = p;
  }
  __syncthreads();
  for (int size = 2; size <= kp2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < kp2; i += blockDim.x) {
        const int j = i ^ stride;
        if (j > i) {
          const bool desc = (i & size) == 0;
          const float li = lamv[i], lj = lamv[j];
          if (desc ? (li < lj) : (li > lj)) {
            lamv[i] = lj;
            lamv[j] = li;
            const int pt = perm[i];
            perm[i] = perm[j];
            perm[j] = pt;
          }
        }
      }
      __syncthreads();
    }
  }
  // Q[i][j] = V(i, perm[j]) = V[perm[j] k + i], through a 32 x 32 shared
  // tile per warp (placed after lamv and perm) so both sides are coalesced
  {
    const int nt = (k + 31) / 32, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float (*tw)[33] = reinterpret_cast<float (*)[33]>(sm + 2 * kp2) + 32 * w;
    for (int tl = w; tl < nt * nt; tl += kThreads / 32) {
      const int bj = tl / nt, bi = tl - bj * nt;   // Q columns 32 bj.., rows 32 bi..
      const int i = 32 * bi + lane;
#pragma unroll 8
      for (int jj = 0; jj < 32; ++jj) {
        const int j = 32 * bj + jj;
        float v = 0.f;
        if (j < k && i < k) {
          int p = perm[j];
          if (p < 0 || p >= k) p = j;  // only reachable with a NaN eigenvalue
          v = b.V[(int64_t)p * k + i];
        }
        tw[jj][lane] = v;
      }
      __syncwarp();
      const int j = 32 * bj + lane;
#pragma unroll 8
      for (int ii = 0; ii < 32; ++ii) {
        const int i2 = 32 * bi + ii;
        if (i2 < k && j < k) b.Q[(int64_t)i2 * k + j] = tw[lane][ii];
      }
      __syncwarp();
    }
  }
  for (int j = threadIdx.x; j < k; j += blockDim.x) lam[j] = lamv[j];
  if (threadIdx.x == 0) {
    float* st = a.stats + 4 * (int64_t)(mi.blk0 + t.blk);
    st[2] = (float)c.sweeps;
    st[3] = (float)c.last_rot;
    if (!c.conv) atomicOr(a.flags + mi.blk0 + t.blk, (uint32_t)DOBB_FLAG_NOT_CONVERGED);
  }
}

// ---------------------------------------------------- orthogonal iteration
// The grid form of the orthogonal-iteration refresh of orth.cu ("Dobb",
// Table 15: one orthogonal-iteration step per refresh; Table 16: Cholesky
// QR): per step T = A V, then two Cholesky QR passes (G = X^T X,
// L = chol(G), V = X L^{-T}), then Lambda_j = v_j^T A v_j and Q = V in the
// column order of the previous basis.  The products are 64 x 64 output tiles
// of the whole batch (one CTA each), the Cholesky factorisation one CTA per
// block, the triangular solve one CTA per 64-row panel.  A block whose Gram
// matrix is not numerically positive definite drops out (ctl.conv = 0, its
// basis untouched) and is redone from its old basis by orth.cu's shifted
// passes.  Buffers: V (the basis) in V0, T in V1, G and L in B.
enum OgProd : int { kOgAV = 0, kOgGramT = 1, kOgGramV = 2 };

__device__ __forceinline__ bool og_ok(const GjCtl& c) { return !c.skip && c.conv; }

__global__ void og_start_kernel(const __grid_constant__ GjArgs a) {
  const int item = blockIdx.x * blockDim.x + threadIdx.x;
  if (item >= a.nitems) return;
  GjCtl& c = a.ctl[item];
  if (c.skip) {
    const Tile t = a.items[item];
    atomicOr(a.flags + a.info[t.mat].blk0 + t.blk, (uint32_t)DOBB_FLAG_NONFINITE_A);
  }
  c.conv = c.skip ? 0 : 1;
}

__global__ void __launch_bounds__(kThreads) og_gemm_kernel(const __grid_constant__ GjArgs a, int prod) {
  extern __shared__ __align__(16) float gs[];
  const int item = blockIdx.y;
  if (!og_ok(a.ctl[item])) return;
  const int k = a.k;
  const int nt = (k + kT - 1) / kT;
  const int ti = blockIdx.x % nt, tj = blockIdx.x / nt;
  if (prod != kOgAV && ti > tj) return;
  const ItemBufs b = bufs_of(a, item);
  if (prod == kOgAV)          // T (in W) = A V
    gemm_tile<false>(b.A, b.V, b.W, nullptr, 1.f, false, false, k, ti, tj, gs);
  else if (prod == kOgGramT)  // G (in B) = T^T T
    gemm_tile<true>(b.W, b.W, b.B, nullptr, 1.f, false, true, k, ti, tj, gs);
  else                        // G (in B) = V^T V
    gemm_tile<true>(b.V, b.V, b.B, nullptr, 1.f, false, true, k, ti, tj, gs);
}

// L = chol(G) in place, one CTA per block.
__global__ void __launch_bounds__(kThreads, 2) og_chol_kernel(const __grid_constant__ GjArgs a) {
  extern __shared__ __align__(16) float sm[];
  __shared__ int s_ok;
  const int item = blockIdx.x;
  GjCtl* c = a.ctl + item;
  if (!og_ok(*c)) return;
  const ItemBufs b = bufs_of(a, item);
  if (!chol_lower(b.B, a.k, sm, &s_ok) && threadIdx.x == 0) c->conv = 0;
}

// V = X L^{-T} for the rows of this CTA's 64-row panel (X = T or V itself).
__global__ void __launch_bounds__(kThreads, 2) og_trsm_kernel(const __grid_constant__ GjArgs a, int from_t) {
  extern __shared__ __align__(16) float sm[];
  const int item = blockIdx.y;
  if (!og_ok(a.ctl[item])) return;
  const int k = a.k, i0 = blockIdx.x * kT;
  if (i0 >= k) return;
  const ItemBufs b = bufs_of(a, item);
  trsm_rows(from_t ? b.W : b.V, b.V, b.B, k, i0, sm);
}

// Lambda_j = v_j . (A v_j), a warp per column (T = A V in W).
__global__ void og_lambda_kernel(const __grid_constant__ GjArgs a) {
  const int item = blockIdx.y;
  if (!og_ok(a.ctl[item])) return;
  const int k = a.k, lane = threadIdx.x & 31;
  const int j = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (j >= k) return;
  const ItemBufs b = bufs_of(a, item);
  const Tile t = a.items[item];
  float d = 0.f;
  for (int i = lane; i < k; i += 32) d = fmaf(b.V[(int64_t)j * k + i], b.W[(int64_t)j * k + i], d);
  d = warp_sum(d);
  if (lane == 0) a.lam[b.mi->lam_off + (int64_t)t.blk * k + j] = d;
}

// Q row-major from V (one 32 x 32 shared tile per warp), and the stats.
__global__ void __launch_bounds__(kThreads) og_finish_kernel(const __grid_constant__ GjArgs a, int steps) {
  __shared__ float tile[kThreads / 32][32][33];
  const int item = blockIdx.y;
  if (!og_ok(a.ctl[item])) return;
  const ItemBufs b = bufs_of(a, item);
  const int k = a.k, nt = (k + 31) / 32, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  float (*tw)[33] = tile[w];
  for (int tl = blockIdx.x * (kThreads / 32) + w; tl < nt * nt; tl += gridDim.x * (kThreads / 32)) {
    const int bj = tl / nt, bi = tl - bj * nt;   // Q columns 32 bj.., rows 32 bi..
    const int i = 32 * bi + lane;
#pragma unroll 8
    for (int jj = 0; jj < 32; ++jj) {
      const int j = 32 * bj + jj;
      tw[jj][lane] = (j < k && i < k) ? b.V[(int64_t)j * k + i] : 0.f;
    }
    __syncwarp();
    const int j = 32 * bj + lane;
#pragma unroll 8
    for (int ii = 0; ii < 32; ++ii) {
      const int i2 = 32 * bi + ii;
      if (i2 < k && j < k) b.Q[(int64_t)i2 * k + j] = tw[lane][ii];
    }
    __syncwarp();
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const Tile t = a.items[item];
    float* st = a.stats + 4 * (int64_t)(b.mi->blk0 + t.blk);
    st[2] = (float)steps;
    st[3] = 0.f;   // shifted Cholesky QR passes: none on this path
  }
}

size_t chol_smem() { return 3 * (size_t)kT * kLd * sizeof(float); }

size_t apply_smem() { return 3 * (size_t)kT * kLdM * sizeof(float); }
size_t gemm_smem() { return (size_t)kGemmFloats * sizeof(float); }

}  // namespace

int64_t gj_rbuf_floats(int k) {
  const Geo G = geo_for(k);
  return (int64_t)G.nT * G.n2 * G.n2;
}

size_t gj_finish_smem(int k) { return (2 * (size_t)pow2_ceil(k) + (kThreads / 32) * 32 * 33) * sizeof(float); }

cudaError_t configure_jacobi_grid(size_t smem_limit) {
  cudaError_t e = cudaFuncSetAttribute(gj_apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)apply_smem());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(og_chol_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)chol_smem());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(og_trsm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)chol_smem());
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gj_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)std::min<size_t>(smem_limit, gj_finish_smem(kMaxK)));
  return e;
}

// The whole refresh of nb batches (each: blocks of one width), batch b on
// streams[b]: the launches of all batches are interleaved round by round, so
// the table solves of one batch (latency-bound) overlap the tile products of
// another (memory- and tensor-bound).  Synchronises the streams once per
// sweep (to read how many blocks still iterate in each batch).
cudaError_t run_jacobi_grid(const GjArgs* batches, int nb, const cudaStream_t* streams,
                            int* host_counts, int64_t* launches) {
  struct Geom {
    Geo G;
    int nt, npair, ctl_blocks;
    dim3 tiles, cgrid;
  };
  Geom gm[kGjMaxBatches];
  if (nb <= 0) return cudaSuccess;
  if (nb > kGjMaxBatches) return cudaErrorInvalidValue;
  const size_t gsm = gemm_smem(), asm_ = apply_smem();
  int64_t n = 0;
  int max_rounds = 0;
  for (int b = 0; b < nb; ++b) {
    const GjArgs& a = batches[b];
    Geom& m = gm[b];
    m.G = geo_for(a.k);
    m.nt = (a.k + kT - 1) / kT;
    m.npair = m.G.nT * (m.G.nT - 1) / 2;
    m.ctl_blocks = (a.nitems + 255) / 256;
    m.tiles = dim3(m.nt * m.nt, a.nitems);
    const int chunks = (int)std::max<int64_t>(1, std::min<int64_t>(256, (int64_t)a.k * a.k / (64 * 1024)));
    m.cgrid = dim3(chunks, a.nitems);
    max_rounds = std::max(max_rounds, m.G.nG - 1);
    const cudaStream_t s = streams[b];
    cudaError_t e = cudaMemsetAsync(a.ctl, 0, sizeof(GjCtl) * (size_t)a.nitems, s);
    if (e != cudaSuccess) return e;
    gj_init_kernel<<<m.cgrid, kThreads, 0, s>>>(a);
    gj_start_kernel<<<m.ctl_blocks, 256, 0, s>>>(a);
    gj_gemm_kernel<<<m.tiles, kThreads, gsm, s>>>(a, kRR1, kActive);
    gj_gemm_kernel<<<m.tiles, kThreads, gsm, s>>>(a, kRR2, kActive);
    n += 4;
    host_counts[b] = a.nitems;
  }
  const int max_sweeps = batches[0].max_sweeps;
  for (int sweep = 0; sweep < max_sweeps; ++sweep) {
    for (int br = 0; br < max_rounds; ++br) {
      for (int b = 0; b < nb; ++b) {
        const GjArgs& a = batches[b];
        const Geom& m = gm[b];
        if (host_counts[b] == 0 || br >= m.G.nG - 1) continue;
        gj_table_kernel<<<dim3(m.G.nT, a.nitems), kTableThreads, 0, streams[b]>>>(a, br);
        gj_apply_kernel<<<dim3(apply_units(a.k), a.nitems), kThreads, asm_, streams[b]>>>(a, br);
        n += 2;
      }
    }
    for (int b = 0; b < nb; ++b) {
      const GjArgs& a = batches[b];
      const Geom& m = gm[b];
      if (host_counts[b] == 0) continue;
      const cudaStream_t s = streams[b];
      cudaError_t e = cudaMemsetAsync(a.active_count, 0, sizeof(int), s);
      if (e != cudaSuccess) return e;
      gj_off_kernel<<<m.cgrid, kThreads, 0, s>>>(a);
      gj_control_kernel<<<m.ctl_blocks, 256, 0, s>>>(a);
      // restart: Newton-Schulz (E into B, V' into W, swap), then RR
      gj_gemm_kernel<<<m.tiles, kThreads, gsm, s>>>(a, kNS1, kRestart);
      gj_gemm_kernel<<<m.tiles, kThreads, gsm, s>>>(a, kNS2, kRestart);
      gj_flip_kernel<<<m.ctl_blocks, 256, 0, s>>>(a, kRestart);
      gj_gemm_kernel<<<m.tiles, kThreads, gsm, s>>>(a, kRR1, kRestart);
      gj_gemm_kernel<<<m.tiles, kThreads, gsm, s>>>(a, kRR2, kRestart);
      n += 7;
      e = cudaMemcpyAsync(host_counts + b, a.active_count, sizeof(int), cudaMemcpyDeviceToHost, s);
      if (e != cudaSuccess) return e;
    }
    bool any = false;
    for (int b = 0; b < nb; ++b) {
      cudaError_t e = cudaStreamSynchronize(streams[b]);
      if (e != cudaSuccess) return e;
    }
    for (int b = 0; b < nb; ++b) any = any || host_counts[b] != 0;
    if (!any) break;
  }
  for (int b = 0; b < nb; ++b) {
    const GjArgs& a = batches[b];
    const Geom& m = gm[b];
    const cudaStream_t s = streams[b];
    gj_diag_kernel<<<dim3((a.k + 255) / 256, a.nitems), 256, 0, s>>>(a);
    gj_gemm_kernel<<<m.tiles, kThreads, gsm, s>>>(a, kNS1, kAlways);
    gj_gemm_kernel<<<m.tiles, kThreads, gsm, s>>>(a, kNS2, kAlways);
    gj_flip_kernel<<<m.ctl_blocks, 256, 0, s>>>(a, kAlways);
    gj_finish_kernel<<<a.nitems, kThreads, gj_finish_smem(a.k), s>>>(a);
    n += 5;
  }
  if (launches) *launches += n;
  return cudaGetLastError();
}

// The orthogonal-iteration refresh of nb batches (batch b on streams[b]),
// each followed on its stream by orth.cu's one-CTA pass over the blocks the
// grid pass left.  No host synchronisation.
cudaError_t run_orth_grid(const GjArgs* batches, int nb, const cudaStream_t* streams, int steps,
                          int sm_count, int64_t* launches) {
  const size_t gsm = gemm_smem(), csm = chol_smem();
  int64_t n = 0;
  for (int b = 0; b < nb; ++b) {
    const GjArgs& a = batches[b];
    const cudaStream_t s = streams[b];
    const int nt = (a.k + kT - 1) / kT;
    const dim3 tiles(nt * nt, a.nitems), panels(nt, a.nitems);
    const int chunks = (int)std::max<int64_t>(1, std::min<int64_t>(256, (int64_t)a.k * a.k / (64 * 1024)));
    const dim3 cgrid(chunks, a.nitems);
    const int ctl_blocks = (a.nitems + 255) / 256;
    cudaError_t e = cudaMemsetAsync(a.ctl, 0, sizeof(GjCtl) * (size_t)a.nitems, s);
    if (e != cudaSuccess) return e;
    gj_init_kernel<<<cgrid, kThreads, 0, s>>>(a);
    og_start_kernel<<<ctl_blocks, 256, 0, s>>>(a);
    n += 2;
    for (int st = 0; st < steps; ++st) {
      og_gemm_kernel<<<tiles, kThreads, gsm, s>>>(a, kOgAV);
      og_gemm_kernel<<<tiles, kThreads, gsm, s>>>(a, kOgGramT);
      og_chol_kernel<<<a.nitems, kThreads, csm, s>>>(a);
      og_trsm_kernel<<<panels, kThreads, csm, s>>>(a, 1);
      og_gemm_kernel<<<tiles, kThreads, gsm, s>>>(a, kOgGramV);   // Cholesky QR2
      og_chol_kernel<<<a.nitems, kThreads, csm, s>>>(a);
      og_trsm_kernel<<<panels, kThreads, csm, s>>>(a, 0);
      n += 7;
    }
    og_gemm_kernel<<<tiles, kThreads, gsm, s>>>(a, kOgAV);
    og_lambda_kernel<<<dim3((a.k + 7) / 8, a.nitems), 256, 0, s>>>(a);
    og_finish_kernel<<<cgrid, kThreads, 0, s>>>(a, steps);
    n += 3;
    EigArgs ea{};
    ea.info = a.info;
    ea.tiles = a.items;
    ea.num_tiles = a.nitems;
    ea.A = a.A;
    ea.Q = a.Q;
    ea.lam = a.lam;
    ea.scratch = a.scratch;
    ea.flags = a.flags;
    ea.stats = a.stats;
    ea.ctl = a.ctl;
    e = launch_orth(ea, steps, std::max(1, std::min(a.nitems, sm_count)), s);
    if (e != cudaSuccess) return e;
    ++n;
  }
  if (launches) *launches += n;
  return cudaGetLastError();
}

}  // namespace dobb
