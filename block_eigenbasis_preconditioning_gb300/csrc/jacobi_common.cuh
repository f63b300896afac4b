// Pieces of the blocked two-sided Jacobi sweep shared by the one-CTA-per-block
// eigensolver (jacobi.cu) and the grid eigensolver (jacobi_grid.cu): the
// round-robin tournament over column groups, the rotation of one table's
// diagonal tile by a team of warps, and the convergence constants.  Included
// inside an anonymous namespace after fp32_tiles.cuh; Golub & Van Loan's 2x2
// symmetric Schur rotation.
#pragma once

constexpr float kEps = 5.9604645e-8f;  // 2^-24, fp32 unit roundoff
constexpr float kColdOff = 3e-4f;      // sweep the same B again while off(B) stays above this
constexpr float kStopOff = 2e-6f;      // default: done when a fresh B's sweep leaves off(B) below this
constexpr float kStallOff = 1e-5f;     // ... or leaves it below this without shrinking (fp32 floor)

__host__ __device__ __forceinline__ int pow2_ceil(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

// Pair i of round r in the circle schedule over kk (even) players.
__host__ __device__ __forceinline__ void rr_pair(int r, int i, int kk, int& p, int& q) {
  if (i == 0) {
    p = kk - 1;
    q = r;
  } else {
    p = (r + i) % (kk - 1);
    q = (r - i + kk - 1) % (kk - 1);
  }
}

// Group geometry of the blocked sweep.
struct Geo {
  int nG;  // groups (even)
  int g;   // columns per group (<= 32)
  int n2;  // columns per table, 2 g
  int nT;  // tables per round, nG / 2
};

__host__ __device__ __forceinline__ Geo geo_for(int k) {
  Geo o;
  o.nG = 2 * ((k + kT - 1) / kT);
  o.g = (k + o.nG - 1) / o.nG;
  o.n2 = 2 * o.g;
  o.nT = o.nG / 2;
  return o;
}

// Column of B for local index a of the table made of groups gI, gJ (k when
// the index lies past the last column).
__device__ __forceinline__ int table_col(int a, int gI, int gJ, int g, int k) {
  const int c = a < g ? gI * g + a : gJ * g + (a - g);
  return c < k ? c : k;
}

// Local pair (p < q) number i of an inner round; false when the pair has an
// index past the group (odd g) or past the last column.
__device__ __forceinline__ bool inner_pair(bool intra, int r, int i, int g, int gI, int gJ, int k,
                                           int& p, int& q) {
  if (intra) {
    const int gp = g + (g & 1), half = gp >> 1;
    const int grp = i / half, ii = i - grp * half;
    rr_pair(r, ii, gp, p, q);
    if (p >= g || q >= g) return false;
    p += grp * g;
    q += grp * g;
  } else {
    p = i;
    q = g + (i + r) % g;
  }
  if (p > q) {
    const int tt = p;
    p = q;
    q = tt;
  }
  return table_col(p, gI, gJ, g, k) < k && table_col(q, gI, gJ, g, k) < k;
}

// Barrier over the nparts warps that solve one table (named barrier id).
__device__ __forceinline__ void team_sync(int id, int nparts) {
  if (nparts == 1)
    __syncwarp();
  else
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nparts * 32) : "memory");
}

// Rotations of one table's diagonal tile by a team of nparts warps (this warp
// is number `part`): each inner round rotates a set of disjoint column pairs
// of S (n2 x n2, row-major, shared memory), S <- J^T S J, and accumulates
// R <- R J.  Every warp of the team computes all the round's rotations, lane
// i for pair i (at most 32 pairs), so indices and rotations stay in
// registers (broadcast by shuffles for the row updates) and the warps need no
// exchange besides the barriers; the row updates are split by pairs and the
// column updates by rows.  Pairs are disjoint, so each lane loads four pairs'
// rows (row update) or four rows (column update) before storing any, which
// keeps several shared-memory loads in flight.  Returns the lane's count of
// rotations (counted by part 0 only).
__device__ int solve_table(float* S, float* R, int br, int t, const Geo& G, int k, float bfloor,
                           int part, int nparts, int bar_id) {
  const int lane = threadIdx.x & 31;
  const int n2 = G.n2;
  int gI, gJ;
  rr_pair(br, t, G.nG, gI, gJ);
  const int gp = G.g + (G.g & 1);
  const int n_intra = br == 0 ? gp - 1 : 0;
  const int perj = (n2 + nparts - 1) / nparts;
  const int j_lo = min(n2, part * perj), j_hi = min(n2, j_lo + perj);
  int rots = 0;
  for (int step = 0; step < n_intra + G.g; ++step) {
    const bool intra = step < n_intra;
    const int r = intra ? step : step - n_intra;
    const int npairs = intra ? gp : G.g;
    int p = 0, q = 0;
    float c = 1.f, s = 0.f;
    if (lane < npairs && inner_pair(intra, r, lane, G.g, gI, gJ, k, p, q)) {
      const float bpq = S[p * n2 + q];
      if (fabsf(bpq) > bfloor) {
        const float ta = (S[q * n2 + q] - S[p * n2 + p]) / (2.f * bpq);
        const float tn = ta >= 0.f ? 1.f / (ta + sqrtf(1.f + ta * ta)) : -1.f / (-ta + sqrtf(1.f + ta * ta));
        c = 1.f / sqrtf(1.f + tn * tn);
        s = tn * c;
        if (part == 0) ++rots;
      }
    }
    team_sync(bar_id, nparts);
    // rows p, q of S for this warp's share of the pairs, lanes along the row
    // (n2 <= 64: two elements per lane)
    const int per = (npairs + nparts - 1) / nparts;
    const int i_lo = min(npairs, part * per), i_hi = min(npairs, i_lo + per);
    for (int i0 = i_lo; i0 < i_hi; i0 += 4) {
      float cu[4], su[4], x[4][2], y[4][2];
      int pu[4], qu[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int src = (i0 + u) & 31;
        cu[u] = __shfl_sync(0xffffffffu, c, src);
        su[u] = __shfl_sync(0xffffffffu, s, src);
        pu[u] = __shfl_sync(0xffffffffu, p, src);
        qu[u] = __shfl_sync(0xffffffffu, q, src);
        if (i0 + u >= i_hi) su[u] = 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = lane + 32 * h;
          const bool ok = su[u] != 0.f && j < n2;
          x[u][h] = ok ? S[pu[u] * n2 + j] : 0.f;
          y[u][h] = ok ? S[qu[u] * n2 + j] : 0.f;
        }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = lane + 32 * h;
          if (su[u] != 0.f && j < n2) {
            S[pu[u] * n2 + j] = cu[u] * x[u][h] - su[u] * y[u][h];
            S[qu[u] * n2 + j] = su[u] * x[u][h] + cu[u] * y[u][h];
          }
        }
    }
    team_sync(bar_id, nparts);
    // columns p, q of S and R for this warp's share of the rows, lane i on
    // pair i, four rows at a time
    if (s != 0.f) {
      for (int j0 = j_lo; j0 < j_hi; j0 += 4) {
        float a[4], b[4], ra[4], rb[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + u < j_hi ? j0 + u : j_hi - 1;
          a[u] = S[j * n2 + p];
          b[u] = S[j * n2 + q];
          ra[u] = R[j * n2 + p];
          rb[u] = R[j * n2 + q];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + u;
          if (j < j_hi) {
            S[j * n2 + p] = c * a[u] - s * b[u];
            S[j * n2 + q] = s * a[u] + c * b[u];
            R[j * n2 + p] = c * ra[u] - s * rb[u];
            R[j * n2 + q] = s * ra[u] + c * rb[u];
          }
        }
      }
    }
    team_sync(bar_id, nparts);
  }
  return rots;
}

// Load an n2 x n2 rotation (row stride n2) into a zero-padded 64 x kLd tile.
__device__ __forceinline__ void load_rot(float* dst, const float* src, int n2) {
  for (int e = threadIdx.x; e < kT * kT; e += blockDim.x) {
    const int a = e / kT, b = e - a * kT;
    dst[a * kLd + b] = (a < n2 && b < n2) ? src[a * n2 + b] : 0.f;
  }
}

