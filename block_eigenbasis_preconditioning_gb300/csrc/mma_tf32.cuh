// 64 x 64 tile products on the warp-level tensor-core path (mma.sync
// m16n8k8, TF32 inputs, fp32 accumulation), for the eigensolver's small
// dense products.  Included inside an anonymous namespace.
//
// Layout: operands staged in shared memory as 64 rows of kLdM floats, row c
// holding the 64 values of reduction index c:  A(m = i, k = c) = P[c kLdM + i],
// B(k = c, n = j) = Q[c kLdM + j].  kLdM = 72 puts the 32 addresses of every
// fragment load (4 reduction rows x 8 consecutive columns) in 32 distinct
// banks.
//
// Eight warps tile the 64 x 64 output: warp w owns rows 16 (w & 3) ... + 16
// and columns 32 (w >> 2) ... + 32, as four 16 x 8 accumulators of four
// floats each (acc[j][0..3] = (row g, col 8 j + 2 t), (g, 8 j + 2 t + 1),
// (g + 8, 8 j + 2 t), (g + 8, 8 j + 2 t + 1) with g = lane / 4, t = lane % 4).
//
// Precision: kPasses = 3 multiplies in split precision, A B ~ Ah Bh + Al Bh +
// Ah Bl with h the TF32 rounding and l = x - h (error ~2^-21 relative to
// |A| |B|); kPasses = 1 in plain TF32 (~2^-11).  The accumulators start from
// whatever the caller loaded, so X + E Y products add the TF32-rounded
// correction onto an fp32 X.
#pragma once

constexpr int kLdM = 72;

__device__ __forceinline__ uint32_t tf32_bits(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void mma_m16n8k8_tf32(float (&d)[4], const uint32_t (&a)[4],
                                                 const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// acc += A B over the first n reduction indices (n <= 64; rows past n of P
// and Q must hold zeros up to the next multiple of 8).
template <int kPasses>
__device__ __forceinline__ void mma_tn_64(const float* P, const float* Q, int n, float (&acc)[4][4]) {
  const int lane = threadIdx.x & 31, warp = (threadIdx.x >> 5) & 7;
  const int g = lane >> 2, t = lane & 3;
  const int m0 = 16 * (warp & 3), nb = 32 * (warp >> 2);
  for (int k0 = 0; k0 < n; k0 += 8) {
    const float* p0 = P + (k0 + t) * kLdM + m0 + g;
    const float* p1 = p0 + 4 * kLdM;
    const float av[4] = {p0[0], p0[8], p1[0], p1[8]};
    uint32_t ah[4], al[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      ah[i] = tf32_bits(av[i]);
      if (kPasses == 3) al[i] = tf32_bits(av[i] - __uint_as_float(ah[i]));
    }
    const float* q0 = Q + (k0 + t) * kLdM + nb + g;
    const float* q1 = q0 + 4 * kLdM;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float b0 = q0[8 * j], b1 = q1[8 * j];
      uint32_t bh[2] = {tf32_bits(b0), tf32_bits(b1)};
      mma_m16n8k8_tf32(acc[j], ah, bh);
      if (kPasses == 3) {
        uint32_t bl[2] = {tf32_bits(b0 - __uint_as_float(bh[0])),
                          tf32_bits(b1 - __uint_as_float(bh[1]))};
        mma_m16n8k8_tf32(acc[j], al, bh);
        mma_m16n8k8_tf32(acc[j], ah, bl);
      }
    }
  }
}

// The element (row, column) held in accumulator slot (j, e) of this thread.
__device__ __forceinline__ void mma_coord(int j, int e, int& row, int& col) {
  const int lane = threadIdx.x & 31, warp = (threadIdx.x >> 5) & 7;
  row = 16 * (warp & 3) + (lane >> 2) + (e >= 2 ? 8 : 0);
  col = 32 * (warp >> 2) + 8 * j + 2 * (lane & 3) + (e & 1);
}

// acc[j][e] = S[row kLdM + col]  (trans = false) or S[col kLdM + row] (true)
template <bool kTrans>
__device__ __forceinline__ void mma_load_acc(const float* S, float (&acc)[4][4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int r, c;
      mma_coord(j, e, r, c);
      acc[j][e] = kTrans ? S[c * kLdM + r] : S[r * kLdM + c];
    }
}

// S[row kLdM + col] = acc (trans = false) or S[col kLdM + row] = acc (true)
template <bool kTrans>
__device__ __forceinline__ void mma_store_acc(float* S, const float (&acc)[4][4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int r, c;
      mma_coord(j, e, r, c);
      if (kTrans) S[c * kLdM + r] = acc[j][e];
      else S[r * kLdM + c] = acc[j][e];
    }
}
