// chunk_bwd_mma.cuh -- the walk's state products on the tensor cores: warp-level
// mma.sync m16n8k8 with TF32 operands and fp32 accumulation.  Each fp32 operand x is split
// into x = hi + lo, both TF32 (round to nearest), and a product takes three MMAs,
// lo*hi + hi*lo + hi*hi (the dropped lo*lo term is about 2^-22 of the product), which keeps
// the products at fp32-level accuracy.
//
// The operands stay where the walk keeps them, fp32 rows in shared memory; the split
// happens in registers as the fragments are loaded (tcgen05 would need the split parts
// staged in shared memory, three times the walk's tiles, which do not fit beside them).
//
// Fragment layout of m16n8k8 (TF32), lane = 4 g + t:
//   A (16 x 8, row-major): a0 (g, t), a1 (g + 8, t), a2 (g, t + 4), a3 (g + 8, t + 4)
//   B (8 x 8, k x n):      b0 (t, g), b1 (t + 4, g)
//   D (16 x 8):            d0 (g, 2t), d1 (g, 2t + 1), d2 (g + 8, 2t), d3 (g + 8, 2t + 1)
//
// Tiles: a product of M x N (M, N multiples of 16 and 8) has MT = M / 16 row tiles and
// NT = N / 8 column tiles.  Warp w takes row tile w % MT and NTW consecutive column tiles
// from (w / MT) NTW, NTW = max(1, MT NT / 8), so that the eight warps cover every tile
// once; with fewer than eight tiles the warps past them idle.  Device code only.
#pragma once

#include <stdint.h>

namespace gdn_bwd {
namespace tc {

struct FragA {
  uint32_t h[4], l[4];
};
struct FragB {
  uint32_t h[2], l[2];
};

__device__ __forceinline__ void split(float x, uint32_t &hi, uint32_t &lo) {
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi) : "f"(x));
  const float r = x - __uint_as_float(hi);
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(lo) : "f"(r));
}

__device__ __forceinline__ void frag_a(FragA &f, float a0, float a1, float a2, float a3) {
  split(a0, f.h[0], f.l[0]);
  split(a1, f.h[1], f.l[1]);
  split(a2, f.h[2], f.l[2]);
  split(a3, f.h[3], f.l[3]);
}

__device__ __forceinline__ void frag_b(FragB &f, float b0, float b1) {
  split(b0, f.h[0], f.l[0]);
  split(b1, f.h[1], f.l[1]);
}

__device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// d += a b in three MMAs, the small terms first
__device__ __forceinline__ void mma3(float (&d)[4], const FragA &a, const FragB &b) {
  mma(d, a.l, b.h);
  mma(d, a.h, b.l);
  mma(d, a.h, b.h);
}

// An operand whose values are exact in TF32 (bf16 inputs widened to fp32: 8 significant bits)
// needs no low part, and its product takes two MMAs.
__device__ __forceinline__ void frag_a_exact(FragA &f, float a0, float a1, float a2, float a3) {
  f.h[0] = __float_as_uint(a0);
  f.h[1] = __float_as_uint(a1);
  f.h[2] = __float_as_uint(a2);
  f.h[3] = __float_as_uint(a3);
}
__device__ __forceinline__ void frag_b_exact(FragB &f, float b0, float b1) {
  f.h[0] = __float_as_uint(b0);
  f.h[1] = __float_as_uint(b1);
}
template <bool AX, bool BX>
__device__ __forceinline__ void mma_x(float (&d)[4], const FragA &a, const FragB &b) {
  if (!AX) mma(d, a.l, b.h);
  if (!BX) mma(d, a.h, b.l);
  mma(d, a.h, b.h);
}

// The warp's tiles of an M x N product (see above): its row tile m0, its first column tile
// n0, and whether it has any.
template <int M, int N>
struct Tiles {
  static constexpr int MT = M / 16, NT = N / 8, NTW = (MT * NT) / 8 > 0 ? (MT * NT) / 8 : 1;
  int m0, n0;
  bool any;
  __device__ __forceinline__ explicit Tiles(int warp) {
    m0 = (warp % MT) * 16;
    n0 = (warp / MT) * NTW * 8;
    any = (warp / MT) * NTW < NT;
  }
};

// The same tiles assigned the other way round: warp w takes column tile w % NT and MTW
// consecutive row tiles from (w / NT) MTW, so that a B fragment serves MTW row tiles.  Better
// where A is cheap to load (exact in TF32) and B must be split.
template <int M, int N>
struct TilesM {
  static constexpr int MT = M / 16, NT = N / 8, MTW = (MT * NT) / 8 > 0 ? (MT * NT) / 8 : 1;
  int m0, n0;
  bool any;
  __device__ __forceinline__ explicit TilesM(int warp) {
    n0 = (warp % NT) * 8;
    m0 = (warp / NT) * MTW * 16;
    any = (warp / NT) * MTW < MT;
  }
};

// The three forms below add to D, over k in [kbeg, kend) (multiples of 8), the products of
// fp32 rows in shared memory; a triangular factor passes the range where it is nonzero.

// D[m][n] += sum_k A[m][k] ka_k B[n][k]: A rows m0 .. (stride lda), with KA its column k
// scaled by ka[k] (ka then holds kend entries; without KA it is not read); B rows n0 + 8 j ..
// (ldb).
// AX, BX: A's (B's) values are exact in TF32 (no split; KA must then be off for A).
template <int NTW, bool KA = false, bool AX = false, bool BX = false>
__device__ __forceinline__ void mma_nt(int lane, const float *A, int lda, const float *ka, const float *B, int ldb,
                                       int m0, int n0, int kbeg, int kend, float (&d)[NTW][4]) {
  static_assert(!(KA && AX), "a scaled operand is not exact");
  const int g = lane >> 2, t = lane & 3;
  const float *a = A + (m0 + g) * lda + t;
  const float *b = B + (n0 + g) * ldb + t;
#pragma unroll 2
  for (int k0 = kbeg; k0 < kend; k0 += 8) {
    const float s0 = KA ? ka[k0 + t] : 1.f, s1 = KA ? ka[k0 + t + 4] : 1.f;
    FragA fa;
    if (AX) frag_a_exact(fa, a[k0], a[8 * lda + k0], a[k0 + 4], a[8 * lda + k0 + 4]);
    else frag_a(fa, s0 * a[k0], s0 * a[8 * lda + k0], s1 * a[k0 + 4], s1 * a[8 * lda + k0 + 4]);
#pragma unroll
    for (int j = 0; j < NTW; ++j) {
      FragB fb;
      if (BX) frag_b_exact(fb, b[8 * j * ldb + k0], b[8 * j * ldb + k0 + 4]);
      else frag_b(fb, b[8 * j * ldb + k0], b[8 * j * ldb + k0 + 4]);
      mma_x<AX, BX>(d[j], fa, fb);
    }
  }
}

// mma_nt over MTW row tiles m0 + 16 i of one column tile n0 (TilesM): D[i][.] += A B^T with
// A exact in TF32 (raw bf16 values, no split) and B split, its fragment loaded once for all
// MTW row tiles.  The same products, in the same order for each tile, as mma_nt.
template <int MTW>
__device__ __forceinline__ void mma_nt_m(int lane, const float *A, int lda, const float *B, int ldb, int m0, int n0,
                                         int kbeg, int kend, float (&d)[MTW][4]) {
  const int g = lane >> 2, t = lane & 3;
  const float *a = A + (m0 + g) * lda + t;
  const float *b = B + (n0 + g) * ldb + t;
#pragma unroll 2
  for (int k0 = kbeg; k0 < kend; k0 += 8) {
    FragB fb;
    frag_b(fb, b[k0], b[k0 + 4]);
#pragma unroll
    for (int i = 0; i < MTW; ++i) {
      const float *ai = a + 16 * i * lda;
      FragA fa;
      frag_a_exact(fa, ai[k0], ai[8 * lda + k0], ai[k0 + 4], ai[8 * lda + k0 + 4]);
      mma_x<true, false>(d[i], fa, fb);
    }
  }
}

// D[m][n] += sum_k mult ra_m A[m][k] kb_k B[k][n]: A rows m0 .. (stride lda) scaled by ra (per
// row), B rows k (stride ldb) scaled by kb (per row k), columns n0 + 8 j ..  BX: B's values
// are exact in TF32 and unscaled (kb is not read), its k-scale then carried by A's columns
// through kb instead.  KB = false: no k-scale (kb is not read; the same as kb all ones).
template <int NTW, bool BX = false, bool KB = true>
__device__ __forceinline__ void mma_nn(int lane, const float *A, int lda, const float *ra, float mult, const float *B,
                                       int ldb, const float *kb, int m0, int n0, int kbeg, int kend,
                                       float (&d)[NTW][4]) {
  const int g = lane >> 2, t = lane & 3;
  const float *a = A + (m0 + g) * lda + t;
  const float *b = B + t * ldb + n0 + g;
  const float r0 = mult * ra[m0 + g], r1 = mult * ra[m0 + g + 8];
#pragma unroll 2
  for (int k0 = kbeg; k0 < kend; k0 += 8) {
    const float s0 = KB ? kb[k0 + t] : 1.f, s1 = KB ? kb[k0 + t + 4] : 1.f;
    FragA fa;
    if (BX) frag_a(fa, r0 * s0 * a[k0], r1 * s0 * a[8 * lda + k0], r0 * s1 * a[k0 + 4], r1 * s1 * a[8 * lda + k0 + 4]);
    else frag_a(fa, r0 * a[k0], r1 * a[8 * lda + k0], r0 * a[k0 + 4], r1 * a[8 * lda + k0 + 4]);
#pragma unroll
    for (int j = 0; j < NTW; ++j) {
      FragB fb;
      if (BX) frag_b_exact(fb, b[k0 * ldb + 8 * j], b[(k0 + 4) * ldb + 8 * j]);
      else frag_b(fb, s0 * b[k0 * ldb + 8 * j], s1 * b[(k0 + 4) * ldb + 8 * j]);
      mma_x<false, BX>(d[j], fa, fb);
    }
  }
}

// D1[m][n] += sum_k r1_m A1[m][k] B[k][n] and D2[m][n] += sum_k mult2 r2_m A2[m][k] B[k][n]: two
// products of the mma_nn form (without a k-scale) that share B, whose fragments are loaded and
// split once for both.  The same sums, term by term, as two mma_nn calls.
template <int NTW>
__device__ __forceinline__ void mma_nn_pair(int lane, const float *A1, const float *A2, int lda, const float *r1,
                                            const float *r2, float mult2, const float *B, int ldb, int m0, int n0,
                                            int kbeg, int kend, float (&d1)[NTW][4], float (&d2)[NTW][4]) {
  const int g = lane >> 2, t = lane & 3;
  const float *a1 = A1 + (m0 + g) * lda + t, *a2 = A2 + (m0 + g) * lda + t;
  const float *b = B + t * ldb + n0 + g;
  const float p0 = r1[m0 + g], p1 = r1[m0 + g + 8];
  const float q0 = mult2 * r2[m0 + g], q1 = mult2 * r2[m0 + g + 8];
#pragma unroll 2
  for (int k0 = kbeg; k0 < kend; k0 += 8) {
    FragA f1, f2;
    frag_a(f1, p0 * a1[k0], p1 * a1[8 * lda + k0], p0 * a1[k0 + 4], p1 * a1[8 * lda + k0 + 4]);
    frag_a(f2, q0 * a2[k0], q1 * a2[8 * lda + k0], q0 * a2[k0 + 4], q1 * a2[8 * lda + k0 + 4]);
#pragma unroll
    for (int j = 0; j < NTW; ++j) {
      FragB fb;
      frag_b(fb, b[k0 * ldb + 8 * j], b[(k0 + 4) * ldb + 8 * j]);
      mma_x<false, false>(d1[j], f1, fb);
      mma_x<false, false>(d2[j], f2, fb);
    }
  }
}

// D[m][n] += sum_k mult ks_k A[k][m] B[k][n]: A stored by rows k (stride lda), so that the
// operand is its transpose, row k scaled by ks[k]; B rows k (stride ldb), columns n0 + 8 j ..
// BX: B's values are exact in TF32 (no split).  KS = false: no row scale (ks is not read;
// the same as ks all ones).
template <int NTW, bool BX = false, bool KS = true>
__device__ __forceinline__ void mma_tn(int lane, const float *A, int lda, const float *ks, float mult, const float *B,
                                       int ldb, int m0, int n0, int kbeg, int kend, float (&d)[NTW][4]) {
  const int g = lane >> 2, t = lane & 3;
  const float *a = A + t * lda + m0 + g;
  const float *b = B + t * ldb + n0 + g;
#pragma unroll 2
  for (int k0 = kbeg; k0 < kend; k0 += 8) {
    const float s0 = KS ? mult * ks[k0 + t] : mult, s1 = KS ? mult * ks[k0 + t + 4] : mult;
    FragA fa;
    frag_a(fa, s0 * a[k0 * lda], s0 * a[k0 * lda + 8], s1 * a[(k0 + 4) * lda], s1 * a[(k0 + 4) * lda + 8]);
#pragma unroll
    for (int j = 0; j < NTW; ++j) {
      FragB fb;
      if (BX) frag_b_exact(fb, b[k0 * ldb + 8 * j], b[(k0 + 4) * ldb + 8 * j]);
      else frag_b(fb, b[k0 * ldb + 8 * j], b[(k0 + 4) * ldb + 8 * j]);
      mma_x<false, BX>(d[j], fa, fb);
    }
  }
}

// The element of tile j that fragment slot e of this lane holds: row m0 + g (+ 8 for e >= 2),
// column n0 + 8 j + 2 t (+ 1 for odd e).
__device__ __forceinline__ int frag_row(int lane, int m0, int e) { return m0 + (lane >> 2) + ((e >> 1) << 3); }
__device__ __forceinline__ int frag_col(int lane, int n0, int j, int e) { return n0 + 8 * j + 2 * (lane & 3) + (e & 1); }

// Four adjacent elements of tile j for one 16-byte vector store or atomic add: lanes t and
// t ^ 1 swap half their fragment, so that an even-t lane holds row g, columns 2t .. 2t + 3 and
// an odd-t lane row g + 8, columns 2t - 2 .. 2t + 1 of the 16 x 8 tile.  row and col are the
// quad's first element within the tile.  Every lane of the warp takes part.
__device__ __forceinline__ void frag_quad(int lane, const float (&d)[4], int &row, int &col, float4 &v) {
  const int t = lane & 3;
  const bool odd = (t & 1) != 0;
  const float r0 = __shfl_xor_sync(0xffffffffu, odd ? d[0] : d[2], 1);
  const float r1 = __shfl_xor_sync(0xffffffffu, odd ? d[1] : d[3], 1);
  row = (lane >> 2) + (odd ? 8 : 0);
  col = odd ? 2 * t - 2 : 2 * t;
  v = odd ? make_float4(r0, r1, d[2], d[3]) : make_float4(d[0], d[1], r0, r1);
}

}  // namespace tc
}  // namespace gdn_bwd
