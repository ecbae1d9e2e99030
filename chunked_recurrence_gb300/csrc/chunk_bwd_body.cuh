// chunk_bwd_body.cuh -- the block bodies of the fp32 backward of the chunked gated delta rule.
//
// Training runs backward through the layer ("[v1] support GDN Ulysses cp", Testing: loss
// alignment over training steps; "feat: hybrid CP for Qwen3.5 MoE (DeltaNet + attention)",
// Test plan: forward/backward passes).  This is the exact gradient of the chunk form
//   gamma = inclusive cumsum of g in the chunk, b = exp(gamma), d = exp(gamma_last - gamma)
//   A  = strictly-lower(diag(beta) (K K^T) * Gamma),  Gamma_ij = exp(gamma_i - gamma_j)
//   Z  = (I + A)^-1,  T = Z diag(beta)
//   U' = T (V - diag(b) K S^T)                  (= T V - W S^T with W = T diag(b) K)
//   O  = scale (diag(b) Q S^T + P U'),  P = (Q K^T) * Gamma, causal incl. the diagonal
//   S1 = b_last S + U'^T diag(d) K
// for upstream gradients dO and dS1, taken back step by step (reverse mode):
//   dU' = diag(d) K dS1^T + P^T Ot   (Ot = scale dO),  dP = Ot U'^T
//   dV  = T^T dU',  dT = dU' (V - diag(b) K S^T)^T,   dA = -Z^T (dT diag(beta)) Z^T
//   dS  = b_last dS1 + Ot^T diag(b) Q - (diag(b) dV)^T K
//   dq  = diag(b) Ot S + (dP * Gamma) K
//   dk  = diag(d) U' dS1 + (dP * Gamma)^T Q - diag(b) dV S + (dKK + dKK^T) K,
//         dKK = diag(beta) dA * Gamma
//   dbeta = colsum(dT * Z) + rowsum(dA * KK * Gamma)
//   dgamma from Gamma (row sums minus column sums of dGamma * Gamma), b and d; dg is the
//   reverse cumulative sum of dgamma.
// The work runs as three kernels:
//   prep  one block per (chunk, v-head), all in parallel: the chunk's state-independent
//         matrices Z = (I + A)^-1, KG = (K K^T) * Gamma (strictly lower) and
//         QG = (Q K^T) * Gamma (lower incl. the diagonal), stored once;
//   walk  one block per (BV state rows, v-head, sequence).  Each row of the state evolves on
//         its own given k, g, beta and its column of v, and so does each row of dS.  A block
//         recomputes its rows' chunk-start states in a forward sweep, then walks the chunks
//         backward carrying its rows of dS.  It completes dv and dh0 of its rows and adds
//         the parts of dq and dk that take S or dS.  dP, dT, dd and db are sums over all
//         state rows: each block adds its rows' share into per-chunk sums;
//   grad  one block per (chunk, v-head), in parallel: from the summed dP, dT, dd and db,
//         everything that is linear in them: dbeta, dgamma and so dg, and the (dP * Gamma)
//         and dKK parts of dq and dk.
// So the C x C work (K K^T, Q K^T, the inversion, Y, dA and the C x C x K products of dq
// and dk) runs once per chunk and head, not once per block of state rows.
//
// The bodies are written against an executor X with three operations: x.par(n, f) runs f(i)
// for i in [0, n), the items independent of each other; x.sync() is a block barrier;
// x.add(p, v) adds v to *p atomically.  The CUDA kernels run items on threads with
// __syncthreads(); a host harness runs the same code with plain loops.
#pragma once

#include <math.h>
#include <stddef.h>
#include <stdint.h>

#if defined(__CUDACC__)
#include "chunk_bwd_mma.cuh"
#define GDN_BWD_FN __device__ __forceinline__
#define GDN_BWD_HD __host__ __device__ inline
#else
#define GDN_BWD_FN inline
#define GDN_BWD_HD inline
#endif

namespace gdn_bwd {

constexpr int C = 64;  // tokens per chunk
constexpr int CP = C + 1;
constexpr float kEps = 1e-6f;  // q/k L2 norm: x / sqrt(sum x^2 + eps)
constexpr size_t kPrep = 3 * (size_t)C * C + 5 * C;  // floats per (chunk, v-head): Z, KG, QG; 5 vectors
constexpr size_t kPrepVec = 3 * (size_t)C * C;       // offset of the vectors gamma, b, d, 1/|k|, 1/|q|
constexpr size_t kSums = 2 * (size_t)C * C + 2 * C;  // floats per (chunk, v-head): dP, dT, dd, db

struct Params {
  const void *q, *k, *v;  // q, k [n_tok][Hqk][K] (token strides qs, ks), v [n_tok][Hv][V] (vs)
  const float *g, *beta;  // [n_tok][Hv]
  const float *h0;        // [n_seq][Hv][V][K] or null
  const float *dout;      // [n_tok][Hv][V]
  const float *dhT;       // [n_seq][Hv][V][K] or null
  const int32_t *cu;      // sequence bounds, or null: rows of row_T tokens
  int64_t row_T, n_tok;
  int n_seqs;
  int Hqk, Hv, K, V;
  int64_t qs, ks, vs;
  float scale;
  int l2norm;
  int vec8;         // q, k, v load as 8-element vectors and d_o as 4-element ones (16-byte aligned
                    // rows and strides)
  // chunk slots: chunk c of sequence s is slot s + start_s / C + c (distinct for every chunk)
  float *states;    // [slot][Hv][V][K]: chunk-start states
  float *fw;        // [slot][Hv][3][C][V]: the forward sweep's U', V - diag(b) K S^T and K S^T
  float *prep;      // [slot][Hv][kPrep]: Z, KG, QG ([C][C] row-major each), then gamma, b = exp(gamma),
                    // d = exp(gamma_last - gamma), 1/|k|, 1/|q| ([C] each)
  float *sums;      // [slot][Hv][kSums]: dP [C][C], dT [C][C], dd [C], db [C]; zero before the walk
  float *dqn, *dkn; // [n_tok][Hqk][K]: gradients of the unit-norm (or raw) q and k, accumulated
  float *dv;        // [n_tok][Hv][V]
  float *dg, *dbeta;  // [n_tok][Hv]
  float *dh0;       // [n_seq][Hv][V][K] or null
  int32_t *status;  // set to GDN_ERR_BOUNDS on a bad sequence range
};

// shared memory of one block, in floats
GDN_BWD_HD size_t prep_smem_floats(int K) { return 2 * (size_t)C * (K + 4) + 2 * (size_t)C * CP + 4 * C; }
GDN_BWD_HD size_t walk_smem_floats(int K, int BV) {
  return 2 * (size_t)C * (K + 4) + 2 * (size_t)BV * (K + 4) + 8 * (size_t)C * (BV + 4) + 2 * (size_t)C * CP + 12 * C;
}
GDN_BWD_HD size_t grad_smem_floats(int K) { return 2 * (size_t)C * (K + 4) + 6 * (size_t)C * (C + 4) + 16 * C; }

GDN_BWD_FN int64_t seq_start(const Params &p, int s) { return p.cu ? (int64_t)p.cu[s] : (int64_t)s * p.row_T; }

GDN_BWD_FN bool seq_bounds(const Params &p, int s, int64_t &start, int64_t &end) {
  start = seq_start(p, s);
  end = p.cu ? (int64_t)p.cu[s + 1] : start + p.row_T;
  return start >= 0 && end >= start && end <= p.n_tok;
}

// The chunk held by a slot: its first token t0 and length n.  False for a slot that no chunk
// uses (slots are distinct, not dense) and for a sequence whose bounds are bad (the walk
// reports those).  Slot s + start_s / C is the first of sequence s, rising with s.
GDN_BWD_FN bool slot_chunk(const Params &p, int64_t slot, int64_t &t0, int &n) {
  int lo = 0, hi = p.n_seqs - 1;
  while (lo < hi) {  // the last sequence whose first slot is at or before this one
    const int mid = (lo + hi + 1) / 2;
    if (mid + seq_start(p, mid) / C <= slot) lo = mid;
    else hi = mid - 1;
  }
  int64_t start, end;
  if (!seq_bounds(p, lo, start, end)) return false;
  const int64_t ci = slot - (lo + start / C);
  if (ci < 0 || ci * C >= end - start) return false;
  t0 = start + ci * C;
  n = (int)(end - t0 < C ? end - t0 : C);
  return true;
}

// Four consecutive floats (16-byte aligned on the device).
GDN_BWD_FN void ld4(const float *p, float *o) {
#if defined(__CUDACC__)
  const float4 v = *reinterpret_cast<const float4 *>(p);
  o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
#else
  for (int e = 0; e < 4; ++e) o[e] = p[e];
#endif
}

// Groups of float4 an item for a copy of nf float4: enough that each thread has several
// loads in flight before its first store (an item's loads all issue before its stores).
GDN_BWD_HD constexpr int per_item(int nf) { return nf >= 1024 ? 4 : (nf >= 512 ? 2 : 1); }

// dst[r][c] = scale * src[r * src_ld + c] for a ROWS x COLS fp32 block (COLS a multiple of 4,
// src and src_ld 16-byte aligned); rows r >= n read as zero when n < ROWS.
template <int ROWS, int COLS, class X>
GDN_BWD_FN void copy_block(X &x, const float *src, size_t src_ld, float *dst, int dst_ld, int n = ROWS,
                           float scale = 1.f) {
  constexpr int NF = ROWS * COLS / 4, PER = per_item(NF), NI = NF / PER;
  static_assert(NF % PER == 0, "whole items");
  x.par(NI, [&](int t) {
    float v[PER][4];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int f = t + u * NI, r = f / (COLS / 4), c = (f % (COLS / 4)) * 4;
      if (r < n) ld4(src + r * src_ld + c, v[u]);
      else v[u][0] = v[u][1] = v[u][2] = v[u][3] = 0.f;
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int f = t + u * NI, r = f / (COLS / 4), c = (f % (COLS / 4)) * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e) dst[r * dst_ld + c + e] = scale * v[u][e];
    }
  });
}

// One item's share of a ROWS x COLS fp32 block copy: float4 pieces t, t + NI, ... of it.
// load() issues the item's loads and store() writes them, so that an item can hold the
// loads of several fills in flight before its first store.  Rows r >= n read as zero.
template <int ROWS, int COLS, int NI>
struct Fill4 {
  static constexpr int NF = ROWS * COLS / 4, PER = (NF + NI - 1) / NI;
  float v[PER][4];
  GDN_BWD_FN void load(int t, const float *src, size_t src_ld, int n) {
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int f = t + u * NI, r = f / (COLS / 4), c = (f % (COLS / 4)) * 4;
      if (f < NF && r < n) ld4(src + r * src_ld + c, v[u]);
      else v[u][0] = v[u][1] = v[u][2] = v[u][3] = 0.f;
    }
  }
  GDN_BWD_FN void store(int t, float *dst, int dst_ld, float scale = 1.f) const {
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int f = t + u * NI, r = f / (COLS / 4), c = (f % (COLS / 4)) * 4;
      if (f < NF)
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[r * dst_ld + c + e] = scale * v[u][e];
    }
  }
};

// The same for rows of q, k or v read as 8-element vectors through LD::vec8: element
// (r, c) of the block is src[base + r * row_stride + c].
template <int ROWS, int COLS, int NI>
struct Fill8 {
  static constexpr int NV = ROWS * COLS / 8, PER = (NV + NI - 1) / NI;
  float v[PER][8];
  template <class LD>
  GDN_BWD_FN void load(LD ld, int t, const void *src, int64_t base, int64_t row_stride, int n) {
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int f = t + u * NI, r = f / (COLS / 8), c = (f % (COLS / 8)) * 8;
#pragma unroll
      for (int e = 0; e < 8; ++e) v[u][e] = 0.f;
      if (f < NV && r < n) ld.vec8(src, base + r * row_stride + c, v[u]);
    }
  }
  GDN_BWD_FN void store(int t, float *dst, int dst_ld) const {
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int f = t + u * NI, r = f / (COLS / 8), c = (f % (COLS / 8)) * 8;
      if (f < NV)
#pragma unroll
        for (int e = 0; e < 8; ++e) dst[r * dst_ld + c + e] = v[u][e];
    }
  }
};

// Rows t0 .. t0 + n - 1 of k (and of q, when Qs is given) of q/k head qh into [C][KP]
// tiles, zero past n.  The L2 norm follows in norm_and_cumsum, after a barrier.
template <int K, int KP = K + 1, class X, class LD>
GDN_BWD_FN void load_keys(X &x, const Params &p, LD ld, float *Ks, float *Qs, int64_t t0, int n, int qh) {
  const bool with_q = Qs != nullptr;
  if (p.vec8) {
    // 8-element vectors, PER of them (of k and of q) an item, all loads before the stores
    constexpr int NV = C * (K / 8), PER = per_item(NV), NI = NV / PER;
    x.par(NI, [&](int t) {
      float kv[PER][8], qv[PER][8];
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int idx = t + u * NI, r = idx / (K / 8), c = (idx % (K / 8)) * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) kv[u][e] = qv[u][e] = 0.f;
        if (r < n) {
          ld.vec8(p.k, (t0 + r) * p.ks + (int64_t)qh * K + c, kv[u]);
          if (with_q) ld.vec8(p.q, (t0 + r) * p.qs + (int64_t)qh * K + c, qv[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < PER; ++u) {
        const int idx = t + u * NI, r = idx / (K / 8), c = (idx % (K / 8)) * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          Ks[r * KP + c + e] = kv[u][e];
          if (with_q) Qs[r * KP + c + e] = qv[u][e];
        }
      }
    });
  } else {
    x.par(C * K, [&](int idx) {
      const int r = idx / K, c = idx % K;
      const bool in = r < n;
      Ks[r * KP + c] = in ? ld(p.k, (t0 + r) * p.ks + (int64_t)qh * K + c) : 0.f;
      if (with_q) Qs[r * KP + c] = in ? ld(p.q, (t0 + r) * p.qs + (int64_t)qh * K + c) : 0.f;
    });
  }
}

template <class X>
GDN_BWD_FN void load_gates(X &x, const Params &p, float *gam, float *bet, int64_t t0, int n, int h) {
  x.par(C, [&](int i) {
    const bool in = i < n;
    gam[i] = in ? p.g[(t0 + i) * p.Hv + h] : 0.f;
    bet[i] = in ? p.beta[(t0 + i) * p.Hv + h] : 0.f;
  });
}

// After the loads' barrier: unit-norm rows of k (and q), gamma = the inclusive cumsum of g.
// The rows past n are zero and stay zero; gamma past n repeats the last token's.
// rin (optional, 2 C floats): the rows' inverse norms, k rows then q rows (1 without the norm).
template <int K, int KP = K + 1, class X>
GDN_BWD_FN void norm_and_cumsum(X &x, const Params &p, float *Ks, float *Qs, float *gam, float *rin = nullptr) {
  if (p.l2norm) {
    x.par(Qs ? 2 * C : C, [&](int r) {
      float *row = r < C ? Ks + r * KP : Qs + (r - C) * KP;
      float ss = 0.f;
      for (int c = 0; c < K; ++c) ss = fmaf(row[c], row[c], ss);
      const float inv = 1.f / sqrtf(ss + kEps);
      for (int c = 0; c < K; ++c) row[c] *= inv;
      if (rin) rin[r] = inv;
    });
  } else if (rin) {
    x.par(Qs ? 2 * C : C, [&](int r) { rin[r] = 1.f; });
  }
  if (x.leader())
    for (int i = 1; i < C; ++i) gam[i] += gam[i - 1];
}

#if defined(__CUDA_ARCH__)
// Z = (I + A)^-1 for the strictly lower C x C A (row stride lda; zero on and above the
// diagonal), by forward substitution swept by columns of A, in registers and without a
// barrier: threads 0-127 each keep an 8 x 4 tile of Z, rows rg + 8 m and columns 16 a + cj
// (one in each 16-column block; rg = lane % 8, cj = 4 warp + lane / 8).  Rows are taken four
// at a time: every thread reads rows k .. k + 3 (updated through row k - 1) from their owners
// by shuffle, finishes them among themselves, and applies all four to its own rows as
// z_i -= sum_j A_ij Z_j; A_ij = 0 for j >= i leaves rows <= k unchanged and makes rows
// k + 1 .. k + 3 final.  Rows of Z are zero right of their diagonal, so rows k .. k + 3 touch
// only the column blocks a <= k / 16 (fixed at compile time).  Writes all of Z, zeros above
// the diagonal included, to Y (row stride ldy); the caller syncs before Y is read.
__device__ __forceinline__ void invert_unit_lower_rt(const float *A, int lda, float *Y, int ldy, int tid) {
  static_assert(C == 64, "the register tiles cover 64 x 64");
  const int lane = tid & 31, rg = lane & 7, cj = (tid >> 5) * 4 + (lane >> 3);
  float y[8][4];
#pragma unroll
  for (int m = 0; m < 8; ++m)
#pragma unroll
    for (int a = 0; a < 4; ++a) y[m][a] = (rg + 8 * m == 16 * a + cj) ? 1.f : 0.f;
  const float *ar = A + rg * lda;
#pragma unroll
  for (int k = 0; k < C; k += 4) {
    const int m0 = k >> 3, na = (k >> 4) + 1;
    float z[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int a = 0; a < na; ++a) z[j][a] = __shfl_sync(0xffffffffu, y[m0][a], ((k + j) & 7) | (lane & 24));
    const float a10 = A[(k + 1) * lda + k], a20 = A[(k + 2) * lda + k], a21 = A[(k + 2) * lda + k + 1];
    const float a30 = A[(k + 3) * lda + k], a31 = A[(k + 3) * lda + k + 1], a32 = A[(k + 3) * lda + k + 2];
#pragma unroll
    for (int a = 0; a < na; ++a) {
      z[1][a] = fmaf(-a10, z[0][a], z[1][a]);
      z[2][a] = fmaf(-a21, z[1][a], fmaf(-a20, z[0][a], z[2][a]));
      z[3][a] = fmaf(-a32, z[2][a], fmaf(-a31, z[1][a], fmaf(-a30, z[0][a], z[3][a])));
    }
#pragma unroll
    for (int m = m0; m < 8; ++m) {
      const float *row = ar + 8 * m * lda + k;
      const float v0 = row[0], v1 = row[1], v2 = row[2], v3 = row[3];
#pragma unroll
      for (int a = 0; a < na; ++a)
        y[m][a] = fmaf(-v3, z[3][a], fmaf(-v2, z[2][a], fmaf(-v1, z[1][a], fmaf(-v0, z[0][a], y[m][a]))));
    }
  }
#pragma unroll
  for (int m = 0; m < 8; ++m)
#pragma unroll
    for (int a = 0; a < 4; ++a) Y[(rg + 8 * m) * ldy + 16 * a + cj] = y[m][a];
}
#endif

// ---- prep: Z, KG and QG of one (chunk, v-head)
template <int KD, class X, class LD>
GDN_BWD_FN void prep_block(X &x, const Params &p, LD ld, float *sm, int64_t slot, int h) {
  constexpr int K = KD, KP = KD + 4;  // rows padded for the tensor-core fragments' loads
  int64_t t0;
  int n;
  if (!slot_chunk(p, slot, t0, n)) return;
  float *Ks = sm;             // [C][KP]
  float *Qs = Ks + C * KP;    // [C][KP]
  float *Am = Qs + C * KP;    // [C][CP]  A (strictly lower)
  float *Zb = Am + C * CP;    // [C][CP]  Z, built row by row
  float *gam = Zb + C * CP;   // [C]
  float *bet = gam + C;       // [C]
  float *kin = bet + C, *qin = kin + C;  // [C] each: 1/|k|, 1/|q|
#if defined(__CUDA_ARCH__)
  constexpr bool RAW = LD::kRawTf32;  // k and q kept raw, their norms in kin / qin
#else
  constexpr bool RAW = false;
#endif
  float *out = p.prep + ((size_t)slot * p.Hv + h) * kPrep;
  float *KGo = out + C * C, *QGo = out + 2 * C * C;
  load_keys<K, KP>(x, p, ld, Ks, Qs, t0, n, h / (p.Hv / p.Hqk));
  load_gates(x, p, gam, bet, t0, n, h);
  x.sync();
  if constexpr (RAW) {  // the inverse norms, the rows left raw
    x.par(2 * C, [&](int r) {
      const float *row = r < C ? Ks + r * KP : Qs + (r - C) * KP;
      float ss = 0.f;
      for (int c = 0; c < K; ++c) ss = fmaf(row[c], row[c], ss);
      (r < C ? kin : qin)[r % C] = p.l2norm ? 1.f / sqrtf(ss + kEps) : 1.f;
    });
    if (x.leader())
      for (int i = 1; i < C; ++i) gam[i] += gam[i - 1];
  } else {
    norm_and_cumsum<K, KP>(x, p, Ks, Qs, gam, kin);  // qin follows kin
  }
  x.sync();
  // K K^T and Q K^T (on the device tensor-core products, on the host 4 x 4 tiles of (i, j) a
  // thread).  Gamma, KG, QG and A = diag(beta) KG follow in the tile's epilogue, which also
  // writes the zeros above the diagonal.
#if defined(__CUDA_ARCH__)
  {
    const int lane = x.tid & 31;
    const tc::Tiles<C, C> tl(x.tid >> 5);
    constexpr int NTW = tc::Tiles<C, C>::NTW;
    if (tl.any) {
      float kk[NTW][4] = {}, qk[NTW][4] = {};
      if (tl.n0 <= tl.m0 + 15) {  // tiles wholly above the diagonal hold zeros
        tc::mma_nt<NTW, false, RAW, RAW>(lane, Ks, KP, nullptr, Ks, KP, tl.m0, tl.n0, 0, K, kk);
        tc::mma_nt<NTW, false, RAW, RAW>(lane, Qs, KP, nullptr, Ks, KP, tl.m0, tl.n0, 0, K, qk);
      }
#pragma unroll
      for (int jt = 0; jt < NTW; ++jt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = tc::frag_row(lane, tl.m0, e), j = tc::frag_col(lane, tl.n0, jt, e);
          const float gij = j <= i ? expf(gam[i] - gam[j]) : 0.f;
          const float kkv = RAW ? kk[jt][e] * kin[i] * kin[j] : kk[jt][e];
          const float qkv = RAW ? qk[jt][e] * qin[i] * kin[j] : qk[jt][e];
          const float kg = j < i ? kkv * gij : 0.f;
          Am[i * CP + j] = bet[i] * kg;
          KGo[i * C + j] = kg;
          QGo[i * C + j] = j <= i ? qkv * gij : 0.f;
        }
    }
  }
#else
  x.par((C / 4) * (C / 4), [&](int t) {
    const int i0 = (t / (C / 4)) * 4, j0 = (t % (C / 4)) * 4;
    float kk[4][4] = {}, qk[4][4] = {};
    if (j0 <= i0 + 3) {  // tiles wholly above the diagonal hold zeros
#pragma unroll 4
      for (int c = 0; c < K; ++c) {
        float ki[4], kj[4], qi[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          ki[r] = Ks[(i0 + r) * KP + c];
          kj[r] = Ks[(j0 + r) * KP + c];
          qi[r] = Qs[(i0 + r) * KP + c];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            kk[a][b] = fmaf(ki[a], kj[b], kk[a][b]);
            qk[a][b] = fmaf(qi[a], kj[b], qk[a][b]);
          }
      }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int i = i0 + a, j = j0 + b;
        const float gij = j <= i ? expf(gam[i] - gam[j]) : 0.f;
        const float kg = j < i ? kk[a][b] * gij : 0.f;
        Am[i * CP + j] = bet[i] * kg;
        KGo[i * C + j] = kg;
        QGo[i * C + j] = j <= i ? qk[a][b] * gij : 0.f;
      }
  });
#endif
#if defined(__CUDA_ARCH__)
  x.sync();  // A is complete
  if (x.tid < 128) invert_unit_lower_rt(Am, CP, Zb, CP, x.tid);
  x.sync();
#else
  x.par(C * C, [&](int idx) {
    const int i = idx / C, j = idx % C;
    Zb[i * CP + j] = i == j ? 1.f : 0.f;
  });
  x.sync();
  // Z = (I + A)^-1 by a row sweep: once row m of Z is final (every row above it applied),
  // each row i below it takes -A_im Z_m.  One barrier a step, a few FMAs a thread.
  for (int m = 0; m < C - 1; ++m) {
    const int cols = m + 1;  // row m of Z is zero right of its diagonal
    x.par((C - 1 - m) * cols, [&](int idx) {
      const int i = m + 1 + idx / cols, j = idx % cols;
      Zb[i * CP + j] = fmaf(-Am[i * CP + m], Zb[m * CP + j], Zb[i * CP + j]);
    });
    x.sync();
  }
#endif
  x.par(C * C, [&](int idx) { out[idx] = Zb[(idx / C) * CP + idx % C]; });
  // gamma, b, d and the inverse norms, for the walk and grad
  x.par(C, [&](int i) {
    float *vo = out + kPrepVec;
    vo[i] = gam[i];
    vo[C + i] = expf(gam[i]);
    vo[2 * C + i] = expf(gam[C - 1] - gam[i]);
    vo[3 * C + i] = kin[i];
    vo[4 * C + i] = qin[i];
  });
}

#if defined(__CUDA_ARCH__)
// Adds the warp's NTW tiles of a C x C product at (m0, n0) into a row-major C x C fp32 sum
// (16-byte aligned), its lower triangle with the diagonal only, as 16-byte vector atomics
// (a quarter of the scalar ones): the elements above the diagonal in a quad add zero.
template <int NTW>
__device__ __forceinline__ void add_lower_quads(int lane, const float (&d)[NTW][4], float *sum, int m0, int n0) {
#pragma unroll
  for (int j = 0; j < NTW; ++j) {
    int r, cb;
    float4 v;
    tc::frag_quad(lane, d[j], r, cb, v);
    const int i = m0 + r, c = n0 + 8 * j + cb;
    if (c > i) continue;  // the quad lies wholly above the diagonal
    v.y = c + 1 <= i ? v.y : 0.f;
    v.z = c + 2 <= i ? v.z : 0.f;
    v.w = c + 3 <= i ? v.w : 0.f;
    atomicAdd(reinterpret_cast<float4 *>(sum + i * C + c), v);
  }
}
// Adds the warp's NTW tiles of a C x K product at (m0, n0) into rows of a global fp32 array
// (row i at base + i * stride, 16-byte aligned), rows i < n only, as 16-byte vector atomics.
template <int NTW>
__device__ __forceinline__ void add_row_quads(int lane, const float (&d)[NTW][4], float *base, size_t stride, int n,
                                              int m0, int n0) {
#pragma unroll
  for (int j = 0; j < NTW; ++j) {
    int r, cb;
    float4 v;
    tc::frag_quad(lane, d[j], r, cb, v);
    const int i = m0 + r;
    if (i < n) atomicAdd(reinterpret_cast<float4 *>(base + (size_t)i * stride + n0 + 8 * j + cb), v);
  }
}
#endif

// ---- walk: the state-dependent steps of BV state rows of one v-head, chunk by chunk
template <int KD, int BV, class X, class LD>
GDN_BWD_FN void walk_block(X &x, const Params &p, LD ld, float *sm, int tile, int h, int s) {
  // rows padded by 4 floats: the tensor-core fragments' loads (lane 4 g + t reads row g,
  // column t) then fall in distinct banks
  constexpr int K = KD, KP = KD + 4, VP = BV + 4;
  const int V = p.V, Hv = p.Hv;
  float *Ks = sm;              // [C][KP]  k of the chunk (unit-norm when l2norm)
  float *Qs = Ks + C * KP;     // [C][KP]  q
  float *Ss = Qs + C * KP;     // [BV][KP] this block's rows of the chunk-start state
  float *dSs = Ss + BV * KP;   // [BV][KP] their gradient, carried from the chunk's end
  float *Vs = dSs + BV * KP;   // [C][VP]  v columns of the block's rows (forward sweep)
  float *Os = Vs + C * VP;     // [C][VP]  scale * dO
  float *Us = Os + C * VP;     // [C][VP]  U'
  float *KdS = Us + C * VP;    // [C][VP]  K dS1^T
  float *dUs = KdS + C * VP;   // [C][VP]  dU'
  float *Ws = dUs + C * VP;    // [C][VP]  V - diag(b) K S^T, then dV
  float *KSs = Ws + C * VP;    // [C][VP]  K S^T
  float *QSs = KSs + C * VP;   // [C][VP]  Q S^T
  float *Zm = QSs + C * VP;    // [C][CP]  Z (from prep)
  float *QGm = Zm + C * CP;    // [C][CP]  QG (from prep)
  float *gam = QGm + C * CP;   // [C] gamma
  float *bet = gam + C;        // [C] beta
  float *bex = bet + C;        // [C] exp(gamma)
  float *dec = bex + C;        // [C] exp(gamma_last - gamma)
  float *prt = dec + C;        // [C] partial sums of <S, dS1>
  float *one = prt + C;        // [C] ones (a unit scale for the tensor-core products)
  // with raw keys (below): 1/|k|, 1/|q| and the row scales that carry them
  float *kin = one + C, *qin = kin + C, *dkn = qin + C, *bkn = dkn + C, *bqn = bkn + C;
#if defined(__CUDA_ARCH__)
  // bf16 inputs widened to fp32 are exact in TF32: the device keeps k and q raw and folds
  // their norms into the tensor-core products' scales, which then need no split of k or q
  constexpr bool RAW = LD::kRawTf32;
#else
  constexpr bool RAW = false;
#endif

  const int qh = h / (Hv / p.Hqk), row0 = tile * BV;
  int64_t start, end;
  if (!seq_bounds(p, s, start, end)) {
    x.fail(p.status);
    return;
  }
  const int64_t slot0 = (int64_t)s + start / C;
  const int n_chunks = (int)((end - start + C - 1) / C);
  const size_t VK = (size_t)V * K, CV = (size_t)C * V;
  // the forward sweep's U', V - diag(b) K S^T and K S^T of the block's columns, [C][V] each
  auto fw_of = [&](int64_t slot) { return p.fw + ((size_t)slot * Hv + h) * 3 * CV + row0; };

  // the chunk's inputs: k (and q), the block's v columns (forward) or scale * dO (backward),
  // the gates, Z (and QG) from prep, and in the backward sweep the block's chunk-start
  // state and the forward sweep's tiles; then the norm, gamma, b and d (with raw keys b, d and
  // the inverse norms come from prep).  Everything but the raw-key scales is ready on return.  With vector loads every fill of a phase is in flight at once (two phases
  // backward, one forward).
  auto load = [&](int64_t slot, int64_t t0, int n, bool bwd) {
    const float *pr = p.prep + ((size_t)slot * Hv + h) * kPrep;
    const float *st = p.states + ((size_t)slot * Hv + h) * VK + (size_t)row0 * K;
    const float *fw = fw_of(slot);
    const int64_t kb = t0 * p.ks + (int64_t)qh * K, qb = t0 * p.qs + (int64_t)qh * K;
    constexpr int NI = 256;
    if (p.vec8 && bwd) {
      x.par(NI, [&](int t) {
        Fill4<BV, K, NI> fs;
        Fill4<C, BV, NI> fu, fwv, fks, fo;
        Fill4<C, C, NI> fz, fq;
        fs.load(t, st, K, BV);
        fu.load(t, fw, V, C);
        fwv.load(t, fw + CV, V, C);
        fks.load(t, fw + 2 * CV, V, C);
        fo.load(t, p.dout + (t0 * Hv + h) * V + row0, (size_t)Hv * V, n);
        fz.load(t, pr, C, C);
        fq.load(t, pr + 2 * C * C, C, C);
        fs.store(t, Ss, KP);
        fu.store(t, Us, VP);
        fwv.store(t, Ws, VP);
        fks.store(t, KSs, VP);
        fo.store(t, Os, VP, p.scale);
        fz.store(t, Zm, CP);
        fq.store(t, QGm, CP);
      });
      x.par(NI, [&](int t) {
        Fill8<C, K, NI> fk, fq;
        fk.load(ld, t, p.k, kb, p.ks, n);
        fq.load(ld, t, p.q, qb, p.qs, n);
        const bool gi = t < C && t < n;
        const float gv = gi ? p.g[(t0 + t) * Hv + h] : 0.f, bv = gi ? p.beta[(t0 + t) * Hv + h] : 0.f;
        float pv[4] = {};  // with raw keys: b, d, 1/|k|, 1/|q| from prep
        if (RAW && t < C)
#pragma unroll
          for (int u = 0; u < 4; ++u) pv[u] = pr[kPrepVec + (u + 1) * C + t];
        fk.store(t, Ks, KP);
        fq.store(t, Qs, KP);
        if (t < C) {
          gam[t] = gv;
          bet[t] = bv;
          if (RAW) {
            bex[t] = pv[0];
            dec[t] = pv[1];
            kin[t] = pv[2];
            qin[t] = pv[3];
          }
        }
      });
    } else if (p.vec8) {
      x.par(NI, [&](int t) {
        Fill8<C, K, NI> fk;
        Fill8<C, BV, NI> fv;
        Fill4<C, C, NI> fz;
        fk.load(ld, t, p.k, kb, p.ks, n);
        fv.load(ld, t, p.v, t0 * p.vs + (int64_t)h * V + row0, p.vs, n);
        fz.load(t, pr, C, C);
        const bool gi = t < C && t < n;
        const float gv = gi ? p.g[(t0 + t) * Hv + h] : 0.f, bv = gi ? p.beta[(t0 + t) * Hv + h] : 0.f;
        float pv[3] = {};  // with raw keys: b, d, 1/|k| from prep
        if (RAW && t < C)
#pragma unroll
          for (int u = 0; u < 3; ++u) pv[u] = pr[kPrepVec + (u + 1) * C + t];
        fk.store(t, Ks, KP);
        fv.store(t, Vs, VP);
        fz.store(t, Zm, CP);
        if (t < C) {
          gam[t] = gv;
          bet[t] = bv;
          if (RAW) {
            bex[t] = pv[0];
            dec[t] = pv[1];
            kin[t] = pv[2];
          }
        }
      });
    } else {
      load_keys<K, KP>(x, p, ld, Ks, bwd ? Qs : nullptr, t0, n, qh);
      x.par(C * BV, [&](int idx) {
        const int r = idx / BV, j = idx % BV;
        const bool in = r < n;
        if (bwd) Os[r * VP + j] = in ? p.scale * p.dout[((t0 + r) * Hv + h) * V + row0 + j] : 0.f;
        else Vs[r * VP + j] = in ? ld(p.v, (t0 + r) * p.vs + (int64_t)h * V + row0 + j) : 0.f;
      });
      load_gates(x, p, gam, bet, t0, n, h);
      if (RAW)
        x.par(C, [&](int i) {
          bex[i] = pr[kPrepVec + C + i];
          dec[i] = pr[kPrepVec + 2 * C + i];
          kin[i] = pr[kPrepVec + 3 * C + i];
          qin[i] = pr[kPrepVec + 4 * C + i];
        });
      copy_block<C, C>(x, pr, C, Zm, CP);
      if (bwd) {
        copy_block<C, C>(x, pr + 2 * C * C, C, QGm, CP);
        copy_block<BV, K>(x, st, K, Ss, KP);
        copy_block<C, BV>(x, fw, V, Us, VP);
        copy_block<C, BV>(x, fw + CV, V, Ws, VP);
        copy_block<C, BV>(x, fw + 2 * CV, V, KSs, VP);
      }
    }
    x.sync();
    if constexpr (RAW) {
      // b, d and the inverse norms came with the fill (prep computed them once per chunk and
      // head); the scales that carry the norms into the state updates are read two phases on,
      // past the next barrier
      x.par(C, [&](int i) {
        dkn[i] = dec[i] * kin[i];
        bkn[i] = bex[i] * kin[i];
        if (bwd) bqn[i] = bex[i] * qin[i];
      });
    } else {
      norm_and_cumsum<K, KP>(x, p, Ks, bwd ? Qs : nullptr, gam);
      x.sync();
      x.par(C, [&](int i) {
        bex[i] = expf(gam[i]);
        dec[i] = expf(gam[C - 1] - gam[i]);
      });
      x.sync();
    }
  };

  // ---- forward sweep: the chunk-start state of every chunk, for this block's rows
  x.par(BV * K, [&](int idx) {
    const int r = idx / K, c = idx % K;
    Ss[r * KP + c] = p.h0 ? p.h0[((size_t)s * Hv + h) * VK + (size_t)(row0 + r) * K + c] : 0.f;
  });
  x.par(C, [&](int i) { one[i] = 1.f; });
  x.sync();
  for (int ci = 0; ci < n_chunks; ++ci) {
    const int64_t t0 = start + (int64_t)ci * C, slot = slot0 + ci;
    const int n = (int)(end - t0 < C ? end - t0 : C);
    float *dst = p.states + ((size_t)slot * Hv + h) * VK + (size_t)row0 * K;
    x.par(BV * K, [&](int idx) { dst[(idx / K) * (size_t)K + idx % K] = Ss[(idx / K) * KP + idx % K]; });
    load(slot, t0, n, false);
    float *fw = fw_of(slot);
    // K S^T; the epilogue forms V - diag(b) K S^T, and both go to the backward sweep (on the
    // device a tensor-core product, on the host 4 x 2 tiles of (i, v) a thread)
#if defined(__CUDA_ARCH__)
    {
      const int lane = x.tid & 31;
      // the tile's (i, v) and its K S^T value: the forms of the raw and the unit-norm keys
      auto epi = [&](int i, int v, float ks) {
        const float w = Vs[i * VP + v] - bex[i] * ks;
        Ws[i * VP + v] = w;
        fw[CV + (size_t)i * V + v] = w;
        fw[2 * CV + (size_t)i * V + v] = ks;
      };
      if constexpr (RAW) {  // raw k exact: a warp takes one column tile, S's fragments split once
        const tc::TilesM<C, BV> tl(x.tid >> 5);
        constexpr int MTW = tc::TilesM<C, BV>::MTW;
        if (tl.any) {
          float d[MTW][4] = {};
          tc::mma_nt_m<MTW>(lane, Ks, KP, Ss, KP, tl.m0, tl.n0, 0, K, d);
#pragma unroll
          for (int r = 0; r < MTW; ++r)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i = tc::frag_row(lane, tl.m0 + 16 * r, e), v = tc::frag_col(lane, tl.n0, 0, e);
              epi(i, v, d[r][e] * kin[i]);
            }
        }
      } else {
        const tc::Tiles<C, BV> tl(x.tid >> 5);
        constexpr int NTW = tc::Tiles<C, BV>::NTW;
        if (tl.any) {
          float d[NTW][4] = {};
          tc::mma_nt<NTW>(lane, Ks, KP, nullptr, Ss, KP, tl.m0, tl.n0, 0, K, d);
#pragma unroll
          for (int j = 0; j < NTW; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              epi(tc::frag_row(lane, tl.m0, e), tc::frag_col(lane, tl.n0, j, e), d[j][e]);
        }
      }
    }
#else
    x.par((C / 4) * (BV / 2), [&](int t) {
      const int i0 = (t / (BV / 2)) * 4, v0 = (t % (BV / 2)) * 2;
      float ks[4][2] = {};
#pragma unroll 4
      for (int c = 0; c < K; ++c) {
        const float s0 = Ss[v0 * KP + c], s1 = Ss[(v0 + 1) * KP + c];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const float kv = Ks[(i0 + a) * KP + c];
          ks[a][0] = fmaf(kv, s0, ks[a][0]);
          ks[a][1] = fmaf(kv, s1, ks[a][1]);
        }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const int i = i0 + a, v = v0 + b;
          const float w = Vs[i * VP + v] - bex[i] * ks[a][b];
          Ws[i * VP + v] = w;
          fw[CV + (size_t)i * V + v] = w;
          fw[2 * CV + (size_t)i * V + v] = ks[a][b];
        }
    });
#endif
    x.sync();
    // U' = Z diag(beta) (V - diag(b) K S^T) (on the device a tensor-core product, on the host
    // 2 x 2 tiles of (i, v) a thread)
#if defined(__CUDA_ARCH__)
    {  // Z is zero right of its diagonal: rows i < m0 + 16 take j < m0 + 16
      const int lane = x.tid & 31;
      const tc::Tiles<C, BV> tl(x.tid >> 5);
      constexpr int NTW = tc::Tiles<C, BV>::NTW;
      if (tl.any) {
        float d[NTW][4] = {};
        tc::mma_nn<NTW>(lane, Zm, CP, one, 1.f, Ws, VP, bet, tl.m0, tl.n0, 0, tl.m0 + 16, d);
#pragma unroll
        for (int j = 0; j < NTW; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = tc::frag_row(lane, tl.m0, e), c = tc::frag_col(lane, tl.n0, j, e);
            Us[i * VP + c] = d[j][e];
            fw[(size_t)i * V + c] = d[j][e];
          }
      }
    }
#else
    x.par((C / 2) * (BV / 2), [&](int t) {
      const int i0 = (t / (BV / 2)) * 2, v0 = (t % (BV / 2)) * 2;
      float acc[2][2] = {};
      for (int j = 0; j <= i0 + 1; ++j) {  // Z is zero right of its diagonal
        const float z0 = Zm[i0 * CP + j] * bet[j], z1 = Zm[(i0 + 1) * CP + j] * bet[j];
        const float w0 = Ws[j * VP + v0], w1 = Ws[j * VP + v0 + 1];
        acc[0][0] = fmaf(z0, w0, acc[0][0]);
        acc[0][1] = fmaf(z0, w1, acc[0][1]);
        acc[1][0] = fmaf(z1, w0, acc[1][0]);
        acc[1][1] = fmaf(z1, w1, acc[1][1]);
      }
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          Us[(i0 + a) * VP + v0 + b] = acc[a][b];
          fw[(size_t)(i0 + a) * V + v0 + b] = acc[a][b];
        }
    });
#endif
    x.sync();
    // S1 = b_last S + U'^T diag(d) K (on the device a tensor-core product, on the host 4 x 4
    // tiles of (v, c) a thread, columns c0 + b K / 4)
#if defined(__CUDA_ARCH__)
    {
      const int lane = x.tid & 31;
      const tc::Tiles<BV, K> tl(x.tid >> 5);
      constexpr int NTW = tc::Tiles<BV, K>::NTW;
      if (tl.any) {
        float d[NTW][4];
#pragma unroll
        for (int j = 0; j < NTW; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            d[j][e] = bex[C - 1] * Ss[tc::frag_row(lane, tl.m0, e) * KP + tc::frag_col(lane, tl.n0, j, e)];
        tc::mma_tn<NTW, RAW>(lane, Us, VP, RAW ? dkn : dec, 1.f, Ks, KP, tl.m0, tl.n0, 0, C, d);
#pragma unroll
        for (int j = 0; j < NTW; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            Ss[tc::frag_row(lane, tl.m0, e) * KP + tc::frag_col(lane, tl.n0, j, e)] = d[j][e];
      }
    }
#else
    x.par((BV / 4) * (K / 4), [&](int t) {
      const int v0 = (t / (K / 4)) * 4, c0 = t % (K / 4);
      float acc[4][4] = {};
      for (int j = 0; j < C; ++j) {
        const float dj = dec[j];
        float u[4], kv[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) u[a] = Us[j * VP + v0 + a] * dj;
#pragma unroll
        for (int b = 0; b < 4; ++b) kv[b] = Ks[j * KP + c0 + b * (K / 4)];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(u[a], kv[b], acc[a][b]);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          float *sp = Ss + (v0 + a) * KP + c0 + b * (K / 4);
          *sp = fmaf(bex[C - 1], *sp, acc[a][b]);
        }
    });
#endif
    x.sync();
  }

  // ---- backward sweep
  x.par(BV * K, [&](int idx) {
    const int r = idx / K, c = idx % K;
    dSs[r * KP + c] = p.dhT ? p.dhT[((size_t)s * Hv + h) * VK + (size_t)(row0 + r) * K + c] : 0.f;
  });
  for (int ci = n_chunks - 1; ci >= 0; --ci) {
    const int64_t t0 = start + (int64_t)ci * C, slot = slot0 + ci;
    const int n = (int)(end - t0 < C ? end - t0 : C);
    float *sums = p.sums + ((size_t)slot * Hv + h) * kSums;
    float *dPsum = sums, *dTsum = sums + C * C, *ddsum = sums + 2 * C * C, *dbsum = ddsum + C;
    load(slot, t0, n, true);
    // Q S^T and K dS1^T (on the device tensor-core products, on the host 4 x 2 tiles of
    // (i, v) a thread)
#if defined(__CUDA_ARCH__)
    if constexpr (RAW) {  // raw q, k exact: a warp takes one column tile, its S fragments split once
      const int lane = x.tid & 31;
      const tc::TilesM<C, BV> tl(x.tid >> 5);
      constexpr int MTW = tc::TilesM<C, BV>::MTW;
      if (tl.any) {
        float dq[MTW][4] = {}, dk[MTW][4] = {};
        tc::mma_nt_m<MTW>(lane, Qs, KP, Ss, KP, tl.m0, tl.n0, 0, K, dq);
        tc::mma_nt_m<MTW>(lane, Ks, KP, dSs, KP, tl.m0, tl.n0, 0, K, dk);
#pragma unroll
        for (int r = 0; r < MTW; ++r)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = tc::frag_row(lane, tl.m0 + 16 * r, e), v = tc::frag_col(lane, tl.n0, 0, e);
            QSs[i * VP + v] = dq[r][e] * qin[i];
            KdS[i * VP + v] = dk[r][e] * kin[i];
          }
      }
    } else {
      const int lane = x.tid & 31;
      const tc::Tiles<C, BV> tl(x.tid >> 5);
      constexpr int NTW = tc::Tiles<C, BV>::NTW;
      if (tl.any) {
        float dq[NTW][4] = {}, dk[NTW][4] = {};
        tc::mma_nt<NTW>(lane, Qs, KP, nullptr, Ss, KP, tl.m0, tl.n0, 0, K, dq);
        tc::mma_nt<NTW>(lane, Ks, KP, nullptr, dSs, KP, tl.m0, tl.n0, 0, K, dk);
#pragma unroll
        for (int j = 0; j < NTW; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = tc::frag_row(lane, tl.m0, e), v = tc::frag_col(lane, tl.n0, j, e);
            QSs[i * VP + v] = dq[j][e];
            KdS[i * VP + v] = dk[j][e];
          }
      }
    }
#else
    x.par((C / 4) * (BV / 2), [&](int t) {
      const int i0 = (t / (BV / 2)) * 4, v0 = (t % (BV / 2)) * 2;
      float qs[4][2] = {}, kd[4][2] = {};
#pragma unroll 2
      for (int c = 0; c < K; ++c) {
        const float s0 = Ss[v0 * KP + c], s1 = Ss[(v0 + 1) * KP + c];
        const float d0 = dSs[v0 * KP + c], d1 = dSs[(v0 + 1) * KP + c];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          const float qv = Qs[(i0 + a) * KP + c], kv = Ks[(i0 + a) * KP + c];
          qs[a][0] = fmaf(qv, s0, qs[a][0]);
          qs[a][1] = fmaf(qv, s1, qs[a][1]);
          kd[a][0] = fmaf(kv, d0, kd[a][0]);
          kd[a][1] = fmaf(kv, d1, kd[a][1]);
        }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          QSs[(i0 + a) * VP + v0 + b] = qs[a][b];
          KdS[(i0 + a) * VP + v0 + b] = kd[a][b];
        }
    });
#endif
    x.sync();
    // this block's share of dP = Ot U'^T (lower incl. the diagonal; 4 x 4 tiles of (i, j):
    // rows i0 .. i0 + 3, columns tj + 16 b) and of dd_i = U'_i . (K dS1^T)_i;
    // dU' = diag(d) K dS1^T + QG^T Ot (2 x 2 tiles of (i, v); row i0 + 1's term at j = i0 has
    // a zero factor, QG being lower)
#if defined(__CUDA_ARCH__)
    {  // tiles wholly above the diagonal skipped
      const int lane = x.tid & 31;
      const tc::Tiles<C, C> tl(x.tid >> 5);
      constexpr int NTW = tc::Tiles<C, C>::NTW;
      if (tl.any && tl.n0 <= tl.m0 + 15) {
        float d[NTW][4] = {};
        tc::mma_nt<NTW>(lane, Os, VP, nullptr, Us, VP, tl.m0, tl.n0, 0, BV, d);
        add_lower_quads<NTW>(lane, d, dPsum, tl.m0, tl.n0);
      }
    }
#else
    x.par((C / 4) * 16, [&](int t) {
      const int i0 = (t / 16) * 4, tj = t % 16;
      if (tj > i0 + 3) return;
      float acc[4][4] = {};
      for (int v = 0; v < BV; ++v) {
        float o[4], u[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          o[a] = Os[(i0 + a) * VP + v];
          u[a] = Us[(tj + 16 * a) * VP + v];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(o[a], u[b], acc[a][b]);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int i = i0 + a, j = tj + 16 * b;
          if (j <= i) x.add(dPsum + i * C + j, acc[a][b]);
        }
    });
#endif
    x.par(C, [&](int i) {
      float acc = 0.f;
      for (int v = 0; v < BV; ++v) acc = fmaf(Us[i * VP + v], KdS[i * VP + v], acc);
      x.add(ddsum + i, acc);
    });
#if defined(__CUDA_ARCH__)
    {  // QG[j][i] is zero for j < i: rows i >= m0 take j >= m0
      const int lane = x.tid & 31;
      const tc::Tiles<C, BV> tl(x.tid >> 5);
      constexpr int NTW = tc::Tiles<C, BV>::NTW;
      if (tl.any) {
        float d[NTW][4];
#pragma unroll
        for (int j = 0; j < NTW; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = tc::frag_row(lane, tl.m0, e), c = tc::frag_col(lane, tl.n0, j, e);
            d[j][e] = dec[i] * KdS[i * VP + c];
          }
        tc::mma_tn<NTW, false, false>(lane, QGm, CP, nullptr, 1.f, Os, VP, tl.m0, tl.n0, tl.m0, C, d);
#pragma unroll
        for (int j = 0; j < NTW; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = tc::frag_row(lane, tl.m0, e), c = tc::frag_col(lane, tl.n0, j, e);
            dUs[i * VP + c] = d[j][e];
          }
      }
    }
#else
    x.par((C / 2) * (BV / 2), [&](int t) {
      const int i0 = (t / (BV / 2)) * 2, v0 = (t % (BV / 2)) * 2;
      float acc[2][2];
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b) acc[a][b] = dec[i0 + a] * KdS[(i0 + a) * VP + v0 + b];
      for (int j = i0; j < C; ++j) {
        const float m0 = QGm[j * CP + i0], m1 = QGm[j * CP + i0 + 1];
        const float o0 = Os[j * VP + v0], o1 = Os[j * VP + v0 + 1];
        acc[0][0] = fmaf(m0, o0, acc[0][0]);
        acc[0][1] = fmaf(m0, o1, acc[0][1]);
        acc[1][0] = fmaf(m1, o0, acc[1][0]);
        acc[1][1] = fmaf(m1, o1, acc[1][1]);
      }
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b) dUs[(i0 + a) * VP + v0 + b] = acc[a][b];
    });
#endif
    x.sync();
    // this block's share of dT = dU' (V - diag(b) K S^T)^T (lower; 4 x 4 tiles, columns
    // tj + 16 b); dV = diag(beta) Z^T dU' (complete for these rows; 2 x 2 tiles, Z being
    // lower), written over V - diag(b) K S^T once dT has read it (after the barrier below)
#if defined(__CUDA_ARCH__)
    {  // tiles wholly above the diagonal skipped
      const int lane = x.tid & 31;
      const tc::Tiles<C, C> tl(x.tid >> 5);
      constexpr int NTW = tc::Tiles<C, C>::NTW;
      if (tl.any && tl.n0 <= tl.m0 + 15) {
        float d[NTW][4] = {};
        tc::mma_nt<NTW>(lane, dUs, VP, nullptr, Ws, VP, tl.m0, tl.n0, 0, BV, d);
        add_lower_quads<NTW>(lane, d, dTsum, tl.m0, tl.n0);
      }
    }
#else
    x.par((C / 4) * 16, [&](int t) {
      const int i0 = (t / 16) * 4, tj = t % 16;
      if (tj > i0 + 3) return;
      float acc[4][4] = {};
      for (int v = 0; v < BV; ++v) {
        float du[4], w[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          du[a] = dUs[(i0 + a) * VP + v];
          w[a] = Ws[(tj + 16 * a) * VP + v];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(du[a], w[b], acc[a][b]);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int i = i0 + a, j = tj + 16 * b;
          if (j <= i) x.add(dTsum + i * C + j, acc[a][b]);
        }
    });
#endif
    // b_last's gradient takes <S, dS1> over the block's rows: 64 partial sums
    x.par(C, [&](int r) {
      float acc = 0.f;
      for (int idx = r; idx < BV * K; idx += C)
        acc = fmaf(Ss[(idx / K) * KP + idx % K], dSs[(idx / K) * KP + idx % K], acc);
      prt[r] = acc;
    });
    x.sync();
#if defined(__CUDA_ARCH__)
    {  // Z[j][i] is zero for j < i: rows i >= m0 take j >= m0
      const int lane = x.tid & 31;
      const tc::Tiles<C, BV> tl(x.tid >> 5);
      constexpr int NTW = tc::Tiles<C, BV>::NTW;
      if (tl.any) {
        float d[NTW][4] = {};
        tc::mma_tn<NTW, false, false>(lane, Zm, CP, nullptr, 1.f, dUs, VP, tl.m0, tl.n0, tl.m0, C, d);
#pragma unroll
        for (int j = 0; j < NTW; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = tc::frag_row(lane, tl.m0, e), c = tc::frag_col(lane, tl.n0, j, e);
            const float r = d[j][e] * bet[i];
            Ws[i * VP + c] = r;
            if (i < n) p.dv[((t0 + i) * Hv + h) * V + row0 + c] = r;
          }
      }
    }
#else
    x.par((C / 2) * (BV / 2), [&](int t) {
      const int i0 = (t / (BV / 2)) * 2, v0 = (t % (BV / 2)) * 2;
      float acc[2][2] = {};
      for (int j = i0; j < C; ++j) {
        const float z0 = Zm[j * CP + i0], z1 = Zm[j * CP + i0 + 1];
        const float d0 = dUs[j * VP + v0], d1 = dUs[j * VP + v0 + 1];
        acc[0][0] = fmaf(z0, d0, acc[0][0]);
        acc[0][1] = fmaf(z0, d1, acc[0][1]);
        acc[1][0] = fmaf(z1, d0, acc[1][0]);
        acc[1][1] = fmaf(z1, d1, acc[1][1]);
      }
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        const int i = i0 + a;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const float r = acc[a][b] * bet[i];
          Ws[i * VP + v0 + b] = r;
          if (i < n) p.dv[((t0 + i) * Hv + h) * V + row0 + v0 + b] = r;
        }
      }
    });
#endif
    x.sync();
    // this block's share of db_j = Ot_j . (Q S^T)_j - dV_j . (K S^T)_j (+ <S, dS1> at the
    // chunk's last row); the S and dS1 parts of dq and dk, dq = diag(b) Ot S,
    // dk = diag(d) U' dS1 - diag(b) dV S (on the device tensor-core products, on the host
    // 4 x 8 tiles of (i, c) a thread, columns c0 + b K / 8)
    x.par(C, [&](int j) {
      float b = 0.f;
      for (int v = 0; v < BV; ++v) b += Os[j * VP + v] * QSs[j * VP + v] - Ws[j * VP + v] * KSs[j * VP + v];
      if (j == C - 1)
        for (int r = 0; r < C; ++r) b += prt[r];
      x.add(dbsum + j, b);
    });
#if defined(__CUDA_ARCH__)
    {
      const int lane = x.tid & 31;
      const tc::Tiles<C, K> tl(x.tid >> 5);
      constexpr int NTW = tc::Tiles<C, K>::NTW;
      if (tl.any) {
        float d[NTW][4] = {};
        float dq[NTW][4] = {};
        tc::mma_nn<NTW, false, false>(lane, Us, VP, dec, 1.f, dSs, KP, nullptr, tl.m0, tl.n0, 0, BV, d);  // diag(d) U' dS1
        // diag(b) Ot S into dq and - diag(b) dV S into dk, S's fragments split once for both
        tc::mma_nn_pair<NTW>(lane, Os, Ws, VP, bex, bex, -1.f, Ss, KP, tl.m0, tl.n0, 0, BV, dq, d);
        add_row_quads<NTW>(lane, dq, p.dqn + ((size_t)t0 * p.Hqk + qh) * K, (size_t)p.Hqk * K, n, tl.m0, tl.n0);
        add_row_quads<NTW>(lane, d, p.dkn + ((size_t)t0 * p.Hqk + qh) * K, (size_t)p.Hqk * K, n, tl.m0, tl.n0);
      }
    }
#else
    x.par((C / 4) * (K / 8), [&](int t) {
      const int i0 = (t / (K / 8)) * 4, c0 = t % (K / 8);
      float sq[4][8] = {}, sk[4][8] = {}, sv[4][8] = {};
      for (int v = 0; v < BV; ++v) {
        float o[4], u[4], w[4], sr[8], dr[8];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          o[a] = Os[(i0 + a) * VP + v];
          u[a] = Us[(i0 + a) * VP + v];
          w[a] = Ws[(i0 + a) * VP + v];
        }
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          sr[b] = Ss[v * KP + c0 + b * (K / 8)];
          dr[b] = dSs[v * KP + c0 + b * (K / 8)];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            sq[a][b] = fmaf(o[a], sr[b], sq[a][b]);
            sk[a][b] = fmaf(u[a], dr[b], sk[a][b]);
            sv[a][b] = fmaf(w[a], sr[b], sv[a][b]);
          }
      }
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        const int i = i0 + a;
        if (i >= n) continue;
        const size_t off = ((size_t)(t0 + i) * p.Hqk + qh) * K + c0;
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          x.add(p.dqn + off + b * (K / 8), bex[i] * sq[a][b]);
          x.add(p.dkn + off + b * (K / 8), dec[i] * sk[a][b] - bex[i] * sv[a][b]);
        }
      }
    });
#endif
    x.sync();
    // dS = b_last dS1 + Ot^T diag(b) Q - (diag(b) dV)^T K (on the device tensor-core products,
    // on the host 4 x 4 tiles of (v, c) a thread, columns c0 + b K / 4)
#if defined(__CUDA_ARCH__)
    {
      const int lane = x.tid & 31;
      const tc::Tiles<BV, K> tl(x.tid >> 5);
      constexpr int NTW = tc::Tiles<BV, K>::NTW;
      if (tl.any) {
        float d[NTW][4];
#pragma unroll
        for (int j = 0; j < NTW; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            d[j][e] = bex[C - 1] * dSs[tc::frag_row(lane, tl.m0, e) * KP + tc::frag_col(lane, tl.n0, j, e)];
        tc::mma_tn<NTW, RAW>(lane, Os, VP, RAW ? bqn : bex, 1.f, Qs, KP, tl.m0, tl.n0, 0, C, d);
        tc::mma_tn<NTW, RAW>(lane, Ws, VP, RAW ? bkn : bex, -1.f, Ks, KP, tl.m0, tl.n0, 0, C, d);
#pragma unroll
        for (int j = 0; j < NTW; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dSs[tc::frag_row(lane, tl.m0, e) * KP + tc::frag_col(lane, tl.n0, j, e)] = d[j][e];
      }
    }
#else
    x.par((BV / 4) * (K / 4), [&](int t) {
      const int v0 = (t / (K / 4)) * 4, c0 = t % (K / 4);
      float acc[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = bex[C - 1] * dSs[(v0 + a) * KP + c0 + b * (K / 4)];
      for (int i = 0; i < C; ++i) {
        const float bi = bex[i];
        float bo[4], bw[4], qv[4], kv[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          bo[a] = bi * Os[i * VP + v0 + a];
          bw[a] = -bi * Ws[i * VP + v0 + a];
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          qv[b] = Qs[i * KP + c0 + b * (K / 4)];
          kv[b] = Ks[i * KP + c0 + b * (K / 4)];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(bw[a], kv[b], fmaf(bo[a], qv[b], acc[a][b]));
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) dSs[(v0 + a) * KP + c0 + b * (K / 4)] = acc[a][b];
    });
#endif
    x.sync();
  }
  if (p.dh0)
    x.par(BV * K, [&](int idx) {
      const int r = idx / K, c = idx % K;
      p.dh0[((size_t)s * Hv + h) * VK + (size_t)(row0 + r) * K + c] = dSs[r * KP + c];
    });
}

// ---- grad: the gradients linear in the summed dP, dT, dd and db of one (chunk, v-head)
template <int KD, class X, class LD>
GDN_BWD_FN void grad_block(X &x, const Params &p, LD ld, float *sm, int64_t slot, int h) {
  // rows padded by 4 floats, so that the tensor-core fragments' loads fall in distinct banks
  constexpr int K = KD, KP = KD + 4, MP = C + 4;
  int64_t t0;
  int n;
  if (!slot_chunk(p, slot, t0, n)) return;
  const int Hv = p.Hv, qh = h / (Hv / p.Hqk);
  float *Ks = sm;              // [C][KP]  k (unit-norm when l2norm)
  float *Qs = Ks + C * KP;     // [C][KP]  q
  float *Zm = Qs + C * KP;     // [C][MP]  Z
  float *KGm = Zm + C * MP;    // [C][MP]  KG
  float *QGm = KGm + C * MP;   // [C][MP]  QG
  float *dPm = QGm + C * MP;   // [C][MP]  dP, then M1 = dP * Gamma
  float *dTm = dPm + C * MP;   // [C][MP]  dT, then dA, then dKK
  float *Ym = dTm + C * MP;    // [C][MP]  Y = (dT diag(beta)) Z^T, then D = dKK + dKK^T
  float *gam = Ym + C * MP;    // [C] gamma
  float *bet = gam + C;        // [C] beta
  float *bex = bet + C;        // [C] exp(gamma)
  float *dec = bex + C;        // [C] exp(gamma_last - gamma)
  float *dd = dec + C;         // [C] dL/dd
  float *db = dd + C;          // [C] dL/db
  float *dbt = db + C;         // [C] dL/dbeta
  float *dgm = dbt + C;        // [C] dL/dgamma, then dg
  float *one = dgm + C;        // [C] ones (a unit scale for the tensor-core products)
  float *kin = one + C, *qin = kin + C;  // [C] each: 1/|k|, 1/|q| with raw keys
  float *gps = qin + C;        // [5][C] the dgamma phase's sums: rA, cA, rP, cP, bA
#if defined(__CUDA_ARCH__)
  constexpr bool RAW = LD::kRawTf32;  // k and q kept raw, their norms in kin / qin
#else
  constexpr bool RAW = false;
#endif
  const float *pr = p.prep + ((size_t)slot * Hv + h) * kPrep;
  const float *sums = p.sums + ((size_t)slot * Hv + h) * kSums;
  if (p.vec8) {  // every fill of the item in flight at once, then every store
    constexpr int NI = 256;
    x.par(NI, [&](int t) {
      Fill4<C, C, NI> fz, fkg, fqg, fdp, fdt;
      Fill8<C, K, NI> fk, fq;
      fz.load(t, pr, C, C);
      fkg.load(t, pr + C * C, C, C);
      fqg.load(t, pr + 2 * C * C, C, C);
      fdp.load(t, sums, C, C);
      fdt.load(t, sums + C * C, C, C);
      fk.load(ld, t, p.k, t0 * p.ks + (int64_t)qh * K, p.ks, n);
      fq.load(ld, t, p.q, t0 * p.qs + (int64_t)qh * K, p.qs, n);
      const float dv = t < C ? sums[2 * C * C + t] : 0.f, sbv = t < C ? sums[2 * C * C + C + t] : 0.f;
      const bool gi = t < C && t < n;
      const float gv = gi ? p.g[(t0 + t) * Hv + h] : 0.f, bv = gi ? p.beta[(t0 + t) * Hv + h] : 0.f;
      float pv[5] = {};  // with raw keys: gamma, b, d, 1/|k|, 1/|q| from prep
      if (RAW && t < C)
#pragma unroll
        for (int u = 0; u < 5; ++u) pv[u] = pr[kPrepVec + u * C + t];
      fz.store(t, Zm, MP);
      fkg.store(t, KGm, MP);
      fqg.store(t, QGm, MP);
      fdp.store(t, dPm, MP);
      fdt.store(t, dTm, MP);
      fk.store(t, Ks, KP);
      fq.store(t, Qs, KP);
      if (t < C) {
        dd[t] = dv;
        db[t] = sbv;
        gam[t] = RAW ? pv[0] : gv;
        bet[t] = bv;
        if (RAW) {
          bex[t] = pv[1];
          dec[t] = pv[2];
          kin[t] = pv[3];
          qin[t] = pv[4];
        }
      }
    });
  } else {
    load_keys<K, KP>(x, p, ld, Ks, Qs, t0, n, qh);
    load_gates(x, p, gam, bet, t0, n, h);
    if (RAW)  // after load_gates' raw g, by the same item
      x.par(C, [&](int i) {
        gam[i] = pr[kPrepVec + i];
        bex[i] = pr[kPrepVec + C + i];
        dec[i] = pr[kPrepVec + 2 * C + i];
        kin[i] = pr[kPrepVec + 3 * C + i];
        qin[i] = pr[kPrepVec + 4 * C + i];
      });
    copy_block<C, C>(x, pr, C, Zm, MP);
    copy_block<C, C>(x, pr + C * C, C, KGm, MP);
    copy_block<C, C>(x, pr + 2 * C * C, C, QGm, MP);
    copy_block<C, C>(x, sums, C, dPm, MP);
    copy_block<C, C>(x, sums + C * C, C, dTm, MP);
    x.par(C, [&](int i) {
      dd[i] = sums[2 * C * C + i];
      db[i] = sums[2 * C * C + C + i];
    });
  }
  x.sync();
  if constexpr (!RAW) {  // with raw keys gamma, b, d and the inverse norms came from prep
    norm_and_cumsum<K, KP>(x, p, Ks, Qs, gam);
    x.sync();
  }
  x.par(C, [&](int i) {
    if (!RAW) {
      bex[i] = expf(gam[i]);
      dec[i] = expf(gam[C - 1] - gam[i]);
    }
    one[i] = 1.f;
  });
  // dbeta from T = Z diag(beta): colsum(dT * Z)
  x.par(C, [&](int j) {
    float acc = 0.f;
    for (int i = j; i < C; ++i) acc = fmaf(dTm[i * MP + j], Zm[i * MP + j], acc);
    dbt[j] = acc;
  });
  // Y = (dT diag(beta)) Z^T (on the device a tensor-core product, on the host 4 x 4 tiles of
  // (i, j) a thread): dT is zero right of its diagonal and Z too, so the terms past min(i, j)
  // add zeros
#if defined(__CUDA_ARCH__)
  {  // terms past min(i, j) are zero: the tile takes m < min(m0 + 16, n0 + its width)
    const int lane = x.tid & 31;
    const tc::Tiles<C, C> tl(x.tid >> 5);
    constexpr int NTW = tc::Tiles<C, C>::NTW;
    if (tl.any) {
      float d[NTW][4] = {};
      const int kend = (tl.m0 + 16 < tl.n0 + 8 * NTW) ? tl.m0 + 16 : tl.n0 + 8 * NTW;
      tc::mma_nt<NTW, true>(lane, dTm, MP, bet, Zm, MP, tl.m0, tl.n0, 0, kend, d);
#pragma unroll
      for (int j = 0; j < NTW; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = tc::frag_row(lane, tl.m0, e), c = tc::frag_col(lane, tl.n0, j, e);
            Ym[i * MP + c] = d[j][e];
          }
    }
  }
#else
  x.par((C / 4) * (C / 4), [&](int t) {
    const int i0 = (t / (C / 4)) * 4, j0 = (t % (C / 4)) * 4;
    const int mend = (i0 < j0 ? i0 : j0) + 4;
    float acc[4][4] = {};
    for (int m = 0; m < mend; ++m) {
      const float bm = bet[m];
      float tr[4], zr[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        tr[a] = dTm[(i0 + a) * MP + m] * bm;
        zr[a] = Zm[(j0 + a) * MP + m];
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(tr[a], zr[b], acc[a][b]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) Ym[(i0 + a) * MP + j0 + b] = acc[a][b];
  });
#endif
  x.sync();
  // dA = -Z^T Y, strictly lower (into dT's place; on the host 4 x 4 tiles): Z^T's column i
  // is zero above row i, so every row of a tile can start at the tile's first row
#if defined(__CUDA_ARCH__)
  {  // Z[m][i] is zero for m < i: rows i >= m0 take m >= m0; tiles above the diagonal write zeros
    const int lane = x.tid & 31;
    const tc::Tiles<C, C> tl(x.tid >> 5);
    constexpr int NTW = tc::Tiles<C, C>::NTW;
    if (tl.any) {
      float d[NTW][4] = {};
      if (tl.n0 <= tl.m0 + 15) tc::mma_tn<NTW, false, false>(lane, Zm, MP, nullptr, 1.f, Ym, MP, tl.m0, tl.n0, tl.m0, C, d);
#pragma unroll
      for (int j = 0; j < NTW; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = tc::frag_row(lane, tl.m0, e), c = tc::frag_col(lane, tl.n0, j, e);
            dTm[i * MP + c] = c < i ? -d[j][e] : 0.f;
          }
    }
  }
#else
  x.par((C / 4) * (C / 4), [&](int t) {
    const int i0 = (t / (C / 4)) * 4, j0 = (t % (C / 4)) * 4;
    float acc[4][4] = {};
    if (j0 < i0 + 3)
      for (int m = i0; m < C; ++m) {
        float zr[4], yr[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          zr[a] = Zm[m * MP + i0 + a];
          yr[a] = Ym[m * MP + j0 + a];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(zr[a], yr[b], acc[a][b]);
      }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int b = 0; b < 4; ++b) dTm[(i0 + a) * MP + j0 + b] = j0 + b < i0 + a ? -acc[a][b] : 0.f;
  });
#endif
  x.sync();
  // dgamma (through Gamma in A and P, b and d) and the rest of dbeta: the row and column sums
  // of dA * KG and dP * QG, one sum kind per item group (a warp pair each on the device)
  x.par(4 * C, [&](int idx) {
    const int i = idx % C, part = idx / C;
    float acc = 0.f, bA = 0.f;
    if (part == 0) {
      for (int j = 0; j < i; ++j) {
        const float t = dTm[i * MP + j] * KGm[i * MP + j];
        bA += t;
        acc = fmaf(bet[i], t, acc);
      }
      gps[4 * C + i] = bA;
    } else if (part == 1) {
      for (int m = i + 1; m < C; ++m) acc = fmaf(bet[m], dTm[m * MP + i] * KGm[m * MP + i], acc);
    } else if (part == 2) {
      for (int j = 0; j <= i; ++j) acc = fmaf(dPm[i * MP + j], QGm[i * MP + j], acc);
    } else {
      for (int m = i; m < C; ++m) acc = fmaf(dPm[m * MP + i], QGm[m * MP + i], acc);
    }
    gps[part * C + i] = acc;
  });
  x.sync();
  x.par(C, [&](int i) {
    const float rA = gps[i], cA = gps[C + i], rP = gps[2 * C + i], cP = gps[3 * C + i];
    dbt[i] += gps[4 * C + i];
    dgm[i] = rP - cP + rA - cA + db[i] * bex[i] - dd[i] * dec[i];
  });
  x.sync();
  if (x.leader()) {
    float sdd = 0.f;
    for (int i = 0; i < C; ++i) sdd = fmaf(dd[i], dec[i], sdd);
    dgm[C - 1] += sdd;
    for (int i = C - 2; i >= 0; --i) dgm[i] += dgm[i + 1];  // dg = reverse cumsum of dgamma
  }
  // dKK = diag(beta) dA * Gamma (strictly lower); M1 = dP * Gamma (lower)
  x.par(C * C, [&](int idx) {
    const int i = idx / C, j = idx % C;
    const float gij = j <= i ? expf(gam[i] - gam[j]) : 0.f;
    dTm[i * MP + j] = j < i ? bet[i] * dTm[i * MP + j] * gij : 0.f;
    dPm[i * MP + j] *= gij;
  });
  x.sync();
  x.par(C, [&](int i) {
    if (i < n) {
      p.dg[(t0 + i) * Hv + h] = dgm[i];
      p.dbeta[(t0 + i) * Hv + h] = dbt[i];
    }
  });
  // D = dKK + dKK^T (symmetric, zero diagonal, in Y's place, free since dA)
  x.par(C * C, [&](int idx) {
    const int i = idx / C, j = idx % C;
    Ym[i * MP + j] = j < i ? dTm[i * MP + j] : (j > i ? dTm[j * MP + i] : 0.f);
  });
  x.sync();
  // the C x C parts of dq and dk (on the device tensor-core products, on the host 4 x 8 tiles
  // of (i, c) a thread, columns c0 + b K / 8):  dq += M1 K,  dk += M1^T Q + D K
#if defined(__CUDA_ARCH__)
  {  // M1 is zero above the diagonal: rows i < m0 + 16 take j < m0 + 16 in dq, j >= m0 in dk
    const int lane = x.tid & 31;
    const tc::Tiles<C, K> tl(x.tid >> 5);
    constexpr int NTW = tc::Tiles<C, K>::NTW;
    if (tl.any) {
      float d[NTW][4] = {};
      // with raw keys the norms scale K's rows and Q's rows; without them there is no scale
      tc::mma_nn<NTW, RAW, RAW>(lane, dPm, MP, one, 1.f, Ks, KP, RAW ? kin : nullptr, tl.m0, tl.n0, 0, tl.m0 + 16, d);
      add_row_quads<NTW>(lane, d, p.dqn + ((size_t)t0 * p.Hqk + qh) * K, (size_t)p.Hqk * K, n, tl.m0, tl.n0);
#pragma unroll
      for (int j = 0; j < NTW; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) d[j][e] = 0.f;
      tc::mma_tn<NTW, RAW, RAW>(lane, dPm, MP, RAW ? qin : nullptr, 1.f, Qs, KP, tl.m0, tl.n0, tl.m0, C, d);
      tc::mma_nn<NTW, RAW, RAW>(lane, Ym, MP, one, 1.f, Ks, KP, RAW ? kin : nullptr, tl.m0, tl.n0, 0, C, d);
      add_row_quads<NTW>(lane, d, p.dkn + ((size_t)t0 * p.Hqk + qh) * K, (size_t)p.Hqk * K, n, tl.m0, tl.n0);
    }
  }
#else
  x.par((C / 4) * (K / 8), [&](int t) {
    const int i0 = (t / (K / 8)) * 4, c0 = t % (K / 8);
    float dq[4][8] = {}, dk[4][8] = {};
    // M1 is zero above the diagonal: row i needs j <= i, column i needs j >= i
    for (int j = 0; j < i0 + 4; ++j) {
      float m[4], kr[8];
#pragma unroll
      for (int a = 0; a < 4; ++a) m[a] = dPm[(i0 + a) * MP + j];
#pragma unroll
      for (int b = 0; b < 8; ++b) kr[b] = Ks[j * KP + c0 + b * (K / 8)];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) dq[a][b] = fmaf(m[a], kr[b], dq[a][b]);
    }
    for (int j = i0; j < C; ++j) {
      float m[4], qr[8];
#pragma unroll
      for (int a = 0; a < 4; ++a) m[a] = dPm[j * MP + i0 + a];
#pragma unroll
      for (int b = 0; b < 8; ++b) qr[b] = Qs[j * KP + c0 + b * (K / 8)];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) dk[a][b] = fmaf(m[a], qr[b], dk[a][b]);
    }
    for (int j = 0; j < C; ++j) {
      float m[4], kr[8];
#pragma unroll
      for (int a = 0; a < 4; ++a) m[a] = Ym[(i0 + a) * MP + j];
#pragma unroll
      for (int b = 0; b < 8; ++b) kr[b] = Ks[j * KP + c0 + b * (K / 8)];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) dk[a][b] = fmaf(m[a], kr[b], dk[a][b]);
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
      const int i = i0 + a;
      if (i >= n) continue;
      const size_t off = ((size_t)(t0 + i) * p.Hqk + qh) * K + c0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        x.add(p.dqn + off + b * (K / 8), dq[a][b]);
        x.add(p.dkn + off + b * (K / 8), dk[a][b]);
      }
    }
  });
#endif
}

// Row r of q or k (token t = r / Hqk, head r % Hqk): the gradient of the unit-norm row taken
// back to the raw row, dx = dxh / n - x (x . dxh) / n^3 with n = sqrt(|x|^2 + eps), or
// copied when there is no norm.
template <class LD>
GDN_BWD_FN void l2_back_row(const void *raw, int64_t stride, int Hqk, int K, int l2norm, LD ld, const float *dn,
                            float *out, int64_t r) {
  const int64_t t = r / Hqk, hh = r % Hqk;
  const int64_t base = t * stride + hh * K;
  const float *dr = dn + r * K;
  float *o = out + r * K;
  if (!l2norm) {
    for (int c = 0; c < K; ++c) o[c] = dr[c];
    return;
  }
  float ss = 0.f, xd = 0.f;
  for (int c = 0; c < K; ++c) {
    const float xv = ld(raw, base + c);
    ss = fmaf(xv, xv, ss);
    xd = fmaf(xv, dr[c], xd);
  }
  const float nn = sqrtf(ss + kEps), inv = 1.f / nn, inv3 = inv * inv * inv;
  for (int c = 0; c < K; ++c) o[c] = dr[c] * inv - ld(raw, base + c) * xd * inv3;
}

}  // namespace gdn_bwd
