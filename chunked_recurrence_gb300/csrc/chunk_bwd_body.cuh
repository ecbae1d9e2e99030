// chunk_bwd_body.cuh -- the block body of the fp32 backward of the chunked gated delta rule.
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
// Each row of the state evolves on its own given k, g, beta and its column of v, and so
// does each row of dS.  So a block owns BV rows of one v-head's state: it recomputes its
// rows' chunk-start states in a forward sweep, then walks the chunks backward carrying its
// rows of dS.  dv and dh0 of its rows are complete in the block; dq, dk, dg and dbeta are
// sums over the blocks of a head (and over the v-heads of a q/k head) and are added
// atomically.
//
// The body is written against an executor X with three operations: x.par(n, f) runs f(i)
// for i in [0, n), the items independent of each other; x.sync() is a block barrier;
// x.add(p, v) adds v to *p atomically.  The CUDA kernel runs items on threads with
// __syncthreads(); a host harness runs the same code with plain loops.
#pragma once

#include <math.h>
#include <stddef.h>
#include <stdint.h>

#if defined(__CUDACC__)
#define GDN_BWD_FN __device__ __forceinline__
#define GDN_BWD_HD __host__ __device__ inline
#else
#define GDN_BWD_FN inline
#define GDN_BWD_HD inline
#endif

namespace gdn_bwd {

constexpr int C = 64;   // tokens per chunk
constexpr int BV = 16;  // state rows per block
constexpr int CP = C + 1, VP = BV + 1;
constexpr float kEps = 1e-6f;  // q/k L2 norm: x / sqrt(sum x^2 + eps)

struct Params {
  const void *q, *k, *v;  // q, k [n_tok][Hqk][K] (token strides qs, ks), v [n_tok][Hv][V] (vs)
  const float *g, *beta;  // [n_tok][Hv]
  const float *h0;        // [n_seq][Hv][V][K] or null
  const float *dout;      // [n_tok][Hv][V]
  const float *dhT;       // [n_seq][Hv][V][K] or null
  const int32_t *cu;      // sequence bounds, or null: rows of row_T tokens
  int64_t row_T, n_tok;
  int Hqk, Hv, K, V;
  int64_t qs, ks, vs;
  float scale;
  int l2norm;
  int vec8;         // q, k, v load as 8-element vectors (16-byte aligned rows and strides)
  float *states;    // [slot][Hv][V][K]: chunk-start states (chunk c of sequence s: slot s + start/C + c)
  float *dqn, *dkn; // [n_tok][Hqk][K]: gradients of the unit-norm (or raw) q and k, accumulated
  float *dv;        // [n_tok][Hv][V]
  float *dg, *dbeta;  // [n_tok][Hv], accumulated
  float *dh0;       // [n_seq][Hv][V][K] or null
  int32_t *status;  // set to GDN_ERR_BOUNDS on a bad sequence range
};

// shared memory of one block, in floats
GDN_BWD_HD size_t smem_floats(int K) {
  const size_t KP = (size_t)K + 1;
  return 2 * C * KP + 2 * BV * KP + 7 * (size_t)C * VP + 7 * (size_t)C * CP + 8 * C;
}

// ld(ptr, i): element i of a q / k / v array as float; ld.vec8(ptr, i, out): elements
// i .. i + 7 (i a multiple of 8, the array 16-byte aligned), used when p.vec8 is set
// KD: the key width (p.K) as a compile-time constant (32, 64 or 128), so that the loops over
// features unroll and row addresses fold into constants.
template <int KD, class X, class LD>
GDN_BWD_FN void block(X &x, const Params &p, LD ld, float *sm, int tile, int h, int s) {
  constexpr int K = KD, KP = KD + 1;
  const int V = p.V, Hv = p.Hv;
  float *Ks = sm;              // [C][KP]  k of the chunk (unit-norm when l2norm)
  float *Qs = Ks + C * KP;     // [C][KP]  q
  float *Ss = Qs + C * KP;     // [BV][KP] this block's rows of the chunk-start state
  float *dSs = Ss + BV * KP;   // [BV][KP] their gradient, carried from the chunk's end
  float *Vs = dSs + BV * KP;   // [C][VP]  v columns of the block's rows
  float *Os = Vs + C * VP;     // [C][VP]  scale * dO
  float *Us = Os + C * VP;     // [C][VP]  U'
  float *dUs = Us + C * VP;    // [C][VP]  K dS1^T, then dU'
  float *dVs = dUs + C * VP;   // [C][VP]  dV
  float *KSs = dVs + C * VP;   // [C][VP]  K S^T
  float *QSs = KSs + C * VP;   // [C][VP]  Q S^T
  float *Zm = QSs + C * VP;    // [C][CP]  A, then Z = (I + A)^-1 (unit lower)
  float *QKm = Zm + C * CP;    // [C][CP]  Q K^T (lower incl. diagonal)
  float *KKm = QKm + C * CP;   // [C][CP]  K K^T (strictly lower)
  float *dPm = KKm + C * CP;   // [C][CP]  dP (lower incl. diagonal)
  float *dTm = dPm + C * CP;   // [C][CP]  dT, then dA, then dKK
  float *Ym = dTm + C * CP;    // [C][CP]  (dT diag(beta)) Z^T
  float *gam = Ym + C * CP;    // [C] gamma
  float *bet = gam + C;        // [C] beta
  float *bex = bet + C;        // [C] exp(gamma)
  float *dec = bex + C;        // [C] exp(gamma_last - gamma)
  float *db = dec + C;         // [C] dL/db
  float *dd = db + C;          // [C] dL/dd
  float *dbt = dd + C;         // [C] dL/dbeta
  float *dgm = dbt + C;        // [C] scratch of the inversion, then dL/dgamma
  float *Gm = dgm + C;         // [C][CP]  Gamma_ij = exp(gamma_i - gamma_j), j <= i (once per chunk)

  const int qh = h / (Hv / p.Hqk), row0 = tile * BV;
  int64_t start, end;
  if (p.cu) {
    start = p.cu[s];
    end = p.cu[s + 1];
  } else {
    start = (int64_t)s * p.row_T;
    end = start + p.row_T;
  }
  if (start < 0 || end < start || end > p.n_tok) {
    x.fail(p.status);
    return;
  }
  const int64_t slot0 = (int64_t)s + start / C;
  const int n_chunks = (int)((end - start + C - 1) / C);
  const size_t VK = (size_t)V * K;
  auto G = [&](int i, int j) { return Gm[i * CP + j]; };  // j <= i

  // ---- the chunk's inputs and its state-independent matrices (with_q: Q, dO, Q K^T too)
  auto prep = [&](int64_t t0, int n, bool with_q) {
    if (p.vec8) {
      // 8 consecutive elements an item (one or two vector loads), so that each thread has
      // several loads in flight instead of one
      x.par(C * (K / 8), [&](int idx) {
        const int r = idx / (K / 8), c = (idx % (K / 8)) * 8;
        const bool in = r < n;
        float kv[8] = {}, qv[8] = {};
        if (in) {
          ld.vec8(p.k, (t0 + r) * p.ks + (int64_t)qh * K + c, kv);
          if (with_q) ld.vec8(p.q, (t0 + r) * p.qs + (int64_t)qh * K + c, qv);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          Ks[r * KP + c + e] = kv[e];
          if (with_q) Qs[r * KP + c + e] = qv[e];
        }
      });
      x.par(C * (BV / 8), [&](int idx) {
        const int r = idx / (BV / 8), j = (idx % (BV / 8)) * 8;
        const bool in = r < n;
        float vv[8] = {}, ov[8] = {};
        if (in) {
          ld.vec8(p.v, (t0 + r) * p.vs + (int64_t)h * V + row0 + j, vv);
          if (with_q) {
            const float *src = p.dout + ((t0 + r) * Hv + h) * V + row0 + j;
#pragma unroll
            for (int e = 0; e < 8; ++e) ov[e] = p.scale * src[e];
          }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          Vs[r * VP + j + e] = vv[e];
          if (with_q) Os[r * VP + j + e] = ov[e];
        }
      });
    } else {
      x.par(C * K, [&](int idx) {
        const int r = idx / K, c = idx % K;
        const bool in = r < n;
        Ks[r * KP + c] = in ? ld(p.k, (t0 + r) * p.ks + (int64_t)qh * K + c) : 0.f;
        if (with_q) Qs[r * KP + c] = in ? ld(p.q, (t0 + r) * p.qs + (int64_t)qh * K + c) : 0.f;
      });
      x.par(C * BV, [&](int idx) {
        const int r = idx / BV, j = idx % BV;
        const bool in = r < n;
        Vs[r * VP + j] = in ? ld(p.v, (t0 + r) * p.vs + (int64_t)h * V + row0 + j) : 0.f;
        if (with_q) Os[r * VP + j] = in ? p.scale * p.dout[((t0 + r) * Hv + h) * V + row0 + j] : 0.f;
      });
    }
    x.par(C, [&](int i) {
      const bool in = i < n;
      gam[i] = in ? p.g[(t0 + i) * Hv + h] : 0.f;
      bet[i] = in ? p.beta[(t0 + i) * Hv + h] : 0.f;
    });
    x.sync();
    if (p.l2norm) {
      x.par(with_q ? 2 * C : C, [&](int r) {
        float *row = r < C ? Ks + r * KP : Qs + (r - C) * KP;
        float ss = 0.f;
        for (int c = 0; c < K; ++c) ss = fmaf(row[c], row[c], ss);
        const float inv = 1.f / sqrtf(ss + kEps);
        for (int c = 0; c < K; ++c) row[c] *= inv;
      });
    }
    if (x.leader())
      for (int i = 1; i < C; ++i) gam[i] += gam[i - 1];
    x.sync();
    x.par(C, [&](int i) {
      bex[i] = expf(gam[i]);
      dec[i] = expf(gam[C - 1] - gam[i]);
    });
    // K K^T (strictly lower) and Q K^T (lower), 4 x 4 tiles of (i, j) a thread: every loaded
    // k or q value feeds four products
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
            qi[r] = with_q ? Qs[(i0 + r) * KP + c] : 0.f;
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
          const float kv = j < i ? kk[a][b] : 0.f;
          Gm[i * CP + j] = gij;
          KKm[i * CP + j] = kv;
          Zm[i * CP + j] = j < i ? bet[i] * gij * kv : 0.f;
          if (with_q) QKm[i * CP + j] = j <= i ? qk[a][b] : 0.f;
        }
    });
    x.sync();
    // Z = (I + A)^-1 by a row sweep: once row m of Z is final (every row above it applied),
    // each row i below it takes -A_im Z_m.  A stays in Zm while Z builds in Ym (free until the
    // backward step's dT), then Z replaces A.  One barrier a step, a few FMAs a thread.
    x.par(C * C, [&](int idx) {
      const int i = idx / C, j = idx % C;
      Ym[i * CP + j] = i == j ? 1.f : 0.f;
    });
    x.sync();
    for (int m = 0; m < C - 1; ++m) {
      const int cols = m + 1;  // row m of Z is zero right of its diagonal
      x.par((C - 1 - m) * cols, [&](int idx) {
        const int i = m + 1 + idx / cols, j = idx % cols;
        Ym[i * CP + j] = fmaf(-Zm[i * CP + m], Ym[m * CP + j], Ym[i * CP + j]);
      });
      x.sync();
    }
    x.par(C * C, [&](int idx) {
      const int i = idx / C, j = idx % C;
      Zm[i * CP + j] = Ym[i * CP + j];
    });
    // K S^T (and Q S^T), 2 x 2 tiles of (i, v) a thread
    x.par((C / 2) * (BV / 2), [&](int t) {
      const int i0 = (t / (BV / 2)) * 2, v0 = (t % (BV / 2)) * 2;
      float ks[2][2] = {}, qs[2][2] = {};
#pragma unroll 4
      for (int c = 0; c < K; ++c) {
        const float k0 = Ks[i0 * KP + c], k1 = Ks[(i0 + 1) * KP + c];
        const float s0 = Ss[v0 * KP + c], s1 = Ss[(v0 + 1) * KP + c];
        ks[0][0] = fmaf(k0, s0, ks[0][0]);
        ks[0][1] = fmaf(k0, s1, ks[0][1]);
        ks[1][0] = fmaf(k1, s0, ks[1][0]);
        ks[1][1] = fmaf(k1, s1, ks[1][1]);
        if (with_q) {
          const float q0 = Qs[i0 * KP + c], q1 = Qs[(i0 + 1) * KP + c];
          qs[0][0] = fmaf(q0, s0, qs[0][0]);
          qs[0][1] = fmaf(q0, s1, qs[0][1]);
          qs[1][0] = fmaf(q1, s0, qs[1][0]);
          qs[1][1] = fmaf(q1, s1, qs[1][1]);
        }
      }
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          KSs[(i0 + a) * VP + v0 + b] = ks[a][b];
          if (with_q) QSs[(i0 + a) * VP + v0 + b] = qs[a][b];
        }
    });
    x.sync();
    // U' = Z diag(beta) (V - diag(b) K S^T): the right factor first (into dV's place, free
    // until the backward step's dV), then 2 x 2 tiles of (i, v) a thread
    x.par(C * BV, [&](int idx) {
      const int j = idx / BV, v = idx % BV;
      dVs[j * VP + v] = Vs[j * VP + v] - bex[j] * KSs[j * VP + v];
    });
    x.sync();
    x.par((C / 2) * (BV / 2), [&](int t) {
      const int i0 = (t / (BV / 2)) * 2, v0 = (t % (BV / 2)) * 2;
      float acc[2][2] = {};
      for (int j = 0; j <= i0 + 1; ++j) {  // Z is zero right of its diagonal
        const float z0 = Zm[i0 * CP + j] * bet[j], z1 = Zm[(i0 + 1) * CP + j] * bet[j];
        const float w0 = dVs[j * VP + v0], w1 = dVs[j * VP + v0 + 1];
        acc[0][0] = fmaf(z0, w0, acc[0][0]);
        acc[0][1] = fmaf(z0, w1, acc[0][1]);
        acc[1][0] = fmaf(z1, w0, acc[1][0]);
        acc[1][1] = fmaf(z1, w1, acc[1][1]);
      }
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b) Us[(i0 + a) * VP + v0 + b] = acc[a][b];
    });
    x.sync();
  };

  // ---- forward sweep: the chunk-start state of every chunk, for this block's rows
  x.par(BV * K, [&](int idx) {
    const int r = idx / K, c = idx % K;
    Ss[r * KP + c] = p.h0 ? p.h0[((size_t)s * Hv + h) * VK + (size_t)(row0 + r) * K + c] : 0.f;
  });
  x.sync();
  for (int ci = 0; ci < n_chunks; ++ci) {
    const int64_t t0 = start + (int64_t)ci * C;
    const int n = (int)(end - t0 < C ? end - t0 : C);
    float *dst = p.states + ((size_t)(slot0 + ci) * Hv + h) * VK + (size_t)row0 * K;
    x.par(BV * K, [&](int idx) { dst[(idx / K) * (size_t)K + idx % K] = Ss[(idx / K) * KP + idx % K]; });
    prep(t0, n, false);
    // S1 = b_last S + U'^T diag(d) K, 2 x 4 tiles of (v, c) a thread (columns c0 + b K / 4,
    // so that neighbouring threads read neighbouring features)
    x.par((BV / 2) * (K / 4), [&](int t) {
      const int v0 = (t / (K / 4)) * 2, c0 = t % (K / 4);
      float acc[2][4] = {};
      for (int j = 0; j < C; ++j) {
        const float u0 = Us[j * VP + v0] * dec[j], u1 = Us[j * VP + v0 + 1] * dec[j];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const float kv = Ks[j * KP + c0 + b * (K / 4)];
          acc[0][b] = fmaf(u0, kv, acc[0][b]);
          acc[1][b] = fmaf(u1, kv, acc[1][b]);
        }
      }
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          float *sp = Ss + (v0 + a) * KP + c0 + b * (K / 4);
          *sp = fmaf(bex[C - 1], *sp, acc[a][b]);
        }
    });
    x.sync();
  }

  // ---- backward sweep
  x.par(BV * K, [&](int idx) {
    const int r = idx / K, c = idx % K;
    dSs[r * KP + c] = p.dhT ? p.dhT[((size_t)s * Hv + h) * VK + (size_t)(row0 + r) * K + c] : 0.f;
  });
  for (int ci = n_chunks - 1; ci >= 0; --ci) {
    const int64_t t0 = start + (int64_t)ci * C;
    const int n = (int)(end - t0 < C ? end - t0 : C);
    const float *src = p.states + ((size_t)(slot0 + ci) * Hv + h) * VK + (size_t)row0 * K;
    x.par(BV * K, [&](int idx) { Ss[(idx / K) * KP + idx % K] = src[(idx / K) * (size_t)K + idx % K]; });
    x.sync();
    prep(t0, n, true);
    // K dS1^T (2 x 2 tiles of (i, v) a thread); dP = Ot U'^T (lower incl. diagonal)
    x.par((C / 2) * (BV / 2), [&](int t) {
      const int i0 = (t / (BV / 2)) * 2, v0 = (t % (BV / 2)) * 2;
      float acc[2][2] = {};
#pragma unroll 4
      for (int c = 0; c < K; ++c) {
        const float k0 = Ks[i0 * KP + c], k1 = Ks[(i0 + 1) * KP + c];
        const float d0 = dSs[v0 * KP + c], d1 = dSs[(v0 + 1) * KP + c];
        acc[0][0] = fmaf(k0, d0, acc[0][0]);
        acc[0][1] = fmaf(k0, d1, acc[0][1]);
        acc[1][0] = fmaf(k1, d0, acc[1][0]);
        acc[1][1] = fmaf(k1, d1, acc[1][1]);
      }
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b) dUs[(i0 + a) * VP + v0 + b] = acc[a][b];
    });
    // (4 x 4 tiles of (i, j): rows i0 .. i0 + 3, columns tj + 16 b)
    x.par((C / 4) * 16, [&](int t) {
      const int i0 = (t / 16) * 4, tj = t % 16;
      float acc[4][4] = {};
      if (tj <= i0 + 3)
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
          dPm[i * CP + j] = j <= i ? acc[a][b] : 0.f;
        }
    });
    x.sync();
    // dd_i = U'_i . (K dS1^T)_i;  dU' = diag(d) K dS1^T + P^T Ot
    x.par(C, [&](int i) {
      float acc = 0.f;
      for (int v = 0; v < BV; ++v) acc = fmaf(Us[i * VP + v], dUs[i * VP + v], acc);
      dd[i] = acc;
    });
    x.sync();
    // (2 x 2 tiles of (i, v); row i0 + 1's term at j = i0 has a zero factor, P being lower)
    x.par((C / 2) * (BV / 2), [&](int t) {
      const int i0 = (t / (BV / 2)) * 2, v0 = (t % (BV / 2)) * 2;
      float acc[2][2];
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 2; ++b) acc[a][b] = dec[i0 + a] * dUs[(i0 + a) * VP + v0 + b];
      for (int j = i0; j < C; ++j) {
        const float m0 = QKm[j * CP + i0] * G(j, i0), m1 = QKm[j * CP + i0 + 1] * G(j, i0 + 1);
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
    x.sync();
    // dV = T^T dU' (complete for these rows); dT = dU' (V - diag(b) K S^T)^T (lower)
    // (dV in 2 x 2 tiles of (i, v), Z being lower; dT in 4 x 4 tiles of (i, j), columns tj + 16 b)
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
          dVs[i * VP + v0 + b] = r;
          if (i < n) p.dv[((t0 + i) * Hv + h) * V + row0 + v0 + b] = r;
        }
      }
    });
    x.par((C / 4) * 16, [&](int t) {
      const int i0 = (t / 16) * 4, tj = t % 16;
      float acc[4][4] = {};
      if (tj <= i0 + 3)
        for (int v = 0; v < BV; ++v) {
          float du[4], w[4];
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            du[a] = dUs[(i0 + a) * VP + v];
            const int j = tj + 16 * a;
            w[a] = Vs[j * VP + v] - bex[j] * KSs[j * VP + v];
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
          dTm[i * CP + j] = j <= i ? acc[a][b] : 0.f;
        }
    });
    x.sync();
    // b_last's gradient takes <S, dS1> over the block's rows: 64 partial sums (in dgm's
    // place, free until dgamma) instead of one thread's 2048-term chain
    x.par(C, [&](int r) {
      float acc = 0.f;
      for (int idx = r; idx < BV * K; idx += C) acc = fmaf(Ss[(idx / K) * KP + idx % K], dSs[(idx / K) * KP + idx % K], acc);
      dgm[r] = acc;
    });
    x.sync();
    // dbeta from T = Z diag(beta); db; Y = (dT diag(beta)) Z^T
    x.par(C, [&](int j) {
      float acc = 0.f;
      for (int i = j; i < C; ++i) acc = fmaf(dTm[i * CP + j], Zm[i * CP + j], acc);
      dbt[j] = acc;
      float b = 0.f;
      for (int v = 0; v < BV; ++v)
        b += Os[j * VP + v] * QSs[j * VP + v] - dVs[j * VP + v] * KSs[j * VP + v];
      if (j == C - 1)
        for (int r = 0; r < C; ++r) b += dgm[r];
      db[j] = b;
    });
    // Y, 4 x 4 tiles of (i, j) a thread: dT is zero right of its diagonal and Z too, so the
    // terms past min(i, j) add zeros
    x.par((C / 4) * (C / 4), [&](int t) {
      const int i0 = (t / (C / 4)) * 4, j0 = (t % (C / 4)) * 4;
      const int mend = (i0 < j0 ? i0 : j0) + 4;
      float acc[4][4] = {};
      for (int m = 0; m < mend; ++m) {
        const float bm = bet[m];
        float tr[4], zr[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          tr[a] = dTm[(i0 + a) * CP + m] * bm;
          zr[a] = Zm[(j0 + a) * CP + m];
        }
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(tr[a], zr[b], acc[a][b]);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) Ym[(i0 + a) * CP + j0 + b] = acc[a][b];
    });
    x.sync();
    // dA = -Z^T Y, strictly lower (into dT's place), 4 x 4 tiles: Z^T's column i is zero
    // above row i, so every row of a tile can start at the tile's first row
    x.par((C / 4) * (C / 4), [&](int t) {
      const int i0 = (t / (C / 4)) * 4, j0 = (t % (C / 4)) * 4;
      float acc[4][4] = {};
      if (j0 < i0 + 3)
        for (int m = i0; m < C; ++m) {
          float zr[4], yr[4];
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            zr[a] = Zm[m * CP + i0 + a];
            yr[a] = Ym[m * CP + j0 + a];
          }
#pragma unroll
          for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(zr[a], yr[b], acc[a][b]);
        }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) dTm[(i0 + a) * CP + j0 + b] = j0 + b < i0 + a ? -acc[a][b] : 0.f;
    });
    x.sync();
    // dgamma (through Gamma in A and P, b and d) and the rest of dbeta
    x.par(C, [&](int i) {
      float rA = 0.f, cA = 0.f, rP = 0.f, cP = 0.f, bA = 0.f;
      for (int j = 0; j < i; ++j) {
        const float t = dTm[i * CP + j] * KKm[i * CP + j] * G(i, j);
        bA += t;
        rA = fmaf(bet[i], t, rA);
      }
      for (int m = i + 1; m < C; ++m) cA = fmaf(bet[m], dTm[m * CP + i] * KKm[m * CP + i] * G(m, i), cA);
      for (int j = 0; j <= i; ++j) rP = fmaf(dPm[i * CP + j], QKm[i * CP + j] * G(i, j), rP);
      for (int m = i; m < C; ++m) cP = fmaf(dPm[m * CP + i], QKm[m * CP + i] * G(m, i), cP);
      dbt[i] += bA;
      dgm[i] = rP - cP + rA - cA + db[i] * bex[i] - dd[i] * dec[i];
    });
    x.sync();
    if (x.leader()) {
      float sdd = 0.f;
      for (int i = 0; i < C; ++i) sdd = fmaf(dd[i], dec[i], sdd);
      dgm[C - 1] += sdd;
      for (int i = C - 2; i >= 0; --i) dgm[i] += dgm[i + 1];  // dg = reverse cumsum of dgamma
    }
    x.sync();
    x.par(C, [&](int i) {
      if (i < n) {
        x.add(p.dg + (t0 + i) * Hv + h, dgm[i]);
        x.add(p.dbeta + (t0 + i) * Hv + h, dbt[i]);
      }
    });
    // dKK = diag(beta) dA * Gamma (strictly lower)
    x.par(C * C, [&](int idx) {
      const int i = idx / C, j = idx % C;
      dTm[i * CP + j] = j < i ? bet[i] * dTm[i * CP + j] * G(i, j) : 0.f;
    });
    x.sync();
    // M1 = dP * Gamma (lower, in dP's place) and D = dKK + dKK^T (symmetric, zero diagonal,
    // in Y's place, free since dA), so that dq and dk are tiled products
    x.par(C * C, [&](int idx) {
      const int i = idx / C, j = idx % C;
      dPm[i * CP + j] = dPm[i * CP + j] * Gm[i * CP + j];
      Ym[i * CP + j] = j < i ? dTm[i * CP + j] : (j > i ? dTm[j * CP + i] : 0.f);
    });
    x.sync();
    // dq and dk of the chunk's tokens, 4 x 8 tiles of (i, c) a thread (columns c0 + b K / 8):
    //   dq = diag(b) Ot S + M1 K,  dk = diag(d) U' dS1 - diag(b) dV S + M1^T Q + D K
    x.par((C / 4) * (K / 8), [&](int t) {
      const int i0 = (t / (K / 8)) * 4, c0 = t % (K / 8);
      float sq[4][8] = {}, sk[4][8] = {}, sv[4][8] = {};
      for (int v = 0; v < BV; ++v) {
        float o[4], u[4], w[4], sr[8], dr[8];
#pragma unroll
        for (int a = 0; a < 4; ++a) {
          o[a] = Os[(i0 + a) * VP + v];
          u[a] = Us[(i0 + a) * VP + v];
          w[a] = dVs[(i0 + a) * VP + v];
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
      float dq[4][8], dk[4][8];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          dq[a][b] = bex[i0 + a] * sq[a][b];
          dk[a][b] = dec[i0 + a] * sk[a][b] - bex[i0 + a] * sv[a][b];
        }
      // M1 is zero above the diagonal: row i needs j <= i, column i needs j >= i
      for (int j = 0; j < i0 + 4; ++j) {
        float m[4], kr[8];
#pragma unroll
        for (int a = 0; a < 4; ++a) m[a] = dPm[(i0 + a) * CP + j];
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
        for (int a = 0; a < 4; ++a) m[a] = dPm[j * CP + i0 + a];
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
        for (int a = 0; a < 4; ++a) m[a] = Ym[(i0 + a) * CP + j];
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
    x.sync();
    // dS = b_last dS1 + Ot^T diag(b) Q - (diag(b) dV)^T K, 2 x 4 tiles of (v, c) a thread
    // (columns c0 + b K / 4)
    x.par((BV / 2) * (K / 4), [&](int t) {
      const int v0 = (t / (K / 4)) * 2, c0 = t % (K / 4);
      float acc[2][4];
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) acc[a][b] = bex[C - 1] * dSs[(v0 + a) * KP + c0 + b * (K / 4)];
      for (int i = 0; i < C; ++i) {
        const float bi = bex[i];
        const float o0 = Os[i * VP + v0], o1 = Os[i * VP + v0 + 1];
        const float w0 = dVs[i * VP + v0], w1 = dVs[i * VP + v0 + 1];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const float qv = Qs[i * KP + c0 + b * (K / 4)], kv = Ks[i * KP + c0 + b * (K / 4)];
          acc[0][b] = fmaf(bi, o0 * qv - w0 * kv, acc[0][b]);
          acc[1][b] = fmaf(bi, o1 * qv - w1 * kv, acc[1][b]);
        }
      }
#pragma unroll
      for (int a = 0; a < 2; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) dSs[(v0 + a) * KP + c0 + b * (K / 4)] = acc[a][b];
    });
    x.sync();
  }
  if (p.dh0)
    x.par(BV * K, [&](int idx) {
      const int r = idx / K, c = idx % K;
      p.dh0[((size_t)s * Hv + h) * VK + (size_t)(row0 + r) * K + c] = dSs[r * KP + c];
    });
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
