// chunk_simt.cu -- fp32 CUDA-core kernel of the chunked gated delta rule.
//
// One block owns (row tile of 32 state rows, v-head, sequence) and walks the
// sequence chunk by chunk (64 tokens), keeping its rows of the fp32 state in
// shared memory.  Inside a chunk it applies the UT/WY form of the recurrence
// (Yang et al., "Gated Delta Networks": chunkwise form of the delta rule):
//   gamma = inclusive cumsum of g in the chunk,  b = exp(gamma)
//   A  = strictly-lower(diag(beta) K K^T * Gamma),  Gamma_ij = exp(gamma_i - gamma_j)
//   T  = (I + A)^-1 diag(beta)                     (forward substitution, fp32)
//   W  = T diag(b) K,   U = T V,   U' = U - W S^T
//   O  = scale * (diag(b) Q S^T + (Q K^T * Gamma, causal incl. diagonal) U')
//   S <- b_last S + U'^T diag(exp(gamma_last - gamma)) K
// Everything is fp32 FFMA: this kernel is the one for fp32 inputs (whose
// tolerance rules out TF32 / bf16 tensor-core operands) and the explicit
// GDN_FLAG_SIMT path for bf16 inputs.
//
// Summary mode computes a segment's (M, S_local) with the same code: the
// block's rows are rows of the augmented state [M; S_local] (K + V rows),
// where the M rows start at the identity and see v = 0, and the S_local rows
// start at zero and see v.  Both evolve by the same per-token map, so
// S_end = S_start M + S_local ("Qwen3.5 cp - #1", Architecture: (b, M) pairs).
#include <math.h>

#include "common.cuh"

using namespace gdn;

namespace {

constexpr int BV = 32;   // state rows per block
constexpr int C = kChunk;
constexpr int NT = 256;  // threads per block
constexpr int CP = C + 1;
constexpr int VP = BV + 1;

struct SimtParams {
  const void *q, *k, *v;
  const float *g, *beta, *h0;
  const int32_t *cu;  // sequence (or segment) bounds, or null
  int64_t row_T;      // tokens per batch row when cu is null
  int64_t n_tok;      // tokens on the token axis: every sequence must lie inside it
  int32_t *status;    // device status word (workspace), set on a bad sequence range
  int Hqk, Hv, K, V;
  int64_t qs, ks, vs;  // token strides (elements)
  float scale;
  int l2norm;
  void *o;
  float *hT;
  float *M, *S_local;  // summary mode outputs
};

size_t simt_smem_bytes(int K) {
  const int KP = K + 1;
  return sizeof(float) * ((size_t)3 * C * KP + (size_t)BV * KP + 2 * C * VP + 2 * C * CP + 4 * C);
}

template <typename T, typename TO, bool SUMMARY>
__global__ void __launch_bounds__(NT) chunk_simt_kernel(const SimtParams p) {
  extern __shared__ float sm[];
  const int K = p.K, KP = K + 1;
  float *Ks = sm;                  // [C][KP]
  float *Qs = Ks + C * KP;         // [C][KP]
  float *Ws = Qs + C * KP;         // [C][KP]
  float *Ss = Ws + C * KP;         // [BV][KP]   fp32 state rows
  float *Vs = Ss + BV * KP;        // [C][VP]
  float *Us = Vs + C * VP;         // [C][VP]    U, then U'
  float *Tm = Us + C * VP;         // [C][CP]    A, then T
  float *Pm = Tm + C * CP;         // [C][CP]    Q K^T * Gamma (causal)
  float *gam = Pm + C * CP;        // [C]
  float *bet = gam + C;            // [C]
  float *bex = bet + C;            // [C] exp(gamma)
  float *dec = bex + C;            // [C] exp(gamma_last - gamma)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
  const int qh = h / (p.Hv / p.Hqk);
  const int row0 = tile * BV;
  const T *qg = (const T *)p.q;
  const T *kg = (const T *)p.k;
  const T *vg = (const T *)p.v;

  int64_t start, end;
  if (p.cu) {
    start = p.cu[s];
    end = p.cu[s + 1];
  } else {
    start = (int64_t)s * p.row_T;
    end = start + p.row_T;
  }
  if (start < 0 || end < start || end > p.n_tok) {  // bad cu_seqlens: report, touch nothing
    if (tid == 0) set_status(p.status, GDN_ERR_BOUNDS);
    return;
  }

  // start state of this block's rows
  for (int idx = tid; idx < BV * K; idx += NT) {
    const int r = idx / K, c = idx % K;
    float val = 0.f;
    if (SUMMARY) {
      const int gr = row0 + r;
      val = (gr < K && gr == c) ? 1.f : 0.f;
    } else if (p.h0) {
      val = p.h0[(((int64_t)s * p.Hv + h) * p.V + row0 + r) * K + c];
    }
    Ss[r * KP + c] = val;
  }

  for (int64_t t0 = start; t0 < end; t0 += C) {
    const int n = (int)min((int64_t)C, end - t0);
    __syncthreads();  // previous chunk done with every buffer
    // ---- loads (rows past the end of the sequence are zero: k = q = v = 0, g = beta = 0)
    for (int idx = tid; idx < C * K; idx += NT) {
      const int r = idx / K, c = idx % K;
      const bool in = r < n;
      Ks[r * KP + c] = in ? to_f32(kg[(t0 + r) * p.ks + (int64_t)qh * K + c]) : 0.f;
      if (!SUMMARY) Qs[r * KP + c] = in ? to_f32(qg[(t0 + r) * p.qs + (int64_t)qh * K + c]) : 0.f;
    }
    for (int idx = tid; idx < C * BV; idx += NT) {
      const int r = idx / BV, j = idx % BV;
      float val = 0.f;
      if (r < n) {
        if (SUMMARY) {
          const int gr = row0 + j;
          if (gr >= K) val = to_f32(vg[(t0 + r) * p.vs + (int64_t)h * p.V + (gr - K)]);
        } else {
          val = to_f32(vg[(t0 + r) * p.vs + (int64_t)h * p.V + row0 + j]);
        }
      }
      Vs[r * VP + j] = val;
    }
    if (tid < C) {
      const bool in = tid < n;
      gam[tid] = in ? p.g[(t0 + tid) * p.Hv + h] : 0.f;
      bet[tid] = in ? p.beta[(t0 + tid) * p.Hv + h] : 0.f;
    }
    __syncthreads();
    // ---- unit-norm q and k (one warp per row, shuffle reduction)
    if (p.l2norm) {
      for (int r = warp; r < 2 * C; r += NT / 32) {
        float *row = (r < C) ? (Ks + r * KP) : (Qs + (r - C) * KP);
        if (SUMMARY && r >= C) continue;
        float ss = 0.f;
        for (int c = lane; c < K; c += 32) ss = fmaf(row[c], row[c], ss);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = 1.f / sqrtf(ss + kL2Eps);
        for (int c = lane; c < K; c += 32) row[c] *= inv;
      }
    }
    // ---- gamma = inclusive cumsum of g (warp 0, two tokens a lane)
    if (warp == 0) {
      const float g0 = gam[2 * lane], g1 = gam[2 * lane + 1];
      float incl = g0 + g1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      gam[2 * lane + 1] = incl;
      gam[2 * lane] = incl - g1;
    }
    __syncthreads();
    if (tid < C) {
      bex[tid] = expf(gam[tid]);
      dec[tid] = expf(gam[C - 1] - gam[tid]);
    }
    // ---- A (strictly lower) and P (lower incl. diagonal); exponents are <= 0
    for (int idx = tid; idx < C * C; idx += NT) {
      const int i = idx / C, j = idx % C;
      float a = 0.f, pq = 0.f;
      if (j <= i) {
        const float gm = expf(gam[i] - gam[j]);
        const float *ki = Ks + i * KP, *kj = Ks + j * KP;
        if (j < i) {
          float d = 0.f;
          for (int c = 0; c < K; ++c) d = fmaf(ki[c], kj[c], d);
          a = bet[i] * gm * d;
        }
        if (!SUMMARY) {
          const float *qi = Qs + i * KP;
          float d = 0.f;
          for (int c = 0; c < K; ++c) d = fmaf(qi[c], kj[c], d);
          pq = gm * d;
        }
      }
      Tm[i * CP + j] = a;
      if (!SUMMARY) Pm[i * CP + j] = pq;
    }
    __syncthreads();
    // ---- X = (I + A)^-1 (unit lower triangular) by forward substitution:
    //      X_i = e_i - sum_{j<i} A_ij X_j, one row at a time, one column a thread.
    //      Tm keeps A in and above row i and X below it; X's unit diagonal is implicit.
    for (int i = 1; i < C; ++i) {
      float x = 0.f;
      if (tid < i) {
        x = Tm[i * CP + tid];  // the j = tid term, X_tid,tid = 1
        for (int j = tid + 1; j < i; ++j) x = fmaf(Tm[i * CP + j], Tm[j * CP + tid], x);
      }
      __syncthreads();
      if (tid < i) Tm[i * CP + tid] = -x;
      __syncthreads();
    }
    // ---- T = X diag(beta)
    for (int idx = tid; idx < C * C; idx += NT) {
      const int i = idx / C, j = idx % C;
      float t = 0.f;
      if (j < i) t = Tm[i * CP + j] * bet[j];
      else if (j == i) t = bet[j];
      Tm[i * CP + j] = t;
    }
    __syncthreads();
    // ---- W = T diag(b) K  and  U = T V
    for (int idx = tid; idx < C * K; idx += NT) {
      const int r = idx / K, c = idx % K;
      float acc = 0.f;
      for (int j = 0; j <= r; ++j) acc = fmaf(Tm[r * CP + j] * bex[j], Ks[j * KP + c], acc);
      Ws[r * KP + c] = acc;
    }
    for (int idx = tid; idx < C * BV; idx += NT) {
      const int r = idx / BV, jv = idx % BV;
      float acc = 0.f;
      for (int j = 0; j <= r; ++j) acc = fmaf(Tm[r * CP + j], Vs[j * VP + jv], acc);
      Us[r * VP + jv] = acc;
    }
    __syncthreads();
    // ---- U' = U - W S^T (and the inter-chunk part of O from the old state)
    constexpr int kPer = C * BV / NT;
    float qs_part[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int idx = tid + u * NT;
      const int r = idx / BV, jv = idx % BV;
      const float *srow = Ss + jv * KP;
      const float *wrow = Ws + r * KP;
      float acc = 0.f;
      for (int c = 0; c < K; ++c) acc = fmaf(wrow[c], srow[c], acc);
      Us[r * VP + jv] -= acc;
      if (!SUMMARY) {
        const float *qrow = Qs + r * KP;
        float aq = 0.f;
        for (int c = 0; c < K; ++c) aq = fmaf(qrow[c], srow[c], aq);
        qs_part[u] = aq;
      }
    }
    __syncthreads();
    // ---- O = scale (diag(b) Q S^T + P U')
    if (!SUMMARY) {
      TO *og = (TO *)p.o;
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int idx = tid + u * NT;
        const int r = idx / BV, jv = idx % BV;
        float acc = bex[r] * qs_part[u];
        for (int j = 0; j <= r; ++j) acc = fmaf(Pm[r * CP + j], Us[j * VP + jv], acc);
        if (r < n) og[(t0 + r) * ((int64_t)p.Hv * p.V) + (int64_t)h * p.V + row0 + jv] =
            from_f32<TO>(p.scale * acc);
      }
    }
    // ---- S <- b_last S + U'^T diag(dec) K
    const float blast = bex[C - 1];
    for (int idx = tid; idx < BV * K; idx += NT) {
      const int jv = idx / K, c = idx % K;
      float acc = 0.f;
      for (int j = 0; j < C; ++j) acc = fmaf(Us[j * VP + jv] * dec[j], Ks[j * KP + c], acc);
      Ss[jv * KP + c] = fmaf(blast, Ss[jv * KP + c], acc);
    }
  }
  __syncthreads();
  // ---- final rows
  for (int idx = tid; idx < BV * K; idx += NT) {
    const int r = idx / K, c = idx % K;
    const float val = Ss[r * KP + c];
    if (SUMMARY) {
      const int gr = row0 + r;
      if (gr < K) p.M[(((int64_t)s * p.Hv + h) * K + gr) * K + c] = val;
      else p.S_local[(((int64_t)s * p.Hv + h) * p.V + (gr - K)) * K + c] = val;
    } else if (p.hT) {
      p.hT[(((int64_t)s * p.Hv + h) * p.V + row0 + r) * K + c] = val;
    }
  }
}

template <typename T, typename TO, bool SUMMARY>
gdn_status launch_simt_t(const SimtParams &p, dim3 grid, size_t smem, cudaStream_t st) {
  auto kern = chunk_simt_kernel<T, TO, SUMMARY>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return GDN_ERR_CUDA;
  kern<<<grid, NT, smem, st>>>(p);
  return launch_status();
}

template <bool SUMMARY>
gdn_status launch_simt(const SimtParams &p, int dtype, bool o_f32, int n_seqs, cudaStream_t st) {
  const size_t smem = simt_smem_bytes(p.K);
  const int rows = SUMMARY ? (p.K + p.V) : p.V;
  const dim3 grid(rows / BV, p.Hv, n_seqs);
  if (dtype == GDN_BF16) {
    if (o_f32) return launch_simt_t<__nv_bfloat16, float, SUMMARY>(p, grid, smem, st);
    return launch_simt_t<__nv_bfloat16, __nv_bfloat16, SUMMARY>(p, grid, smem, st);
  }
  return launch_simt_t<float, float, SUMMARY>(p, grid, smem, st);
}

}  // namespace

namespace gdn {

gdn_status chunk_fwd_simt(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, const float *h0, const int32_t *cu,
                          const gdn_shape &sh, float scale, uint32_t flags, void *o, float *h_T,
                          int32_t *status, cudaStream_t st) {
  SimtParams p{};
  p.n_tok = cu ? sh.T : (int64_t)sh.B * sh.T;
  p.status = status;
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.h0 = h0; p.cu = cu;
  p.row_T = sh.T;
  p.Hqk = sh.Hqk; p.Hv = sh.Hv; p.K = sh.K; p.V = sh.V;
  p.qs = sh.q_stride; p.ks = sh.k_stride; p.vs = sh.v_stride;
  p.scale = scale;
  p.l2norm = (flags & GDN_FLAG_QK_L2NORM) ? 1 : 0;
  p.o = o; p.hT = h_T;
  return launch_simt<false>(p, sh.dtype, (flags & GDN_FLAG_O_F32) != 0, sh.n_seqs, st);
}

gdn_status segment_summary_simt(const void *k, const void *v, const float *g, const float *beta,
                                const int32_t *bounds, int n_seg, const gdn_shape &sh,
                                uint32_t flags, float *M, float *S_local, int32_t *status,
                                cudaStream_t st) {
  SimtParams p{};
  p.n_tok = sh.T;
  p.status = status;
  p.k = k; p.v = v; p.g = g; p.beta = beta; p.cu = bounds;
  p.Hqk = sh.Hqk; p.Hv = sh.Hv; p.K = sh.K; p.V = sh.V;
  p.qs = sh.q_stride; p.ks = sh.k_stride; p.vs = sh.v_stride;
  p.l2norm = (flags & GDN_FLAG_QK_L2NORM) ? 1 : 0;
  p.M = M; p.S_local = S_local;
  return launch_simt<true>(p, sh.dtype, false, n_seg, st);
}

}  // namespace gdn
