// chunk_bwd.cu -- the fp32 CUDA-core backward of the chunked gated delta rule
// (gdn_chunk_bwd).  The arithmetic is the block bodies in chunk_bwd_body.cuh, run as three
// kernels of 256 threads: prep (one block per chunk and v-head), walk (one block per 32 or 16
// state rows, v-head and sequence) and grad (one block per chunk and v-head).  A fourth
// kernel takes the gradients of the unit-norm q and k back through the L2 norm.
#include <algorithm>

#include "chunk_bwd_body.cuh"
#include "chunk_common.cuh"

using namespace gdn;

namespace {

constexpr int kThreads = 256;

struct DevExec {
  int tid;
  template <class F>
  __device__ __forceinline__ void par(int n, F &&f) {
    for (int i = tid; i < n; i += kThreads) f(i);
  }
  __device__ __forceinline__ void sync() { __syncthreads(); }
  __device__ __forceinline__ bool leader() const { return tid == 0; }
  __device__ __forceinline__ void add(float *p, float v) { atomicAdd(p, v); }
  __device__ __forceinline__ void fail(int32_t *status) {
    if (tid == 0) set_status(status, GDN_ERR_BOUNDS);
  }
};

template <typename T>
struct DevLoad {
  static constexpr bool kRawTf32 = sizeof(T) == 2;  // bf16 values are exact in TF32
  __device__ __forceinline__ float operator()(const void *p, int64_t i) const {
    return to_f32<T>(reinterpret_cast<const T *>(p)[i]);
  }
  __device__ __forceinline__ void vec8(const void *p, int64_t i, float *out) const {
    if constexpr (sizeof(T) == 2) {
      const uint4 r = __ldg(reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(p) + i));
      const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        out[2 * e] = __uint_as_float(w[e] << 16);
        out[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
      }
    } else {
      const float4 *q = reinterpret_cast<const float4 *>(reinterpret_cast<const T *>(p) + i);
      const float4 a = __ldg(q), b = __ldg(q + 1);
      out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
      out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
    }
  }
};

template <typename T, int KD>
__global__ void __launch_bounds__(kThreads, 2) chunk_bwd_prep_kernel(const gdn_bwd::Params p) {
  extern __shared__ float sm[];
  DevExec x{(int)threadIdx.x};
  gdn_bwd::prep_block<KD>(x, p, DevLoad<T>{}, sm, (int64_t)blockIdx.x, (int)blockIdx.y);
}

template <typename T, int KD, int BV>
__global__ void __launch_bounds__(kThreads) chunk_bwd_walk_kernel(const gdn_bwd::Params p) {
  extern __shared__ float sm[];
  DevExec x{(int)threadIdx.x};
  gdn_bwd::walk_block<KD, BV>(x, p, DevLoad<T>{}, sm, (int)blockIdx.x, (int)blockIdx.y, (int)blockIdx.z);
}

template <typename T, int KD>
__global__ void __launch_bounds__(kThreads) chunk_bwd_grad_kernel(const gdn_bwd::Params p) {
  extern __shared__ float sm[];
  DevExec x{(int)threadIdx.x};
  gdn_bwd::grad_block<KD>(x, p, DevLoad<T>{}, sm, (int64_t)blockIdx.x, (int)blockIdx.y);
}

template <class KF>
bool set_smem(KF kernel, size_t smem) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) == cudaSuccess;
}

// the three launches; the walk takes 32 state rows a block when V allows, else 16
template <typename T, int KD>
gdn_status launch_bwd(const gdn_bwd::Params &p, int64_t n_slots, cudaStream_t st) {
  const int bv = p.V % 32 == 0 ? 32 : 16;
  const size_t s_prep = gdn_bwd::prep_smem_floats(KD) * sizeof(float);
  const size_t s_walk = gdn_bwd::walk_smem_floats(KD, bv) * sizeof(float);
  const size_t s_grad = gdn_bwd::grad_smem_floats(KD) * sizeof(float);
  const dim3 cgrid((unsigned)n_slots, (unsigned)p.Hv);
  const dim3 wgrid((unsigned)(p.V / bv), (unsigned)p.Hv, (unsigned)p.n_seqs);
  if (!set_smem(chunk_bwd_prep_kernel<T, KD>, s_prep) || !set_smem(chunk_bwd_grad_kernel<T, KD>, s_grad))
    return GDN_ERR_CUDA;
  chunk_bwd_prep_kernel<T, KD><<<cgrid, kThreads, s_prep, st>>>(p);
  if (bv == 32) {
    if (!set_smem(chunk_bwd_walk_kernel<T, KD, 32>, s_walk)) return GDN_ERR_CUDA;
    chunk_bwd_walk_kernel<T, KD, 32><<<wgrid, kThreads, s_walk, st>>>(p);
  } else {
    if (!set_smem(chunk_bwd_walk_kernel<T, KD, 16>, s_walk)) return GDN_ERR_CUDA;
    chunk_bwd_walk_kernel<T, KD, 16><<<wgrid, kThreads, s_walk, st>>>(p);
  }
  chunk_bwd_grad_kernel<T, KD><<<cgrid, kThreads, s_grad, st>>>(p);
  return GDN_OK;
}

template <typename T>
gdn_status launch_bwd_k(const gdn_bwd::Params &p, int64_t n_slots, cudaStream_t st) {
  switch (p.K) {
    case 32: return launch_bwd<T, 32>(p, n_slots, st);
    case 64: return launch_bwd<T, 64>(p, n_slots, st);
    default: return launch_bwd<T, 128>(p, n_slots, st);
  }
}

// One warp per row of q or k (rows of q first): the gradient of the unit-norm row taken back
// to the raw row, dx = dxh / n - x (x . dxh) / n^3 with n = sqrt(|x|^2 + eps), or copied when
// there is no norm (gdn_bwd::l2_back_row's arithmetic, the row's two sums reduced across
// the warp so that the loads coalesce).
template <typename T>
__global__ void __launch_bounds__(256) l2_back_kernel(const void *q, const void *k, int64_t qs, int64_t ks, int Hqk,
                                                      int K, int l2norm, const float *dqn, const float *dkn,
                                                      float *dq, float *dk, int64_t rows) {
  const int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= 2 * rows) return;  // whole warps
  const bool is_q = r < rows;
  const int64_t rr = is_q ? r : r - rows;
  const void *raw = is_q ? q : k;
  const int64_t base = (rr / Hqk) * (is_q ? qs : ks) + (rr % Hqk) * K;
  const float *dr = (is_q ? dqn : dkn) + rr * K;
  float *o = (is_q ? dq : dk) + rr * K;
  const int per = K / 32;  // 1, 2 or 4
  if (!l2norm) {
    for (int e = 0; e < per; ++e) o[lane + 32 * e] = dr[lane + 32 * e];
    return;
  }
  DevLoad<T> ld;
  float xv[4] = {}, dv[4] = {}, ss = 0.f, xd = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (e < per) {
      xv[e] = ld(raw, base + lane + 32 * e);
      dv[e] = dr[lane + 32 * e];
      ss = fmaf(xv[e], xv[e], ss);
      xd = fmaf(xv[e], dv[e], xd);
    }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    ss += __shfl_xor_sync(0xffffffffu, ss, m);
    xd += __shfl_xor_sync(0xffffffffu, xd, m);
  }
  const float nn = sqrtf(ss + gdn_bwd::kEps), inv = 1.f / nn, inv3 = inv * inv * inv;
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (e < per) o[lane + 32 * e] = dv[e] * inv - xv[e] * xd * inv3;
}

constexpr size_t kHeader = 256;

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// the workspace after its header: chunk-start states, the forward sweep's U', V - diag(b) K S^T
// and K S^T, prep's matrices, the walk's sums, then the accumulated gradients of the unit-norm
// q and k
struct BwdLayout {
  size_t states, fw, prep, sums, acc;
  BwdLayout(int64_t n_tok, int n_seqs, int Hqk, int Hv, int K, int V) {
    const size_t slots_h = n_slots(n_tok, n_seqs) * (size_t)Hv;
    states = round256(slots_h * V * K * sizeof(float));
    fw = round256(slots_h * 3 * gdn_bwd::C * V * sizeof(float));
    prep = round256(slots_h * gdn_bwd::kPrep * sizeof(float));
    sums = round256(slots_h * gdn_bwd::kSums * sizeof(float));
    acc = round256((size_t)n_tok * Hqk * K * sizeof(float));
  }
  size_t total() const { return kHeader + states + fw + prep + sums + 2 * acc; }
};

size_t bwd_workspace_bytes(int64_t n_tok, int n_seqs, int Hqk, int Hv, int K, int V) {
  return BwdLayout(n_tok, n_seqs, Hqk, Hv, K, V).total();
}

bool bwd_shape_ok(const gdn_shape *sh) {
  if (!sh) return false;
  if (sh->dtype != GDN_F32 && sh->dtype != GDN_BF16) return false;
  if (sh->B <= 0 || sh->T < 0 || sh->n_seqs < 0 || sh->Hqk <= 0 || sh->Hv <= 0) return false;
  if (sh->Hv % sh->Hqk != 0) return false;
  if (!(sh->K == 32 || sh->K == 64 || sh->K == 128)) return false;
  if (sh->V % 16 != 0 || sh->V <= 0 || sh->V > 256) return false;
  if (sh->n_seqs > 65535 || sh->Hv > 65535) return false;
  return true;
}

}  // namespace

extern "C" size_t gdn_chunk_bwd_workspace_bytes(const gdn_shape *shape) {
  if (!bwd_shape_ok(shape)) return 0;
  const int64_t n_tok = (int64_t)shape->B * shape->T;
  return bwd_workspace_bytes(n_tok, shape->n_seqs, shape->Hqk, shape->Hv, shape->K, shape->V);
}

extern "C" gdn_status gdn_chunk_bwd(const void *q, const void *k, const void *v, const float *g, const float *beta,
                                    const float *h0, const int32_t *cu_seqlens, const gdn_shape *shape, float scale,
                                    uint32_t flags, const float *d_o, const float *dh_T, float *dq, float *dk,
                                    float *dv, float *dg, float *dbeta, float *dh0, void *workspace,
                                    size_t workspace_bytes, void *stream) {
  if (!shape) return GDN_ERR_INVALID_ARG;
  if (!bwd_shape_ok(shape)) {
    const bool valid = (shape->dtype == GDN_F32 || shape->dtype == GDN_BF16) && shape->B > 0 && shape->T >= 0 &&
                       shape->n_seqs >= 0 && shape->Hqk > 0 && shape->Hv > 0 && shape->Hv % shape->Hqk == 0;
    return valid ? GDN_ERR_UNSUPPORTED : GDN_ERR_INVALID_ARG;
  }
  if (flags & ~GDN_FLAG_QK_L2NORM) return GDN_ERR_INVALID_ARG;
  const gdn_shape &sh = *shape;
  if (cu_seqlens) {
    if (sh.B != 1) return GDN_ERR_INVALID_ARG;
  } else if (sh.n_seqs != sh.B) {
    return GDN_ERR_INVALID_ARG;
  }
  const int64_t n_tok = cu_seqlens ? sh.T : (int64_t)sh.B * sh.T;
  const int64_t qs = sh.q_stride ? sh.q_stride : (int64_t)sh.Hqk * sh.K;
  const int64_t ks = sh.k_stride ? sh.k_stride : (int64_t)sh.Hqk * sh.K;
  const int64_t vs = sh.v_stride ? sh.v_stride : (int64_t)sh.Hv * sh.V;
  if (qs < (int64_t)sh.Hqk * sh.K || ks < (int64_t)sh.Hqk * sh.K || vs < (int64_t)sh.Hv * sh.V)
    return GDN_ERR_INVALID_ARG;
  const size_t need = bwd_workspace_bytes(n_tok, sh.n_seqs, sh.Hqk, sh.Hv, sh.K, sh.V);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return GDN_ERR_WORKSPACE;
  if (sh.n_seqs == 0) return GDN_OK;
  if (n_tok > 0 && (!q || !k || !v || !g || !beta || !d_o || !dq || !dk || !dv || !dg || !dbeta))
    return GDN_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  uint8_t *ws = (uint8_t *)workspace;
  const BwdLayout L(n_tok, sh.n_seqs, sh.Hqk, sh.Hv, sh.K, sh.V);
  const int64_t slots = (int64_t)n_slots(n_tok, sh.n_seqs);
  gdn_bwd::Params p{};
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.h0 = h0; p.dout = d_o; p.dhT = dh_T;
  p.cu = cu_seqlens;
  p.row_T = sh.T;
  p.n_tok = n_tok;
  p.n_seqs = sh.n_seqs;
  p.Hqk = sh.Hqk; p.Hv = sh.Hv; p.K = sh.K; p.V = sh.V;
  p.qs = qs; p.ks = ks; p.vs = vs;
  p.scale = scale;
  p.l2norm = (flags & GDN_FLAG_QK_L2NORM) ? 1 : 0;
  p.vec8 = aligned(q, 16) && aligned(k, 16) && aligned(v, 16) && aligned(d_o, 16) && qs % 8 == 0 && ks % 8 == 0 &&
           vs % 8 == 0 && (sh.dtype == GDN_BF16 || (qs % 4 == 0 && ks % 4 == 0 && vs % 4 == 0));
  uint8_t *cur = ws + kHeader;
  p.states = (float *)cur;
  p.fw = (float *)(cur += L.states);
  p.prep = (float *)(cur += L.fw);
  p.sums = (float *)(cur += L.prep);
  p.dqn = (float *)(cur += L.sums);
  p.dkn = (float *)(cur += L.acc);
  p.dv = dv; p.dg = dg; p.dbeta = dbeta; p.dh0 = dh0;
  p.status = (int32_t *)workspace;
  // the accumulated outputs and the walk's sums start at zero; dv, dg and dbeta too, so
  // tokens outside every sequence read 0
  const size_t tok_hk = (size_t)n_tok * sh.Hqk * sh.K * sizeof(float);
  const size_t tok_h = (size_t)n_tok * sh.Hv * sizeof(float);
  if (cudaMemsetAsync(p.sums, 0, (size_t)slots * sh.Hv * gdn_bwd::kSums * sizeof(float), st) != cudaSuccess)
    return GDN_ERR_CUDA;
  if (n_tok > 0 &&
      (cudaMemsetAsync(p.dqn, 0, tok_hk, st) != cudaSuccess || cudaMemsetAsync(p.dkn, 0, tok_hk, st) != cudaSuccess ||
       cudaMemsetAsync(dg, 0, tok_h, st) != cudaSuccess || cudaMemsetAsync(dbeta, 0, tok_h, st) != cudaSuccess ||
       cudaMemsetAsync(dv, 0, (size_t)n_tok * sh.Hv * sh.V * sizeof(float), st) != cudaSuccess))
    return GDN_ERR_CUDA;
  const int64_t rows = n_tok * sh.Hqk;
  const unsigned lgrid = (unsigned)((2 * rows * 32 + 255) / 256);  // a warp per row
  if (sh.dtype == GDN_BF16) {
    const gdn_status r = launch_bwd_k<__nv_bfloat16>(p, slots, st);
    if (r != GDN_OK) return r;
    if (rows > 0)
      l2_back_kernel<__nv_bfloat16><<<lgrid, 256, 0, st>>>(q, k, qs, ks, sh.Hqk, sh.K, p.l2norm, p.dqn, p.dkn, dq,
                                                           dk, rows);
  } else {
    const gdn_status r = launch_bwd_k<float>(p, slots, st);
    if (r != GDN_OK) return r;
    if (rows > 0)
      l2_back_kernel<float><<<lgrid, 256, 0, st>>>(q, k, qs, ks, sh.Hqk, sh.K, p.l2norm, p.dqn, p.dkn, dq, dk, rows);
  }
  return launch_status();
}
