// chunk_bwd.cu -- the fp32 CUDA-core backward of the chunked gated delta rule
// (gdn_chunk_bwd).  The arithmetic is the block body in chunk_bwd_body.cuh: one block
// per (16 state rows, v-head, sequence), 256 threads.  A second kernel takes the
// gradients of the unit-norm q and k back through the L2 norm.
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
__global__ void __launch_bounds__(kThreads) chunk_bwd_kernel(const gdn_bwd::Params p) {
  extern __shared__ float sm[];
  DevExec x{(int)threadIdx.x};
  gdn_bwd::block<KD>(x, p, DevLoad<T>{}, sm, blockIdx.x, blockIdx.y, blockIdx.z);
}

template <typename T, int KD>
gdn_status launch_bwd(const gdn_bwd::Params &p, dim3 grid, size_t smem, cudaStream_t st) {
  if (cudaFuncSetAttribute(chunk_bwd_kernel<T, KD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return GDN_ERR_CUDA;
  chunk_bwd_kernel<T, KD><<<grid, kThreads, smem, st>>>(p);
  return GDN_OK;
}

template <typename T>
gdn_status launch_bwd_k(const gdn_bwd::Params &p, dim3 grid, size_t smem, cudaStream_t st) {
  switch (p.K) {
    case 32: return launch_bwd<T, 32>(p, grid, smem, st);
    case 64: return launch_bwd<T, 64>(p, grid, smem, st);
    default: return launch_bwd<T, 128>(p, grid, smem, st);
  }
}

template <typename T>
__global__ void __launch_bounds__(256) l2_back_kernel(const void *q, const void *k, int64_t qs, int64_t ks, int Hqk,
                                                      int K, int l2norm, const float *dqn, const float *dkn,
                                                      float *dq, float *dk, int64_t rows) {
  const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= 2 * rows) return;
  if (r < rows) gdn_bwd::l2_back_row(q, qs, Hqk, K, l2norm, DevLoad<T>{}, dqn, dq, r);
  else gdn_bwd::l2_back_row(k, ks, Hqk, K, l2norm, DevLoad<T>{}, dkn, dk, r - rows);
}

constexpr size_t kHeader = 256;

size_t bwd_workspace_bytes(int64_t n_tok, int n_seqs, int Hqk, int Hv, int K, int V) {
  const size_t states = n_slots(n_tok, n_seqs) * (size_t)Hv * V * K * sizeof(float);
  const size_t acc = (size_t)n_tok * Hqk * K * sizeof(float);
  return kHeader + ((states + 255) / 256) * 256 + 2 * ((acc + 255) / 256) * 256;
}

bool bwd_shape_ok(const gdn_shape *sh) {
  if (!sh) return false;
  if (sh->dtype != GDN_F32 && sh->dtype != GDN_BF16) return false;
  if (sh->B <= 0 || sh->T < 0 || sh->n_seqs < 0 || sh->Hqk <= 0 || sh->Hv <= 0) return false;
  if (sh->Hv % sh->Hqk != 0) return false;
  if (!(sh->K == 32 || sh->K == 64 || sh->K == 128)) return false;
  if (sh->V % gdn_bwd::BV != 0 || sh->V <= 0 || sh->V > 256) return false;
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
  const size_t states_bytes = ((n_slots(n_tok, sh.n_seqs) * (size_t)sh.Hv * sh.V * sh.K * sizeof(float) + 255) / 256) * 256;
  const size_t acc_bytes = (((size_t)n_tok * sh.Hqk * sh.K * sizeof(float) + 255) / 256) * 256;
  gdn_bwd::Params p{};
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta; p.h0 = h0; p.dout = d_o; p.dhT = dh_T;
  p.cu = cu_seqlens;
  p.row_T = sh.T;
  p.n_tok = n_tok;
  p.Hqk = sh.Hqk; p.Hv = sh.Hv; p.K = sh.K; p.V = sh.V;
  p.qs = qs; p.ks = ks; p.vs = vs;
  p.scale = scale;
  p.l2norm = (flags & GDN_FLAG_QK_L2NORM) ? 1 : 0;
  p.vec8 = aligned(q, 16) && aligned(k, 16) && aligned(v, 16) && qs % 8 == 0 && ks % 8 == 0 && vs % 8 == 0 &&
           (sh.dtype == GDN_BF16 || (qs % 4 == 0 && ks % 4 == 0 && vs % 4 == 0));
  p.states = (float *)(ws + kHeader);
  p.dqn = (float *)(ws + kHeader + states_bytes);
  p.dkn = (float *)(ws + kHeader + states_bytes + acc_bytes);
  p.dv = dv; p.dg = dg; p.dbeta = dbeta; p.dh0 = dh0;
  p.status = (int32_t *)workspace;
  // the accumulated outputs start at zero; dv too, so tokens outside every sequence read 0
  const size_t tok_hk = (size_t)n_tok * sh.Hqk * sh.K * sizeof(float);
  const size_t tok_h = (size_t)n_tok * sh.Hv * sizeof(float);
  if (n_tok > 0 &&
      (cudaMemsetAsync(p.dqn, 0, tok_hk, st) != cudaSuccess || cudaMemsetAsync(p.dkn, 0, tok_hk, st) != cudaSuccess ||
       cudaMemsetAsync(dg, 0, tok_h, st) != cudaSuccess || cudaMemsetAsync(dbeta, 0, tok_h, st) != cudaSuccess ||
       cudaMemsetAsync(dv, 0, (size_t)n_tok * sh.Hv * sh.V * sizeof(float), st) != cudaSuccess))
    return GDN_ERR_CUDA;
  const size_t smem = gdn_bwd::smem_floats(sh.K) * sizeof(float);
  const dim3 grid((unsigned)(sh.V / gdn_bwd::BV), (unsigned)sh.Hv, (unsigned)sh.n_seqs);
  const int64_t rows = n_tok * sh.Hqk;
  const unsigned lgrid = (unsigned)((2 * rows + 255) / 256);
  if (sh.dtype == GDN_BF16) {
    const gdn_status r = launch_bwd_k<__nv_bfloat16>(p, grid, smem, st);
    if (r != GDN_OK) return r;
    if (rows > 0)
      l2_back_kernel<__nv_bfloat16><<<lgrid, 256, 0, st>>>(q, k, qs, ks, sh.Hqk, sh.K, p.l2norm, p.dqn, p.dkn, dq,
                                                           dk, rows);
  } else {
    const gdn_status r = launch_bwd_k<float>(p, grid, smem, st);
    if (r != GDN_OK) return r;
    if (rows > 0)
      l2_back_kernel<float><<<lgrid, 256, 0, st>>>(q, k, qs, ks, sh.Hqk, sh.K, p.l2norm, p.dqn, p.dkn, dq, dk, rows);
  }
  return launch_status();
}
