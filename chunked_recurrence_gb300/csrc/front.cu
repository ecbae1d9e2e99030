// front.cu -- the elementwise / stencil steps in front of the recurrence
// (gate prep, varlen causal conv1d, cu_seqlens from position_ids), the fp32
// chain reduce of segment summaries, and the small ABI helpers.
#include <math.h>

#include "common.cuh"
#include "gates.cuh"

using namespace gdn;

// ----------------------------------------------------------------- helpers

extern "C" const char *gdn_status_string(int status) {
  switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
    case GDN_ERR_BOUNDS: return "GDN_ERR_BOUNDS";
    default: return "GDN_ERR_UNKNOWN";
  }
}

extern "C" int32_t gdn_version(void) { return (1 << 16) | 2; }

extern "C" gdn_status gdn_workspace_reset(void *workspace, size_t workspace_bytes, void *stream) {
  if (!workspace || workspace_bytes < sizeof(int32_t)) return GDN_ERR_WORKSPACE;
  if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), (cudaStream_t)stream) != cudaSuccess)
    return GDN_ERR_CUDA;
  return GDN_OK;
}

extern "C" gdn_status gdn_workspace_status(const void *workspace, int32_t *status_out, void *stream) {
  if (!workspace || !status_out) return GDN_ERR_INVALID_ARG;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, (cudaStream_t)stream) !=
      cudaSuccess)
    return GDN_ERR_CUDA;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GDN_ERR_CUDA;
  *status_out = v;
  return GDN_OK;
}

// --------------------------------------------------------------- gate prep

// g = -exp(A_log[h]) * softplus(a + dt_bias[h]), beta = sigmoid(b), 4 elements a thread.
template <typename T>
__global__ void __launch_bounds__(256) gate_prep_kernel(const T *__restrict__ a, const T *__restrict__ b,
                                                        const float *__restrict__ A_log,
                                                        const float *__restrict__ dt_bias, int64_t n,
                                                        int Hv, float *__restrict__ g,
                                                        float *__restrict__ beta) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x * 4;
  for (int64_t i0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; i0 < n; i0 += stride) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u;
      if (i < n) {
        const int h = (int)(i % Hv);
        gdn_gates(to_f32(a[i]), to_f32(b[i]), A_log[h], dt_bias[h], g[i], beta[i]);
      }
    }
  }
}

extern "C" gdn_status gdn_gate_prep(const void *a, const void *b, int32_t ab_dtype,
                                    const float *A_log, const float *dt_bias, int64_t n_tokens,
                                    int32_t Hv, float *g, float *beta, void *stream) {
  if (n_tokens < 0 || Hv <= 0) return GDN_ERR_INVALID_ARG;
  if (ab_dtype != GDN_F32 && ab_dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (n_tokens == 0) return GDN_OK;
  if (!a || !b || !A_log || !dt_bias || !g || !beta) return GDN_ERR_INVALID_ARG;
  const int64_t n = n_tokens * Hv;
  const int threads = 256;
  int64_t blocks = (n + threads * 4 - 1) / (threads * 4);
  if (blocks > 152 * 16) blocks = 152 * 16;
  cudaStream_t st = (cudaStream_t)stream;
  if (ab_dtype == GDN_BF16)
    gate_prep_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, st>>>(
        (const __nv_bfloat16 *)a, (const __nv_bfloat16 *)b, A_log, dt_bias, n, Hv, g, beta);
  else
    gate_prep_kernel<float><<<(unsigned)blocks, threads, 0, st>>>((const float *)a, (const float *)b,
                                                                  A_log, dt_bias, n, Hv, g, beta);
  return launch_status();
}

// ------------------------------------------------------------------- conv

// Each thread owns VEC adjacent channels (16 bytes of input) and a run of
// kRun tokens, keeping the last W-1 inputs of its channels in registers.  At
// a sequence start the history is zero.  A warp covers 32 * 16 contiguous
// bytes of one token row, so loads and stores are fully coalesced.
constexpr int kRun = 32;
constexpr int kMaxW = 8;

template <typename T, int VEC>
struct Vec;
template <>
struct Vec<__nv_bfloat16, 8> {
  using raw = uint4;
  __device__ static raw load_raw(const __nv_bfloat16 *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }
  __device__ static void cvt(const raw &r, float *f) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(h[i]);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
  __device__ static void load(const __nv_bfloat16 *p, float *f) {
    const uint4 r = *reinterpret_cast<const uint4 *>(p);
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(h[i]);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
  __device__ static void store(__nv_bfloat16 *p, const float *f) {
    uint4 r;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&r);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    *reinterpret_cast<uint4 *>(p) = r;
  }
};
template <>
struct Vec<float, 4> {
  using raw = float4;
  __device__ static raw load_raw(const float *p) { return __ldg(reinterpret_cast<const float4 *>(p)); }
  __device__ static void cvt(const raw &r, float *f) {
    f[0] = r.x; f[1] = r.y; f[2] = r.z; f[3] = r.w;
  }
  __device__ static void load(const float *p, float *f) {
    const float4 r = *reinterpret_cast<const float4 *>(p);
    f[0] = r.x; f[1] = r.y; f[2] = r.z; f[3] = r.w;
  }
  __device__ static void store(float *p, const float *f) {
    *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
};
template <typename T>
struct Vec<T, 1> {
  using raw = T;
  __device__ static raw load_raw(const T *p) { return *p; }
  __device__ static void cvt(const raw &r, float *f) { f[0] = to_f32(r); }
  __device__ static void load(const T *p, float *f) { f[0] = to_f32(*p); }
  __device__ static void store(T *p, const float *f) { *p = from_f32<T>(f[0]); }
};

template <typename T, int VEC, int W>
__global__ void __launch_bounds__(128, 4) conv1d_kernel(const T *__restrict__ x, const T *__restrict__ w,
                                                     const T *__restrict__ bias,
                                                     const int32_t *__restrict__ cu, int n_seqs,
                                                     int64_t row_T, int64_t n_tok, int C, int act,
                                                     T *__restrict__ y) {
  const int c0 = (blockIdx.y * blockDim.x + threadIdx.x) * VEC;
  if (c0 >= C) return;
  const int64_t t0 = (int64_t)blockIdx.x * kRun;
  if (t0 >= n_tok) return;
  const int64_t t1 = min(t0 + (int64_t)kRun, n_tok);

  float wt[W][VEC], bs[VEC];
#pragma unroll
  for (int v = 0; v < VEC; ++v) {
#pragma unroll
    for (int j = 0; j < W; ++j) wt[j][v] = to_f32(w[(int64_t)(c0 + v) * W + j]);
    bs[v] = bias ? to_f32(bias[c0 + v]) : 0.f;
  }
  // sequence bounds of t0
  int s = 0;
  int64_t start, end;
  if (cu) {
    s = seq_of_token(cu, n_seqs, t0);
    while (s + 1 < n_seqs && (int64_t)cu[s + 1] <= t0) ++s;  // skip empty sequences
    start = max((int64_t)cu[s], (int64_t)0);  // a malformed cu_seqlens never makes a read go negative
    end = cu[s + 1];
  } else {
    start = (t0 / row_T) * row_T;
    end = start + row_T;
  }
  // history: hist[j] holds x[t - (W-1) + j] for j < W-1
  float hist[W > 1 ? W - 1 : 1][VEC];
#pragma unroll
  for (int j = 0; j < W - 1; ++j) {
    const int64_t src = t0 - (W - 1) + j;
    if (src >= start) Vec<T, VEC>::load(x + src * C + c0, hist[j]);
    else {
#pragma unroll
      for (int v = 0; v < VEC; ++v) hist[j][v] = 0.f;
    }
  }
  // tokens in batches of kAhead: all of a batch's loads are in flight before its first use
  constexpr int kAhead = 8;
  for (int64_t tb = t0; tb < t1; tb += kAhead) {
    typename Vec<T, VEC>::raw raw[kAhead];
#pragma unroll
    for (int u = 0; u < kAhead; ++u)
      if (tb + u < t1) raw[u] = Vec<T, VEC>::load_raw(x + (tb + u) * C + c0);
#pragma unroll
    for (int u = 0; u < kAhead; ++u) {
      const int64_t t = tb + u;
      if (t >= t1) break;
      if (t >= end) {  // a new sequence begins at t: zero history
        if (cu) {
          while (s + 1 < n_seqs && (int64_t)cu[s + 1] <= t) ++s;
          start = max((int64_t)cu[s], (int64_t)0);
          end = cu[s + 1];
        } else {
          start = t;
          end = t + row_T;
        }
#pragma unroll
        for (int j = 0; j < W - 1; ++j)
#pragma unroll
          for (int v = 0; v < VEC; ++v) hist[j][v] = 0.f;
      }
      float cur[VEC], out[VEC];
      Vec<T, VEC>::cvt(raw[u], cur);
#pragma unroll
      for (int v = 0; v < VEC; ++v) {
        float acc = bs[v];
#pragma unroll
        for (int j = 0; j < W - 1; ++j) acc = fmaf(wt[j][v], hist[j][v], acc);
        acc = fmaf(wt[W - 1][v], cur[v], acc);
        // SiLU with the fast exponential and division: their error (a few ulp of fp32) is
        // far below the rounding of y to the input dtype
        out[v] = act ? __fdividef(acc, 1.f + __expf(-acc)) : acc;
      }
      Vec<T, VEC>::store(y + t * C + c0, out);
#pragma unroll
      for (int j = 0; j + 1 < W - 1; ++j)
#pragma unroll
        for (int v = 0; v < VEC; ++v) hist[j][v] = hist[j + 1][v];
      if (W > 1) {
#pragma unroll
        for (int v = 0; v < VEC; ++v) hist[W > 1 ? W - 2 : 0][v] = cur[v];
      }
    }
  }
}

template <typename T, int VEC>
static void launch_conv_w(int W, dim3 grid, dim3 block, cudaStream_t st, const T *x, const T *w,
                          const T *bias, const int32_t *cu, int n_seqs, int64_t row_T,
                          int64_t n_tok, int C, int act, T *y) {
#define GDN_CONV_CASE(WW)                                                                 \
  case WW:                                                                                \
    conv1d_kernel<T, VEC, WW><<<grid, block, 0, st>>>(x, w, bias, cu, n_seqs, row_T, n_tok, \
                                                      C, act, y);                         \
    break;
  switch (W) {
    GDN_CONV_CASE(1) GDN_CONV_CASE(2) GDN_CONV_CASE(3) GDN_CONV_CASE(4)
    GDN_CONV_CASE(5) GDN_CONV_CASE(6) GDN_CONV_CASE(7) GDN_CONV_CASE(8)
    default: break;
  }
#undef GDN_CONV_CASE
}

extern "C" gdn_status gdn_conv1d_varlen(const void *x, const void *w, const void *bias, int32_t dtype,
                                        const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens,
                                        int32_t C, int32_t width, int32_t act, void *y, void *stream) {
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (n_tokens < 0 || C <= 0 || width < 1 || width > kMaxW || (act != 0 && act != 1))
    return GDN_ERR_INVALID_ARG;
  if (n_seqs < 0 || (n_tokens > 0 && n_seqs < 1)) return GDN_ERR_INVALID_ARG;
  if (n_tokens == 0) return GDN_OK;
  if (!x || !w || !y) return GDN_ERR_INVALID_ARG;
  if (!cu_seqlens && n_tokens % n_seqs != 0) return GDN_ERR_INVALID_ARG;
  const int64_t row_T = cu_seqlens ? 0 : n_tokens / n_seqs;
  const int64_t runs = (n_tokens + kRun - 1) / kRun;
  if (runs > 2147483647LL) return GDN_ERR_UNSUPPORTED;
  cudaStream_t st = (cudaStream_t)stream;
  const dim3 block(128);
  if (dtype == GDN_BF16) {
    using T = __nv_bfloat16;
    const bool vec = (C % 8 == 0) && aligned(x, 16) && aligned(y, 16);
    const int per = vec ? 8 : 1;
    const dim3 grid((unsigned)runs, (unsigned)((C / per + 127) / 128));
    if (grid.y > 65535u) return GDN_ERR_UNSUPPORTED;
    if (vec)
      launch_conv_w<T, 8>(width, grid, block, st, (const T *)x, (const T *)w, (const T *)bias,
                          cu_seqlens, n_seqs, row_T, n_tokens, C, act, (T *)y);
    else
      launch_conv_w<T, 1>(width, grid, block, st, (const T *)x, (const T *)w, (const T *)bias,
                          cu_seqlens, n_seqs, row_T, n_tokens, C, act, (T *)y);
  } else {
    using T = float;
    const bool vec = (C % 4 == 0) && aligned(x, 16) && aligned(y, 16);
    const int per = vec ? 4 : 1;
    const dim3 grid((unsigned)runs, (unsigned)((C / per + 127) / 128));
    if (grid.y > 65535u) return GDN_ERR_UNSUPPORTED;
    if (vec)
      launch_conv_w<T, 4>(width, grid, block, st, (const T *)x, (const T *)w, (const T *)bias,
                          cu_seqlens, n_seqs, row_T, n_tokens, C, act, (T *)y);
    else
      launch_conv_w<T, 1>(width, grid, block, st, (const T *)x, (const T *)w, (const T *)bias,
                          cu_seqlens, n_seqs, row_T, n_tokens, C, act, (T *)y);
  }
  return launch_status();
}

// -------------------------------------------------- cu_seqlens from position_ids

// One block walks the token axis in tiles of blockDim.x tokens; a sample
// starts at token 0 and wherever position_ids is 0.  Start offsets are
// compacted in order with a block-wide exclusive scan of the start flags.
__global__ void __launch_bounds__(1024) cu_from_pos_kernel(const int64_t *__restrict__ pos, int64_t n,
                                                           int32_t *__restrict__ cu,
                                                           int32_t *__restrict__ n_seqs) {
  __shared__ int warp_off[32];
  __shared__ int base;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if (threadIdx.x == 0) base = 0;
  __syncthreads();
  for (int64_t t0 = 0; t0 < n; t0 += blockDim.x) {
    const int64_t t = t0 + threadIdx.x;
    const int flag = (t < n) && (t == 0 || pos[t] == 0);
    const unsigned m = __ballot_sync(0xffffffffu, flag);
    const int in_warp = __popc(m & ((1u << lane) - 1u));
    if (lane == 0) warp_off[wid] = __popc(m);
    __syncthreads();
    if (wid == 0) {
      const int v = lane < nw ? warp_off[lane] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      if (lane < nw) warp_off[lane] = incl - v;
    }
    __syncthreads();
    const int idx = base + warp_off[wid] + in_warp;
    if (flag) cu[idx] = (int32_t)t;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) base = idx + flag;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    cu[base] = (int32_t)n;
    *n_seqs = base;
  }
}

extern "C" gdn_status gdn_cu_seqlens_from_position_ids(const int64_t *position_ids, int64_t n_tokens,
                                                       int32_t *cu_seqlens, int32_t *n_seqs,
                                                       void *stream) {
  if (n_tokens < 0 || n_tokens > 2147483647LL) return GDN_ERR_INVALID_ARG;
  if (!cu_seqlens || !n_seqs || (n_tokens > 0 && !position_ids)) return GDN_ERR_INVALID_ARG;
  cu_from_pos_kernel<<<1, 1024, 0, (cudaStream_t)stream>>>(position_ids, n_tokens, cu_seqlens,
                                                           n_seqs);
  return launch_status();
}

// ------------------------------------------------------------ chain reduce

// S_start[0] = h0; S_start[i+1] = S_start[i] M_i + S_local_i, in fp32 FFMA.
// Rows of S evolve independently (row a: s_a <- s_a M + l_a), so a block owns
// kChainRows rows of one head's state and walks the segments in order, with
// the segment's K x K transition staged in shared memory.
constexpr int kChainRows = 8;

__global__ void __launch_bounds__(256) chain_reduce_kernel(const float *__restrict__ M,
                                                           const float *__restrict__ S_local,
                                                           const float *__restrict__ h0, int n_seg,
                                                           int Hv, int K, int V,
                                                           float *__restrict__ S_start,
                                                           float *__restrict__ h_T) {
  extern __shared__ float sm[];
  float *Ms = sm;                   // K * K
  float *Sr = Ms + (size_t)K * K;   // kChainRows * K
  const int h = blockIdx.y, r0 = blockIdx.x * kChainRows;
  const int rows = min(kChainRows, V - r0);
  for (int idx = threadIdx.x; idx < kChainRows * K; idx += blockDim.x) {
    const int r = idx / K, c = idx % K;
    Sr[idx] = (r < rows && h0) ? h0[((size_t)h * V + r0 + r) * K + c] : 0.f;
  }
  __syncthreads();
  for (int i = 0; i < n_seg; ++i) {
    const float *Mi = M + ((size_t)i * Hv + h) * K * K;
    for (int idx = threadIdx.x; idx < K * K; idx += blockDim.x) Ms[idx] = Mi[idx];
    const size_t base = ((size_t)i * Hv + h) * V * K;
    for (int idx = threadIdx.x; idx < rows * K; idx += blockDim.x) {
      const int r = idx / K, c = idx % K;
      S_start[base + (size_t)(r0 + r) * K + c] = Sr[idx];
    }
    __syncthreads();
    float acc[(kChainRows * 128 + 255) / 256];
    int n_out = 0;
    for (int idx = threadIdx.x; idx < rows * K; idx += blockDim.x, ++n_out) {
      const int r = idx / K, c = idx % K;
      float a = S_local[base + (size_t)(r0 + r) * K + c];
      const float *srow = Sr + r * K;
      for (int m = 0; m < K; ++m) a = fmaf(srow[m], Ms[m * K + c], a);
      acc[n_out] = a;
    }
    __syncthreads();
    n_out = 0;
    for (int idx = threadIdx.x; idx < rows * K; idx += blockDim.x, ++n_out) Sr[idx] = acc[n_out];
    __syncthreads();
  }
  if (h_T)
    for (int idx = threadIdx.x; idx < rows * K; idx += blockDim.x) {
      const int r = idx / K, c = idx % K;
      h_T[((size_t)h * V + r0 + r) * K + c] = Sr[idx];
    }
}

extern "C" gdn_status gdn_chain_reduce(const float *M, const float *S_local, const float *h0,
                                       int32_t n_seg, int32_t Hv, int32_t K, int32_t V,
                                       float *S_start, float *h_T, void *stream) {
  if (n_seg < 0 || Hv <= 0 || K <= 0 || V <= 0) return GDN_ERR_INVALID_ARG;
  if (K > 128) return GDN_ERR_UNSUPPORTED;
  if (n_seg > 0 && (!M || !S_local || !S_start)) return GDN_ERR_INVALID_ARG;
  if (n_seg == 0 && !h_T) return GDN_OK;
  const size_t smem = ((size_t)K * K + (size_t)kChainRows * K) * sizeof(float);
  if (cudaFuncSetAttribute(chain_reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return GDN_ERR_CUDA;
  const dim3 grid((V + kChainRows - 1) / kChainRows, Hv);
  chain_reduce_kernel<<<grid, 256, smem, (cudaStream_t)stream>>>(M, S_local, h0, n_seg, Hv, K, V,
                                                                 S_start, h_T);
  return launch_status();
}
