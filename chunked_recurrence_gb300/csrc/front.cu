// front.cu -- the elementwise / stencil steps in front of the recurrence
// (gate prep, varlen causal conv1d, cu_seqlens from position_ids), the fp32
// chain reduce of segment summaries, and the small ABI helpers.
#include <math.h>

#include <algorithm>

#include "common.cuh"
#include "conv_tap.cuh"
#include "gates.cuh"
#include "sm100.cuh"

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
  const size_t n = workspace_bytes >= 2 * sizeof(int32_t) ? 2 * sizeof(int32_t) : sizeof(int32_t);
  if (cudaMemsetAsync(workspace, 0, n, (cudaStream_t)stream) != cudaSuccess) return GDN_ERR_CUDA;
  return GDN_OK;
}

extern "C" gdn_status gdn_workspace_path(const void *workspace, int32_t *path_out, void *stream) {
  if (!workspace || !path_out) return GDN_ERR_INVALID_ARG;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, (const int32_t *)workspace + 1, sizeof(v), cudaMemcpyDeviceToHost,
                      (cudaStream_t)stream) != cudaSuccess ||
      cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess)
    return GDN_ERR_CUDA;
  *path_out = v;
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

// The bf16 conv with its input staged in shared memory.  A block owns 1024 channels (eight
// a thread) of a run of tokens; whole token rows of those channels (2 KB each) arrive by bulk
// async copies into a ring of kStages stages of kStageRows rows, each stage with its own
// mbarrier, so three stages of loads stay in flight while the block computes on the fourth.
// The run starts W-1 tokens early (at most back to its sequence's start) so the history
// comes through the same ring.  Runs are sized so that the grid is about one wave of
// resident blocks.  Each row's arithmetic is conv_row8 (packed fp32x2 taps in the scalar
// chain's order, SiLU on the hardware exponential and reciprocal), which the chunk operand
// kernel's fused front end shares.  A wait that gives up (only a failed copy can make it)
// leaves NaN in the outputs the block did not compute.
constexpr int kStageRows = 8, kStages = 4, kStagedCols = 1024;
constexpr uint32_t kStagedSmem = kStages * kStageRows * kStagedCols * 2;
constexpr uint32_t kConvSpin = 1u << 22;

// The layer's gates, computed by the conv's blocks over their run of tokens, the elements of
// a run spread over its channel blocks (gdn_layer_fwd): the same values as gdn_gate_prep, one
// launch fewer.
struct ConvGates {
  const __nv_bfloat16 *a, *b;  // [n_tok][Hv]
  const float *A_log, *dt_bias;
  float *g, *beta;
  int Hv;
};

template <int W>
__global__ void __launch_bounds__(128, 3) conv1d_staged_kernel(const __nv_bfloat16 *__restrict__ x,
                                                               const __nv_bfloat16 *__restrict__ w,
                                                               const __nv_bfloat16 *__restrict__ bias,
                                                               const int32_t *__restrict__ cu, int n_seqs,
                                                               int64_t row_T, int64_t n_tok, int C, int run,
                                                               int act, __nv_bfloat16 *__restrict__ y,
                                                               const ConvGates gates) {
  using namespace gdn::sm100;
  constexpr int VEC = 8, HW = W > 1 ? W - 1 : 1;
  extern __shared__ __align__(128) uint4 ring[];  // [kStages][kStageRows][kStagedCols / 8]
  __shared__ __align__(8) uint64_t full[kStages];
  const int tid = threadIdx.x;
  const int cbase = blockIdx.y * kStagedCols, c0 = cbase + tid * VEC;
  const bool mine = c0 < C;
  const uint32_t row_bytes = (uint32_t)min(kStagedCols, C - cbase) * 2;
  const int64_t t0 = (int64_t)blockIdx.x * run;
  if (t0 >= n_tok) return;
  const int64_t t1 = min(t0 + (int64_t)run, n_tok);
  if (gates.g) {  // the run's gates, spread over its channel blocks
    const int64_t n_g = (t1 - t0) * gates.Hv;
    for (int64_t e = (int64_t)blockIdx.y * blockDim.x + tid; e < n_g; e += (int64_t)gridDim.y * blockDim.x) {
      const int64_t i = t0 * gates.Hv + e;
      const int hh = (int)(i % gates.Hv);
      gdn_gates(__bfloat162float(gates.a[i]), __bfloat162float(gates.b[i]), gates.A_log[hh], gates.dt_bias[hh],
                gates.g[i], gates.beta[i]);
    }
  }
  int s = 0;
  int64_t start, end;
  if (cu) {
    s = seq_of_token(cu, n_seqs, t0);
    while (s + 1 < n_seqs && (int64_t)cu[s + 1] <= t0) ++s;  // skip empty sequences
    start = max((int64_t)cu[s], (int64_t)0);
    end = cu[s + 1];
  } else {
    start = (t0 / row_T) * row_T;
    end = start + row_T;
  }
  // loaded rows: the history tokens of t0 inside its sequence, then the run
  const int64_t ts = max(t0 - (W - 1), min(start, t0));
  const int nst = (int)((t1 - ts + kStageRows - 1) / kStageRows);
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto issue = [&](int k) {  // stage k: rows ts + k kStageRows ...
    const int st = k % kStages;
    const int64_t a = ts + (int64_t)k * kStageRows;
    const int m = (int)min((int64_t)kStageRows, t1 - a);
    mbar_arrive_expect_tx(&full[st], (uint32_t)m * row_bytes);
    for (int i = 0; i < m; ++i)
      bulk_load(ring + (st * kStageRows + i) * (kStagedCols / 8), x + (a + i) * C + cbase, row_bytes, &full[st]);
  };
  if (tid == 0)
    for (int k = 0; k < min(kStages, nst); ++k) issue(k);
  // taps, bias and history as fp32 pairs (channels c0 + 2i, c0 + 2i + 1)
  uint64_t wt[W][VEC / 2], bs[VEC / 2], hist[HW][VEC / 2];
#pragma unroll
  for (int i = 0; i < VEC / 2; ++i) {
    const int64_t ca = c0 + 2 * i, cb = ca + 1;
#pragma unroll
    for (int j = 0; j < W; ++j)
      wt[j][i] = mine ? f2_pack(to_f32(w[ca * W + j]), to_f32(w[cb * W + j])) : 0ull;
    bs[i] = (mine && bias) ? f2_pack(to_f32(bias[ca]), to_f32(bias[cb])) : 0ull;
#pragma unroll
    for (int j = 0; j < HW; ++j) hist[j][i] = 0ull;
  }
  int k = 0;
  for (; k < nst; ++k) {
    const int st = k % kStages;
    const bool ok = mbar_wait(&full[st], (uint32_t)(k / kStages) & 1, kConvSpin);
    if (__syncthreads_or(!ok)) break;
    const int64_t a = ts + (int64_t)k * kStageRows;
    const int m = (int)min((int64_t)kStageRows, t1 - a);
    const uint4 *rows = ring + st * kStageRows * (kStagedCols / 8) + tid;
    // one token row: its conv output (when `emit`) and the history shift
    auto conv_row = [&](const uint4 &raw, int64_t t, bool emit) {
      uint64_t cur[VEC / 2];
      unpack8p(raw, cur);
      if (emit) {
        uint64_t out[VEC / 2];
        conv_row8p<W, HW>(wt, bs, hist, cur, act != 0, out);
        *reinterpret_cast<uint4 *>(y + t * C + c0) = pack8p(out);
      }
      if (W > 1) conv_shift8p<HW>(hist, cur);
    };
    if (m == kStageRows && a >= t0 && a + kStageRows <= end && mine) {
      // the whole stage lies inside one sequence and past the history rows: straight-line
      // rows with no per-row test, so the rows' arithmetic can interleave
      uint4 raw[kStageRows];
#pragma unroll
      for (int i = 0; i < kStageRows; ++i) raw[i] = rows[i * (kStagedCols / 8)];
#pragma unroll
      for (int i = 0; i < kStageRows; ++i) conv_row(raw[i], a + i, true);
    } else {
#pragma unroll
      for (int i = 0; i < kStageRows; ++i) {
        if (i >= m) break;
        const int64_t t = a + i;
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
          for (int j = 0; j < HW; ++j)
#pragma unroll
            for (int v = 0; v < VEC / 2; ++v) hist[j][v] = 0ull;
        }
        conv_row(rows[i * (kStagedCols / 8)], t, t >= t0 && mine);
      }
    }
    __syncthreads();  // every read of stage st is done before it is refilled
    if (tid == 0 && k + kStages < nst) issue(k + kStages);
  }
  if (k < nst) {  // a wait gave up: NaN where nothing was computed, and the copies land first
    if (mine) {
      float nan[VEC];
#pragma unroll
      for (int v = 0; v < VEC; ++v) nan[v] = __int_as_float(0x7fc00000);
      for (int64_t t = max(t0, ts + (int64_t)k * kStageRows); t < t1; ++t) Vec<__nv_bfloat16, VEC>::store(y + t * C + c0, nan);
    }
    if (tid == 0)
      for (int j = k; j < min(nst, k + kStages); ++j) (void)mbar_wait(&full[j % kStages], (uint32_t)(j / kStages) & 1, kConvSpin);
    __syncthreads();
  }
}

// Launches the staged bf16 conv; returns false (nothing launched) where it does not apply.
static bool launch_conv_staged(int W, cudaStream_t st, const __nv_bfloat16 *x, const __nv_bfloat16 *w,
                               const __nv_bfloat16 *bias, const int32_t *cu, int n_seqs, int64_t row_T,
                               int64_t n_tok, int C, int act, __nv_bfloat16 *y, gdn_status *status,
                               const ConvGates &gates = ConvGates{}) {
  int dev = 0, sms = 0, smem_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess) {
    *status = GDN_ERR_CUDA;
    return true;
  }
  const int64_t ncb = (C + kStagedCols - 1) / kStagedCols;
  if (ncb > 65535) return false;
  const int per_sm = std::max(1, std::min(3, smem_sm / (int)(kStagedSmem + 1024)));
  const int64_t per_wave = std::max<int64_t>(1, (int64_t)sms * per_sm / ncb);  // runs in one wave
  const int64_t run = std::max<int64_t>(16, (n_tok + per_wave - 1) / per_wave);
  if (run > 2147483647LL) return false;
  const dim3 grid((unsigned)((n_tok + run - 1) / run), (unsigned)ncb);
#define GDN_STAGED_CASE(WW)                                                                          \
  case WW:                                                                                           \
    if (cudaFuncSetAttribute(conv1d_staged_kernel<WW>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             (int)kStagedSmem) != cudaSuccess) {                                     \
      *status = GDN_ERR_CUDA;                                                                        \
      return true;                                                                                   \
    }                                                                                                \
    conv1d_staged_kernel<WW><<<grid, 128, kStagedSmem, st>>>(x, w, bias, cu, n_seqs, row_T, n_tok, C, \
                                                             (int)run, act, y, gates);               \
    break;
  switch (W) {
    GDN_STAGED_CASE(1) GDN_STAGED_CASE(2) GDN_STAGED_CASE(3) GDN_STAGED_CASE(4)
    GDN_STAGED_CASE(5) GDN_STAGED_CASE(6)
    default: return false;  // wider convs hold more history than fit 3 blocks an SM: the register kernel
  }
#undef GDN_STAGED_CASE
  *status = launch_status();
  return true;
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

namespace gdn {

// gdn_layer_fwd's front steps: the conv (SiLU) and the gates.  bf16 with the staged conv
// takes both in one launch; otherwise gdn_gate_prep and gdn_conv1d_varlen run.
gdn_status layer_conv_and_gates(const void *x, const void *w, const void *bias, int32_t dtype,
                                const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens, int32_t C,
                                int32_t width, void *y, const void *a, const void *b, const float *A_log,
                                const float *dt_bias, int32_t Hv, float *g, float *beta, void *stream) {
  const bool staged = dtype == GDN_BF16 && n_tokens > 0 && width >= 1 && width <= 6 && C % 8 == 0 &&
                      aligned(x, 16) && aligned(y, 16) && n_seqs >= 1 && (cu_seqlens || n_tokens % n_seqs == 0) &&
                      a && b && A_log && dt_bias && g && beta && Hv > 0;
  if (staged) {
    const int64_t row_T = cu_seqlens ? 0 : n_tokens / n_seqs;
    const ConvGates gates{(const __nv_bfloat16 *)a, (const __nv_bfloat16 *)b, A_log, dt_bias, g, beta, Hv};
    gdn_status st = GDN_OK;
    if (launch_conv_staged(width, (cudaStream_t)stream, (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)w,
                           (const __nv_bfloat16 *)bias, cu_seqlens, n_seqs, row_T, n_tokens, C, 1,
                           (__nv_bfloat16 *)y, &st, gates))
      return st;
  }
  gdn_status st = gdn_gate_prep(a, b, dtype, A_log, dt_bias, n_tokens, Hv, g, beta, stream);
  if (st != GDN_OK) return st;
  return gdn_conv1d_varlen(x, w, bias, dtype, cu_seqlens, n_seqs, n_tokens, C, width, 1, y, stream);
}

}  // namespace gdn

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
    gdn_status staged = GDN_OK;
    if (vec && launch_conv_staged(width, st, (const T *)x, (const T *)w, (const T *)bias, cu_seqlens, n_seqs,
                                  row_T, n_tokens, C, act, (T *)y, &staged))
      return staged;
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
// kChainRows rows of one head's state and walks the segments in order.  Each thread
// keeps a 2-row x 4-column tile of the product (8 independent sums; one float4 of M
// feeds 8 FMAs), and the next segment's K x K transition streams into the second of two
// shared-memory buffers (cp.async) while the current one is used.
constexpr int kChainRows = 16;

__global__ void __launch_bounds__(256) chain_reduce_kernel(const float *__restrict__ M,
                                                           const float *__restrict__ S_local,
                                                           const float *__restrict__ h0, int n_seg,
                                                           int Hv, int K, int V,
                                                           float *__restrict__ S_start,
                                                           float *__restrict__ h_T) {
  extern __shared__ float4 sm4[];
  float *Ms = reinterpret_cast<float *>(sm4);  // 2 x K * K
  float *Sr = Ms + 2 * (size_t)K * K;         // kChainRows * K
  const int tid = threadIdx.x;
  const int h = blockIdx.y, r0 = blockIdx.x * kChainRows;
  const int rows = min(kChainRows, V - r0);
  const int cg = tid & 31, rg = tid >> 5;     // columns 4 cg .. 4 cg + 3, rows 2 rg, 2 rg + 1
  const int c0 = 4 * cg;
  const bool col_ok = c0 < K;                  // K is a multiple of 4 (32, 64 or 128)
  const int n4 = K * K / 4;
  auto prefetch = [&](int i, int buf) {
    const float4 *src = reinterpret_cast<const float4 *>(M + ((size_t)i * Hv + h) * K * K);
    float4 *dst = reinterpret_cast<float4 *>(Ms + (size_t)buf * K * K);
    for (int idx = tid; idx < n4; idx += blockDim.x) cp_async16(dst + idx, src + idx);
    cp_async_commit();
  };
  if (n_seg > 0) prefetch(0, 0);
  for (int idx = tid; idx < kChainRows * K; idx += blockDim.x) {
    const int r = idx / K, c = idx % K;
    Sr[idx] = (r < rows && h0) ? h0[((size_t)h * V + r0 + r) * K + c] : 0.f;
  }
  for (int i = 0; i < n_seg; ++i) {
    const size_t base = ((size_t)i * Hv + h) * V * K;
    cp_async_wait_all();
    __syncthreads();  // M_i and the rows are in place; the other buffer is free
    if (i + 1 < n_seg) prefetch(i + 1, (i + 1) & 1);
    for (int idx = tid; idx < rows * K; idx += blockDim.x) {
      const int r = idx / K, c = idx % K;
      S_start[base + (size_t)(r0 + r) * K + c] = Sr[idx];
    }
    const float *Mi = Ms + (size_t)(i & 1) * K * K;
    float acc[2][4];
    const int ra = 2 * rg, rb = 2 * rg + 1;
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) acc[e][cc] = 0.f;
    if (col_ok && ra < rows) {
      const float4 la = *reinterpret_cast<const float4 *>(S_local + base + (size_t)(r0 + ra) * K + c0);
      acc[0][0] = la.x; acc[0][1] = la.y; acc[0][2] = la.z; acc[0][3] = la.w;
      if (rb < rows) {
        const float4 lb = *reinterpret_cast<const float4 *>(S_local + base + (size_t)(r0 + rb) * K + c0);
        acc[1][0] = lb.x; acc[1][1] = lb.y; acc[1][2] = lb.z; acc[1][3] = lb.w;
      }
      const float *sa = Sr + ra * K, *sb = Sr + rb * K;
#pragma unroll 8
      for (int m = 0; m < K; ++m) {
        const float4 mv = *reinterpret_cast<const float4 *>(Mi + (size_t)m * K + c0);
        const float xa = sa[m], xb = sb[m];
        acc[0][0] = fmaf(xa, mv.x, acc[0][0]);
        acc[0][1] = fmaf(xa, mv.y, acc[0][1]);
        acc[0][2] = fmaf(xa, mv.z, acc[0][2]);
        acc[0][3] = fmaf(xa, mv.w, acc[0][3]);
        acc[1][0] = fmaf(xb, mv.x, acc[1][0]);
        acc[1][1] = fmaf(xb, mv.y, acc[1][1]);
        acc[1][2] = fmaf(xb, mv.z, acc[1][2]);
        acc[1][3] = fmaf(xb, mv.w, acc[1][3]);
      }
    }
    __syncthreads();  // every read of Sr is done
    if (col_ok && ra < rows) {
      *reinterpret_cast<float4 *>(Sr + ra * K + c0) = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
      if (rb < rows)
        *reinterpret_cast<float4 *>(Sr + rb * K + c0) = make_float4(acc[1][0], acc[1][1], acc[1][2], acc[1][3]);
    }
  }
  __syncthreads();
  if (h_T)
    for (int idx = tid; idx < rows * K; idx += blockDim.x) {
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
  if (K % 4 != 0) return GDN_ERR_UNSUPPORTED;
  if (!aligned(M, 16) || !aligned(S_local, 16) || !aligned(S_start, 16)) return GDN_ERR_INVALID_ARG;
  const size_t smem = (2 * (size_t)K * K + (size_t)kChainRows * K) * sizeof(float);
  if (cudaFuncSetAttribute(chain_reduce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return GDN_ERR_CUDA;
  const dim3 grid((V + kChainRows - 1) / kChainRows, Hv);
  chain_reduce_kernel<<<grid, 256, smem, (cudaStream_t)stream>>>(M, S_local, h0, n_seg, Hv, K, V,
                                                                 S_start, h_T);
  return launch_status();
}
