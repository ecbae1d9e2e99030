// chunk_tc.cu -- tensor-core path of gdn_chunk_fwd for bf16 inputs (K = 128),
// tcgen05 MMAs with TMEM accumulators, TMA-staged 64-token tiles.
//
// The chunk form (UT/WY transform of the gated delta rule, "Gated Delta
// Networks", chunkwise algorithm), per chunk of C = 64 tokens, v-head h and
// start state S (V x K, fp32), with unit-norm keys/queries k_hat = k / |k|:
//   gamma = inclusive cumsum of g,  b = exp(gamma),  d = exp(gamma_last - gamma)
//   A  = strictly-lower(diag(beta) K_hat K_hat^T * Gamma),  Gamma_ij = exp(gamma_i - gamma_j)
//   T  = (I + A)^-1 diag(beta)
//   W  = T diag(b) K_hat,  U = T V,  U' = U - W S^T
//   O  = scale diag(b) Q_hat S^T + P U',  P = scale (Q_hat K_hat^T * Gamma), j <= i
//   S <- b_last S + U'^T diag(d) K_hat
//
// Precision: the bf16 inputs q, k, v are exact bf16 values, so the MMAs read
// them unchanged and the 1/|q|, 1/|k| factors are applied in fp32 where they
// are cheapest (inside A and P, and folded into operands that are rounded to
// bf16 anyway).  T is kept in fp32 between the kernels and enters the MMAs as
// a hi + lo pair of bf16 matrices; the diagonal of P (the largest term of
// the largest outputs) is added in fp32 outside the MMA.
//
// Two kernels:
//  * chunk_prep_kernel (fully parallel over chunk x q/k head): K K^T on the
//    tensor core, then per v-head the 64 x 64 forward substitution for T in
//    fp32 on CUDA cores; T is written packed (lower triangle incl. diagonal,
//    fp32, 8320 bytes per chunk and v-head) to the workspace.  It is the only
//    state-independent step that is sequential inside a chunk, so it runs off
//    the state chain.
//  * chunk_tc_kernel (one block per sequence x v-head x 32 value columns):
//    walks the chunks in order with the fp32 state transposed in registers
//    (thread f holds row f of S^T, one TMEM lane per key feature), TMA
//    prefetching chunk c+1 while chunk c runs, and every contraction on
//    tcgen05: Q K^T, W, U, U' = U - W S^T, Q S^T, P U', K^T diag(d) U'.
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "sm100.cuh"

using namespace gdn;
using namespace gdn::sm100;

namespace {

constexpr int C = kChunk;   // 64 tokens per chunk
constexpr int KD = 128;     // key width handled by this path
constexpr int BVT = 32;     // value columns per block (N of the chain MMAs)
constexpr int NT = 128;     // threads per block: one per TMEM lane
constexpr uint32_t kSpin = 1u << 22;  // bounded waits (~0.2 s) before reporting a timeout

// ---------------------------------------------------------------- workspace
// [0, 256): status word.  Then T for (slot, v-head): the lower triangle of the
// 64 x 64 fp32 matrix including its diagonal, row by row (entry (i, j) at
// i(i+1)/2 + j).  Chunk c of sequence s (start token t_s) uses slot
// s + floor(t_s / 64) + c, which is unique over all chunks and below
// n_seqs + ceil(n_tok / 64).
constexpr size_t kWsHeader = 256;
constexpr int kTPacked = C * (C + 1) / 2;                  // 2080 floats
constexpr size_t kTBytes = (size_t)kTPacked * sizeof(float);  // 8320 bytes, a multiple of 16

inline size_t n_slots(int64_t n_tok, int n_seqs) { return (size_t)n_seqs + (size_t)((n_tok + C - 1) / C); }

__device__ __forceinline__ void seq_range(const int32_t *cu, int64_t row_T, int s, int64_t &start,
                                          int64_t &end) {
  if (cu) {
    start = cu[s];
    end = cu[s + 1];
  } else {
    start = (int64_t)s * row_T;
    end = start + row_T;
  }
}

__device__ __forceinline__ int64_t slot_base(const int32_t *cu, int64_t row_T, int s) {
  const int64_t st = cu ? (int64_t)cu[s] : (int64_t)s * row_T;
  return (int64_t)s + st / C;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&u);
  return __bfloat1622float2(h);
}

// ============================================================ prep kernel

struct PrepParams {
  const __nv_bfloat16 *k;
  int64_t ks;  // token stride of k (elements)
  const float *g, *beta;
  const int32_t *cu;
  int64_t row_T, n_tok;
  int n_seqs, Hqk, Hv, l2norm;
  float *T;  // workspace T region (packed fp32)
  int32_t *status;
};

constexpr int kAP = C + 1;  // padded fp32 row of the A / X matrices
constexpr size_t kPrepSmem = 1024 + 16384 + sizeof(float) * (C * kAP * 3 + 5 * C);

__global__ void __launch_bounds__(NT) chunk_prep_kernel(const PrepParams p) {
  extern __shared__ uint8_t smraw[];
  uint8_t *sm = (uint8_t *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  uint8_t *Ks = sm;                                // [2 fb][64 rows][128 B] raw bf16 k, SW128
  float *KK = (float *)(sm + 16384);               // [64][kAP]  k_hat k_hat^T
  float *X0 = KK + C * kAP;                        // [64][kAP]  A then X, v-head of half 0
  float *X1 = X0 + C * kAP;                        // [64][kAP]  half 1
  float *gm = X1 + C * kAP;                        // [2][64] gamma per half
  float *bt = gm + 2 * C;                          // [2][64] beta per half
  float *kinv = bt + 2 * C;                        // [64] 1 / |k| per token
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int qh = blockIdx.y;
  const int64_t slot = blockIdx.x;
  // sequence of this slot: largest s with slot_base(s) <= slot
  int lo = 0, hi = p.n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (slot_base(p.cu, p.row_T, mid) <= slot) lo = mid; else hi = mid - 1;
  }
  const int s = lo;
  int64_t start, end;
  seq_range(p.cu, p.row_T, s, start, end);
  if (start < 0 || end < start || end > p.n_tok) {
    if (tid == 0) set_status(p.status, GDN_ERR_BOUNDS);
    return;
  }
  const int64_t c = slot - slot_base(p.cu, p.row_T, s);
  const int64_t t0 = start + c * C;
  if (c < 0 || t0 >= end) return;  // slot past this sequence's last chunk
  const int n = (int)min((int64_t)C, end - t0);

  // ---- raw k rows into a K-major SW128 tile (two threads per row) and 1/|k|
  {
    const int r = tid >> 1, fb = tid & 1;
    float ss = 0.f;
    uint4 raw[8];
    if (r < n) {
      const uint4 *src = reinterpret_cast<const uint4 *>(p.k + (t0 + r) * p.ks + (int64_t)qh * KD + fb * 64);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        raw[j] = src[j];
        const uint32_t *w = reinterpret_cast<const uint32_t *>(&raw[j]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = unpack_bf16(w[e]);
          ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) raw[j] = make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) *reinterpret_cast<uint4 *>(Ks + fb * 8192 + sw128_off(r, j * 8)) = raw[j];
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    if (fb == 0) kinv[r] = p.l2norm ? 1.f / sqrtf(ss + kL2Eps) : 1.f;
  }
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(&tbase, 64);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tbase;
  // ---- K K^T (M = 64, N = 64, K = 128) on the tensor core
  if (tid == 0) {
    const uint32_t a0 = smem_u32(Ks);
    const uint32_t id = idesc_bf16(64, 64, false, false);
#pragma unroll
    for (int ks = 0; ks < KD / 16; ++ks) {
      const uint32_t off = (ks >> 2) * 8192 + (ks & 3) * 32;
      umma_bf16(tm, smem_desc(a0 + off, 16, 1024, 2), smem_desc(a0 + off, 16, 1024, 2), id, ks > 0);
    }
    umma_commit(&bar);
  }
  const bool ok = mbar_wait(&bar, 0, kSpin);
  if (__syncthreads_or(!ok)) {
    if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT);
    (void)mbar_wait(&bar, 0, kSpin);  // let an MMA still in flight land before TMEM is freed
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 64);
    return;
  }
  tc_fence_after();
  // rows of an M = 64 result sit in lanes 0-15 of each 32-lane quarter
  {
    const bool has_row = lane < 16;
    const int r = warp * 16 + lane;
    const float ir = has_row ? kinv[r] : 0.f;
#pragma unroll
    for (int c0 = 0; c0 < C; c0 += 16) {
      float v[16];
      tmem_ld16(tm + ((uint32_t)(warp * 32) << 16) + c0, v);
      tmem_wait_ld();
      if (has_row)
#pragma unroll
        for (int i = 0; i < 16; ++i) KK[r * kAP + c0 + i] = v[i] * ir * kinv[c0 + i];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, 64);

  // ---- per v-head: A, forward substitution, T = X diag(beta); two v-heads at a time
  const int rh = p.Hv / p.Hqk;
  const int half = tid >> 6, lt = tid & 63;
  float *X = half ? X1 : X0;
  float *gh = gm + half * C, *bh = bt + half * C;
  for (int j0 = 0; j0 < rh; j0 += 2) {
    const int j = j0 + half;
    const bool active = j < rh;  // uniform per half (64 threads)
    const int hv = qh * rh + (active ? j : 0);
    if (active) {
      gh[lt] = lt < n ? p.g[(t0 + lt) * p.Hv + hv] : 0.f;
      bh[lt] = lt < n ? p.beta[(t0 + lt) * p.Hv + hv] : 0.f;
    }
    __syncthreads();
    if (active && (lt >> 5) == 0) {  // inclusive cumsum by the first warp of the half
      const float g0 = gh[2 * lt], g1 = gh[2 * lt + 1];
      float incl = g0 + g1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lt >= o) incl += u;
      }
      gh[2 * lt + 1] = incl;
      gh[2 * lt] = incl - g1;
    }
    __syncthreads();
    // column lt of A: A[i][lt] = beta_i exp(gamma_i - gamma_lt) (k_hat_i . k_hat_lt), i > lt
    if (active) {
      const float gl = gh[lt];
      for (int i = 0; i < C; ++i)
        X[i * kAP + lt] = (i > lt) ? bh[i] * expf(gh[i] - gl) * KK[i * kAP + lt] : 0.f;
    }
    __syncthreads();
    // X = (I + A)^-1 by forward substitution, row by row, one column a thread;
    // rows < i of X already replaced A's rows.
    for (int i = 1; i < C; ++i) {
      float x = 0.f;
      if (active && lt < i) {
        x = X[i * kAP + lt];
        for (int m = lt + 1; m < i; ++m) x = fmaf(X[i * kAP + m], X[m * kAP + lt], x);
      }
      __syncthreads();
      if (active && lt < i) X[i * kAP + lt] = -x;
      __syncthreads();
    }
    // T row lt = X row lt scaled by beta per column (unit diagonal -> beta), packed fp32
    if (active) {
      float *dst = p.T + ((size_t)slot * p.Hv + hv) * kTPacked + lt * (lt + 1) / 2;
      for (int c0 = 0; c0 < lt; ++c0) dst[c0] = X[lt * kAP + c0] * bh[c0];
      dst[lt] = bh[lt];
    }
    __syncthreads();
  }
}

// ============================================================ main kernel

struct TcParams {
  const int32_t *cu;
  int64_t row_T, n_tok;
  int Hqk, Hv, V;
  const float *g, *h0;
  const float *T;  // packed fp32 T per (slot, v-head) from chunk_prep_kernel
  float scale;
  int l2norm;
  void *o;
  int o_f32;
  float *hT;
  int32_t *status;
};

// dynamic shared memory map (offsets from a 1024-aligned base)
constexpr uint32_t OFF_QK = 0;          // 2 stages x 32 KB: [fb][rows 0-63 k | 64-127 q][128 B], raw bf16
constexpr uint32_t OFF_V = 65536;       // 2 stages x 4 KB:  [64 tok][32 v] SW64
constexpr uint32_t OFF_TP = 73728;      // 2 stages x 8448 B: packed fp32 T
constexpr uint32_t kTPStride = 8448;
constexpr uint32_t OFF_TH = 91136;      // 8 KB T hi            [64][128 B] SW128
constexpr uint32_t OFF_TL = 99328;      // 8 KB T lo
constexpr uint32_t OFF_TPH = 107520;    // 8 KB T diag(b/|k|) hi
constexpr uint32_t OFF_TPL = 115712;    // 8 KB T diag(b/|k|) lo
constexpr uint32_t OFF_NW = 123904;     // 16 KB -W              [fb][64][128 B]
constexpr uint32_t OFF_QT = 140288;     // 16 KB scale diag(b/|q|) q
constexpr uint32_t OFF_PT = 156672;     // 8 KB  P without its diagonal [64][128 B]
constexpr uint32_t OFF_ST = 164864;     // 8 KB  S^T (bf16)      [128 feat][32 v] SW64
constexpr uint32_t OFF_UP = 173056;     // 4 KB  U' hi           [64 tok][32 v] SW64
constexpr uint32_t OFF_DU = 177152;     // 4 KB  diag(d/|k|) U' hi
constexpr uint32_t OFF_UPL = 181248;    // 4 KB  U' lo
constexpr uint32_t OFF_DUL = 185344;    // 4 KB  diag(d/|k|) U' lo
constexpr uint32_t kTcSmem = 189440 + 1024;
constexpr uint32_t kStageBytes = 4 * 8192 + 4096 + (uint32_t)kTBytes;  // k, q (2 boxes each), v, T

// TMEM columns
constexpr uint32_t COL_QK = 0, COL_W = 64, COL_U = 192, COL_O = 224, COL_S = 256, kTmemCols = 512;

__device__ __forceinline__ void put_bf16(uint8_t *tile, int row, int col, float x) {
  *reinterpret_cast<__nv_bfloat16 *>(tile + sw128_off(row, col)) = __float2bfloat16_rn(x);
}

__global__ void __launch_bounds__(NT, 1)
    chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
  extern __shared__ uint8_t smraw[];
  uint8_t *sm = (uint8_t *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  __shared__ uint64_t bar_tma[2], bar_mma;
  __shared__ uint32_t tbase;
  __shared__ float gam[C], bex[C], dec[C], kinv[C], qinv[C];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int v0 = blockIdx.x * BVT, h = blockIdx.y, s = blockIdx.z;
  const int qh = h / (p.Hv / p.Hqk);
  int64_t start, end;
  seq_range(p.cu, p.row_T, s, start, end);
  if (start < 0 || end < start || end > p.n_tok) {
    if (tid == 0) set_status(p.status, GDN_ERR_BOUNDS);
    return;
  }
  const int n_chunks = (int)((end - start + C - 1) / C);
  const int64_t sbase = (int64_t)s + start / C;
  const uint32_t sb = smem_u32(sm);

  if (tid == 0) {
    mbar_init(&bar_tma[0], 1);
    mbar_init(&bar_tma[1], 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 0) {
    tmem_alloc(&tbase, kTmemCols);
    tmem_relinquish();
  }
  // the four T tiles keep a zero upper triangle: clear them once
  for (uint32_t i = tid; i < 4 * 8192 / 16; i += NT)
    reinterpret_cast<uint4 *>(sm + OFF_TH)[i] = make_uint4(0, 0, 0, 0);
  // fp32 state, transposed: thread f holds S[v0 + v][f] for v < 32
  float S[BVT];
  const float *h0p = p.h0 ? p.h0 + (((size_t)s * p.Hv + h) * p.V + v0) * KD + tid : nullptr;
#pragma unroll
  for (int v = 0; v < BVT; ++v) S[v] = h0p ? h0p[(size_t)v * KD] : 0.f;
  auto write_state_bf16 = [&]() {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 o = make_uint4(pack_bf16(S[q * 8 + 0], S[q * 8 + 1]), pack_bf16(S[q * 8 + 2], S[q * 8 + 3]),
                           pack_bf16(S[q * 8 + 4], S[q * 8 + 5]), pack_bf16(S[q * 8 + 6], S[q * 8 + 7]));
      *reinterpret_cast<uint4 *>(sm + OFF_ST + sw64_off(tid, q * 8)) = o;
    }
  };
  write_state_bf16();
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tbase;
  const uint32_t tl = tm + ((uint32_t)(warp * 32) << 16);  // this warp's lane quarter

  auto issue_tma = [&](int ci, int st) {
    const int64_t t0 = start + (int64_t)ci * C;
    const float *tsrc = p.T + ((size_t)(sbase + ci) * p.Hv + h) * kTPacked;
    uint8_t *qk = sm + OFF_QK + st * 32768;
    mbar_arrive_expect_tx(&bar_tma[st], kStageBytes);
    tma_load_3d(qk, &tm_k, &bar_tma[st], 0, qh, (int32_t)t0);
    tma_load_3d(qk + 16384, &tm_k, &bar_tma[st], 64, qh, (int32_t)t0);
    tma_load_3d(qk + 8192, &tm_q, &bar_tma[st], 0, qh, (int32_t)t0);
    tma_load_3d(qk + 16384 + 8192, &tm_q, &bar_tma[st], 64, qh, (int32_t)t0);
    tma_load_3d(sm + OFF_V + st * 4096, &tm_v, &bar_tma[st], v0, h, (int32_t)t0);
    bulk_load(sm + OFF_TP + st * kTPStride, tsrc, (uint32_t)kTBytes, &bar_tma[st]);
  };
  if (tid == 0 && n_chunks > 0) issue_tma(0, 0);
  // what is in flight, tracked identically by every thread (the issuing thread is tid 0)
  bool tma_inflight[2] = {n_chunks > 0, false};
  bool mma_inflight = false;
  uint32_t ph_tma[2] = {0u, 0u}, ph_mma = 0;
  bool failed = false;
  auto commit_mma = [&]() {
    if (tid == 0) umma_commit(&bar_mma);
    mma_inflight = true;
  };
  auto wait_mma = [&]() -> bool {
    const bool ok = mbar_wait(&bar_mma, ph_mma, kSpin);
    if (__syncthreads_or(!ok)) return false;
    ph_mma ^= 1u;
    mma_inflight = false;
    return true;
  };
  auto sync_smem_for_mma = [&]() {
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  };

  const bool lane_row = lane < 16;      // rows of M = 64 results: lanes 0-15 of each quarter
  const int mrow = warp * 16 + lane;    // the token row this thread holds in M = 64 results
  const int row = mrow & 63;            // in-range index for the threads without a row
  const size_t o_tok_stride = (size_t)p.Hv * p.V;

  for (int ci = 0; ci < n_chunks && !failed; ++ci) {
    const int st = ci & 1;
    const int64_t t0 = start + (int64_t)ci * C;
    const int n = (int)min((int64_t)C, end - t0);
    const uint8_t *qk = sm + OFF_QK + st * 32768;
    const uint32_t qk_a = sb + OFF_QK + st * 32768;
    const uint32_t v_a = sb + OFF_V + st * 4096;
    const float *tp = reinterpret_cast<const float *>(sm + OFF_TP + st * kTPStride);
    if (ci + 1 < n_chunks) {
      if (tid == 0) issue_tma(ci + 1, st ^ 1);
      tma_inflight[st ^ 1] = true;
    }
    // ---- gates of this chunk: gamma (cumsum), b = exp(gamma), d = exp(gamma_last - gamma)
    if (tid < C) gam[tid] = tid < n ? p.g[(t0 + tid) * p.Hv + h] : 0.f;
    __syncthreads();
    if (warp == 0) {
      const float g0 = gam[2 * lane], g1 = gam[2 * lane + 1];
      float incl = g0 + g1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      const float last = __shfl_sync(0xffffffffu, incl, 31);
      const float ga = incl - g1, gb = incl;
      gam[2 * lane] = ga;
      gam[2 * lane + 1] = gb;
      bex[2 * lane] = expf(ga);
      bex[2 * lane + 1] = expf(gb);
      dec[2 * lane] = expf(last - ga);
      dec[2 * lane + 1] = expf(last - gb);
    }
    // ---- wait for this chunk's tiles
    {
      const bool ok = mbar_wait(&bar_tma[st], ph_tma[st], kSpin);
      if (__syncthreads_or(!ok)) { failed = true; break; }
      ph_tma[st] ^= 1u;
      tma_inflight[st] = false;
    }
    // ---- 1/|k| and 1/|q| per token (threads 0-63 k rows, 64-127 q rows);
    //      q rows also give the bf16 operand scale * b / |q| * q
    {
      const int r = tid & 63;
      const bool isq = tid >= 64;
      const uint8_t *rowbase = qk + (isq ? 8192 : 0);
      float ss = 0.f;
#pragma unroll
      for (int fb = 0; fb < 2; ++fb)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 u = *reinterpret_cast<const uint4 *>(rowbase + fb * 16384 + sw128_off(r, j * 8));
          const uint32_t *w = reinterpret_cast<const uint32_t *>(&u);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = unpack_bf16(w[e]);
            ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
          }
        }
      const float inv = p.l2norm ? 1.f / sqrtf(ss + kL2Eps) : 1.f;
      if (!isq) {
        kinv[r] = inv;
      } else {
        qinv[r] = inv;
        const float sc = p.scale * bex[r] * inv;
#pragma unroll
        for (int fb = 0; fb < 2; ++fb)
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 u = *reinterpret_cast<const uint4 *>(rowbase + fb * 16384 + sw128_off(r, j * 8));
            const uint32_t *w = reinterpret_cast<const uint32_t *>(&u);
            uint4 b;
            uint32_t *bw = reinterpret_cast<uint32_t *>(&b);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = unpack_bf16(w[e]);
              bw[e] = pack_bf16(f.x * sc, f.y * sc);
            }
            *reinterpret_cast<uint4 *>(sm + OFF_QT + fb * 8192 + sw128_off(r, j * 8)) = b;
          }
      }
    }
    __syncthreads();
    // ---- T (fp32, packed) -> bf16 hi/lo tiles of T and of T diag(b / |k|)
    for (int idx = tid; idx < kTPacked; idx += NT) {
      int i = (int)((sqrtf(8.f * (float)idx + 1.f) - 1.f) * 0.5f);
      while ((i + 1) * (i + 2) / 2 <= idx) ++i;
      while (i * (i + 1) / 2 > idx) --i;
      const int j = idx - i * (i + 1) / 2;
      const float t = tp[idx];
      const float th = __bfloat162float(__float2bfloat16_rn(t));
      const float t2 = t * bex[j] * kinv[j];
      const float t2h = __bfloat162float(__float2bfloat16_rn(t2));
      put_bf16(sm + OFF_TH, i, j, th);
      put_bf16(sm + OFF_TL, i, j, t - th);
      put_bf16(sm + OFF_TPH, i, j, t2h);
      put_bf16(sm + OFF_TPL, i, j, t2 - t2h);
    }
    sync_smem_for_mma();
    // ---- state-independent MMAs: Q K^T, W = T diag(b/|k|) K (hi + lo), U = T V (hi + lo)
    if (tid == 0) {
      const uint32_t id_qk = idesc_bf16(64, 64, false, false);
#pragma unroll
      for (int ks = 0; ks < KD / 16; ++ks) {
        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
        umma_bf16(tm + COL_QK, smem_desc(qk_a + 8192 + off, 16, 1024, 2),
                  smem_desc(qk_a + off, 16, 1024, 2), id_qk, ks > 0);
      }
      const uint32_t id_w = idesc_bf16(64, 128, false, true);
      const uint32_t id_u = idesc_bf16(64, BVT, false, true);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks) {
        const uint64_t kb = smem_desc(qk_a + ks * 2048, 16384, 1024, 2);
        const uint64_t vb = smem_desc(v_a + ks * 1024, 2048, 512, 4);
        umma_bf16(tm + COL_W, smem_desc(sb + OFF_TPH + ks * 32, 16, 1024, 2), kb, id_w, ks > 0);
        umma_bf16(tm + COL_W, smem_desc(sb + OFF_TPL + ks * 32, 16, 1024, 2), kb, id_w, 1);
        umma_bf16(tm + COL_U, smem_desc(sb + OFF_TH + ks * 32, 16, 1024, 2), vb, id_u, ks > 0);
        umma_bf16(tm + COL_U, smem_desc(sb + OFF_TL + ks * 32, 16, 1024, 2), vb, id_u, 1);
      }
    }
    commit_mma();
    if (!wait_mma()) { failed = true; break; }
    tc_fence_after();
    // ---- P = scale (Q_hat K_hat^T * Gamma), strictly lower part -> bf16 tile, diagonal kept
    //      in fp32; -W -> bf16 tile
    float pdiag = 0.f;
    {
      const float gr = gam[row], qr = p.scale * qinv[row];
#pragma unroll
      for (int c0 = 0; c0 < C; c0 += 16) {
        float v[16];
        tmem_ld16(tl + COL_QK + c0, v);
        tmem_wait_ld();
        if (lane_row) {
          uint32_t w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j0 = c0 + 2 * e, j1 = j0 + 1;
            const float a = (j0 < mrow) ? qr * kinv[j0] * expf(gr - gam[j0]) * v[2 * e] : 0.f;
            const float b = (j1 < mrow) ? qr * kinv[j1] * expf(gr - gam[j1]) * v[2 * e + 1] : 0.f;
            if (j0 == mrow) pdiag = qr * kinv[j0] * v[2 * e];
            if (j1 == mrow) pdiag = qr * kinv[j1] * v[2 * e + 1];
            w[e] = pack_bf16(a, b);
          }
          *reinterpret_cast<uint4 *>(sm + OFF_PT + sw128_off(mrow, c0)) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4 *>(sm + OFF_PT + sw128_off(mrow, c0 + 8)) = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
#pragma unroll
      for (int c0 = 0; c0 < KD; c0 += 16) {
        float v[16];
        tmem_ld16(tl + COL_W + c0, v);
        tmem_wait_ld();
        if (lane_row) {
          uint32_t w[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) w[e] = pack_bf16(-v[2 * e], -v[2 * e + 1]);
          const int fb = c0 >> 6, cc = c0 & 63;
          *reinterpret_cast<uint4 *>(sm + OFF_NW + fb * 8192 + sw128_off(mrow, cc)) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4 *>(sm + OFF_NW + fb * 8192 + sw128_off(mrow, cc + 8)) = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    }
    sync_smem_for_mma();
    // ---- state chain, round 1: U' = U - W S^T ; O = scale diag(b/|q|) Q S^T
    if (tid == 0) {
      const uint32_t id = idesc_bf16(64, BVT, false, true);
#pragma unroll
      for (int ks = 0; ks < KD / 16; ++ks) {
        const uint32_t off = (ks >> 2) * 8192 + (ks & 3) * 32;
        const uint64_t bs = smem_desc(sb + OFF_ST + ks * 1024, 2048, 512, 4);
        umma_bf16(tm + COL_U, smem_desc(sb + OFF_NW + off, 16, 1024, 2), bs, id, 1);
        umma_bf16(tm + COL_O, smem_desc(sb + OFF_QT + off, 16, 1024, 2), bs, id, ks > 0);
      }
    }
    commit_mma();
    if (!wait_mma()) { failed = true; break; }
    tc_fence_after();
    float up[BVT];  // U' row of this thread (fp32), reused for the diagonal term of O
    tmem_ld16(tl + COL_U, *reinterpret_cast<float(*)[16]>(up));
    tmem_ld16(tl + COL_U + 16, *reinterpret_cast<float(*)[16]>(up + 16));
    tmem_wait_ld();
    if (lane_row) {
      const float dr = dec[mrow] * kinv[mrow];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c0 = q * 8;
        uint32_t uh[4], ul[4], dh[4], dl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = up[c0 + 2 * e], b = up[c0 + 2 * e + 1];
          const float ah = __bfloat162float(__float2bfloat16_rn(a));
          const float bh = __bfloat162float(__float2bfloat16_rn(b));
          uh[e] = pack_bf16(ah, bh);
          ul[e] = pack_bf16(a - ah, b - bh);
          const float da = dr * a, db = dr * b;
          const float dah = __bfloat162float(__float2bfloat16_rn(da));
          const float dbh = __bfloat162float(__float2bfloat16_rn(db));
          dh[e] = pack_bf16(dah, dbh);
          dl[e] = pack_bf16(da - dah, db - dbh);
        }
        const uint32_t off = sw64_off(mrow, c0);
        *reinterpret_cast<uint4 *>(sm + OFF_UP + off) = make_uint4(uh[0], uh[1], uh[2], uh[3]);
        *reinterpret_cast<uint4 *>(sm + OFF_UPL + off) = make_uint4(ul[0], ul[1], ul[2], ul[3]);
        *reinterpret_cast<uint4 *>(sm + OFF_DU + off) = make_uint4(dh[0], dh[1], dh[2], dh[3]);
        *reinterpret_cast<uint4 *>(sm + OFF_DUL + off) = make_uint4(dl[0], dl[1], dl[2], dl[3]);
      }
    }
    sync_smem_for_mma();
    // ---- state chain, round 2: O += P U' (strictly lower P) ; dS^T = K^T diag(d/|k|) U'
    //      (U' as a hi + lo pair of bf16 operands)
    if (tid == 0) {
      const uint32_t id_o = idesc_bf16(64, BVT, false, true);
      const uint32_t id_s = idesc_bf16(128, BVT, true, true);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks) {
        const uint64_t pa = smem_desc(sb + OFF_PT + ks * 32, 16, 1024, 2);
        const uint64_t ka = smem_desc(qk_a + ks * 2048, 16384, 1024, 2);
        umma_bf16(tm + COL_O, pa, smem_desc(sb + OFF_UP + ks * 1024, 2048, 512, 4), id_o, 1);
        umma_bf16(tm + COL_O, pa, smem_desc(sb + OFF_UPL + ks * 1024, 2048, 512, 4), id_o, 1);
        umma_bf16(tm + COL_S, ka, smem_desc(sb + OFF_DU + ks * 1024, 2048, 512, 4), id_s, ks > 0);
        umma_bf16(tm + COL_S, ka, smem_desc(sb + OFF_DUL + ks * 1024, 2048, 512, 4), id_s, 1);
      }
    }
    commit_mma();
    if (!wait_mma()) { failed = true; break; }
    tc_fence_after();
    {
      const float blast = bex[C - 1];
      float ds[BVT], ov[BVT];
      tmem_ld16(tl + COL_S, *reinterpret_cast<float(*)[16]>(ds));
      tmem_ld16(tl + COL_S + 16, *reinterpret_cast<float(*)[16]>(ds + 16));
      tmem_ld16(tl + COL_O, *reinterpret_cast<float(*)[16]>(ov));
      tmem_ld16(tl + COL_O + 16, *reinterpret_cast<float(*)[16]>(ov + 16));
      tmem_wait_ld();
#pragma unroll
      for (int v = 0; v < BVT; ++v) S[v] = fmaf(blast, S[v], ds[v]);
      write_state_bf16();
      if (lane_row && mrow < n) {
#pragma unroll
        for (int v = 0; v < BVT; ++v) ov[v] = fmaf(pdiag, up[v], ov[v]);
        const size_t off = (size_t)(t0 + mrow) * o_tok_stride + (size_t)h * p.V + v0;
        if (p.o_f32) {
          float4 *dst = reinterpret_cast<float4 *>((float *)p.o + off);
#pragma unroll
          for (int q = 0; q < BVT / 4; ++q) dst[q] = make_float4(ov[4 * q], ov[4 * q + 1], ov[4 * q + 2], ov[4 * q + 3]);
        } else {
          uint4 *dst = reinterpret_cast<uint4 *>((__nv_bfloat16 *)p.o + off);
#pragma unroll
          for (int q = 0; q < BVT / 8; ++q)
            dst[q] = make_uint4(pack_bf16(ov[8 * q], ov[8 * q + 1]), pack_bf16(ov[8 * q + 2], ov[8 * q + 3]),
                                pack_bf16(ov[8 * q + 4], ov[8 * q + 5]), pack_bf16(ov[8 * q + 6], ov[8 * q + 7]));
        }
      }
    }
    sync_smem_for_mma();
  }
  if (failed) {
    if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT);
    // copies or MMAs still in flight land before shared memory and TMEM are released
    for (int i = 0; i < 2; ++i)
      if (tma_inflight[i]) (void)mbar_wait(&bar_tma[i], ph_tma[i], kSpin);
    if (mma_inflight) (void)mbar_wait(&bar_mma, ph_mma, kSpin);
  } else if (p.hT) {
    float *dst = p.hT + (((size_t)s * p.Hv + h) * p.V + v0) * KD + tid;
#pragma unroll
    for (int v = 0; v < BVT; ++v) dst[(size_t)v * KD] = S[v];
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, kTmemCols);
}

// ============================================================ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 3-D bf16 map over [n_tok][heads][width] with token stride `tok_stride` elements.
bool make_map3(CUtensorMap *m, const void *base, int width, int heads, int64_t n_tok,
               int64_t tok_stride, int box_w, CUtensorMapSwizzle swz) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)heads, (cuuint64_t)n_tok};
  cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)tok_stride * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_w, 1, (cuuint32_t)C};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace gdn {

// Whether the tensor-core path takes this call (else the CUDA-core kernel runs).
bool chunk_tc_supported(const void *q, const void *k, const void *v, const gdn_shape &sh) {
  if (sh.dtype != GDN_BF16 || sh.K != KD || sh.V % BVT != 0) return false;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16)) return false;
  if ((sh.q_stride * 2) % 16 || (sh.k_stride * 2) % 16 || (sh.v_stride * 2) % 16) return false;
  const int64_t n_tok = (int64_t)sh.B * sh.T;
  if (n_tok >= (1LL << 31)) return false;
  return true;
}

size_t chunk_tc_workspace_bytes(const gdn_shape &sh, int64_t n_tok) {
  return kWsHeader + n_slots(n_tok, sh.n_seqs) * (size_t)sh.Hv * kTBytes;
}

gdn_status chunk_fwd_tc(const void *q, const void *k, const void *v, const float *g,
                        const float *beta, const float *h0, const int32_t *cu,
                        const gdn_shape &sh, float scale, uint32_t flags, void *o, float *h_T,
                        void *workspace, size_t ws_bytes, cudaStream_t st) {
  const int64_t n_tok = cu ? sh.T : (int64_t)sh.B * sh.T;
  if (ws_bytes < chunk_tc_workspace_bytes(sh, n_tok)) return GDN_ERR_WORKSPACE;
  int32_t *status = (int32_t *)workspace;
  float *Tws = (float *)((uint8_t *)workspace + kWsHeader);
  const size_t slots = n_slots(n_tok, sh.n_seqs);
  const int l2 = (flags & GDN_FLAG_QK_L2NORM) ? 1 : 0;
  if (n_tok > 0) {
    PrepParams pp{};
    pp.k = (const __nv_bfloat16 *)k;
    pp.ks = sh.k_stride;
    pp.g = g;
    pp.beta = beta;
    pp.cu = cu;
    pp.row_T = sh.T;
    pp.n_tok = n_tok;
    pp.n_seqs = sh.n_seqs;
    pp.Hqk = sh.Hqk;
    pp.Hv = sh.Hv;
    pp.l2norm = l2;
    pp.T = Tws;
    pp.status = status;
    if (cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kPrepSmem) != cudaSuccess)
      return GDN_ERR_CUDA;
    if (slots > 2147483647ULL) return GDN_ERR_UNSUPPORTED;
    chunk_prep_kernel<<<dim3((unsigned)slots, sh.Hqk), NT, kPrepSmem, st>>>(pp);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
  }
  CUtensorMap mq, mk, mv;
  const int64_t map_tok = n_tok > 0 ? n_tok : 1;
  if (!make_map3(&mq, q ? q : k, KD, sh.Hqk, map_tok, sh.q_stride, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map3(&mk, k, KD, sh.Hqk, map_tok, sh.k_stride, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map3(&mv, v, sh.V, sh.Hv, map_tok, sh.v_stride, BVT, CU_TENSOR_MAP_SWIZZLE_64B))
    return GDN_ERR_CUDA;
  TcParams tp{};
  tp.cu = cu;
  tp.row_T = sh.T;
  tp.n_tok = n_tok;
  tp.Hqk = sh.Hqk;
  tp.Hv = sh.Hv;
  tp.V = sh.V;
  tp.g = g;
  tp.h0 = h0;
  tp.T = Tws;
  tp.scale = scale;
  tp.l2norm = l2;
  tp.o = o;
  tp.o_f32 = (flags & GDN_FLAG_O_F32) ? 1 : 0;
  tp.hT = h_T;
  tp.status = status;
  if (cudaFuncSetAttribute(chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kTcSmem) != cudaSuccess)
    return GDN_ERR_CUDA;
  chunk_tc_kernel<<<dim3(sh.V / BVT, sh.Hv, sh.n_seqs), NT, kTcSmem, st>>>(mq, mk, mv, tp);
  return launch_status();
}

}  // namespace gdn
