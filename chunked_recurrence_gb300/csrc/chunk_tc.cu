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
// This is the compact-workspace pair (only T of every chunk is kept between the
// kernels; chunk_scan.cu holds the split pair used when the workspace has room
// for full operand records):
//  * chunk_prep_kernel (fully parallel over chunk x q/k head): K K^T on the
//    tensor core, then per v-head the 64 x 64 forward substitution for T in
//    fp32 on CUDA cores; T is written packed (lower triangle incl. diagonal,
//    fp32, 8320 bytes per chunk and v-head) to the workspace.
//  * chunk_ws_kernel (one block per sequence x v-head x 32 value columns):
//    one warpgroup rebuilds chunk c+1's operands from T while the other walks
//    the state chain of chunk c, with the fp32 state transposed in registers
//    (thread f holds row f of S^T, one TMEM lane per key feature) and every
//    contraction on tcgen05: Q K^T, W, U, U' = U - W S^T, Q S^T, P U', K^T diag(d) U'.
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "sm100.cuh"
#include "chunk_common.cuh"

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

constexpr int kAP = C + 4;  // fp32 row of the A / X matrices, padded to keep rows 16-byte aligned
// dynamic shared memory: 1024 alignment slack + the bf16 k tile (16 KB) + fp32 KK, X0, X1
// (3 x 64 x kAP) + gamma, beta (2 x 64 each), 1/|k| (64) and exp(g) (2 x 64) = 7 x 64 floats
constexpr size_t kPrepSmem = 1024 + 16384 + sizeof(float) * (C * kAP * 3 + 7 * C);

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
  float *al = kinv + C;                            // [2][64] exp(g) per half
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
    // shared loads before any store: interleaved, each load would wait for the previous
    // store (the compiler cannot rule out aliasing between the two arrays)
    float kv[C];
#pragma unroll
    for (int c = 0; c < C; ++c) kv[c] = kinv[c];
#pragma unroll
    for (int c0 = 0; c0 < C; c0 += 16) {
      float v[16];
      tmem_ld16(tm + ((uint32_t)(warp * 32) << 16) + c0, v);
      tmem_wait_ld();
      if (has_row)
#pragma unroll
        for (int i = 0; i < 16; ++i) KK[r * kAP + c0 + i] = v[i] * ir * kv[c0 + i];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, 64);

  // ---- per v-head: A, forward substitution, T = X diag(beta); two v-heads at a time
  const int rh = p.Hv / p.Hqk;
  const int half = tid >> 6, lt = tid & 63;
  float *X = half ? X1 : X0;
  float *gh = gm + half * C, *bh = bt + half * C, *ah = al + half * C;
  for (int j0 = 0; j0 < rh; j0 += 2) {
    const int j = j0 + half;
    const bool active = j < rh;  // uniform per half (64 threads)
    const int hv = qh * rh + (active ? j : 0);
    if (active) {
      const float gv = lt < n ? p.g[(t0 + lt) * p.Hv + hv] : 0.f;
      gh[lt] = gv;
      ah[lt] = expf(gv);  // per-token decay exp(g)
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
      // exp(gamma_i - gamma_lt) = prod_{m = lt+1..i} exp(g_m): a running product down the
      // column; all loads come before the stores (see the K K^T unpacking above)
      float col[C];
      float gp = 1.f;
#pragma unroll
      for (int i = 0; i < C; ++i) {
        if (i > lt) gp *= ah[i];
        col[i] = (i > lt) ? bh[i] * gp * KK[i * kAP + lt] : 0.f;
      }
#pragma unroll
      for (int i = 0; i < C; ++i) X[i * kAP + lt] = col[i];
    }
    __syncthreads();
    // X = (I + A)^-1, one column per thread, held in registers: x_r = delta_rc - sum_{j<r} A_rj x_j.
    // Every thread walks the same (r, j) sequence, so the A_rj reads are warp-wide broadcasts and
    // no barrier is needed; entries above the diagonal of the column are zero and add nothing.
    if (active) {
      float x[C];
#pragma unroll
      for (int r = 0; r < C; ++r) x[r] = 0.f;
      x[0] = (lt == 0) ? 1.f : 0.f;
#pragma unroll
      for (int r = 1; r < C; ++r) {
        const float4 *Ar = reinterpret_cast<const float4 *>(X + r * kAP);  // rows are 16-byte aligned
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int j = 0; j < r; j += 4) {  // columns < 64 of row r; entries past r are not used
          const float4 a = Ar[j >> 2];
          a0 = fmaf(a.x, x[j], a0);
          if (j + 1 < r) a1 = fmaf(a.y, x[j + 1], a1);
          if (j + 2 < r) a2 = fmaf(a.z, x[j + 2], a2);
          if (j + 3 < r) a3 = fmaf(a.w, x[j + 3], a3);
        }
        x[r] = (r == lt) ? 1.f : -((a0 + a1) + (a2 + a3));
      }
      // T[r][lt] = x_r beta_lt for r >= lt (x_lt = 1 gives the diagonal beta_lt), packed rows;
      // for a fixed r the 32 lanes write 32 consecutive floats.
      float *dst = p.T + ((size_t)slot * p.Hv + hv) * kTPacked;
      const float bl = bh[lt];
#pragma unroll
      for (int r = 0; r < C; ++r)
        if (r >= lt) dst[r * (r + 1) / 2 + lt] = x[r] * bl;
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
  // segment-summary mode: state columns [0, K) are M (start I, v = 0), [K, K + V) S_local
  int summary;
  float *M, *S_local;
};

constexpr uint32_t kTmemCols = 512;

// ======================================== warp-specialised main kernel
//
// Two warpgroups per block (256 threads) overlap consecutive chunks:
//  * WG0 (warps 0-3) prepares chunk c+1's state-independent operands: gates,
//    1/|k| and 1/|q|, the bf16 hi/lo split of T and T diag(b/|k|), the MMAs
//    Q K^T, W = T diag(b/|k|) K and U = T V, then the bf16 tiles P (strictly
//    lower) and -W.  It hands them over through double-buffered shared memory
//    and TMEM, signalling `full[b]`.
//  * WG1 (warps 4-7) runs chunk c's state chain: U' = U - W S^T and Q S^T,
//    the U' epilogue, P U' and K^T diag(d/|k|) U', then the fp32 state update
//    and the output, signalling `empty[b]` when chunk c's buffers may be reused.
// Raw k | q tiles sit in a 3-stage TMA ring (both groups read them); v tiles
// in a 2-stage ring of WG0; T is prefetched from global into registers one
// chunk ahead.

constexpr int NT2 = 256;
constexpr uint32_t W_KQ = 0;                 // 3 stages x 32 KB: [fb][rows 0-63 k | 64-127 q][128 B]
constexpr uint32_t W_V = 98304;              // 2 x 4 KB: [64 tok][32 v] SW64
constexpr uint32_t W_TH = 106496, W_TL = 114688, W_TPH = 122880, W_TPL = 131072;  // 4 x 8 KB, SW128
constexpr uint32_t W_NW = 139264;            // 2 x 16 KB: -W [fb][64][128 B]
constexpr uint32_t W_PT = 172032;            // 2 x 8 KB: P (strictly lower) [64][128 B]
constexpr uint32_t W_ST = 188416;            // 8 KB: S^T bf16 [128 feat][32 v] SW64
constexpr uint32_t W_UP = 196608, W_DU = 200704, W_UPL = 204800, W_DUL = 208896;  // 4 x 4 KB, SW64
constexpr uint32_t kWsSmem = 212992 + 1024;
constexpr uint32_t WC_QK = 0, WC_W = 64, WC_U = 192, WC_OA = 256, WC_OB = 288, WC_S = 320;

struct WsShared {
  uint64_t kq_full[3], v_full[2], pre_done, chain_done, out_done, full[2], empty[2];
  uint32_t tbase;
  int abort;
  int kq_issued[3], kq_seen[3], v_issued[2], v_seen[2];
  int pre_inflight, chain_inflight, out_inflight;
  uint32_t ph_pre, ph_chain, ph_out;
  float gam[C], gl2[C], bex[C], dec[C], kinv[C], qinv[C], alf[C + 1];  // WG0 working set
  float dk[2][C], alpha[2][C], pdiag[2][C], blast[2];      // handed to WG1 per buffer
  int nvalid[2];
};

__global__ void __launch_bounds__(NT2, 1)
    chunk_ws_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
  extern __shared__ uint8_t smraw[];
  uint8_t *sm = (uint8_t *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  __shared__ WsShared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int wg = tid >> 7, wt = tid & 127, quarter = warp & 3;
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
  volatile int *abort_flag = &sh.abort;
  // summary mode: M's columns see v = 0 (their v tiles stay zero and are never loaded);
  // S_local's columns read v at column v0 - K
  const bool m_cols = p.summary && v0 < KD;
  const bool load_v = !m_cols;
  const int vcol = p.summary ? v0 - KD : v0;

  auto issue_kq = [&](int ci, int st) {  // raw k and q tiles of chunk ci into ring stage st
    const int32_t t0 = (int32_t)(start + (int64_t)ci * C);
    uint8_t *qk = sm + W_KQ + st * 32768;
    mbar_arrive_expect_tx(&sh.kq_full[st], 4 * 8192);
    tma_load_3d(qk, &tm_k, &sh.kq_full[st], 0, qh, t0);
    tma_load_3d(qk + 16384, &tm_k, &sh.kq_full[st], 64, qh, t0);
    tma_load_3d(qk + 8192, &tm_q, &sh.kq_full[st], 0, qh, t0);
    tma_load_3d(qk + 16384 + 8192, &tm_q, &sh.kq_full[st], 64, qh, t0);
    sh.kq_issued[st] += 1;
  };
  auto issue_v = [&](int ci, int vb) {
    const int32_t t0 = (int32_t)(start + (int64_t)ci * C);
    mbar_arrive_expect_tx(&sh.v_full[vb], 4096);
    tma_load_3d(sm + W_V + vb * 4096, &tm_v, &sh.v_full[vb], vcol, h, t0);
    sh.v_issued[vb] += 1;
  };
  auto fail = [&]() {
    *abort_flag = 1;
    set_status(p.status, GDN_ERR_TIMEOUT);
  };

  if (tid == 0) {
    for (int i = 0; i < 3; ++i) mbar_init(&sh.kq_full[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.v_full[i], 1);
      mbar_init(&sh.full[i], 1);
      mbar_init(&sh.empty[i], 1);
      sh.v_issued[i] = sh.v_seen[i] = 0;
    }
    mbar_init(&sh.pre_done, 1);
    mbar_init(&sh.chain_done, 1);
    mbar_init(&sh.out_done, 1);
    for (int i = 0; i < 3; ++i) sh.kq_issued[i] = sh.kq_seen[i] = 0;
    sh.abort = 0;
    sh.pre_inflight = sh.chain_inflight = sh.out_inflight = 0;
    sh.ph_pre = sh.ph_chain = sh.ph_out = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    for (int ci = 0; ci < 3 && ci < n_chunks; ++ci) issue_kq(ci, ci);
    if (n_chunks > 0 && load_v) issue_v(0, 0);
  }
  if (m_cols)  // v = 0 for M's columns: both v buffers stay zero
    for (int i = tid; i < 2 * 4096 / 16; i += NT2) reinterpret_cast<uint4 *>(sm + W_V)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 0) {
    tmem_alloc(&sh.tbase, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = sh.tbase;
  const uint32_t tl = tm + ((uint32_t)(quarter * 32) << 16);  // this warp's lane quarter
  const bool lane_row = lane < 16;                             // M = 64 rows: lanes 0-15 of a quarter
  const int mrow = quarter * 16 + lane;

  if (wg == 0) {
    // ===================================================== WG0: operands
    float gnext = 0.f;
    if (n_chunks > 0 && wt < C && start + wt < end) gnext = p.g[(start + wt) * p.Hv + h];
    const int tr = wt & 63, tcb = (wt >> 6) * 32;  // T row and 32-column half of this thread
    float tpre[32];
    auto load_T = [&](int ci) {
      const float *trow = p.T + ((size_t)(sbase + ci) * p.Hv + h) * kTPacked + tr * (tr + 1) / 2;
#pragma unroll
      for (int u = 0; u < 32; ++u) tpre[u] = (tcb + u <= tr) ? trow[tcb + u] : 0.f;
    };
    if (n_chunks > 0) load_T(0);
    for (int ci = 0; ci < n_chunks; ++ci) {
      const int b = ci & 1, st = ci % 3;
      const int64_t t0 = start + (int64_t)ci * C;
      const int n = (int)min((int64_t)C, end - t0);
      const uint32_t qk_a = sb + W_KQ + st * 32768;
      const uint8_t *qk = sm + W_KQ + st * 32768;
      // chunk ci-2's buffers (same parity) must be released by WG1
      {
        // one thread polls; the others wait in the hardware barrier of the vote below
        const bool ok = ci < 2 || wt != 0 || mbar_wait_abortable(&sh.empty[b], ((ci - 2) >> 1) & 1, kSpin, abort_flag);
        if (named_bar_any(1, 128, !ok)) {
          if (wt == 0) fail();
          break;
        }
      }
      if (wt == 0 && ci + 1 < n_chunks && load_v) issue_v(ci + 1, (ci + 1) & 1);
      // ---- gates
      if (wt < C) sh.gam[wt] = gnext;
      if (ci + 1 < n_chunks && wt < C) {
        const int64_t t1 = t0 + C;
        gnext = (t1 + wt < end) ? p.g[(t1 + wt) * p.Hv + h] : 0.f;
      }
      named_bar_sync(1, 128);
      if (warp == 0) {
        const float g0 = sh.gam[2 * lane], g1 = sh.gam[2 * lane + 1];
        float incl = g0 + g1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float u = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += u;
        }
        const float last = __shfl_sync(0xffffffffu, incl, 31);
        const float ga = incl - g1, gb = incl;
        sh.gam[2 * lane] = ga;
        sh.gam[2 * lane + 1] = gb;
        sh.gl2[2 * lane] = ga * 1.4426950408889634f;
        sh.gl2[2 * lane + 1] = gb * 1.4426950408889634f;
        sh.bex[2 * lane] = expf(ga);
        sh.bex[2 * lane + 1] = expf(gb);
        sh.dec[2 * lane] = expf(last - ga);
        sh.dec[2 * lane + 1] = expf(last - gb);
        sh.alf[2 * lane] = expf(g0);  // per-token decay exp(g)
        sh.alf[2 * lane + 1] = expf(g1);
        if (lane == 31) {
          sh.blast[b] = expf(last);
          sh.alf[C] = 1.f;
        }
      }
      // ---- this chunk's k | q and v tiles
      {
        bool ok = wt != 0 || mbar_wait_abortable(&sh.kq_full[st], (ci / 3) & 1, kSpin, abort_flag);
        if (load_v) ok = ok && (wt != 0 || mbar_wait_abortable(&sh.v_full[b], (ci >> 1) & 1, kSpin, abort_flag));
        if (named_bar_any(1, 128, !ok)) {
          if (wt == 0) fail();
          break;
        }
        if (wt == 0) {
          sh.kq_seen[st] += 1;
          if (load_v) sh.v_seen[b] += 1;
        }
      }
      named_bar_sync(1, 128);
      // ---- 1/|k|, 1/|q|; alpha = scale b / |q|
      {
        const int r = wt & 63;
        const bool isq = wt >= 64;
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
          sh.kinv[r] = inv;
        } else {
          sh.qinv[r] = inv;
          sh.alpha[b][r] = p.scale * sh.bex[r] * inv;
        }
      }
      named_bar_sync(1, 128);
      if (wt < C) sh.dk[b][wt] = sh.dec[wt] * sh.kinv[wt];
      // ---- T and T diag(b/|k|) as bf16 hi/lo tiles (row tr, columns tcb..tcb+31);
      //      the column factors are read before any tile store: interleaved, every shared
      //      load would wait for the preceding store (the compiler cannot rule out aliasing)
      float cf[32];
#pragma unroll
      for (int u = 0; u < 32; ++u) cf[u] = sh.bex[tcb + u] * sh.kinv[tcb + u];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int c0 = tcb + q * 8;
        uint32_t wh[4], wl[4], xh[4], xl[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float t_0 = tpre[q * 8 + 2 * e], t_1 = tpre[q * 8 + 2 * e + 1];
          const float u_0 = t_0 * cf[q * 8 + 2 * e], u_1 = t_1 * cf[q * 8 + 2 * e + 1];
          const float h0 = __bfloat162float(__float2bfloat16_rn(t_0));
          const float h1 = __bfloat162float(__float2bfloat16_rn(t_1));
          const float g0 = __bfloat162float(__float2bfloat16_rn(u_0));
          const float g1 = __bfloat162float(__float2bfloat16_rn(u_1));
          wh[e] = pack_bf16(h0, h1);
          wl[e] = pack_bf16(t_0 - h0, t_1 - h1);
          xh[e] = pack_bf16(g0, g1);
          xl[e] = pack_bf16(u_0 - g0, u_1 - g1);
        }
        const uint32_t off = sw128_off(tr, c0);
        *reinterpret_cast<uint4 *>(sm + W_TH + off) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        *reinterpret_cast<uint4 *>(sm + W_TL + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        *reinterpret_cast<uint4 *>(sm + W_TPH + off) = make_uint4(xh[0], xh[1], xh[2], xh[3]);
        *reinterpret_cast<uint4 *>(sm + W_TPL + off) = make_uint4(xl[0], xl[1], xl[2], xl[3]);
      }
      if (ci + 1 < n_chunks) load_T(ci + 1);
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(1, 128);
      tc_fence_after();
      // ---- Q K^T, W = T diag(b/|k|) K, U = T V (hi + lo)
      if (wt == 0) {
        const uint32_t id_qk = idesc_bf16(64, 64, false, false);
#pragma unroll
        for (int ks = 0; ks < KD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
          umma_bf16(tm + WC_QK, smem_desc(qk_a + 8192 + off, 16, 1024, 2),
                    smem_desc(qk_a + off, 16, 1024, 2), id_qk, ks > 0);
        }
        const uint32_t id_w = idesc_bf16(64, 128, false, true);
        const uint32_t id_u = idesc_bf16(64, BVT, false, true);
        const uint32_t v_a = sb + W_V + b * 4096;
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks) {
          const uint64_t kb = smem_desc(qk_a + ks * 2048, 16384, 1024, 2);
          const uint64_t vb = smem_desc(v_a + ks * 1024, 2048, 512, 4);
          umma_bf16(tm + WC_W, smem_desc(sb + W_TPH + ks * 32, 16, 1024, 2), kb, id_w, ks > 0);
          umma_bf16(tm + WC_W, smem_desc(sb + W_TPL + ks * 32, 16, 1024, 2), kb, id_w, 1);
          umma_bf16(tm + WC_U + b * BVT, smem_desc(sb + W_TH + ks * 32, 16, 1024, 2), vb, id_u, ks > 0);
          umma_bf16(tm + WC_U + b * BVT, smem_desc(sb + W_TL + ks * 32, 16, 1024, 2), vb, id_u, 1);
        }
        umma_commit(&sh.pre_done);
        sh.pre_inflight = 1;
      }
      {
        const bool ok = wt != 0 || mbar_wait_abortable(&sh.pre_done, ci & 1, kSpin, abort_flag);
        if (named_bar_any(1, 128, !ok)) {
          if (wt == 0) fail();
          break;
        }
      }
      if (wt == 0) {
        sh.pre_inflight = 0;
        sh.ph_pre = (ci + 1) & 1;
      }
      tc_fence_after();
      // ---- P (strictly lower, bf16) with its diagonal kept in fp32; -W (bf16)
      {
        const int row = mrow & 63;
        const float qr = p.scale * sh.qinv[row];
        uint8_t *pt = sm + W_PT + b * 8192;
        uint8_t *nw = sm + W_NW + b * 16384;
        // Q K^T and the first half of W in one TMEM round trip, the second half of W in another
        float qk[64], w64[64];
        tmem_ld64(tl + WC_QK, qk);
        tmem_ld64(tl + WC_W, w64);
        tmem_wait_ld();
        if (lane_row) {
          // Gamma_{r,j} = exp(gamma_r - gamma_j) = prod_{i=j+1..r} exp(g_i) for j < r: a running
          // product walking j downwards, one multiply per column and no exponential.  All shared
          // loads come before the stores (see the T conversion).
          float gprod = 1.f, vd = 0.f;
#pragma unroll
          for (int j = C - 1; j >= 0; --j) {
            const float aj = sh.alf[j + 1], kj = sh.kinv[j];
            vd = (j == mrow) ? qk[j] : vd;
            if (j < mrow) gprod *= aj;
            qk[j] = (j < mrow) ? qr * kj * gprod * qk[j] : 0.f;
          }
          const float pdv = qr * sh.kinv[mrow] * vd;
#pragma unroll
          for (int c0 = 0; c0 < C; c0 += 8)
            *reinterpret_cast<uint4 *>(pt + sw128_off(mrow, c0)) =
                make_uint4(pack_bf16(qk[c0], qk[c0 + 1]), pack_bf16(qk[c0 + 2], qk[c0 + 3]),
                           pack_bf16(qk[c0 + 4], qk[c0 + 5]), pack_bf16(qk[c0 + 6], qk[c0 + 7]));
          sh.pdiag[b][mrow] = pdv;
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 8)
            *reinterpret_cast<uint4 *>(nw + sw128_off(mrow, c0)) =
                make_uint4(pack_bf16(-w64[c0], -w64[c0 + 1]), pack_bf16(-w64[c0 + 2], -w64[c0 + 3]),
                           pack_bf16(-w64[c0 + 4], -w64[c0 + 5]), pack_bf16(-w64[c0 + 6], -w64[c0 + 7]));
        }
        tmem_ld64(tl + WC_W + 64, w64);
        tmem_wait_ld();
        if (lane_row) {
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 8)
            *reinterpret_cast<uint4 *>(nw + 8192 + sw128_off(mrow, c0)) =
                make_uint4(pack_bf16(-w64[c0], -w64[c0 + 1]), pack_bf16(-w64[c0 + 2], -w64[c0 + 3]),
                           pack_bf16(-w64[c0 + 4], -w64[c0 + 5]), pack_bf16(-w64[c0 + 6], -w64[c0 + 7]));
        }
      }
      if (wt == 0) sh.nvalid[b] = n;
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(1, 128);
      if (wt == 0) mbar_arrive(&sh.full[b]);
    }
  } else {
    // ===================================================== WG1: state chain
    float S[BVT];
    if (m_cols) {  // M starts at the identity: S[v0 + v][f] = (v0 + v == f)
#pragma unroll
      for (int v = 0; v < BVT; ++v) S[v] = (v0 + v == wt) ? 1.f : 0.f;
    } else {
      const float *h0p = (p.h0 && !p.summary) ? p.h0 + (((size_t)s * p.Hv + h) * p.V + v0) * KD + wt : nullptr;
#pragma unroll
      for (int v = 0; v < BVT; ++v) S[v] = h0p ? h0p[(size_t)v * KD] : 0.f;
    }
    auto write_state_bf16 = [&]() {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 o = make_uint4(pack_bf16(S[q * 8 + 0], S[q * 8 + 1]), pack_bf16(S[q * 8 + 2], S[q * 8 + 3]),
                             pack_bf16(S[q * 8 + 4], S[q * 8 + 5]), pack_bf16(S[q * 8 + 6], S[q * 8 + 7]));
        *reinterpret_cast<uint4 *>(sm + W_ST + sw64_off(wt, q * 8)) = o;
      }
    };
    write_state_bf16();
    fence_proxy_async_smem();
    named_bar_sync(2, 128);
    const size_t o_tok_stride = (size_t)p.Hv * p.V;
    uint32_t ph_chain = 0;
    bool ok_all = true;
    for (int ci = 0; ci < n_chunks; ++ci) {
      const int b = ci & 1, st = ci % 3;
      const int64_t t0 = start + (int64_t)ci * C;
      const uint32_t qk_a = sb + W_KQ + st * 32768;
      {
        const bool ok = wt != 0 || mbar_wait_abortable(&sh.full[b], (ci >> 1) & 1, kSpin, abort_flag);
        if (named_bar_any(2, 128, !ok)) {
          if (wt == 0) fail();
          ok_all = false;
          break;
        }
      }
      tc_fence_after();
      // ---- MMA group 1: U' = U - W S^T ; Q S^T
      if (wt == 0) {
        const uint32_t id = idesc_bf16(64, BVT, false, true);
#pragma unroll
        for (int ks = 0; ks < KD / 16; ++ks) {
          const uint32_t off = (ks >> 2) * 8192 + (ks & 3) * 32;
          umma_bf16(tm + WC_U + b * BVT, smem_desc(sb + W_NW + b * 16384 + off, 16, 1024, 2),
                    smem_desc(sb + W_ST + ks * 1024, 2048, 512, 4), id, 1);
        }
        umma_commit(&sh.chain_done);  // the state path waits for U' only
        sh.chain_inflight = 1;
#pragma unroll
        for (int ks = 0; ks < (p.summary ? 0 : KD / 16); ++ks) {
          const uint32_t qoff = 8192 + (ks >> 2) * 16384 + (ks & 3) * 32;
          umma_bf16(tm + WC_OA, smem_desc(qk_a + qoff, 16, 1024, 2),
                    smem_desc(sb + W_ST + ks * 1024, 2048, 512, 4), id, ks > 0);
        }
      }
      {
        const bool ok = wt != 0 || mbar_wait_abortable(&sh.chain_done, ph_chain, kSpin, abort_flag);
        if (named_bar_any(2, 128, !ok)) {
          if (wt == 0) fail();
          ok_all = false;
          break;
        }
      }
      ph_chain ^= 1u;
      tc_fence_after();
      float up[BVT];
      tmem_ld16(tl + WC_U + b * BVT, *reinterpret_cast<float(*)[16]>(up));
      tmem_ld16(tl + WC_U + b * BVT + 16, *reinterpret_cast<float(*)[16]>(up + 16));
      tmem_wait_ld();
      if (lane_row) {
        const float dr = sh.dk[b][mrow];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c0 = q * 8;
          uint32_t uh[4], ul[4], dh[4], dl[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a = up[c0 + 2 * e], bb = up[c0 + 2 * e + 1];
            const float ah = __bfloat162float(__float2bfloat16_rn(a));
            const float bh = __bfloat162float(__float2bfloat16_rn(bb));
            uh[e] = pack_bf16(ah, bh);
            ul[e] = pack_bf16(a - ah, bb - bh);
            const float da = dr * a, db = dr * bb;
            const float dah = __bfloat162float(__float2bfloat16_rn(da));
            const float dbh = __bfloat162float(__float2bfloat16_rn(db));
            dh[e] = pack_bf16(dah, dbh);
            dl[e] = pack_bf16(da - dah, db - dbh);
          }
          const uint32_t off = sw64_off(mrow, c0);
          *reinterpret_cast<uint4 *>(sm + W_UP + off) = make_uint4(uh[0], uh[1], uh[2], uh[3]);
          *reinterpret_cast<uint4 *>(sm + W_UPL + off) = make_uint4(ul[0], ul[1], ul[2], ul[3]);
          *reinterpret_cast<uint4 *>(sm + W_DU + off) = make_uint4(dh[0], dh[1], dh[2], dh[3]);
          *reinterpret_cast<uint4 *>(sm + W_DUL + off) = make_uint4(dl[0], dl[1], dl[2], dl[3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(2, 128);
      tc_fence_after();
      // ---- MMA group 2: P U' (hi + lo) ; dS^T = K^T diag(d/|k|) U' (hi + lo)
      if (wt == 0) {
        const uint32_t id_o = idesc_bf16(64, BVT, false, true);
        const uint32_t id_s = idesc_bf16(128, BVT, true, true);
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks) {
          const uint64_t ka = smem_desc(qk_a + ks * 2048, 16384, 1024, 2);
          umma_bf16(tm + WC_S, ka, smem_desc(sb + W_DU + ks * 1024, 2048, 512, 4), id_s, ks > 0);
          umma_bf16(tm + WC_S, ka, smem_desc(sb + W_DUL + ks * 1024, 2048, 512, 4), id_s, 1);
        }
        umma_commit(&sh.chain_done);  // the state update waits for dS^T only
#pragma unroll
        for (int ks = 0; ks < (p.summary ? 0 : C / 16); ++ks) {
          const uint64_t pa = smem_desc(sb + W_PT + b * 8192 + ks * 32, 16, 1024, 2);
          umma_bf16(tm + WC_OB, pa, smem_desc(sb + W_UP + ks * 1024, 2048, 512, 4), id_o, ks > 0);
          umma_bf16(tm + WC_OB, pa, smem_desc(sb + W_UPL + ks * 1024, 2048, 512, 4), id_o, 1);
        }
        if (!p.summary) {
          umma_commit(&sh.out_done);  // Q S^T and P U' of this chunk
          sh.out_inflight = 1;
        }
      }
      {
        const bool ok = wt != 0 || mbar_wait_abortable(&sh.chain_done, ph_chain, kSpin, abort_flag);
        if (named_bar_any(2, 128, !ok)) {
          if (wt == 0) fail();
          ok_all = false;
          break;
        }
      }
      ph_chain ^= 1u;
      if (wt == 0) sh.chain_inflight = 0;
      tc_fence_after();
      {
        const float blast = sh.blast[b];
        float ds[BVT];
        tmem_ld16(tl + WC_S, *reinterpret_cast<float(*)[16]>(ds));
        tmem_ld16(tl + WC_S + 16, *reinterpret_cast<float(*)[16]>(ds + 16));
        tmem_wait_ld();
#pragma unroll
        for (int v = 0; v < BVT; ++v) S[v] = fmaf(blast, S[v], ds[v]);
        write_state_bf16();
      }
      if (!p.summary) {
        const bool ok = wt != 0 || mbar_wait_abortable(&sh.out_done, sh.ph_out, kSpin, abort_flag);
        if (named_bar_any(2, 128, !ok)) {
          if (wt == 0) fail();
          ok_all = false;
          break;
        }
        if (wt == 0) {
          sh.ph_out ^= 1u;
          sh.out_inflight = 0;
        }
      }
      tc_fence_after();
      {
        float oa[BVT], ob[BVT];
        tmem_ld16(tl + WC_OA, *reinterpret_cast<float(*)[16]>(oa));
        tmem_ld16(tl + WC_OA + 16, *reinterpret_cast<float(*)[16]>(oa + 16));
        tmem_ld16(tl + WC_OB, *reinterpret_cast<float(*)[16]>(ob));
        tmem_ld16(tl + WC_OB + 16, *reinterpret_cast<float(*)[16]>(ob + 16));
        tmem_wait_ld();
        if (!p.summary && lane_row && mrow < sh.nvalid[b]) {
          const float al = sh.alpha[b][mrow], pd = sh.pdiag[b][mrow];
#pragma unroll
          for (int v = 0; v < BVT; ++v) oa[v] = fmaf(al, oa[v], fmaf(pd, up[v], ob[v]));
          const size_t off = (size_t)(t0 + mrow) * o_tok_stride + (size_t)h * p.V + v0;
          if (p.o_f32) {
            float4 *dst = reinterpret_cast<float4 *>((float *)p.o + off);
#pragma unroll
            for (int q = 0; q < BVT / 4; ++q) dst[q] = make_float4(oa[4 * q], oa[4 * q + 1], oa[4 * q + 2], oa[4 * q + 3]);
          } else {
            uint4 *dst = reinterpret_cast<uint4 *>((__nv_bfloat16 *)p.o + off);
#pragma unroll
            for (int q = 0; q < BVT / 8; ++q)
              dst[q] = make_uint4(pack_bf16(oa[8 * q], oa[8 * q + 1]), pack_bf16(oa[8 * q + 2], oa[8 * q + 3]),
                                  pack_bf16(oa[8 * q + 4], oa[8 * q + 5]), pack_bf16(oa[8 * q + 6], oa[8 * q + 7]));
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      named_bar_sync(2, 128);
      if (wt == 0) {
        mbar_arrive(&sh.empty[b]);
        if (ci + 3 < n_chunks) issue_kq(ci + 3, st);
      }
    }
    if (ok_all && p.summary) {
      float *dst = m_cols ? p.M + (((size_t)s * p.Hv + h) * KD + v0) * KD + wt
                          : p.S_local + (((size_t)s * p.Hv + h) * p.V + vcol) * KD + wt;
#pragma unroll
      for (int v = 0; v < BVT; ++v) dst[(size_t)v * KD] = S[v];
    } else if (ok_all && p.hT) {
      float *dst = p.hT + (((size_t)s * p.Hv + h) * p.V + v0) * KD + wt;
#pragma unroll
      for (int v = 0; v < BVT; ++v) dst[(size_t)v * KD] = S[v];
    }
    if (wt == 0) sh.ph_chain = ph_chain;
  }
  __syncthreads();
  if (tid == 0 && sh.abort) {
    // let copies and MMAs still in flight land before shared memory and TMEM are released
    for (int i = 0; i < 3; ++i)
      if (sh.kq_issued[i] > sh.kq_seen[i]) (void)mbar_wait(&sh.kq_full[i], sh.kq_seen[i] & 1, kSpin);
    for (int i = 0; i < 2; ++i)
      if (sh.v_issued[i] > sh.v_seen[i]) (void)mbar_wait(&sh.v_full[i], sh.v_seen[i] & 1, kSpin);
    if (sh.pre_inflight) (void)mbar_wait(&sh.pre_done, sh.ph_pre, kSpin);
    if (sh.chain_inflight) (void)mbar_wait(&sh.chain_done, sh.ph_chain, kSpin);
    if (sh.out_inflight) (void)mbar_wait(&sh.out_done, sh.ph_out, kSpin);
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

// Both kernels of the tensor-core path: the prep kernel (T for every chunk and
// v-head into the workspace), then the warp-specialised chunk kernel over
// (state-column tiles, v-heads, sequences).
static gdn_status run_tc(const void *q, const void *k, const void *v, const float *g, const float *beta,
                  const float *h0, const int32_t *cu, int n_seqs, int64_t n_tok, const gdn_shape &sh,
                  float scale, uint32_t flags, void *o, float *h_T, bool summary, float *M,
                  float *S_local, void *workspace, size_t ws_bytes, cudaStream_t st) {
  const size_t slots = n_slots(n_tok, n_seqs);
  if (ws_bytes < kWsHeader + slots * (size_t)sh.Hv * kTBytes) return GDN_ERR_WORKSPACE;
  if (slots > 2147483647ULL) return GDN_ERR_UNSUPPORTED;
  int32_t *status = (int32_t *)workspace;
  float *Tws = (float *)((uint8_t *)workspace + kWsHeader);
  const int l2 = (flags & GDN_FLAG_QK_L2NORM) ? 1 : 0;
  PrepParams pp{};
  pp.k = (const __nv_bfloat16 *)k;
  pp.ks = sh.k_stride;
  pp.g = g;
  pp.beta = beta;
  pp.cu = cu;
  pp.row_T = sh.T;
  pp.n_tok = n_tok;
  pp.n_seqs = n_seqs;
  pp.Hqk = sh.Hqk;
  pp.Hv = sh.Hv;
  pp.l2norm = l2;
  pp.T = Tws;
  pp.status = status;
  if (cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kPrepSmem) != cudaSuccess)
    return GDN_ERR_CUDA;
  chunk_prep_kernel<<<dim3((unsigned)slots, sh.Hqk), NT, kPrepSmem, st>>>(pp);
  if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
  CUtensorMap mq, mk, mv;
  if (!make_map3(&mq, q, KD, sh.Hqk, n_tok, summary ? sh.k_stride : sh.q_stride, 64,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map3(&mk, k, KD, sh.Hqk, n_tok, sh.k_stride, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map3(&mv, v, sh.V, sh.Hv, n_tok, sh.v_stride, BVT, CU_TENSOR_MAP_SWIZZLE_64B))
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
  tp.summary = summary ? 1 : 0;
  tp.M = M;
  tp.S_local = S_local;
  if (cudaFuncSetAttribute(chunk_ws_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kWsSmem) != cudaSuccess)
    return GDN_ERR_CUDA;
  const int cols = summary ? KD + sh.V : sh.V;
  chunk_ws_kernel<<<dim3(cols / BVT, sh.Hv, n_seqs), NT2, kWsSmem, st>>>(mq, mk, mv, tp);
  return launch_status();
}

gdn_status chunk_fwd_tc(const void *q, const void *k, const void *v, const float *g,
                        const float *beta, const float *h0, const int32_t *cu,
                        const gdn_shape &sh, float scale, uint32_t flags, void *o, float *h_T,
                        void *workspace, size_t ws_bytes, cudaStream_t st) {
  const int64_t n_tok = cu ? sh.T : (int64_t)sh.B * sh.T;
  return run_tc(q, k, v, g, beta, h0, cu, sh.n_seqs, n_tok, sh, scale, flags, o, h_T, false,
                nullptr, nullptr, workspace, ws_bytes, st);
}

gdn_status summary_tc(const void *k, const void *v, const float *g, const float *beta,
                      const int32_t *bounds, int n_seg, const gdn_shape &sh, uint32_t flags,
                      float *M, float *S_local, void *workspace, size_t ws_bytes, cudaStream_t st) {
  return run_tc(k, k, v, g, beta, nullptr, bounds, n_seg, sh.T, sh, 1.f, flags, nullptr, nullptr,
                true, M, S_local, workspace, ws_bytes, st);
}

}  // namespace gdn
