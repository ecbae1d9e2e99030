// chunk_scan.cu -- tensor-core path of gdn_chunk_fwd split by dependence on the
// state: a fully parallel operand kernel, then a lean state scan.
//
// The chunk form of the gated delta rule ("Gated Delta Networks", chunkwise
// algorithm; the UT/WY transform), per chunk of C = 64 tokens, v-head h and
// start state S (V x K, fp32), with unit-norm keys and queries:
//   gamma = inclusive cumsum of g,  b = exp(gamma),  d = exp(gamma_last - gamma)
//   A  = strictly-lower(diag(beta) K_hat K_hat^T * Gamma),  Gamma_ij = exp(gamma_i - gamma_j)
//   T  = (I + A)^-1 diag(beta)
//   W  = T diag(b) K_hat,  U = T V                          (state-independent)
//   U' = U - W S^T                                          (state step 1)
//   O  = scale diag(b) Q_hat S^T + P U',  P = scale (Q_hat K_hat^T * Gamma), j <= i
//   S <- b_last S + U'^T diag(d) K_hat                      (state step 2)
//
// chunk_operand_kernel (one block per chunk x v-head, all chunks at once)
// computes everything that does not depend on S and stores it in a record of
// the workspace laid out as the scan kernel's shared-memory tiles:
//   -W (bf16, K-major 128-byte-swizzled images, two 64-feature halves), P
//   without its diagonal (bf16, same layout), U (fp32, 32-column slices) and
//   the vectors alpha = scale b / |q|, diag(P) (fp32), d / |k| and b_last.
// chunk_scan_kernel (one block per sequence x v-head x 32 value columns) then
// walks the chunks with three small tcgen05 MMA groups per chunk:
//   [Q; -W] S^T                   (M = 128: raw q rows, then -W rows)
//   K^T [dU'_hi | dU'_lo]         (M = 128 key features, N = 2 x 32)
//   [P; -] [U'_hi | U'_lo]        (rows 0-63 used)
// Operands of three chunks are in flight (TMA and bulk copies) ahead of the scan.
// with the fp32 state in registers (one key feature per thread) and a bf16
// copy of S^T in shared memory as the MMA operand.
//
// Precision: q and k enter the MMAs as their exact bf16 values (1/|q|, 1/|k|
// applied in fp32); T enters as a hi + lo pair of bf16 matrices; U' and
// diag(d/|k|) U' enter as hi + lo pairs; the diagonal of P stays fp32.
#include <cudaTypedefs.h>

#include <algorithm>
#include <math.h>

#include "chunk_common.cuh"
#include "common.cuh"
#include "conv_tap.cuh"
#include "gates.cuh"
#include "sm100.cuh"

using namespace gdn;
using namespace gdn::sm100;

namespace {

constexpr int C = kChunk;   // 64 tokens per chunk
constexpr int KD = 128;     // key width of this path
constexpr int VS = 32;      // value columns per scan block
constexpr uint32_t kSpin = 1u << 22;  // bounded waits before reporting a timeout
constexpr size_t kHeader = 256;       // status word + padding

// ------------------------------------------------------------ records
// One record per (chunk slot, v-head), 1 KB aligned pieces:
constexpr uint32_t REC_NW = 0;       // -W: [2 feature halves][64 rows][128 B] bf16, SW128 images
constexpr uint32_t REC_P = 16384;    // P (strictly lower): [64 rows][128 B] bf16, SW128 image
constexpr uint32_t REC_VEC = 24576;  // alpha[64], pdiag[64], dk[64] fp32, b_last, n
constexpr uint32_t REC_U = 25600;    // U: [V / 32 slices][64 tokens][32] fp32; the 16-byte
                                     // piece m of token row r sits at piece m ^ (r % 8)
constexpr uint32_t VEC_ALPHA = 0, VEC_PDIAG = 64, VEC_DK = 128, VEC_BLAST = 192, VEC_N = 193;  // floats

__host__ __device__ constexpr size_t rec_bytes(int V) { return (size_t)REC_U + (size_t)V * C * 4; }

// ============================================================ operand kernel

struct OpParams {
  const __nv_bfloat16 *q, *k, *v;
  int64_t qs, ks, vs;  // token strides (elements)
  const float *g, *beta;
  const int32_t *cu;
  int64_t row_T, n_tok;
  int n_seqs, Hqk, Hv, l2norm;
  float scale;
  uint8_t *rec;
  size_t rec_bytes;
  int64_t n_items;  // chunk slots x v-heads
  int32_t *status;
  // Fused front end (the layer's Q|K|V projections x before the conv): the maps read the
  // raw q, k and v channels of x, the tiles are conv'd (+ SiLU) in place in shared memory,
  // the gates come from a and b, and the first v-head of every q/k head writes the conv'd
  // q and k rows that the scan reads.
  int front, width;                   // width 1..4 (taps before the last W zero-padded)
  const __nv_bfloat16 *x, *cw, *cbias;  // x [n_tok][Cx]; weights [Cx][width]; bias [Cx] or null
  int64_t Cx;
  const __nv_bfloat16 *ga, *gb;       // a, b [n_tok][Hv]
  const float *A_log, *dt_bias;       // [Hv]
  __nv_bfloat16 *qc, *kc;             // conv'd q, k [n_tok][Hqk][128]
  unsigned long long *claim;          // front end: item-group counter, zero at launch
  int quit;                           // GDN_FLAG_TEST_NO_WAIT: a wait that misses its first poll gives up
};

constexpr int kXP = C + 4;  // fp32 row of A, padded (rows stay 16-byte aligned)
constexpr uint32_t OP_KQ = 0;      // [2 halves][128 rows][128 B]: rows 0-63 raw k, 64-127 raw q;
                                   // once Q K^T is done, T hi and T lo take the q rows' places
constexpr uint32_t OP_TH = 8192, OP_TL = 24576;
// Raw v ([V / 64 blocks][64 tokens][128 B], SW128).  Up to V = 128 it is loaded late, into
// the k rows once W = T diag(b/|k|) K has read them (blocks 16 KB apart), which keeps a
// block at 50 KB of shared memory so that four fit on an SM; wider v has its own region.
__host__ __device__ constexpr bool op_late_v(int V) { return V <= 128; }
__host__ __device__ constexpr uint32_t op_vt(int V) { return op_late_v(V) ? 0u : 32768u; }
__host__ __device__ constexpr uint32_t op_vt_stride(int V) { return op_late_v(V) ? 16384u : 8192u; }
// A, then (I + A)^-1, both row-major (row stride kXP), then the T diag(b/|k|) hi / lo tiles
__host__ __device__ constexpr uint32_t op_x(int V) { return op_late_v(V) ? 32768u : 32768u + (uint32_t)V * 128; }
__host__ __device__ constexpr uint32_t op_smem(int V) { return op_x(V) + 17408u + 1024; }

__device__ __forceinline__ uint4 ldg_nc_v4(const __nv_bfloat16 *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }
// Conv taps of channels chan .. chan + 7 as four taps of fp32 pairs: a width below 4 leaves
// the first 4 - width taps zero (they multiply finite history rows, so the sums are those of
// the narrower conv).
__device__ __forceinline__ void front_weights(const OpParams &p, int64_t chan, uint64_t (&wt)[4][4], uint64_t (&bs)[4]) {
  const int W = p.width;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t ca = chan + 2 * i, cb = ca + 1;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      wt[j][i] = (j >= 4 - W) ? f2_pack(__bfloat162float(p.cw[ca * W + j - (4 - W)]),
                                                     __bfloat162float(p.cw[cb * W + j - (4 - W)]))
                                           : 0ull;
    bs[i] = p.cbias ? f2_pack(__bfloat162float(p.cbias[ca]), __bfloat162float(p.cbias[cb])) : 0ull;
  }
}

// Y = (I + A)^-1 for the strictly lower 64 x 64 A in X, by forward substitution swept
// by columns of A: y_i = delta_ij - sum_{k<i} A_ik y_k, and once row k of Y is final every
// row below it takes the rank-1 term -A_ik Y_kj.  Each thread keeps an 8 x 4 tile of Y in
// registers: rows rg + 8 m (m = 0..7) and columns 16 a + cj (a = 0..3), one in each
// 16-column block, with rg = lane % 8 and cj = 4 warp + lane / 8, so the eight owners of
// one column set sit in one warp.
// The sweep takes the rows four at a time, k = 4 b .. 4 b + 3: every thread reads those
// rows (updated through row k - 1) from their owners by shuffle, finishes them among
// themselves (rows k + 1 .. k + 3 take the terms of rows k .. k + 2: six FMAs a column),
// and then applies all four to its own rows as y_i -= sum_j A_ij Y_j, with A_i,k..k+3 one
// 16-byte load.  A_ij = 0 for j >= i, so the same update leaves rows <= k unchanged and
// turns rows k + 1 .. k + 3 into their final values.  Rows of Y are zero right of their
// diagonal, so block b touches only the column blocks a <= k / 16, a bound fixed at compile
// time with the loop unrolled, the same for every warp.  No barrier between steps.  Y is
// left in X, row-major, zero above the diagonal.
__device__ __forceinline__ void invert_unit_lower(float *X, int tid) {
  const int lane = tid & 31, rg = lane & 7, cj = (tid >> 5) * 4 + (lane >> 3);
  float y[8][4];
#pragma unroll
  for (int m = 0; m < 8; ++m)
#pragma unroll
    for (int a = 0; a < 4; ++a) y[m][a] = (rg + 8 * m == 16 * a + cj) ? 1.f : 0.f;
  const float *xr = X + rg * kXP;
#pragma unroll
  for (int k = 0; k < C; k += 4) {
    const int m0 = k >> 3, na = (k >> 4) + 1;
    float z[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int a = 0; a < na; ++a) z[j][a] = __shfl_sync(0xffffffffu, y[m0][a], ((k + j) & 7) | (lane & 24));
    const float4 r1 = *reinterpret_cast<const float4 *>(X + (k + 1) * kXP + k);
    const float4 r2 = *reinterpret_cast<const float4 *>(X + (k + 2) * kXP + k);
    const float4 r3 = *reinterpret_cast<const float4 *>(X + (k + 3) * kXP + k);
#pragma unroll
    for (int a = 0; a < na; ++a) {
      z[1][a] = fmaf(-r1.x, z[0][a], z[1][a]);
      z[2][a] = fmaf(-r2.y, z[1][a], fmaf(-r2.x, z[0][a], z[2][a]));
      z[3][a] = fmaf(-r3.z, z[2][a], fmaf(-r3.y, z[1][a], fmaf(-r3.x, z[0][a], z[3][a])));
    }
#pragma unroll
    for (int m = m0; m < 8; ++m) {
      const float4 av = *reinterpret_cast<const float4 *>(xr + 8 * m * kXP + k);
#pragma unroll
      for (int a = 0; a < na; ++a)
        y[m][a] = fmaf(-av.w, z[3][a], fmaf(-av.z, z[2][a], fmaf(-av.y, z[1][a], fmaf(-av.x, z[0][a], y[m][a]))));
    }
  }
  __syncthreads();  // every read of A is done
#pragma unroll
  for (int m = 0; m < 8; ++m)
#pragma unroll
    for (int a = 0; a < 4; ++a) X[(rg + 8 * m) * kXP + 16 * a + cj] = y[m][a];
  __syncthreads();
}

template <int V, bool FRONT>
__global__ void __launch_bounds__(128, 4)
    chunk_operand_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_qc,
                         const __grid_constant__ CUtensorMap tm_kc, const OpParams p) {
  constexpr int NVB = V / 64;                       // 64-column blocks of v
  constexpr uint32_t kCols = (V <= 128) ? 128u : 256u;
  extern __shared__ uint8_t smraw[];
  uint8_t *sm = (uint8_t *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  // per-token vectors, 16-byte aligned so that runs of four load as one: gam, then
  // bex = b, dec = d, als[j] = exp(g_{j+1}) (1 at j = C - 1), 1/|k|, 1/|q|, beta, b/|k|
  __shared__ __align__(16) float gam[C], bex[C], dec[C], als[C], kinv[C], qinv[C], bet[C], bk[C];
  __shared__ float blast_s;
  __shared__ uint64_t bar, ld_bar;
  __shared__ uint32_t tbase;
  // front end: the conv history rows of the chunk's first tokens, as 8-channel pieces:
  // [row][0-15 k, 16-31 q, 32-47 v]
  __shared__ uint4 halo[3][48];
  __shared__ int64_t claim_s[2];
  // the front end's code lives only in its own instantiation (V = 128), so that the plain
  // kernel's instruction footprint stays small
  constexpr bool kFront = FRONT && V == 128;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // A resident block walks the (chunk slot, v-head) items with the grid's stride: TMEM and
  // the barriers are set up once, and the phases of the barriers are counted across items.
  if (tid == 0) {
    mbar_init(&ld_bar, 1);
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tbase, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tbase;
  uint32_t ldp = 0, mp = 0;  // completed phases of ld_bar and bar
  if (kFront && blockIdx.x == 0 && tid == 0) atomicOr(p.status + 1, GDN_PATH_FRONT);
  // every block is resident (the grid is one wave): the state scan may start its prologue
  // on SMs this grid leaves, and waits for the whole grid before reading what it wrote
  launch_dependents();
  // In front mode blocks claim groups of G consecutive items from a counter (G = the v-heads
  // of one q/k head) and walk each group in order: the group's first item convs the q/k
  // head's tiles and writes them out, and the later items load them back.
  // Each claim is made one group ahead (thread 32, into the other of two slots), so its
  // latency overlaps the current group's work.
  const int G = kFront ? p.Hv / p.Hqk : 1;
  int64_t group = 0;
  int jg = G, slot_par = 0;  // item of the current group to run next; slot of its claim
  // Without the front end (G = 1) the blocks stride over the items instead.
  if (G > 1 && tid == 32) claim_s[0] = (int64_t)atomicAdd(p.claim, 1ull);
  bool first = true;
#pragma unroll 1
  for (;;) {
  if (jg == G) {
    if (G == 1) {
      group = first ? (int64_t)blockIdx.x : group + gridDim.x;
      first = false;
    } else {
      __syncthreads();  // this group's claim is stored; the slot the next claim reuses is read
      group = claim_s[slot_par];
      slot_par ^= 1;
      if (tid == 32) claim_s[slot_par] = (int64_t)atomicAdd(p.claim, 1ull);
    }
    jg = 0;
    if (group * G >= p.n_items) break;
  }
  const int jv = jg++;  // this item's place in its group
  const int64_t item = group * G + jv;
  int h;
  int64_t slot;
  if (p.n_items <= 0x7fffffff) {  // 32-bit division (the 64-bit one is a long software routine)
    const uint32_t it = (uint32_t)item, hv = (uint32_t)p.Hv;
    slot = it / hv;
    h = (int)(it - (uint32_t)slot * hv);
  } else {
    h = (int)(item % p.Hv);
    slot = item / p.Hv;
  }
  const int qh = h / (p.Hv / p.Hqk);
  int lo = 0, hi = p.n_seqs - 1;  // sequence of this slot: largest s with slot_base(s) <= slot
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (slot_base(p.cu, p.row_T, mid) <= slot) lo = mid; else hi = mid - 1;
  }
  const int s = lo;
  int64_t start, end;
  seq_range(p.cu, p.row_T, s, start, end);
  if (start < 0 || end < start || end > p.n_tok) {
    if (tid == 0) set_status(p.status, GDN_ERR_BOUNDS);
    break;
  }
  const int64_t c = slot - slot_base(p.cu, p.row_T, s);
  const int64_t t0 = start + c * C;
  if (c < 0 || t0 >= end) continue;  // slot past this sequence's last chunk: never read
  const int n = (int)min((int64_t)C, end - t0);
  uint8_t *rec = p.rec + ((size_t)slot * p.Hv + h) * p.rec_bytes;
  float *vec = reinterpret_cast<float *>(rec + REC_VEC);
  float *X = reinterpret_cast<float *>(sm + op_x(V));

  // ---- raw k, q and v tiles by TMA (rows past the chunk's end hold finite data of the
  //      next sequence or zeros: beta = 0 there keeps them out of every result); gates
  if (tid == 0) {
    const int32_t tt = (int32_t)t0;
    mbar_arrive_expect_tx(&ld_bar, (4 + (op_late_v(V) ? 0 : NVB)) * 8192);
    const CUtensorMap *mk = jv ? &tm_kc : &tm_k, *mq = jv ? &tm_qc : &tm_q;
    tma_load_3d(sm + OP_KQ, mk, &ld_bar, 0, qh, tt);
    tma_load_3d(sm + OP_KQ + 16384, mk, &ld_bar, 64, qh, tt);
    tma_load_3d(sm + OP_KQ + 8192, mq, &ld_bar, 0, qh, tt);
    tma_load_3d(sm + OP_KQ + 24576, mq, &ld_bar, 64, qh, tt);
    if (!op_late_v(V))
#pragma unroll
      for (int nb = 0; nb < NVB; ++nb) tma_load_3d(sm + op_vt(V) + nb * 8192, &tm_v, &ld_bar, nb * 64, h, tt);
  }
  if (!kFront) {
    if (tid < C) gam[tid] = (tid < n) ? p.g[(t0 + tid) * p.Hv + h] : 0.f;
    else bet[tid - C] = (tid - C < n) ? p.beta[(t0 + tid - C) * p.Hv + h] : 0.f;
  } else {
    // gates of the chunk's tokens (gdn_gate_prep's arithmetic), and the conv history rows
    // of the chunk's first tokens: zero at the sequence's start, else x's previous rows
    if (tid < C) {
      float gg = 0.f, bb = 0.f;
      if (tid < n) {
        const int64_t ai = (t0 + tid) * p.Hv + h;
        gdn_gates(__bfloat162float(p.ga[ai]), __bfloat162float(p.gb[ai]), p.A_log[h], p.dt_bias[h], gg, bb);
      }
      gam[tid] = gg;
      bet[tid] = bb;
    }
    for (int e = tid + (jv ? 96 : 0); e < 3 * 48; e += 128) {  // later items: v pieces only
      const int j = (jv ? e - 96 : e) / (jv ? 16 : 48), pc = jv ? 32 + (e - 96) % 16 : e % 48;
      const int64_t chan = pc < 16 ? (int64_t)(p.Hqk + qh) * KD + pc * 8
                         : pc < 32 ? (int64_t)qh * KD + (pc - 16) * 8
                                   : (int64_t)2 * p.Hqk * KD + (int64_t)h * V + (pc - 32) * 8;
      halo[j][pc] = (c > 0) ? ldg_nc_v4(p.x + (t0 - 3 + j) * p.Cx + chan) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  {
    const bool ok = tid != 0 || mbar_wait_q(&ld_bar, ldp & 1, kSpin, p.quit != 0);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT);
      (void)mbar_wait(&ld_bar, ldp & 1, kSpin);  // the copies land before shared memory is released
      break;
    }
    ++ldp;
  }
  if (kFront && jv == 0) {
    // ---- conv (+ SiLU) of the k and q tiles in place: warp w takes rows 16 w .. 16 w + 15,
    //      lanes 0-15 the k tile and 16-31 the q tile, eight channels a lane
    const int tile = lane >> 4, pc = lane & 15;
    const int64_t chan = (int64_t)(tile ? qh : p.Hqk + qh) * KD + pc * 8;
    uint8_t *base = sm + OP_KQ + (pc >> 3) * 16384 + tile * 8192;
    const int cin = (pc & 7) * 8;
    uint64_t wt[4][4], bs[4], hist[3][4];
    front_weights(p, chan, wt, bs);
#pragma unroll
    for (int j = 0; j < 3; ++j)
      unpack8p(warp == 0 ? halo[j][(tile ? 16 : 0) + pc]
                         : *reinterpret_cast<const uint4 *>(base + sw128_off(16 * warp - 3 + j, cin)),
               hist[j]);
    __syncthreads();  // every history row is read before any row is overwritten
    // the conv'd rows this item owns go to the scan's q / k arrays (past the last
    // sequence's end, the chunk's remaining rows too)
    const int64_t last_end = p.cu ? (int64_t)p.cu[p.n_seqs] : p.n_tok;
    const int64_t lim = (end >= last_end) ? p.n_tok : end;
    __nv_bfloat16 *dst = (tile ? p.qc : p.kc) + (int64_t)qh * KD + pc * 8;
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      const int row = 16 * warp + r;
      uint4 *cell = reinterpret_cast<uint4 *>(base + sw128_off(row, cin));
      uint64_t cur[4], out[4];
      unpack8p(*cell, cur);
      conv_row8p<4, 3>(wt, bs, hist, cur, true, out);
      const uint4 y = pack8p(out);
      *cell = y;
      if (t0 + row < lim) *reinterpret_cast<uint4 *>(dst + (t0 + row) * (int64_t)p.Hqk * KD) = y;
      conv_shift8p<3>(hist, cur);
    }
    // the MMAs read the conv'd tiles, and the group's later items load the written rows
    fence_proxy_async_all();
    __syncthreads();
  } else if (kFront && n < C) {
    // ---- rows past this sequence's end in tiles loaded back: they may not be written yet
    for (int e = tid; e < (C - n) * 32; e += 128) {
      const int r = n + (e >> 5), pcs = e & 31;  // 32 pieces of 16 bytes: k and q, both halves
      *reinterpret_cast<uint4 *>(sm + OP_KQ + (pcs >> 4) * 16384 + ((pcs >> 3) & 1) * 8192 +
                                 sw128_off(r, (pcs & 7) * 8)) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
    __syncthreads();
  }
  // ---- 1/|k| and 1/|q| from the tiles (two threads per token)
  {
    const int r = tid >> 1, hf = tid & 1;
    float sk = 0.f, sq = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint4 kr = *reinterpret_cast<const uint4 *>(sm + OP_KQ + hf * 16384 + sw128_off(r, j * 8));
      const uint4 qr = *reinterpret_cast<const uint4 *>(sm + OP_KQ + hf * 16384 + 8192 + sw128_off(r, j * 8));
      const uint32_t wk[4] = {kr.x, kr.y, kr.z, kr.w}, wq[4] = {qr.x, qr.y, qr.z, qr.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 a = unpack_bf16(wk[e]), b = unpack_bf16(wq[e]);
        sk = fmaf(a.x, a.x, fmaf(a.y, a.y, sk));
        sq = fmaf(b.x, b.x, fmaf(b.y, b.y, sq));
      }
    }
    sk += __shfl_xor_sync(0xffffffffu, sk, 1);
    sq += __shfl_xor_sync(0xffffffffu, sq, 1);
    if (hf == 0) {
      kinv[r] = p.l2norm ? 1.f / sqrtf(sk + kL2Eps) : 1.f;
      qinv[r] = p.l2norm ? 1.f / sqrtf(sq + kL2Eps) : 1.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t kq_a = smem_u32(sm + OP_KQ);
  // ---- [K; Q] K^T: M = 128 (k rows, then q rows), N = 64, K = 128 on the tensor core
  if (tid == 0) {
    const uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
    for (int ks = 0; ks < KD / 16; ++ks) {
      const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
      umma_bf16(tm, smem_desc(kq_a + off, 16, 1024, 2), smem_desc(kq_a + off, 16, 1024, 2), id, ks > 0);
    }
    umma_commit(&bar);
  }
  // ---- gates: inclusive cumsum of g and the exponentials the chunk form uses
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
    if (lane > 0) als[2 * lane - 1] = expf(g0);
    als[2 * lane] = expf(g1);
    bk[2 * lane] = bex[2 * lane] * kinv[2 * lane];
    bk[2 * lane + 1] = bex[2 * lane + 1] * kinv[2 * lane + 1];
    if (lane == 31) {
      blast_s = expf(last);
      als[C - 1] = 1.f;
    }
  }
  __syncthreads();
  if (tid < C) {
    vec[VEC_ALPHA + tid] = p.scale * bex[tid] * qinv[tid];
    vec[VEC_DK + tid] = (tid < n) ? dec[tid] * kinv[tid] : 0.f;
    if (tid == 0) {
      vec[VEC_BLAST] = blast_s;
      reinterpret_cast<int *>(vec)[VEC_N] = n;
    }
  }
  {
    const bool ok = tid != 0 || mbar_wait_q(&bar, mp & 1, kSpin, p.quit != 0);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT);
      (void)mbar_wait(&bar, mp & 1, kSpin);  // an MMA still in flight lands before TMEM is freed
      break;
    }
    ++mp;
  }
  tc_fence_after();
  // ---- rows of K K^T (lanes 0-63) become rows of A; rows of Q K^T (lanes 64-127) rows of P
  {
    const int i = tid & 63;
    const bool isq = tid >= 64;
    float r64[64];
    tmem_ld64(tm + ((uint32_t)(warp * 32) << 16), r64);
    tmem_wait_ld();
    const float bi = isq ? p.scale * qinv[i] : bet[i] * kinv[i];
    // Gamma_ij = prod_{m=j+1..i} exp(g_m) for j < i: a running product walking j down.
    // Every shared load comes before the stores below (interleaved, each load would wait for
    // the previous store: the compiler cannot rule out aliasing).
    float gprod = 1.f, vd = 0.f;
#pragma unroll
    for (int j = C - 1; j >= 0; --j) {
      const float aj = als[j], kj = kinv[j];
      vd = (j == i) ? r64[j] : vd;
      if (j < i) gprod *= aj;
      r64[j] = (j < i) ? bi * kj * gprod * r64[j] : 0.f;
    }
    if (!isq) {
      float4 *xr = reinterpret_cast<float4 *>(X + i * kXP);
#pragma unroll
      for (int m = 0; m < C / 4; ++m) xr[m] = make_float4(r64[4 * m], r64[4 * m + 1], r64[4 * m + 2], r64[4 * m + 3]);
    } else {
      const float pd = bi * kinv[i] * vd;
      uint8_t *pimg = rec + REC_P;
#pragma unroll
      for (int c0 = 0; c0 < C; c0 += 8)
        *reinterpret_cast<uint4 *>(pimg + sw128_off(i, c0)) =
            make_uint4(pack_bf16(r64[c0], r64[c0 + 1]), pack_bf16(r64[c0 + 2], r64[c0 + 3]),
                       pack_bf16(r64[c0 + 4], r64[c0 + 5]), pack_bf16(r64[c0 + 6], r64[c0 + 7]));
      vec[VEC_PDIAG + i] = pd;
    }
  }
  __syncthreads();
  // ---- T = (I + A)^-1 diag(beta)
  invert_unit_lower(X, tid);
  // ---- T and T diag(b/|k|) as bf16 hi/lo K-major tiles (row r, columns cb..cb+31): T's
  //      tiles replace the raw q rows (Q K^T no longer needs them), T diag(b/|k|)'s tiles
  //      replace A once every thread has read its row of the inverse
  {
    const int r = tid & 63, cb = (tid >> 6) * 32;
    float t[32], cf[32];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float4 a = reinterpret_cast<const float4 *>(X + r * kXP + cb)[m];
      t[4 * m] = a.x;
      t[4 * m + 1] = a.y;
      t[4 * m + 2] = a.z;
      t[4 * m + 3] = a.w;
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const float4 b4 = reinterpret_cast<const float4 *>(bet + cb)[m], c4 = reinterpret_cast<const float4 *>(bk + cb)[m];
      const float bu[4] = {b4.x, b4.y, b4.z, b4.w}, cu[4] = {c4.x, c4.y, c4.z, c4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int u = 4 * m + e;
        t[u] = (cb + u <= r) ? t[u] * bu[e] : 0.f;
        cf[u] = cu[e];
      }
    }
    __syncthreads();  // X is free
    uint8_t *TP = reinterpret_cast<uint8_t *>(X);
#pragma unroll
    for (int q8 = 0; q8 < 4; ++q8) {
      uint32_t wh[4], wl[4], xh[4], xl[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int u = q8 * 8 + 2 * e;
        const float t_0 = t[u], t_1 = t[u + 1];
        const float u_0 = t_0 * cf[u], u_1 = t_1 * cf[u + 1];
        const float h0 = __bfloat162float(__float2bfloat16_rn(t_0));
        const float h1 = __bfloat162float(__float2bfloat16_rn(t_1));
        const float g0 = __bfloat162float(__float2bfloat16_rn(u_0));
        const float g1 = __bfloat162float(__float2bfloat16_rn(u_1));
        wh[e] = pack_bf16(h0, h1);
        wl[e] = pack_bf16(t_0 - h0, t_1 - h1);
        xh[e] = pack_bf16(g0, g1);
        xl[e] = pack_bf16(u_0 - g0, u_1 - g1);
      }
      const uint32_t off = sw128_off(r, cb + q8 * 8);
      *reinterpret_cast<uint4 *>(sm + OP_TH + off) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
      *reinterpret_cast<uint4 *>(sm + OP_TL + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
      *reinterpret_cast<uint4 *>(TP + off) = make_uint4(xh[0], xh[1], xh[2], xh[3]);
      *reinterpret_cast<uint4 *>(TP + 8192 + off) = make_uint4(xl[0], xl[1], xl[2], xl[3]);
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // ---- W = T diag(b/|k|) K, then U = T V, each hi + lo, in the same TMEM columns
  const uint32_t tl = tm + ((uint32_t)(warp * 32) << 16);
  const int rr = warp * 16 + lane;  // rows of an M = 64 result sit in lanes 0-15 of a quarter
  const bool has_row = lane < 16;
  bool dead = false;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    if (op_late_v(V) && pass == 1) {
      const bool ok = tid != 0 || mbar_wait_q(&ld_bar, ldp & 1, kSpin, p.quit != 0);
      if (__syncthreads_or(!ok)) {
        if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT);
        (void)mbar_wait(&ld_bar, ldp & 1, kSpin);  // the copy lands before shared memory is released
        dead = true;
        break;
      }
      ++ldp;
      if (kFront) {
        // ---- conv (+ SiLU) of the v tile in place: rows 8 (tid / 16) .. + 7, eight
        //      channels (tid % 16) a thread; the first row group's history from halo
        const int rg = tid >> 4, pc = tid & 15;
        uint8_t *base = sm + op_vt(V) + (pc >> 3) * op_vt_stride(V);
        const int cin = (pc & 7) * 8;
        uint64_t wt[4][4], bs[4], hist[3][4];
        front_weights(p, (int64_t)2 * p.Hqk * KD + (int64_t)h * V + pc * 8, wt, bs);
#pragma unroll
        for (int j = 0; j < 3; ++j)
          unpack8p(rg == 0 ? halo[j][32 + pc] : *reinterpret_cast<const uint4 *>(base + sw128_off(8 * rg - 3 + j, cin)),
                   hist[j]);
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          uint4 *cell = reinterpret_cast<uint4 *>(base + sw128_off(8 * rg + r, cin));
          uint64_t cur[4], out[4];
          unpack8p(*cell, cur);
          conv_row8p<4, 3>(wt, bs, hist, cur, true, out);
          *cell = pack8p(out);
          conv_shift8p<3>(hist, cur);
        }
        fence_proxy_async_smem();
        __syncthreads();
      }
    }
    if (tid == 0) {
      if (pass == 0) {
        const uint32_t tp_a = smem_u32(X);
        const uint32_t id_w = idesc_bf16(64, 128, false, true);
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks) {
          const uint64_t kb = smem_desc(kq_a + ks * 2048, 16384, 1024, 2);
          umma_bf16(tm, smem_desc(tp_a + ks * 32, 16, 1024, 2), kb, id_w, ks > 0);
          umma_bf16(tm, smem_desc(tp_a + 8192 + ks * 32, 16, 1024, 2), kb, id_w, 1);
        }
      } else {
        const uint32_t vt_a = smem_u32(sm + op_vt(V));
        const uint32_t id_u = idesc_bf16(64, V, false, true);
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks) {
          const uint64_t vb = smem_desc(vt_a + ks * 2048, op_vt_stride(V), 1024, 2);
          umma_bf16(tm, smem_desc(kq_a + OP_TH + ks * 32, 16, 1024, 2), vb, id_u, ks > 0);
          umma_bf16(tm, smem_desc(kq_a + OP_TL + ks * 32, 16, 1024, 2), vb, id_u, 1);
        }
      }
      umma_commit(&bar);
    }
    {
      const uint32_t par = mp & 1;
      bool ok = tid != 0 || mbar_wait_q(&bar, par, kSpin, p.quit != 0);
      if (op_late_v(V) && pass == 0 && tid == 0 && ok) {
        // W has read the k rows: v goes there while -W drains
        const int32_t tt = (int32_t)t0;
        mbar_arrive_expect_tx(&ld_bar, NVB * 8192);
#pragma unroll
        for (int nb = 0; nb < NVB; ++nb)
          tma_load_3d(sm + op_vt(V) + nb * op_vt_stride(V), &tm_v, &ld_bar, nb * 64, h, tt);
      }
      if (__syncthreads_or(!ok)) {
        if (tid == 0) set_status(p.status, GDN_ERR_TIMEOUT);
        (void)mbar_wait(&bar, par, kSpin);
        dead = true;
        break;
      }
      ++mp;
    }
    tc_fence_after();
    float w64[64];
    if (pass == 0) {  // -W as bf16 K-major images of the two 64-feature halves
#pragma unroll
      for (int fb = 0; fb < 2; ++fb) {
        tmem_ld64(tl + fb * 64, w64);
        tmem_wait_ld();
        if (has_row) {
          uint8_t *dst = rec + REC_NW + fb * 8192;
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 8)
            *reinterpret_cast<uint4 *>(dst + sw128_off(rr, c0)) =
                make_uint4(pack_bf16(-w64[c0], -w64[c0 + 1]), pack_bf16(-w64[c0 + 2], -w64[c0 + 3]),
                           pack_bf16(-w64[c0 + 4], -w64[c0 + 5]), pack_bf16(-w64[c0 + 6], -w64[c0 + 7]));
        }
      }
    } else {  // U as fp32 32-column slices
#pragma unroll
      for (int vb = 0; vb < NVB; ++vb) {
        tmem_ld64(tl + vb * 64, w64);
        tmem_wait_ld();
        if (has_row) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float4 *dst = reinterpret_cast<float4 *>(rec + REC_U + (size_t)(2 * vb + half) * 8192 + rr * 128);
#pragma unroll
            for (int m = 0; m < 8; ++m)
              dst[m ^ (rr & 7)] = make_float4(w64[half * 32 + 4 * m], w64[half * 32 + 4 * m + 1],
                                   w64[half * 32 + 4 * m + 2], w64[half * 32 + 4 * m + 3]);
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();  // the columns are free for the next pass
    tc_fence_after();
  }
  if (dead) break;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, kCols);
}

// ============================================================ scan kernel

struct ScanParams {
  const int32_t *cu;
  int64_t row_T, n_tok;
  int Hqk, Hv, V;
  const float *h0;
  const uint8_t *rec;
  size_t rec_bytes;
  void *o;
  int o_f32;
  float *hT;
  int32_t *status;
  // segment-summary mode: state columns [0, K) are M (start I, v = 0), [K, K + V) are
  // S_local (start 0); no output, q unused
  int summary;
  float *M, *S_local;
  // gated RMS norm of o in the output epilogue: the V / 32 blocks of one (v-head, sequence)
  // form a cluster and exchange each token's partial sum of squares
  int norm;
  const __nv_bfloat16 *z, *nw;  // z [n_tok][Hv][V]; the norm weight [V] or null (ones)
  float eps;
  int quit;  // GDN_FLAG_TEST_NO_WAIT: the abort flag starts set, so waits give up after 32 polls;
             // drains keep the full bound
};

// warps 0-7: state path; 8, 9, 12, 13: outputs; 10: copies; 11: MMAs
constexpr int NTS = 448;
// one stage of chunk operands (offsets inside the stage; each stage is 1 KB aligned)
constexpr uint32_t ST_AQW = 0;      // [2 halves][128 rows][128 B]: rows 0-63 raw q, rows 64-127 -W
constexpr uint32_t ST_K = 32768;    // [2 halves][64 tokens][128 B] raw k
constexpr uint32_t ST_P = 49152;    // [64][128 B] P; the 8 KB after it stand in as the unused
                                    // rows 64-127 of the M = 128 operand
constexpr uint32_t ST_U = 57344;    // [64 tokens][32] fp32 U slice (16-byte pieces swizzled)
constexpr uint32_t ST_VEC = 65536;  // alpha, pdiag, dk, b_last, n
constexpr uint32_t kStage = 66560;
constexpr uint32_t kStageTx = 16384 + 16384 + 16384 + 8192 + 8192 + 1024;
constexpr int kStages = 3;                 // chunks of operands in flight
constexpr uint32_t SC_ST = kStages * kStage;  // S^T bf16 [128 features][32 values] SW64
constexpr uint32_t SC_UP = SC_ST + 8192;      // [U'_hi | U'_lo] [64 tokens][64] SW128
constexpr uint32_t SC_DU = SC_UP + 8192;      // [dU'_hi | dU'_lo] [64 tokens][64] SW128
constexpr uint32_t SC_NP = SC_DU + 8192;      // norm: [2 chunk slots][4 ranks][2 halves][64 tokens] fp32
constexpr int kNormRanks = 4;                 // the norm epilogue takes V <= 128
constexpr uint32_t kScanSmem = SC_NP + 2 * kNormRanks * 2 * 64 * 4 + 1024;
// TMEM columns
constexpr uint32_t TC_A = 0;    // 3 x 32: q S^T in lanes 0-63, -W S^T in lanes 64-127
constexpr uint32_t TC_O = 96;   // 64: [P U'_hi | P U'_lo] in lanes 0-63
constexpr uint32_t TC_S = 160;  // 64: [K^T dU'_hi | K^T dU'_lo], one lane per key feature
constexpr uint32_t kScanCols = 256;

struct ScanShared {
  uint64_t full[kStages], empty[kStages], ga, b1, b2, epa, epa2, epb, outd, nbar[2];
  uint32_t tbase;
  int abort;
  int fills[kStages];    // loads issued into each stage
  uint64_t *mma_bar;     // barrier of the last MMA commit and its phase parity
  uint32_t mma_par;
};

// x0, x1 as a packed bf16 pair (hi) and the packed bf16 pair of what it leaves (lo).
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<uint32_t *>(&h);
  lo = *reinterpret_cast<uint32_t *>(&l);
}

// One arrival for the whole warp, after every lane's shared-memory writes and fences.
__device__ __forceinline__ void warp_arrive(uint64_t *bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// Every lane waits (bounded by `spin` polls); the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint32_t spin, volatile int *abort) {
  const bool ok = mbar_wait_spin(bar, parity, spin, abort);
  return __all_sync(0xffffffffu, ok);
}

// NORM: the gated-norm epilogue (its code only in that instantiation; NORM is set with it)
template <bool NORM>
__global__ void __launch_bounds__(NTS, 1)
    chunk_scan_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const ScanParams p) {
  extern __shared__ uint8_t smraw[];
  uint8_t *sm = (uint8_t *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  __shared__ ScanShared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int v0 = blockIdx.x * VS, h = blockIdx.y, s = blockIdx.z;
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
  const bool summary = p.summary != 0;
  const bool m_cols = summary && v0 < KD;   // columns of M: v = 0, so U = 0 and nothing is loaded
  const int uslice = (summary ? v0 - KD : v0) / VS;
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&sh.full[i], 1);
      mbar_init(&sh.empty[i], 12);
      sh.fills[i] = 0;
    }
    mbar_init(&sh.ga, 1);
    mbar_init(&sh.b1, 1);
    mbar_init(&sh.b2, 1);
    mbar_init(&sh.epa, 4);  // epilogue barriers count warps: lane 0 arrives for its warp
    mbar_init(&sh.epa2, 4);
    mbar_init(&sh.epb, 8);
    mbar_init(&sh.outd, 4);
    if (NORM) {  // one local arrival a chunk (with the bytes the cluster's partials bring)
      mbar_init(&sh.nbar[0], 1);
      mbar_init(&sh.nbar[1], 1);
    }
    sh.abort = p.quit ? 1 : 0;  // test mode: every wait gives up after 32 polls
    sh.mma_bar = nullptr;
    sh.mma_par = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&sh.tbase, kScanCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (NORM) cluster_sync_all();  // the peers' barriers are initialised before any remote arrival
  grid_dependency_wait();  // the operand kernel's records (and conv'd q, k) are complete and visible
  if (NORM && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && tid == 0)
    atomicOr(p.status + 1, GDN_PATH_NORM);
  const uint32_t tm = sh.tbase;
  auto fail = [&]() {
    *abort_flag = 1;
    set_status(p.status, GDN_ERR_TIMEOUT);
  };

  if (warp == 10) {
    // ===================================================== copies
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      for (int ci = 0; ci < n_chunks; ++ci) {
        const int st = ci % kStages;
        if (ci >= kStages && !mbar_wait_spin(&sh.empty[st], ((ci - kStages) / kStages) & 1, kSpin, abort_flag)) {
          fail();
          break;
        }
        const int32_t t0 = (int32_t)(start + (int64_t)ci * C);
        const uint8_t *r = p.rec + ((size_t)(sbase + ci) * p.Hv + h) * p.rec_bytes;
        uint8_t *sg = sm + st * kStage;
        uint64_t *fb = &sh.full[st];
        mbar_arrive_expect_tx(fb, kStageTx - (summary ? 16384u : 0u) - (m_cols ? 8192u : 0u));
        if (!summary) {  // the summary has no output: the q rows stay unused
          tma_load_3d(sg + ST_AQW, &tm_q, fb, 0, qh, t0);
          tma_load_3d(sg + ST_AQW + 16384, &tm_q, fb, 64, qh, t0);
        }
        bulk_load(sg + ST_AQW + 8192, r + REC_NW, 8192, fb);
        bulk_load(sg + ST_AQW + 24576, r + REC_NW + 8192, 8192, fb);
        tma_load_3d(sg + ST_K, &tm_k, fb, 0, qh, t0);
        tma_load_3d(sg + ST_K + 8192, &tm_k, fb, 64, qh, t0);
        bulk_load(sg + ST_P, r + REC_P, 8192, fb);
        if (!m_cols) bulk_load(sg + ST_U, r + REC_U + (size_t)uslice * 8192, 8192, fb);
        bulk_load(sg + ST_VEC, r + REC_VEC, 1024, fb);
        sh.fills[st] += 1;
      }
    }
  } else if (warp == 11) {
    // ===================================================== MMAs
    if (lane == 0) {
      const uint32_t id_a = idesc_bf16(128, VS, false, true);
      const uint32_t id_s = idesc_bf16(128, 64, true, true);
      const uint32_t id_o = idesc_bf16(128, 64, false, true);
      // descriptors of stage 0; a byte offset moves a descriptor by offset / 16
      const uint64_t d_aqw = smem_desc(sb + ST_AQW, 16, 1024, 2);
      const uint64_t d_st = smem_desc(sb + SC_ST, 2048, 512, 4);
      const uint64_t d_k = smem_desc(sb + ST_K, 8192, 1024, 2);
      const uint64_t d_du = smem_desc(sb + SC_DU, 8192, 1024, 2);
      const uint64_t d_p = smem_desc(sb + ST_P, 16, 1024, 2);
      const uint64_t d_up = smem_desc(sb + SC_UP, 8192, 1024, 2);
      int outd_seen = 0;  // outputs known to be done; out_done phases are consumed in order
      auto outputs_done = [&](int need) {
        while (outd_seen < need) {
          if (!mbar_wait_spin(&sh.outd, outd_seen & 1, kSpin, abort_flag)) return false;
          ++outd_seen;
        }
        return true;
      };
      // [P; -] [U'_hi | U'_lo] of chunk cj: the output path, one chunk behind the state path
      auto issue_b2 = [&](int cj) {
        if (!mbar_wait_spin(&sh.epa2, cj & 1, kSpin, abort_flag) || !outputs_done(cj)) return false;
        tc_fence_after();
        const uint64_t sj = (uint64_t)((cj % kStages) * kStage) >> 4;
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks)
          umma_bf16(tm + TC_O, d_p + sj + ((ks * 32) >> 4), d_up + ((ks * 2048) >> 4), id_o, ks > 0);
        umma_commit(&sh.b2);
        sh.mma_bar = &sh.b2;
        sh.mma_par = cj & 1;
        return true;
      };
      bool mok = true;
      for (int ci = 0; ci < n_chunks && mok; ++ci) {
        const int st = ci % kStages;
        // chunk ci's operands, the state after chunk ci-1, and the output of chunk ci-3
        // (whose accumulator columns [q; -W] S^T reuses) done
        if (!mbar_wait_spin(&sh.full[st], (ci / kStages) & 1, kSpin, abort_flag) ||
            !mbar_wait_spin(&sh.epb, ci & 1, kSpin, abort_flag) || (!summary && !outputs_done(ci - 2))) {
          mok = false;
          break;
        }
        tc_fence_after();
        const uint64_t so = (uint64_t)(st * kStage) >> 4;
        // [q; -W] S^T
#pragma unroll
        for (int ks = 0; ks < KD / 16; ++ks)
          umma_bf16(tm + TC_A + (ci % 3) * 32, d_aqw + so + (((ks >> 2) * 16384 + (ks & 3) * 32) >> 4),
                    d_st + ((ks * 1024) >> 4), id_a, ks > 0);
        umma_commit(&sh.ga);
        sh.mma_bar = &sh.ga;
        sh.mma_par = ci & 1;
        if ((!summary && ci > 0 && !issue_b2(ci - 1)) || !mbar_wait_spin(&sh.epa, ci & 1, kSpin, abort_flag)) {
          mok = false;
          break;
        }
        tc_fence_after();
        // K^T [dU'_hi | dU'_lo]: the state path
#pragma unroll
        for (int ks = 0; ks < C / 16; ++ks)
          umma_bf16(tm + TC_S, d_k + so + ((ks * 2048) >> 4), d_du + ((ks * 2048) >> 4), id_s, ks > 0);
        umma_commit(&sh.b1);
        sh.mma_bar = &sh.b1;
        sh.mma_par = ci & 1;
      }
      if (mok && !summary && n_chunks > 0) mok = issue_b2(n_chunks - 1);
      if (!mok) fail();
    }
  } else if (warp < 8) {
    // ===================================================== state path (warps 0-7)
    // warp w reads TMEM lanes 32 (w % 4) .. +31 and handles value columns 16 (w / 4) .. +15
    const int quarter = warp & 3, hc = warp >> 2;
    const uint32_t lq = (uint32_t)(quarter * 32) << 16;
    const int f = quarter * 32 + lane;  // key feature of this thread's state row
    const int cb = hc * 16;             // first value column of this thread (inside the block)
    float S[16];
    if (m_cols) {  // M starts at the identity
#pragma unroll
      for (int j = 0; j < 16; ++j) S[j] = (v0 + cb + j == f) ? 1.f : 0.f;
    } else {
      const float *h0p = (p.h0 && !summary) ? p.h0 + (((size_t)s * p.Hv + h) * p.V + v0 + cb) * KD + f : nullptr;
#pragma unroll
      for (int j = 0; j < 16; ++j) S[j] = h0p ? h0p[(size_t)j * KD] : 0.f;
    }
    auto write_state = [&]() {
#pragma unroll
      for (int m = 0; m < 2; ++m)
        *reinterpret_cast<uint4 *>(sm + SC_ST + sw64_off(f, cb + 8 * m)) =
            make_uint4(pack_bf16(S[8 * m], S[8 * m + 1]), pack_bf16(S[8 * m + 2], S[8 * m + 3]),
                       pack_bf16(S[8 * m + 4], S[8 * m + 5]), pack_bf16(S[8 * m + 6], S[8 * m + 7]));
    };
    write_state();
    fence_proxy_async_smem();
    warp_arrive(&sh.epb);
    bool ok = true;
    for (int ci = 0; ci < n_chunks; ++ci) {
      const int st = ci % kStages;
      const uint8_t *sg = sm + st * kStage;
      const float *vec = reinterpret_cast<const float *>(sg + ST_VEC);
      if (!warp_wait(&sh.full[st], (ci / kStages) & 1, kSpin, abort_flag)) {
        ok = false;
        break;
      }
      const int i = (quarter - 2) * 32 + lane;  // token of this lane (warps on lanes 64-127)
      float x[16];
      if (quarter >= 2) {
        // ---- U' = U - W S^T for tokens i: diag(d/|k|) U' hi/lo for the state path
        if (!warp_wait(&sh.ga, ci & 1, kSpin, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_ld16(tm + lq + TC_A + (ci % 3) * 32 + cb, x);
        const float4 *ur = reinterpret_cast<const float4 *>(sg + ST_U + i * 128);
        float4 u4[4];
#pragma unroll
        for (int m = 0; m < 4; ++m)  // rows are swizzled; M's columns have U = 0
          u4[m] = m_cols ? make_float4(0.f, 0.f, 0.f, 0.f) : ur[((cb >> 2) + m) ^ (i & 7)];
        const float dk = vec[VEC_DK + i];
        tmem_wait_ld();
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          x[4 * m] += u4[m].x;
          x[4 * m + 1] += u4[m].y;
          x[4 * m + 2] += u4[m].z;
          x[4 * m + 3] += u4[m].w;
        }
        uint32_t dh[8], dl[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) split_bf16(dk * x[2 * e], dk * x[2 * e + 1], dh[e], dl[e]);
        uint8_t *du = sm + SC_DU;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          *reinterpret_cast<uint4 *>(du + sw128_off(i, cb + 8 * m)) =
              make_uint4(dh[4 * m], dh[4 * m + 1], dh[4 * m + 2], dh[4 * m + 3]);
          *reinterpret_cast<uint4 *>(du + sw128_off(i, 32 + cb + 8 * m)) =
              make_uint4(dl[4 * m], dl[4 * m + 1], dl[4 * m + 2], dl[4 * m + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        warp_arrive(&sh.epa);
      }
      // ---- S <- b_last S + dS (fp32), and its bf16 copy for the next chunk's MMAs
      if (!warp_wait(&sh.b1, ci & 1, kSpin, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      {
        float dh[16], dl[16];
        tmem_ld16(tm + lq + TC_S + cb, dh);
        tmem_ld16(tm + lq + TC_S + 32 + cb, dl);
        const float bl = vec[VEC_BLAST];
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) S[j] = fmaf(bl, S[j], dh[j] + dl[j]);
        write_state();
        fence_proxy_async_smem();
        tc_fence_before();
        warp_arrive(&sh.epb);
      }
      if (quarter >= 2 && !summary) {
        // ---- U' hi/lo for the output path, once the previous chunk's output has read its tile
        if (ci > 0 && !warp_wait(&sh.outd, (ci - 1) & 1, kSpin, abort_flag)) {
          ok = false;
          break;
        }
        uint32_t uh[8], ul[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) split_bf16(x[2 * e], x[2 * e + 1], uh[e], ul[e]);
        uint8_t *up = sm + SC_UP;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          *reinterpret_cast<uint4 *>(up + sw128_off(i, cb + 8 * m)) =
              make_uint4(uh[4 * m], uh[4 * m + 1], uh[4 * m + 2], uh[4 * m + 3]);
          *reinterpret_cast<uint4 *>(up + sw128_off(i, 32 + cb + 8 * m)) =
              make_uint4(ul[4 * m], ul[4 * m + 1], ul[4 * m + 2], ul[4 * m + 3]);
        }
        fence_proxy_async_smem();
        warp_arrive(&sh.epa2);
      }
      tc_fence_before();
      warp_arrive(&sh.empty[st]);
    }
    if (!ok && lane == 0) fail();
    float *dst = nullptr;
    if (m_cols) dst = p.M + (((size_t)s * p.Hv + h) * KD + v0 + cb) * KD + f;
    else if (summary) dst = p.S_local + (((size_t)s * p.Hv + h) * p.V + uslice * VS + cb) * KD + f;
    else if (p.hT) dst = p.hT + (((size_t)s * p.Hv + h) * p.V + v0 + cb) * KD + f;
    if (ok && dst) {
#pragma unroll
      for (int j = 0; j < 16; ++j) dst[(size_t)j * KD] = S[j];
    }
  } else {
    // ===================================================== outputs (warps 8, 9, 12, 13)
    // o = alpha (q S^T) + P U' + diag(P) U' for tokens i = lanes 0-63
    const int quarter = warp & 3, hc = (warp >> 2) & 1;
    const uint32_t lq = (uint32_t)(quarter * 32) << 16;
    const int cb = hc * 16;
    const int i = quarter * 32 + lane;
    const size_t o_tok = (size_t)p.Hv * p.V;
    const uint32_t rank = NORM ? cluster_ctarank() : 0u, n_ranks = gridDim.x;
    float wv[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) wv[j] = (NORM && p.nw) ? __bfloat162float(p.nw[v0 + cb + j]) : 1.f;
    // the norm's z of this token's 16 columns, loaded a chunk ahead of its use
    auto load_z = [&](int cj, uint4 &za, uint4 &zb) {
      za = zb = make_uint4(0u, 0u, 0u, 0u);
      const int64_t tj = start + (int64_t)cj * C + i;
      if (cj < n_chunks && tj < end) {
        const uint4 *zp = reinterpret_cast<const uint4 *>(p.z + (size_t)tj * o_tok + (size_t)h * p.V + v0 + cb);
        za = __ldg(zp);
        zb = __ldg(zp + 1);
      }
    };
    uint4 zc0 = make_uint4(0u, 0u, 0u, 0u), zc1 = zc0;
    if (NORM && !summary) load_z(0, zc0, zc1);
    bool ok = true;
    for (int ci = 0; ci < n_chunks; ++ci) {
      const int st = ci % kStages;
      const uint8_t *sg = sm + st * kStage;
      const float *vec = reinterpret_cast<const float *>(sg + ST_VEC);
      if (!warp_wait(&sh.full[st], (ci / kStages) & 1, kSpin, abort_flag)) {
        ok = false;
        break;
      }
      if (summary) {  // no output: only release the stage
        tc_fence_before();
        warp_arrive(&sh.empty[st]);
        continue;
      }
      if (!warp_wait(&sh.b2, ci & 1, kSpin, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint4 zn0 = zc0, zn1 = zc1;
      if (NORM) load_z(ci + 1, zn0, zn1);
      float qs[16], ph[16], pl[16];
      tmem_ld16(tm + lq + TC_A + (ci % 3) * 32 + cb, qs);
      tmem_ld16(tm + lq + TC_O + cb, ph);
      tmem_ld16(tm + lq + TC_O + 32 + cb, pl);
      const uint8_t *up = sm + SC_UP;
      float uo[16];
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const uint4 hv = *reinterpret_cast<const uint4 *>(up + sw128_off(i, cb + 8 * m));
        const uint4 lv = *reinterpret_cast<const uint4 *>(up + sw128_off(i, 32 + cb + 8 * m));
        const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w}, lw[4] = {lv.x, lv.y, lv.z, lv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 a = unpack_bf16(hw[e]), b = unpack_bf16(lw[e]);
          uo[8 * m + 2 * e] = a.x + b.x;
          uo[8 * m + 2 * e + 1] = a.y + b.y;
        }
      }
      const float al = vec[VEC_ALPHA + i], pd = vec[VEC_PDIAG + i];
      const int64_t t0 = start + (int64_t)ci * C;
      const int nv = (int)min((int64_t)C, end - t0);
      tmem_wait_ld();
      float ov[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) ov[j] = fmaf(al, qs[j], fmaf(pd, uo[j], ph[j] + pl[j]));
      // o is in registers: the accumulator columns, the U' tile and the stage are free
      tc_fence_before();
      warp_arrive(&sh.outd);
      warp_arrive(&sh.empty[st]);
      if (NORM) {
        // ---- y = o / sqrt(mean_v o^2 + eps) * w * silu(z): this thread's 16 columns' sum of
        //      squares goes to every block of the cluster (slot ci % 2), whose barrier for that
        //      slot completes once all of a token's partials are in
        const uint4 zr0 = zc0, zr1 = zc1;
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) ss = fmaf(ov[j], ov[j], ss);
        const int slot = ci & 1;
        const uint32_t np_mine = sb + SC_NP + (uint32_t)((((slot * kNormRanks + (int)rank) * 2 + hc) * 64 + i) * 4);
        const uint32_t bar_mine = smem_u32(&sh.nbar[slot]);
        // this block's barrier for the slot expects every partial of the cluster: 128 output
        // threads a block, 4 bytes each (one arrival, by warp 8's lane 0)
        if (warp == 8 && lane == 0) mbar_arrive_expect_tx(&sh.nbar[slot], 128u * 4u * n_ranks);
        for (uint32_t r = 0; r < n_ranks; ++r) st_async_cluster_f32(mapa_shared(np_mine, r), ss, mapa_shared(bar_mine, r));
        const bool got = mbar_wait_cluster_spin(&sh.nbar[slot], (uint32_t)(ci >> 1) & 1, kSpin, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          ok = false;
          break;
        }
        const float *np = reinterpret_cast<const float *>(sm + SC_NP) + slot * kNormRanks * 2 * 64 + i;
        float tot = 0.f;  // the same order in every block
        for (uint32_t r = 0; r < n_ranks; ++r) tot += np[(r * 2) * 64] + np[(r * 2 + 1) * 64];
        const float inv = 1.f / sqrtf(tot * (1.f / (float)p.V) + p.eps);
        const uint32_t zw[8] = {zr0.x, zr0.y, zr0.z, zr0.w, zr1.x, zr1.y, zr1.z, zr1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 zz = unpack_bf16(zw[e]);
          ov[2 * e] = ov[2 * e] * inv * wv[2 * e] * __fdividef(zz.x, 1.f + __expf(-zz.x));
          ov[2 * e + 1] = ov[2 * e + 1] * inv * wv[2 * e + 1] * __fdividef(zz.y, 1.f + __expf(-zz.y));
        }
      }
      if (i < nv) {
        const size_t off = (size_t)(t0 + i) * o_tok + (size_t)h * p.V + v0 + cb;
        if (p.o_f32) {
          float4 *dst = reinterpret_cast<float4 *>((float *)p.o + off);
#pragma unroll
          for (int m = 0; m < 4; ++m) dst[m] = make_float4(ov[4 * m], ov[4 * m + 1], ov[4 * m + 2], ov[4 * m + 3]);
        } else {
          uint4 *dst = reinterpret_cast<uint4 *>((__nv_bfloat16 *)p.o + off);
#pragma unroll
          for (int m = 0; m < 2; ++m)
            dst[m] = make_uint4(pack_bf16(ov[8 * m], ov[8 * m + 1]), pack_bf16(ov[8 * m + 2], ov[8 * m + 3]),
                                pack_bf16(ov[8 * m + 4], ov[8 * m + 5]), pack_bf16(ov[8 * m + 6], ov[8 * m + 7]));
        }
      }
      zc0 = zn0;
      zc1 = zn1;
    }
    if (!ok && lane == 0) fail();
  }
  __syncthreads();
  if (tid == 0 && sh.abort) {
    // copies and MMAs still in flight land before shared memory and TMEM are released
    for (int i = 0; i < kStages; ++i)
      if (sh.fills[i] > 0) (void)mbar_wait(&sh.full[i], (sh.fills[i] - 1) & 1, kSpin);
    if (sh.mma_bar) (void)mbar_wait(sh.mma_bar, sh.mma_par, kSpin);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, kScanCols);
  if (NORM) cluster_sync_all();  // no block leaves while a peer may still write into it
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

}  // namespace

namespace gdn {

// [n_tok][heads][width] bf16 map with token stride `tok_stride` elements; 64 x 64 boxes, SW128.
bool make_tile_map(CUtensorMap *m, const void *base, int width, int heads, int64_t n_tok, int64_t tok_stride) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)heads, (cuuint64_t)n_tok};
  cuuint64_t strides[2] = {(cuuint64_t)width * 2, (cuuint64_t)tok_stride * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)C};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace gdn

namespace {

template <int V, bool FRONT = false>
gdn_status launch_operands(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                           const CUtensorMap &mqc, const CUtensorMap &mkc, const OpParams &op, size_t slots,
                           cudaStream_t st) {
  const size_t smem = op_smem(V);
  if (cudaFuncSetAttribute(chunk_operand_kernel<V, FRONT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess ||
      cudaFuncSetAttribute(chunk_operand_kernel<V, FRONT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return GDN_ERR_CUDA;
  const size_t items = slots * (size_t)op.Hv;
  if (items == 0) return GDN_OK;
  // resident blocks only: each walks the items with the grid's stride
  int dev = 0, sms = 0, smem_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess)
    return GDN_ERR_CUDA;
  // blocks an SM holds: shared memory (dynamic + 2 KB static + 1 KB reserved), at most 4
  // (128 registers x 128 threads each)
  const int per_sm = std::max(1, std::min(4, smem_sm / (int)(smem + 3072)));
  size_t grid = std::min(items, (size_t)sms * (size_t)per_sm);
  if (!op.front) {  // as few blocks as give the same number of rounds (strided items)
    const size_t rounds = (items + grid - 1) / grid;
    grid = (items + rounds - 1) / rounds;
  }
  OpParams q = op;
  q.n_items = (int64_t)items;
  if (q.front && cudaMemsetAsync(q.claim, 0, sizeof(*q.claim), st) != cudaSuccess) return GDN_ERR_CUDA;
  chunk_operand_kernel<V, FRONT><<<(unsigned)grid, 128, smem, st>>>(mq, mk, mv, mqc, mkc, q);
  return launch_status();
}

}  // namespace

namespace gdn {

// The split path handles bf16, K = 128 and V a multiple of 64 up to 256.
bool chunk_scan_supported(const void *q, const void *k, const void *v, const gdn_shape &sh) {
  if (sh.dtype != GDN_BF16 || sh.K != KD || sh.V % 64 != 0 || sh.V > 256) return false;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16)) return false;
  if ((sh.q_stride * 2) % 16 || (sh.k_stride * 2) % 16 || (sh.v_stride * 2) % 16) return false;
  const int64_t n_tok = (int64_t)sh.B * sh.T;
  return n_tok < (1LL << 31);
}

size_t chunk_scan_workspace_bytes(const gdn_shape &sh, int64_t n_tok) {
  return kHeader + n_slots(n_tok, sh.n_seqs) * (size_t)sh.Hv * rec_bytes(sh.V);
}

// The fused front end applies to the Qwen3.5 layer's shape on this path: bf16, K = V = 128,
// conv width up to 4, and x, the weights, a and b 16-byte aligned (bias and a/b rows any).
bool chunk_front_supported(const void *x, const void *w, int width, const gdn_shape &sh) {
  if (sh.dtype != GDN_BF16 || sh.K != KD || sh.V != 128 || width < 1 || width > 4) return false;
  if (!aligned(x, 16) || !aligned(w, 2)) return false;
  const int64_t n_tok = (int64_t)sh.B * sh.T;
  return n_tok < (1LL << 31);
}

size_t chunk_front_workspace_bytes(const gdn_shape &sh, int64_t n_tok) {
  return chunk_scan_workspace_bytes(sh, n_tok) + 2 * front_qk_bytes(sh, n_tok);
}


// Both kernels of the split path over `n_seqs` sequences (cu_seqlens `cu`, or rows of
// sh.T tokens): the operand records, then the state scan over (value-column blocks,
// v-heads, sequences).  Summary mode scans the K + V columns of [M; S_local] instead.
// With `fr` (the fused front end) q, k and v are unused: the operand kernel reads x, and the
// conv'd q and k it writes after the records feed the scan.
static gdn_status run_scan(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, const float *h0, const int32_t *cu, int n_seqs,
                           int64_t n_tok, const gdn_shape &sh, int64_t q_stride, float scale,
                           uint32_t flags, void *o, float *h_T, bool summary, float *M,
                           float *S_local, void *workspace, size_t ws_bytes, cudaStream_t st,
                           const FrontArgs *fr = nullptr, const NormArgs *nm = nullptr) {
  const size_t slots = n_slots(n_tok, n_seqs);
  const size_t rec_end = kHeader + slots * (size_t)sh.Hv * rec_bytes(sh.V);
  const size_t qk_bytes = fr ? front_qk_bytes(sh, n_tok) : 0;
  if (ws_bytes < rec_end + 2 * qk_bytes) return GDN_ERR_WORKSPACE;
  int32_t *status = (int32_t *)workspace;
  OpParams op{};
  op.q = (const __nv_bfloat16 *)q;
  op.k = (const __nv_bfloat16 *)k;
  op.v = (const __nv_bfloat16 *)v;
  op.qs = q_stride;
  op.ks = sh.k_stride;
  op.vs = sh.v_stride;
  op.g = g;
  op.beta = beta;
  op.cu = cu;
  op.row_T = sh.T;
  op.n_tok = n_tok;
  op.n_seqs = n_seqs;
  op.Hqk = sh.Hqk;
  op.Hv = sh.Hv;
  op.l2norm = (flags & GDN_FLAG_QK_L2NORM) ? 1 : 0;
  op.scale = scale;
  op.rec = (uint8_t *)workspace + kHeader;
  op.rec_bytes = rec_bytes(sh.V);
  op.status = status;
  op.claim = reinterpret_cast<unsigned long long *>((uint8_t *)workspace + 8);  // header bytes 8-15
  op.quit = (flags & GDN_FLAG_TEST_NO_WAIT) ? 1 : 0;
  CUtensorMap mq, mk, mv;
  if (fr) {
    const __nv_bfloat16 *x = (const __nv_bfloat16 *)fr->x;
    const int64_t Cx = (int64_t)2 * sh.Hqk * KD + (int64_t)sh.Hv * sh.V;
    op.front = 1;
    op.width = fr->width;
    op.x = x;
    op.cw = (const __nv_bfloat16 *)fr->w;
    op.cbias = (const __nv_bfloat16 *)fr->bias;
    op.Cx = Cx;
    op.ga = (const __nv_bfloat16 *)fr->a;
    op.gb = (const __nv_bfloat16 *)fr->b;
    op.A_log = fr->A_log;
    op.dt_bias = fr->dt_bias;
    op.qc = (__nv_bfloat16 *)((uint8_t *)workspace + rec_end);
    op.kc = (__nv_bfloat16 *)((uint8_t *)workspace + rec_end + qk_bytes);
    if (!make_tile_map(&mq, x, KD, sh.Hqk, n_tok, Cx) ||
        !make_tile_map(&mk, x + (int64_t)sh.Hqk * KD, KD, sh.Hqk, n_tok, Cx) ||
        !make_tile_map(&mv, x + (int64_t)2 * sh.Hqk * KD, sh.V, sh.Hv, n_tok, Cx))
      return GDN_ERR_CUDA;
  } else if (!make_tile_map(&mq, q, KD, sh.Hqk, n_tok, q_stride) ||
             !make_tile_map(&mk, k, KD, sh.Hqk, n_tok, sh.k_stride) ||
             !make_tile_map(&mv, v, sh.V, sh.Hv, n_tok, sh.v_stride)) {
    return GDN_ERR_CUDA;
  }
  // the front end's later items load the conv'd q and k back from the workspace
  CUtensorMap mqc = mq, mkc = mk;
  if (fr && (!make_tile_map(&mqc, op.qc, KD, sh.Hqk, n_tok, (int64_t)sh.Hqk * KD) ||
             !make_tile_map(&mkc, op.kc, KD, sh.Hqk, n_tok, (int64_t)sh.Hqk * KD)))
    return GDN_ERR_CUDA;
  gdn_status r;
  switch (sh.V) {
    case 64: r = launch_operands<64>(mq, mk, mv, mqc, mkc, op, slots, st); break;
    case 128:
      r = fr ? launch_operands<128, true>(mq, mk, mv, mqc, mkc, op, slots, st)
             : launch_operands<128>(mq, mk, mv, mqc, mkc, op, slots, st);
      break;
    case 192: r = launch_operands<192>(mq, mk, mv, mqc, mkc, op, slots, st); break;
    case 256: r = launch_operands<256>(mq, mk, mv, mqc, mkc, op, slots, st); break;
    default: return GDN_ERR_UNSUPPORTED;
  }
  if (r != GDN_OK) return r;
  ScanParams sp{};
  sp.cu = cu;
  sp.row_T = sh.T;
  sp.n_tok = n_tok;
  sp.Hqk = sh.Hqk;
  sp.Hv = sh.Hv;
  sp.V = sh.V;
  sp.h0 = h0;
  sp.rec = op.rec;
  sp.rec_bytes = op.rec_bytes;
  sp.o = o;
  sp.o_f32 = (flags & GDN_FLAG_O_F32) ? 1 : 0;
  sp.hT = h_T;
  sp.status = status;
  sp.summary = summary ? 1 : 0;
  sp.quit = op.quit;
  sp.M = M;
  sp.S_local = S_local;
  if (cudaFuncSetAttribute(chunk_scan_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kScanSmem) != cudaSuccess ||
      cudaFuncSetAttribute(chunk_scan_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kScanSmem) != cudaSuccess)
    return GDN_ERR_CUDA;
  const int cols = summary ? KD + sh.V : sh.V;
  if (fr) {
    mq = mqc;
    mk = mkc;
  }
  const dim3 grid(cols / VS, sh.Hv, n_seqs);
  // a programmatic dependent of the operand kernel only when that kernel ran (no items: no
  // launch, and the previous kernel on the stream is someone else's)
  const bool pdl = slots * (size_t)sh.Hv > 0;
  if (nm && !summary) {
    // the norm epilogue: the blocks of one (v-head, sequence) as one cluster
    sp.norm = 1;
    sp.z = (const __nv_bfloat16 *)nm->z;
    sp.nw = (const __nv_bfloat16 *)nm->w;
    sp.eps = nm->eps;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(NTS);
    cfg.dynamicSmemBytes = kScanSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = grid.x;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, chunk_scan_kernel<true>, mq, mk, sp) != cudaSuccess) return GDN_ERR_CUDA;
    return launch_status();
  }
  // launched as a programmatic dependent of the operand kernel: its launch and prologue overlap
  // that kernel's last items
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(NTS);
  cfg.dynamicSmemBytes = kScanSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, chunk_scan_kernel<false>, mq, mk, sp) != cudaSuccess) return GDN_ERR_CUDA;
  return launch_status();
}

// Whether a cluster of `ranks` scan blocks can be resident at once on the current device
// (asked once per device and cluster size).
static bool scan_cluster_fits(int ranks) {
  static int cached[8][kNormRanks + 1] = {};  // 0 unknown, 1 fits, 2 does not
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 8 || ranks < 1 || ranks > kNormRanks) return false;
  if (cached[dev][ranks] == 0) {
    bool fits = cudaFuncSetAttribute(chunk_scan_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)kScanSmem) == cudaSuccess;
    if (fits) {
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(ranks, 1, 1);
      cfg.blockDim = dim3(NTS);
      cfg.dynamicSmemBytes = kScanSmem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = ranks;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      fits = cudaOccupancyMaxActiveClusters(&n, chunk_scan_kernel<true>, &cfg) == cudaSuccess && n >= 1;
    }
    (void)cudaGetLastError();  // a refused query is an answer, not an error to report later
    cached[dev][ranks] = fits ? 1 : 2;
  }
  return cached[dev][ranks] == 1;
}

// The norm epilogue applies to the split scan's bf16 output with V <= 128 (V / 32 blocks of a
// head in one cluster, at most four) where such a cluster fits the device.
bool chunk_norm_supported(const gdn_shape &sh, uint32_t flags, const NormArgs &nm) {
  return sh.dtype == GDN_BF16 && sh.V % 64 == 0 && sh.V / VS <= kNormRanks && !(flags & GDN_FLAG_O_F32) &&
         aligned(nm.z, 16) && scan_cluster_fits(sh.V / VS);
}

gdn_status chunk_fwd_scan(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, const float *h0, const int32_t *cu,
                          const gdn_shape &sh, float scale, uint32_t flags, void *o, float *h_T,
                          void *workspace, size_t ws_bytes, cudaStream_t st, const NormArgs *nm) {
  const int64_t n_tok = cu ? sh.T : (int64_t)sh.B * sh.T;
  return run_scan(q, k, v, g, beta, h0, cu, sh.n_seqs, n_tok, sh, sh.q_stride, scale, flags, o,
                  h_T, false, nullptr, nullptr, workspace, ws_bytes, st, nullptr, nm);
}

// gdn_segment_summary on the split path: k stands in for q (no output is formed).
gdn_status summary_scan(const void *k, const void *v, const float *g, const float *beta,
                        const int32_t *bounds, int n_seg, const gdn_shape &sh, uint32_t flags,
                        float *M, float *S_local, void *workspace, size_t ws_bytes,
                        cudaStream_t st) {
  return run_scan(k, k, v, g, beta, nullptr, bounds, n_seg, sh.T, sh, sh.k_stride, 1.f, flags,
                  nullptr, nullptr, true, M, S_local, workspace, ws_bytes, st);
}

// gdn_layer_fwd's fused front end: conv, SiLU and gates inside the operand kernel.
gdn_status chunk_fwd_front(const FrontArgs &fr, const float *h0, const int32_t *cu, const gdn_shape &sh,
                           float scale, uint32_t flags, void *o, float *h_T, void *workspace,
                           size_t ws_bytes, cudaStream_t st, const NormArgs *nm) {
  const int64_t n_tok = cu ? sh.T : (int64_t)sh.B * sh.T;
  return run_scan(nullptr, nullptr, nullptr, nullptr, nullptr, h0, cu, sh.n_seqs, n_tok, sh, 0, scale,
                  flags | GDN_FLAG_QK_L2NORM, o, h_T, false, nullptr, nullptr, workspace, ws_bytes, st, &fr,
                  nm);
}

}  // namespace gdn
