// chunk_fused.cu -- gdn_chunk_fwd (bf16, K = V = 128, GDN_FLAG_FUSED) as one persistent
// kernel in which per-head state chains are fed by chunk builders running beside them.
//
// The chunk form of the gated delta rule ("Gated Delta Networks", chunkwise
// algorithm with the UT/WY transform), per chunk of C = 64 tokens and v-head,
// with raw (unnormalised) bf16 q, k and 1/|q|, 1/|k| applied in fp32:
//   gamma = inclusive cumsum of g,  b = exp(gamma),  d = exp(gamma_last - gamma)
//   A  = strictly-lower(diag(beta) K_hat K_hat^T * Gamma),  Gamma_ij = exp(gamma_i - gamma_j)
//   T  = (I + A)^-1 diag(beta),  W = T diag(b) K_hat,  U = T V
//   P  = scale (Q_hat K_hat^T * Gamma) on and below the diagonal
// and, with the chunk's start state S (V x K, fp32),
//   O      = scale diag(b) Q_hat S^T + P (U - W S^T)  =  Qt S^T + P U,  Qt = alpha Q - P W
//   S_next = b_last S + (U - W S^T)^T diag(d) K_hat    =  b_last S + Ut^T K - S What
// with alpha = scale b / |q|, Ut = diag(d / |k|) U and What = W^T diag(d / |k|) K.
// Written this way a chunk costs the state chain ONE dependent product, S What
// (K x K, whatever the chunk length), instead of two (W S^T, then U'^T D K).
//
// Roles (one CTA per SM, all resident: cooperative launch):
//  * chain CTAs, one per (sequence, v-head) item at a time: hold S in fp32 registers
//    and a bf16 copy of S in tensor memory as the A operand of
//        D   = Ut^T K  +  S_bf16 (-What)      (tcgen05, fp32 accumulate)
//        O^T = S_bf16 Qt^T  (+ the P U part computed by the builder)
//    then S <- b_last S + D in fp32.
//  * builder CTAs, two independent 128-thread lanes each: for one (chain, chunk)
//    unit at a time they load k, q, v by TMA, form the norms, the gates, [K;Q]K^T
//    (tcgen05), A, T by forward substitution, U and W (tcgen05), then What, (P W)^T,
//    (P U)^T (tcgen05) and write a record: -What, Ut (hi + lo bf16), Qt^T (bf16),
//    (P U)^T (fp32) and b_last, into a ring slot in the workspace that the chain
//    reads a few chunks later (the ring stays in L2).
// Hand-off: a builder waits until the chain has consumed the slot's previous
// record, writes, then releases the slot's ready flag (stream position + 1); the
// chain acquires it, bulk-copies the record into shared memory, and releases its
// consumed count once the output of that chunk is stored.  Every wait is bounded
// and ends the kernel with GDN_ERR_TIMEOUT in the status word.
//
// Precision (chosen by an emulation of every rounding point): T as hi + lo bf16
// for U, T diag(b/|k|) as bf16 for W; P as hi + lo in the P U product (its
// diagonal carries most of o under strong decay); Ut as bf16 with its lo half
// added on the last chunk of each sequence, so h_T keeps the fp32 increment;
// What, Qt, S as bf16 operands; every accumulation fp32; the state fp32.
#include <cooperative_groups.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <math.h>

#include "chunk_common.cuh"
#include "common.cuh"
#include "sm100.cuh"

using namespace gdn;
using namespace gdn::sm100;

namespace {

constexpr int C = kChunk;  // 64 tokens per chunk
constexpr int KD = 128;    // key width
constexpr int VD = 128;    // value width
constexpr int NT = 320;    // threads per CTA: 10 warps
constexpr uint32_t kSpinDefault = 1u << 22;
constexpr size_t kHeader = 256;  // status word + padding

// ------------------------------------------------------------ ring record
// One record per (chain, stream position), in a ring slot of the workspace.  The first
// REC_SMEM bytes are laid out exactly as the chain's shared-memory stage (1 KB aligned
// images, 128-byte swizzle), so one bulk copy moves them.
constexpr uint32_t REC_WN = 0;        // -What: [2 f-halves][128 k rows][128 B] bf16 (B operand, N-major)
constexpr uint32_t REC_UTH = 32768;   // Ut hi: [2 v-halves][64 token rows][128 B] (A operand, M-major)
constexpr uint32_t REC_UTL = 49152;   // Ut lo, same layout
constexpr uint32_t REC_QT = 65536;    // Qt^T: [128 k rows][128 B = 64 tokens] (B operand, N-major)
constexpr uint32_t REC_VEC = 81920;   // b_last (fp32) and padding
constexpr uint32_t REC_K = 82944;     // raw k: [2 f-halves][64 token rows][128 B] (B operand, N-major)
constexpr uint32_t REC_SMEM = 99328;  // bytes the chain copies to shared memory
constexpr uint32_t REC_OP = 99328;    // (P U)^T: [128 v][64 tokens] fp32, read by the chain's output warps
constexpr uint32_t REC_BYTES = 132096;

// chain stage in shared memory: the record's first REC_SMEM bytes
constexpr uint32_t ST_K = REC_K;
constexpr uint32_t kStage = REC_SMEM;
constexpr int kStages = 2;
// chain TMEM columns
constexpr uint32_t T_DCH = 0;    // 2 x 128: D = Ut^T K - S What, lane = v, column = key feature
constexpr uint32_t T_DOUT = 256; // 2 x 64: O^T's S part, lane = v, column = token
constexpr uint32_t T_SHI = 384;  // 2 x 64: S as packed bf16 pairs, lane = v (A operand)

// builder lane region in shared memory (two lanes per CTA)
constexpr uint32_t B_KQ = 0;        // [2 halves][128 rows][128 B]: rows 0-63 raw k (later d/|k| k), 64-127 raw q
constexpr uint32_t B_V = 32768;     // [2 halves][64 rows][128 B] raw v; later U hi (same layout)
constexpr uint32_t B_X = 49152;     // A, then (I + A)^-1: fp32 [64][68]; later U lo
constexpr uint32_t B_TH = 66560;    // T hi [64][128 B]; with B_TL later W bf16 [2 halves][64 rows][128 B]
constexpr uint32_t B_TL = 74752;    // T lo
constexpr uint32_t B_TPH = 82944;   // T diag(b/|k|) as bf16
constexpr uint32_t B_PH = 91136;    // P hi [64 rows][128 B]
constexpr uint32_t B_PL = 99328;    // P lo
constexpr uint32_t B_SMALL = 107520;
constexpr uint32_t kLane = 110592;  // bytes per builder lane (1 KB multiple)
constexpr uint32_t kDynSmem = 2 * kLane + 1024;
constexpr int kXP = C + 4;          // padded fp32 row of A

static_assert(kStages * kStage <= 2 * kLane, "chain stages fit in the builder footprint");
static_assert(B_X + C * kXP * 4 <= B_TH, "A fits its region");
static_assert(B_X + 16384 <= B_TH, "U lo fits A's region");
static_assert(REC_OP + 128 * 64 * 4 == REC_BYTES, "record size");
static_assert(REC_BYTES % 1024 == 0 && REC_SMEM % 16 == 0, "record alignment");

// small per-lane vectors (float offsets inside B_SMALL)
constexpr int SM_GAM = 0, SM_BEX = 64, SM_DEC = 128, SM_ALF = 192, SM_KINV = 260, SM_QINV = 324,
              SM_BET = 388, SM_ALPHA = 452, SM_DK = 516, SM_MISC = 580;  // misc: blast, unit ints
constexpr int SM_BAR = 640;  // two mbarriers (8-byte aligned: float index 640 = byte 2560)
static_assert(SM_MISC + 2 * 8 + 1 <= SM_BAR, "unit words and b_last");
static_assert(SM_BAR * 4 + 16 <= 3072, "small region");

struct FfCtl {  // at the start of the fused path's control area
  int32_t counter;  // next unit to claim
  int32_t maxN;     // longest chain stream
  int32_t abort;    // set by any CTA that gave up
  int32_t pad;
};

struct FfParams {
  const float *g, *beta, *h0;
  const int32_t *cu;
  int64_t row_T, n_tok;
  int n_seqs, Hqk, Hv, n_items, n_chain, R;
  float scale;
  int l2norm, o_f32;
  void *o;
  float *hT;
  FfCtl *ctl;
  int32_t *consumed, *ready, *P0, *nch, *chainN;
  uint8_t *ring;
  int32_t *status;
  uint32_t spin;  // polls of every bounded wait (0: give up at once; a test mode)
};

// ------------------------------------------------------------ small helpers

__device__ __forceinline__ int ld_acquire(const int32_t *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int32_t *p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed(int32_t *p, int v) {
  asm volatile("st.relaxed.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }

// Waits until *flag >= want (acquire), polling at most `limit` times; gives up early when
// another CTA has aborted.  Returns false on give-up.
__device__ __forceinline__ bool wait_flag_ge(const int32_t *flag, int want, uint32_t limit,
                                             const FfCtl *ctl) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (ld_acquire(flag) >= want) return true;
    if ((i & 63) == 63 && *(volatile const int32_t *)&ctl->abort) return false;
    if (i > 16) __nanosleep(64);
  }
  return false;
}

__device__ __forceinline__ void give_up(FfParams &p, volatile int *local_abort) {
  if (local_abort) *local_abort = 1;
  *(volatile int32_t *)&p.ctl->abort = 1;
  set_status(p.status, GDN_ERR_TIMEOUT);
}

// D[tmem] (+)= A[tmem] * B[smem]: the A operand read from tensor memory.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 32 columns of 32-bit data to TMEM (thread i of the warp writes lane quarter + i).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// 32 lanes x 32 columns of 32-bit TMEM data (thread i of the warp reads lane quarter + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<uint32_t *>(&h);
  lo = *reinterpret_cast<uint32_t *>(&l);
}

__device__ __forceinline__ void warp_arrive(uint64_t *bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// The item (sequence s, v-head h) and chunk of stream position `pos` of chain `ci`, or
// false when the chain's stream is shorter.
struct Unit {
  int s, h, c, last;
  int64_t t0;
  int n;
};
__device__ __forceinline__ bool decode_unit(const FfParams &p, int ci, int pos, Unit &u) {
  if (pos >= p.chainN[ci]) return false;
  const int n_r = (p.n_items - ci + p.n_chain - 1) / p.n_chain;  // items of this chain
  int lo = 0, hi = n_r - 1;  // largest r with P0[ci + r n_chain] <= pos
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.P0[ci + mid * p.n_chain] <= pos) lo = mid; else hi = mid - 1;
  }
  const int j = ci + lo * p.n_chain;
  u.s = j / p.Hv;
  u.h = j % p.Hv;
  u.c = pos - p.P0[j];
  u.last = (u.c == p.nch[j] - 1);
  int64_t start, end;
  seq_range(p.cu, p.row_T, u.s, start, end);
  u.t0 = start + (int64_t)u.c * C;
  u.n = (int)min((int64_t)C, end - u.t0);
  return true;
}

// Y = (I + A)^-1 for the strictly lower 64 x 64 A in X (row stride kXP), by forward
// substitution swept over the columns of A; each of the lane's 128 threads keeps an
// 8 x 4 tile of Y (rows rg + 8 m, columns 16 a + cj: one in each 16-column block) and reads
// row k of Y from its owner by shuffle.  Row k is zero right of column k, so step k updates
// only the blocks a <= k / 16, a bound fixed at compile time and the same for every warp.
// Y is left in X, zero above the diagonal.  `bar` syncs the lane's threads.
template <typename Bar>
__device__ __forceinline__ void invert_unit_lower(float *X, int tid, Bar bar) {
  const int lane = tid & 31, rg = lane & 7, cj = (tid >> 5) * 4 + (lane >> 3);
  float y[8][4];
#pragma unroll
  for (int m = 0; m < 8; ++m)
#pragma unroll
    for (int a = 0; a < 4; ++a) y[m][a] = (rg + 8 * m == 16 * a + cj) ? 1.f : 0.f;
  const float *xr = X + rg * kXP;
#pragma unroll
  for (int k = 0; k < C - 1; ++k) {
    float yk[4];
#pragma unroll
    for (int a = 0; a <= (k >> 4); ++a) yk[a] = __shfl_sync(0xffffffffu, y[k >> 3][a], (k & 7) | (lane & 24));
#pragma unroll
    for (int m = k >> 3; m < 8; ++m) {
      const float av = xr[8 * m * kXP + k];
#pragma unroll
      for (int a = 0; a <= (k >> 4); ++a) y[m][a] = fmaf(-av, yk[a], y[m][a]);
    }
  }
  bar();
#pragma unroll
  for (int m = 0; m < 8; ++m)
#pragma unroll
    for (int a = 0; a < 4; ++a) X[(rg + 8 * m) * kXP + 16 * a + cj] = y[m][a];
  bar();
}

// ============================================================ builder lane

// bulk copies shared -> global, tracked per issuing thread in bulk async-groups
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(ssrc)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// every committed group has finished reading shared memory
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// all but the newest committed group have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// every committed group has completed its writes
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// decoded unit (ints): valid (1) or none left (-1), chain, position, v-head, tokens, first token
constexpr int U_VALID = 0, U_CI = 1, U_POS = 2, U_H = 3, U_N = 4, U_T0 = 5, U_WORDS = 8;
// mbarriers of a builder lane (in its small region, 8-byte aligned)
constexpr int BB_LD = 0, BB_MMA = 1, BB_CLAIMED = 2 /* two: even and odd units */, BB_STAGED_A = 4,
              BB_UFREE = 5, BB_STAGED_B = 6, BB_KSAVED = 7, BB_COUNT = 8;
static_assert(SM_BAR * 4 + BB_COUNT * 8 <= 3072, "lane barriers fit the small region");

// Claims units until one is real (a chain's stream can be shorter than the longest).
__device__ __forceinline__ void claim_unit(const FfParams &p, int64_t total, int *u_out) {
  int valid = -1;
  Unit un{};
  int ci = 0, pos = 0;
  while (!*(volatile int32_t *)&p.ctl->abort) {
    const int u = atomicAdd(&p.ctl->counter, 1);
    if ((int64_t)u >= total) break;
    ci = u % p.n_chain;
    pos = u / p.n_chain;
    if (decode_unit(p, ci, pos, un)) {
      valid = 1;
      break;
    }
  }
  u_out[U_CI] = ci;
  u_out[U_POS] = pos;
  u_out[U_H] = un.h;
  u_out[U_N] = un.n;
  u_out[U_T0] = (int)un.t0;
  u_out[U_VALID] = valid;
}

// A bounded wait that also gives up once any CTA has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, uint32_t limit, const FfCtl *ctl) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 63 && *(volatile const int32_t *)&ctl->abort) return false;
    if (i > 64) __nanosleep(32);
  }
  return false;
}

struct LaneRefs {
  float *smf;
  int *ring;  // [2][U_WORDS]: units 2 i and 2 i + 1 alternate
  float *blast;
  uint64_t *bars;
};
__device__ __forceinline__ LaneRefs lane_refs(uint8_t *sm) {
  LaneRefs r;
  r.smf = reinterpret_cast<float *>(sm + B_SMALL);
  r.ring = reinterpret_cast<int *>(r.smf + SM_MISC);
  r.blast = r.smf + SM_MISC + 2 * U_WORDS;
  r.bars = reinterpret_cast<uint64_t *>(r.smf + SM_BAR);
  return r;
}

// The helper of a builder lane (one thread): claims units two ahead, loads each unit's
// k, q, v tiles by TMA, writes each staged record to its ring slot by bulk copies (after the
// chain has consumed the slot's previous record) and releases the slot's ready flag once the
// copies have landed.  The lane itself only computes and stages.
__device__ void builder_helper(const CUtensorMap *tm_q, const CUtensorMap *tm_k, const CUtensorMap *tm_v,
                               FfParams &p, uint8_t *sm) {
  LaneRefs L = lane_refs(sm);
  uint64_t *ld_bar = L.bars + BB_LD;
  const int64_t total = (int64_t)p.n_chain * (int64_t)p.ctl->maxN;
  auto issue_tma = [&](const int *u) {
    const int h = u[U_H], qh = h / (p.Hv / p.Hqk);
    const int32_t tt = u[U_T0];
    mbar_arrive_expect_tx(ld_bar, 6 * 8192);
    tma_load_3d(sm + B_KQ, tm_k, ld_bar, 0, qh, tt);
    tma_load_3d(sm + B_KQ + 16384, tm_k, ld_bar, 64, qh, tt);
    tma_load_3d(sm + B_KQ + 8192, tm_q, ld_bar, 0, qh, tt);
    tma_load_3d(sm + B_KQ + 24576, tm_q, ld_bar, 64, qh, tt);
    tma_load_3d(sm + B_V, tm_v, ld_bar, 0, h, tt);
    tma_load_3d(sm + B_V + 8192, tm_v, ld_bar, 64, h, tt);
  };
  claim_unit(p, total, L.ring);
  mbar_arrive(L.bars + BB_CLAIMED);
  claim_unit(p, total, L.ring + U_WORDS);
  mbar_arrive(L.bars + BB_CLAIMED + 1);
  int tma_issued = 0;
  if (L.ring[U_VALID] > 0) {
    issue_tma(L.ring);
    tma_issued = 1;
  }
  bool ok = true;
  for (int i = 0;; ++i) {
    int *u = L.ring + (i & 1) * U_WORDS;
    if (u[U_VALID] <= 0) break;
    const int ci = u[U_CI], pos = u[U_POS], slot = pos % p.R;
    uint8_t *rec = p.ring + ((size_t)ci * p.R + slot) * REC_BYTES;
    // the slot is free and the unit's tiles have landed: the raw k rows go to the record
    // before the lane scales them in place
    ok = wait_flag_ge(p.consumed + ci, pos - p.R + 1, p.spin, p.ctl) && wait_bar(ld_bar, i & 1, p.spin, p.ctl);
    if (!ok) break;
    bulk_store(rec + REC_K, sm + B_KQ, 8192);
    bulk_store(rec + REC_K + 8192, sm + B_KQ + 16384, 8192);
    bulk_commit();
    bulk_wait_read0();
    mbar_arrive(L.bars + BB_KSAVED);
    if (!wait_bar(L.bars + BB_STAGED_A, i & 1, p.spin, p.ctl)) {
      ok = false;
      break;
    }
    bulk_store(rec + REC_UTH, sm + B_V, 16384);
    bulk_store(rec + REC_UTL, sm + B_X, 16384);
    bulk_commit();
    bulk_store(rec + REC_WN, sm + B_TH, 32768);
    bulk_store(rec + REC_QT, sm + B_KQ, 8192);
    bulk_store(rec + REC_QT + 8192, sm + B_KQ + 16384, 8192);
    bulk_commit();
    *reinterpret_cast<float *>(rec + REC_VEC) = *L.blast;
    bulk_wait_read1();  // the U images have been read: the lane may put (P U)^T there
    mbar_arrive(L.bars + BB_UFREE);
    claim_unit(p, total, u);  // unit i + 2 into the entry unit i used
    mbar_arrive(L.bars + BB_CLAIMED + (i & 1));
    if (!wait_bar(L.bars + BB_STAGED_B, i & 1, p.spin, p.ctl)) {
      ok = false;
      break;
    }
    bulk_store(rec + REC_OP, sm + B_V, 32768);
    bulk_commit();
    bulk_wait_read0();  // the lane's tiles are free for the next unit
    const int *un = L.ring + ((i + 1) & 1) * U_WORDS;
    if (un[U_VALID] > 0) {
      issue_tma(un);
      ++tma_issued;
    }
    bulk_wait_all();
    fence_proxy_async_all();
    __threadfence();
    st_release(p.ready + (size_t)ci * p.R + slot, pos + 1);
  }
  if (!ok) give_up(p, nullptr);
  bulk_wait_all();  // no copy may still read shared memory when the CTA exits
  if (tma_issued > 0) (void)mbar_wait(ld_bar, (tma_issued - 1) & 1, kSpinDefault);
}

__device__ void builder_lane(FfParams &p, uint8_t *sm, uint32_t tm, int lane_id) {
  const int tid = threadIdx.x - 128 * lane_id;  // 0..127 inside the lane
  const int lane = tid & 31, wq = tid >> 5;      // wq = TMEM lane quarter of this warp
  const uint32_t bid = 1 + lane_id;              // named barrier of the lane
  auto bar = [&]() { named_bar_sync(bid, 128); };
  LaneRefs L = lane_refs(sm);
  float *smf = L.smf;
  float *gam = smf + SM_GAM, *bex = smf + SM_BEX, *dec = smf + SM_DEC, *alf = smf + SM_ALF;
  float *kinv = smf + SM_KINV, *qinv = smf + SM_QINV, *bet = smf + SM_BET, *alpha = smf + SM_ALPHA;
  float *dk = smf + SM_DK;
  uint64_t *ld_bar = L.bars + BB_LD, *mma_bar = L.bars + BB_MMA;
  float *X = reinterpret_cast<float *>(sm + B_X);
  const uint32_t sb = smem_u32(sm);
  const uint32_t lq = (uint32_t)(wq * 32) << 16;
  const uint32_t R0 = tm, R1 = tm + 128;
  uint32_t mp = 0;
  // thread 0 waits on an mbarrier phase; every thread learns the outcome.  An MMA or copy
  // still in flight after a give-up lands before the lane leaves.
  auto lane_wait = [&](uint64_t *b, uint32_t parity, bool drain) -> bool {
    bool ok = true;
    if (tid == 0) ok = wait_bar(b, parity, p.spin, p.ctl);
    if (named_bar_any(bid, 128, !ok)) {
      if (tid == 0) {
        give_up(p, nullptr);
        if (drain) (void)mbar_wait(b, parity, kSpinDefault);
      }
      return false;
    }
    return true;
  };
  // gates of a unit: zero past the chunk's end (beta = 0 keeps those rows out of every result,
  // g = 0 keeps the decays of the real rows)
  auto gate_of = [&](const int *u) -> float {
    const int n = u[U_N], h = u[U_H];
    const int64_t t0 = u[U_T0];
    if (tid < C) return (tid < n) ? p.g[(t0 + tid) * p.Hv + h] : 0.f;
    return (tid - C < n) ? p.beta[(t0 + tid - C) * p.Hv + h] : 0.f;
  };
  float gnext = 0.f;
  bool failed_mid = false;
#pragma unroll 1
  for (int i = 0;; ++i) {
    if (!lane_wait(L.bars + BB_CLAIMED + (i & 1), (i >> 1) & 1, false)) break;
    const int *u = L.ring + (i & 1) * U_WORDS;
    if (u[U_VALID] <= 0) break;
    const int n = u[U_N];
    const float gv = i == 0 ? gate_of(u) : gnext;
    if (tid < C) gam[tid] = gv;
    else bet[tid - C] = gv;
    if (!lane_wait(ld_bar, i & 1, false)) break;

    // ---- 1/|k| and 1/|q| (two threads per token)
    {
      const int r = tid >> 1, hf = tid & 1;
      float sk = 0.f, sq = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 kr = *reinterpret_cast<const uint4 *>(sm + B_KQ + hf * 16384 + sw128_off(r, j * 8));
        const uint4 qr = *reinterpret_cast<const uint4 *>(sm + B_KQ + hf * 16384 + 8192 + sw128_off(r, j * 8));
        const uint32_t wk[4] = {kr.x, kr.y, kr.z, kr.w}, wqv[4] = {qr.x, qr.y, qr.z, qr.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 a = unpack_bf16(wk[e]), b = unpack_bf16(wqv[e]);
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
    bar();
    tc_fence_after();
    const uint32_t kq = sb + B_KQ;
    // ---- [K; Q] K^T: M = 128 (k rows, then q rows), N = 64, K = 128
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
      for (int ks = 0; ks < KD / 16; ++ks) {
        const uint32_t off = (ks >> 2) * 16384 + (ks & 3) * 32;
        umma_bf16(R0, smem_desc(kq + off, 16, 1024, 2), smem_desc(kq + off, 16, 1024, 2), id, ks > 0);
      }
      umma_commit(mma_bar);
    }
    // ---- gates: inclusive cumsum of g and the exponentials
    if (wq == 0) {
      const float g0 = gam[2 * lane], g1 = gam[2 * lane + 1];
      float incl = g0 + g1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float uu = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += uu;
      }
      const float last = __shfl_sync(0xffffffffu, incl, 31);
      const float ga = incl - g1, gb = incl;
      gam[2 * lane] = ga;  // the inclusive cumulative sum from here on
      gam[2 * lane + 1] = gb;
      bex[2 * lane] = expf(ga);
      bex[2 * lane + 1] = expf(gb);
      dec[2 * lane] = expf(last - ga);
      dec[2 * lane + 1] = expf(last - gb);
      alf[2 * lane] = expf(g0);
      alf[2 * lane + 1] = expf(g1);
      if (lane == 31) {
        *L.blast = expf(last);
        alf[C] = 1.f;
      }
    }
    if (!lane_wait(mma_bar, mp & 1, true)) break;
    ++mp;
    tc_fence_after();
    if (tid < C) {
      alpha[tid] = p.scale * bex[tid] * qinv[tid];
      dk[tid] = (tid < n) ? dec[tid] * kinv[tid] : 0.f;
    }
    // ---- rows of K K^T (lanes 0-63) become rows of A; rows of Q K^T (lanes 64-127) rows of P
    {
      const int ii = tid & 63;
      const bool isq = tid >= 64;
      float r64[64];
      tmem_ld64(R0 + lq, r64);
      tmem_wait_ld();
      const float bi = isq ? p.scale * qinv[ii] : bet[ii] * kinv[ii];
      const float gi = gam[ii];
      // Gamma_ij = exp(gamma_i - gamma_j) <= 1 for j <= i (every g <= 0), each independent
#pragma unroll
      for (int j = 0; j < C; ++j) {
        const bool keep = isq ? (j <= ii) : (j < ii);
        r64[j] = keep ? bi * kinv[j] * expf(gi - gam[j]) * r64[j] : 0.f;
      }
      if (!isq) {
        float4 *xr = reinterpret_cast<float4 *>(X + ii * kXP);
#pragma unroll
        for (int m = 0; m < C / 4; ++m) xr[m] = make_float4(r64[4 * m], r64[4 * m + 1], r64[4 * m + 2], r64[4 * m + 3]);
      } else {
#pragma unroll
        for (int c0 = 0; c0 < C; c0 += 8) {
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split2(r64[c0 + 2 * e], r64[c0 + 2 * e + 1], hw[e], lw[e]);
          *reinterpret_cast<uint4 *>(sm + B_PH + sw128_off(ii, c0)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4 *>(sm + B_PL + sw128_off(ii, c0)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
    }
    bar();
    // ---- (I + A)^-1
    invert_unit_lower(X, tid, bar);
    // ---- T = (I + A)^-1 diag(beta) as hi + lo bf16, T diag(b/|k|) as bf16 (K-major images)
    {
      const int r = tid & 63, cb = (tid >> 6) * 32;
      float t[32];
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        const float4 a = reinterpret_cast<const float4 *>(X + r * kXP + cb)[m];
        t[4 * m] = a.x;
        t[4 * m + 1] = a.y;
        t[4 * m + 2] = a.z;
        t[4 * m + 3] = a.w;
      }
#pragma unroll
      for (int q8 = 0; q8 < 4; ++q8) {
        uint32_t wh[4], wl[4], xh[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int u0 = q8 * 8 + 2 * e, c0 = cb + u0;
          const float t_0 = (c0 <= r) ? t[u0] * bet[c0] : 0.f;
          const float t_1 = (c0 + 1 <= r) ? t[u0 + 1] * bet[c0 + 1] : 0.f;
          split2(t_0, t_1, wh[e], wl[e]);
          xh[e] = pack_bf16(t_0 * bex[c0] * kinv[c0], t_1 * bex[c0 + 1] * kinv[c0 + 1]);
        }
        const uint32_t off = sw128_off(r, cb + q8 * 8);
        *reinterpret_cast<uint4 *>(sm + B_TH + off) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        *reinterpret_cast<uint4 *>(sm + B_TL + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        *reinterpret_cast<uint4 *>(sm + B_TPH + off) = make_uint4(xh[0], xh[1], xh[2], xh[3]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    bar();
    tc_fence_after();
    // ---- U = T V (hi + lo) into R0, W = T diag(b/|k|) K into R1 (M = 64, N = 128)
    if (tid == 0) {
      const uint32_t id = idesc_bf16(64, 128, false, true);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks) {
        const uint64_t vb = smem_desc(sb + B_V + ks * 2048, 8192, 1024, 2);
        umma_bf16(R0, smem_desc(sb + B_TH + ks * 32, 16, 1024, 2), vb, id, ks > 0);
        umma_bf16(R0, smem_desc(sb + B_TL + ks * 32, 16, 1024, 2), vb, id, 1);
      }
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks)
        umma_bf16(R1, smem_desc(sb + B_TPH + ks * 32, 16, 1024, 2), smem_desc(kq + ks * 2048, 16384, 1024, 2),
                  id, ks > 0);
      umma_commit(mma_bar);
    }
    if (!lane_wait(mma_bar, mp & 1, true)) break;
    ++mp;
    tc_fence_after();
    // ---- rows of U (hi + lo) and W (bf16) into shared memory (an M = 64 result: lanes 0-15
    //      of each quarter); k rows become diag(d/|k|) k for What = W^T diag(d/|k|) K
    {
      const int rr = wq * 16 + lane;
      const bool has_row = lane < 16;
#pragma unroll 1
      for (int hv = 0; hv < 2; ++hv) {
        float uu[64];
        tmem_ld64(R0 + lq + hv * 64, uu);
        tmem_wait_ld();
        if (has_row) {
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 8) {
            uint32_t uh[4], ul[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) split2(uu[c0 + 2 * e], uu[c0 + 2 * e + 1], uh[e], ul[e]);
            const uint32_t off = hv * 8192 + sw128_off(rr, c0);
            *reinterpret_cast<uint4 *>(sm + B_V + off) = make_uint4(uh[0], uh[1], uh[2], uh[3]);
            *reinterpret_cast<uint4 *>(sm + B_X + off) = make_uint4(ul[0], ul[1], ul[2], ul[3]);
          }
        }
        tmem_ld64(R1 + lq + hv * 64, uu);
        tmem_wait_ld();
        if (has_row) {
#pragma unroll
          for (int c0 = 0; c0 < 64; c0 += 8)
            *reinterpret_cast<uint4 *>(sm + B_TH + hv * 8192 + sw128_off(rr, c0)) =
                make_uint4(pack_bf16(uu[c0], uu[c0 + 1]), pack_bf16(uu[c0 + 2], uu[c0 + 3]),
                           pack_bf16(uu[c0 + 4], uu[c0 + 5]), pack_bf16(uu[c0 + 6], uu[c0 + 7]));
        }
      }
      if (!lane_wait(L.bars + BB_KSAVED, i & 1, false)) {
        failed_mid = true;
      } else {
        const int r = tid >> 1, hf = tid & 1;
        const float sc = dk[r];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint4 *ptr = reinterpret_cast<uint4 *>(sm + B_KQ + hf * 16384 + sw128_off(r, j * 8));
          const uint4 kr = *ptr;
          const float2 a = unpack_bf16(kr.x), b = unpack_bf16(kr.y), c = unpack_bf16(kr.z), d = unpack_bf16(kr.w);
          *ptr = make_uint4(pack_bf16(sc * a.x, sc * a.y), pack_bf16(sc * b.x, sc * b.y), pack_bf16(sc * c.x, sc * c.y),
                            pack_bf16(sc * d.x, sc * d.y));
        }
      }
    }
    if (failed_mid) break;
    fence_proxy_async_smem();
    tc_fence_before();
    bar();
    tc_fence_after();
    // ---- (P U)^T and (P W)^T into R0 (N = 64 each), What = W^T diag(d/|k|) K into R1
    if (tid == 0) {
      const uint32_t id_p = idesc_bf16(128, 64, true, false);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks) {
        const uint64_t ph = smem_desc(sb + B_PH + ks * 32, 16, 1024, 2);
        const uint64_t pl = smem_desc(sb + B_PL + ks * 32, 16, 1024, 2);
        const uint64_t uh = smem_desc(sb + B_V + ks * 2048, 8192, 1024, 2);
        const uint64_t ul = smem_desc(sb + B_X + ks * 2048, 8192, 1024, 2);
        umma_bf16(R0, uh, ph, id_p, ks > 0);
        umma_bf16(R0, ul, ph, id_p, 1);
        umma_bf16(R0, uh, pl, id_p, 1);
      }
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks)
        umma_bf16(R0 + 64, smem_desc(sb + B_TH + ks * 2048, 8192, 1024, 2),
                  smem_desc(sb + B_PH + ks * 32, 16, 1024, 2), id_p, ks > 0);
      const uint32_t id_w = idesc_bf16(128, 128, true, true);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks)
        umma_bf16(R1, smem_desc(sb + B_TH + ks * 2048, 8192, 1024, 2), smem_desc(kq + ks * 2048, 16384, 1024, 2),
                  id_w, ks > 0);
      umma_commit(mma_bar);
    }
    // the next unit's gates, loaded while the MMAs run (its claim was made a unit earlier)
    if (!lane_wait(L.bars + BB_CLAIMED + ((i + 1) & 1), ((i + 1) >> 1) & 1, false)) {
      if (tid == 0) (void)mbar_wait(mma_bar, mp & 1, kSpinDefault);
      break;
    }
    {
      const int *un = L.ring + ((i + 1) & 1) * U_WORDS;
      if (un[U_VALID] > 0) gnext = gate_of(un);
    }
    if (!lane_wait(mma_bar, mp & 1, true)) break;
    ++mp;
    tc_fence_after();
    // ---- the record, staged in shared memory for the helper's bulk copies:
    // (1) Ut = diag(d/|k|) U as hi + lo, in place over the U images (16-byte pieces)
#pragma unroll 2
    for (int c16 = tid; c16 < 1024; c16 += 128) {
      const uint32_t off = (uint32_t)c16 * 16;
      const float sc = dk[(off & 8191) >> 7];
      uint4 *ph = reinterpret_cast<uint4 *>(sm + B_V + off), *pl = reinterpret_cast<uint4 *>(sm + B_X + off);
      const uint4 h4 = *ph, l4 = *pl;
      const uint32_t hw[4] = {h4.x, h4.y, h4.z, h4.w}, lw[4] = {l4.x, l4.y, l4.z, l4.w};
      uint32_t oh[4], ol[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 a = unpack_bf16(hw[e]), b = unpack_bf16(lw[e]);
        split2(sc * (a.x + b.x), sc * (a.y + b.y), oh[e], ol[e]);
      }
      *ph = make_uint4(oh[0], oh[1], oh[2], oh[3]);
      *pl = make_uint4(ol[0], ol[1], ol[2], ol[3]);
    }
    const int m = wq * 32 + lane;  // TMEM lane: v for (P U)^T, key feature for the others
    // (2) -What from R1 into the free T and P images (rows m, [2 f-halves][128 rows][128 B])
#pragma unroll 1
    for (int fh = 0; fh < 2; ++fh) {
      float x[64];
      tmem_ld64(R1 + lq + fh * 64, x);
      tmem_wait_ld();
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 8)
        *reinterpret_cast<uint4 *>(sm + B_TH + fh * 16384 + sw128_off(m, c0)) =
            make_uint4(pack_bf16(-x[c0], -x[c0 + 1]), pack_bf16(-x[c0 + 2], -x[c0 + 3]),
                       pack_bf16(-x[c0 + 4], -x[c0 + 5]), pack_bf16(-x[c0 + 6], -x[c0 + 7]));
    }
    // (3) Qt^T = alpha Q^T - (P W)^T into the k rows (rows 0-63 of the image in the first
    //     half's k rows, rows 64-127 in the second half's)
    {
      float x[64];
      tmem_ld64(R0 + lq + 64, x);
      tmem_wait_ld();
      const uint8_t *qcol = sm + B_KQ + (m >> 6) * 16384;
      const int f = m & 63;
      uint8_t *dst = sm + B_KQ + (m >> 6) * 16384;
#pragma unroll
      for (int t8 = 0; t8 < 64; t8 += 8) {
        uint32_t w4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = t8 + 2 * e;
          const float q0 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(qcol + sw128_off(64 + t, f)));
          const float q1 = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(qcol + sw128_off(65 + t, f)));
          w4[e] = pack_bf16(fmaf(alpha[t], q0, -x[t]), fmaf(alpha[t + 1], q1, -x[t + 1]));
        }
        *reinterpret_cast<uint4 *>(dst + sw128_off(f, t8)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    bar();
    if (tid == 0) mbar_arrive(L.bars + BB_STAGED_A);
    // (4) (P U)^T fp32, row v = m: 16-byte piece j at (j ^ (v % 16)) of its 256-byte row, over
    //     the U images once the helper's copies have read them
    if (!lane_wait(L.bars + BB_UFREE, i & 1, false)) break;
    {
      float x[64];
      tmem_ld64(R0 + lq, x);
      tmem_wait_ld();
      uint8_t *row = sm + B_V + (size_t)m * 256;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        *reinterpret_cast<float4 *>(row + ((j ^ (m & 15)) << 4)) =
            make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    bar();
    if (tid == 0) mbar_arrive(L.bars + BB_STAGED_B);
  }
}

// ============================================================ chain CTA

struct ChainShared {
  uint64_t full[kStages], empty[kStages], s_ready, chain_done[2], out_done[2], out_free[2];
  int abort;
  int fills[kStages];
  uint64_t *mma_bar;
  uint32_t mma_par;
};

constexpr int kEpiWarps = 8;         // state and output warps of a chain CTA
constexpr uint32_t CH_TILE = kStages * kStage;  // bf16 [64 tokens][128 v] output tile

__device__ void chain_cta(FfParams &p, uint8_t *sm, uint32_t tm, ChainShared &sh, int ci) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t sb = smem_u32(sm);
  volatile int *abort_flag = &sh.abort;
  const int n_r = (p.n_items - ci + p.n_chain - 1) / p.n_chain;

  if (warp == kEpiWarps) {
    // ===================================================== loads
    if (lane == 0) {
      int pos = 0;
      bool ok = true;
      for (int r = 0; r < n_r && ok; ++r) {
        const int nc = p.nch[ci + r * p.n_chain];
        for (int c = 0; c < nc; ++c, ++pos) {
          const int st = pos % kStages;
          const int slot = pos % p.R;
          // the record's flag first (usually set long before), then the stage
          if (!wait_flag_ge(p.ready + (size_t)ci * p.R + slot, pos + 1, p.spin, p.ctl) ||
              (pos >= kStages &&
               !mbar_wait_spin(&sh.empty[st], ((pos - kStages) / kStages) & 1, p.spin, abort_flag))) {
            ok = false;
            break;
          }
          fence_proxy_async_all();
          uint8_t *sg = sm + st * kStage;
          const uint8_t *rec = p.ring + ((size_t)ci * p.R + slot) * REC_BYTES;
          const bool last = c == nc - 1;  // Ut lo is only read on a sequence's last chunk
          mbar_arrive_expect_tx(&sh.full[st], REC_UTL + (REC_SMEM - REC_QT) + (last ? 16384u : 0u));
          bulk_load(sg, rec, REC_UTL, &sh.full[st]);
          bulk_load(sg + REC_QT, rec + REC_QT, REC_SMEM - REC_QT, &sh.full[st]);
          if (last) bulk_load(sg + REC_UTL, rec + REC_UTL, 16384, &sh.full[st]);
          sh.fills[st] += 1;
        }
      }
      if (!ok) give_up(p, abort_flag);
    }
  } else if (warp == kEpiWarps + 1) {
    // ===================================================== MMAs
    if (lane == 0) {
      const uint32_t id_u = idesc_bf16(128, 128, true, true);
      const uint32_t id_c = idesc_bf16(128, 128, false, true);
      const uint32_t id_o = idesc_bf16(128, 64, false, true);
      int pos = 0;
      bool ok = true;
      for (int r = 0; r < n_r && ok; ++r) {
        const int j = ci + r * p.n_chain;
        const int nc = p.nch[j];
        for (int c = 0; c < nc; ++c, ++pos) {
          const int st = pos % kStages, b = pos & 1;
          if (!mbar_wait_spin(&sh.full[st], (pos / kStages) & 1, p.spin, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sg = sb + st * kStage;
          const uint32_t dch = tm + T_DCH + b * 128, dout = tm + T_DOUT + b * 64, shi = tm + T_SHI + b * 64;
          // D = Ut^T K (hi; + lo on the last chunk of the sequence)
#pragma unroll
          for (int ks = 0; ks < C / 16; ++ks)
            umma_bf16(dch, smem_desc(sg + REC_UTH + ks * 2048, 8192, 1024, 2),
                      smem_desc(sg + ST_K + ks * 2048, 8192, 1024, 2), id_u, ks > 0);
          if (c == nc - 1) {
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks)
              umma_bf16(dch, smem_desc(sg + REC_UTL + ks * 2048, 8192, 1024, 2),
                        smem_desc(sg + ST_K + ks * 2048, 8192, 1024, 2), id_u, 1);
          }
          // S of this chunk written
          if (!mbar_wait_spin(&sh.s_ready, pos & 1, p.spin, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // D += S (-What): the state chain
#pragma unroll
          for (int ks = 0; ks < KD / 16; ++ks)
            umma_bf16_ts(dch, shi + ks * 8, smem_desc(sg + REC_WN + ks * 2048, 16384, 1024, 2), id_c, 1);
          umma_commit(&sh.chain_done[b]);
          sh.mma_bar = &sh.chain_done[b];
          sh.mma_par = (pos >> 1) & 1;
          // O^T = S Qt^T once the epilogue warps are done with this accumulator (chunk pos - 2)
          if (pos >= 2 && !mbar_wait_spin(&sh.out_free[b], ((pos - 2) >> 1) & 1, p.spin, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < KD / 16; ++ks)
            umma_bf16_ts(dout, shi + ks * 8, smem_desc(sg + REC_QT + ks * 2048, 8192, 1024, 2), id_o, ks > 0);
          umma_commit(&sh.out_done[b]);
          umma_commit(&sh.empty[st]);
          sh.mma_bar = &sh.out_done[b];  // completes with the MMA alone (count 1)
          sh.mma_par = (pos >> 1) & 1;
        }
      }
      if (!ok) give_up(p, abort_flag);
    }
  } else {
    // ===================================================== state and outputs (warps 0-7)
    // thread: value row v = 32 (warp % 4) + lane; key features [64 g, +64) of the state and
    // tokens [32 g, +32) of the output, g = warp / 4
    const int quarter = warp & 3, g = warp >> 2;
    const int v = quarter * 32 + lane;
    const uint32_t lq = (uint32_t)(quarter * 32) << 16;
    const size_t o_tok = (size_t)p.Hv * VD;
    __nv_bfloat16 *tile = reinterpret_cast<__nv_bfloat16 *>(sm + CH_TILE);
    float S[64];
    int pos = 0;
    bool ok = true;
    auto write_shi = [&](int b) {
      uint32_t pk[32];
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) pk[jj] = pack_bf16(S[2 * jj], S[2 * jj + 1]);
      tmem_st32(tm + lq + T_SHI + b * 64 + g * 32, pk);
      tmem_wait_st();
      tc_fence_before();
      warp_arrive(&sh.s_ready);
    };
    for (int r = 0; r < n_r && ok; ++r) {
      const int j = ci + r * p.n_chain, s = j / p.Hv, h = j % p.Hv;
      const int nc = p.nch[j];
      if (nc == 0) continue;
      int64_t start, end;
      seq_range(p.cu, p.row_T, s, start, end);
      const size_t srow = (((size_t)s * p.Hv + h) * VD + v) * KD + g * 64;
      if (p.h0) {
        const float4 *src = reinterpret_cast<const float4 *>(p.h0 + srow);
#pragma unroll
        for (int m = 0; m < 16; ++m) {
          const float4 a = src[m];
          S[4 * m] = a.x;
          S[4 * m + 1] = a.y;
          S[4 * m + 2] = a.z;
          S[4 * m + 3] = a.w;
        }
      } else {
#pragma unroll
        for (int m = 0; m < 64; ++m) S[m] = 0.f;
      }
      write_shi(pos & 1);
      for (int c = 0; c < nc; ++c, ++pos) {
        const int b = pos & 1, st = pos % kStages, slot = pos % p.R;
        // ---- the state: S <- b_last S + D
        {
          // the warp's lanes agree on the outcome: the TMEM loads below need the whole warp
          const bool got = mbar_wait_spin(&sh.chain_done[b], (pos >> 1) & 1, p.spin, abort_flag) &&
                           mbar_wait_spin(&sh.full[st], (pos / kStages) & 1, p.spin, abort_flag);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
        }
        const float bl = *reinterpret_cast<const float *>(sm + st * kStage + REC_VEC);
        tc_fence_after();
        {
          float D[64];
          tmem_ld64(tm + lq + T_DCH + b * 128 + g * 64, D);
          tmem_wait_ld();
#pragma unroll
          for (int m = 0; m < 64; ++m) S[m] = fmaf(bl, S[m], D[m]);
        }
        tc_fence_before();
        warp_arrive(&sh.empty[st]);
        if (c + 1 < nc) {
          write_shi(b ^ 1);
        } else if (p.hT) {
          float4 *dst = reinterpret_cast<float4 *>(p.hT + srow);
#pragma unroll
          for (int m = 0; m < 16; ++m) dst[m] = make_float4(S[4 * m], S[4 * m + 1], S[4 * m + 2], S[4 * m + 3]);
        }
        // (P U)^T of this chunk from the ring slot, loaded now so that the loads overlap the
        // wait for the output MMA.  The slot's ready flag was acquired by the loader before its
        // copies, whose completion these warps observed on full[st]: the reads see the record.
        float x[32];
        {
          const uint8_t *prow = p.ring + ((size_t)ci * p.R + slot) * REC_BYTES + REC_OP + (size_t)v * 256;
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(prow + (((g * 8 + jj) ^ (v & 15)) << 4)));
            x[4 * jj] = a.x;
            x[4 * jj + 1] = a.y;
            x[4 * jj + 2] = a.z;
            x[4 * jj + 3] = a.w;
          }
        }
        // ---- the output of this chunk: o[t][v] = O^T[v][t] + (P U)^T[v][t] for tokens [32 g, +32)
        const bool got = mbar_wait_spin(&sh.out_done[b], (pos >> 1) & 1, p.spin, abort_flag);
        // the epilogue warps agree before any of them leaves: one that left alone would
        // strand the others at the named barriers below
        if (named_bar_any(3, 32 * kEpiWarps, !got)) {
          ok = false;
          break;
        }
        tc_fence_after();
        {
          float d[32];
          tmem_ld32(tm + lq + T_DOUT + b * 64 + g * 32, d);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] += d[i];
        }
        tc_fence_before();
        warp_arrive(&sh.out_free[b]);
        const int64_t t0 = start + (int64_t)c * C;
        const int n = (int)min((int64_t)C, end - t0);
        const size_t base = (size_t)t0 * o_tok + (size_t)h * VD;
        if (p.o_f32) {
          float *o = reinterpret_cast<float *>(p.o) + base + v;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (g * 32 + i < n) o[(size_t)(g * 32 + i) * o_tok] = x[i];
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) tile[(g * 32 + i) * VD + v] = __float2bfloat16_rn(x[i]);
          named_bar_sync(3, 32 * kEpiWarps);
          // rows of 256 bytes: 16 threads per row, 16 rows per pass
          const int tr = tid >> 4, tc = tid & 15;
#pragma unroll
          for (int pass = 0; pass < 4; ++pass) {
            const int t = pass * 16 + tr;
            if (t < n)
              *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.o) + base + (size_t)t * o_tok + tc * 8) =
                  *reinterpret_cast<const uint4 *>(tile + t * VD + tc * 8);
          }
        }
        // every epilogue thread has read the slot and the tile: both may be reused.  The
        // flag orders nothing but loads that have returned, so it needs no release fence
        // (which would wait for the output stores above).
        named_bar_sync(3, 32 * kEpiWarps);
        if (tid == 0) st_relaxed(p.consumed + ci, pos + 1);
      }
    }
    if (!ok && lane == 0) give_up(p, abort_flag);
  }
}

__global__ void __launch_bounds__(NT, 1)
    chunk_fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, FfParams p) {
  extern __shared__ uint8_t smraw[];
  uint8_t *sm = (uint8_t *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
  __shared__ ChainShared sh;
  __shared__ uint32_t tbase;
  const int tid = threadIdx.x, warp = tid >> 5;
  if (*(volatile int32_t *)&p.ctl->abort) return;  // the set-up found a bad sequence range
  const bool is_chain = (int)blockIdx.x < p.n_chain;
  if (tid == 0) {
    if (is_chain) {
      for (int i = 0; i < kStages; ++i) {
        mbar_init(&sh.full[i], 1);
        mbar_init(&sh.empty[i], 1 + kEpiWarps);  // the MMA commit and the warps that read b_last
        sh.fills[i] = 0;
      }
      mbar_init(&sh.s_ready, kEpiWarps);
      for (int i = 0; i < 2; ++i) {
        mbar_init(&sh.chain_done[i], 1);
        mbar_init(&sh.out_done[i], 1);
        mbar_init(&sh.out_free[i], kEpiWarps);
      }
    }
    if (!is_chain) {
      for (int l = 0; l < 2; ++l) {
        uint64_t *bars = lane_refs(sm + l * kLane).bars;
        for (int b = 0; b < BB_COUNT; ++b) mbar_init(bars + b, 1);
      }
    }
    sh.abort = 0;
    sh.mma_bar = nullptr;
    sh.mma_par = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tbase, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tbase;
  if (is_chain) {
    chain_cta(p, sm, tm, sh, blockIdx.x);
  } else if (warp < 8) {
    const int lane_id = warp >> 2;
    builder_lane(p, sm + lane_id * kLane, tm + lane_id * 256, lane_id);
  } else if ((tid & 31) == 0) {  // warps 8 and 9: the helpers of lanes 0 and 1
    builder_helper(&tm_q, &tm_k, &tm_v, p, sm + (warp - 8) * kLane);
  }
  __syncthreads();
  if (is_chain && tid == 0 && sh.abort) {
    // copies and MMAs still in flight land before shared memory and TMEM are released
    for (int i = 0; i < kStages; ++i)
      if (sh.fills[i] > 0) (void)mbar_wait(&sh.full[i], (sh.fills[i] - 1) & 1, kSpinDefault);
    if (sh.mma_bar) (void)mbar_wait(sh.mma_bar, sh.mma_par, kSpinDefault);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, 512);
}

// Set-up (one block): zero the ring flags and the unit counter, count each item's chunks,
// lay the items of each chain end to end (P0 = first stream position of an item), and
// write h_T = h0 (or 0) for empty sequences, which no chain visits.
__global__ void chunk_fused_setup_kernel(FfParams p) {
  const int tid = threadIdx.x;
  __shared__ int bad, mx;
  if (tid == 0) {
    bad = 0;
    mx = 0;
    p.ctl->counter = 0;
    p.ctl->abort = 0;
    p.status[1] = GDN_PATH_FUSED;  // the workspace header's path word
  }
  for (int i = tid; i < p.n_chain * p.R; i += blockDim.x) p.ready[i] = 0;
  for (int i = tid; i < p.n_chain; i += blockDim.x) p.consumed[i] = 0;
  __syncthreads();
  for (int j = tid; j < p.n_items; j += blockDim.x) {
    const int s = j / p.Hv;
    int64_t start, end;
    seq_range(p.cu, p.row_T, s, start, end);
    if (start < 0 || end < start || end > p.n_tok) {
      bad = 1;
      p.nch[j] = 0;
    } else {
      p.nch[j] = (int)((end - start + C - 1) / C);
    }
  }
  __syncthreads();
  for (int i = tid; i < p.n_chain; i += blockDim.x) {
    int acc = 0;
    for (int j = i; j < p.n_items; j += p.n_chain) {
      p.P0[j] = acc;
      acc += p.nch[j];
    }
    p.chainN[i] = acc;
    atomicMax(&mx, acc);
  }
  __syncthreads();
  if (tid == 0) {
    p.ctl->maxN = mx;
    if (bad) {
      p.ctl->abort = 1;
      set_status(p.status, GDN_ERR_BOUNDS);
    }
  }
  if (bad || !p.hT) return;
  for (int j = 0; j < p.n_items; ++j) {
    if (p.nch[j] != 0) continue;
    const int s = j / p.Hv, h = j % p.Hv;
    const size_t base = ((size_t)s * p.Hv + h) * VD * KD;
    for (int e = tid; e < VD * KD; e += blockDim.x) p.hT[base + e] = p.h0 ? p.h0[base + e] : 0.f;
  }
}

// control area of the fused path, after the status header: FfCtl, consumed, ready, P0, nch,
// chainN (int32 each), then the ring at a 1 KB boundary
struct FfLayout {
  size_t consumed, ready, P0, nch, chainN, ring, total;
};
FfLayout ff_layout(int n_chain, int R, int n_items) {
  FfLayout L;
  size_t off = kHeader + sizeof(FfCtl);
  L.consumed = off;
  off += (size_t)n_chain * 4;
  L.ready = off;
  off += (size_t)n_chain * R * 4;
  L.P0 = off;
  off += (size_t)n_items * 4;
  L.nch = off;
  off += (size_t)n_items * 4;
  L.chainN = off;
  off += (size_t)n_chain * 4;
  off = (off + 1023) & ~(size_t)1023;
  L.ring = off;
  L.total = off + (size_t)n_chain * R * REC_BYTES;
  return L;
}

constexpr int kMaxChains = 32;  // chains at once; the other SMs build
constexpr int kMaxRing = 12;    // records per chain in flight

}  // namespace

namespace gdn {

bool make_tile_map(CUtensorMap *m, const void *base, int width, int heads, int64_t n_tok, int64_t tok_stride);

// The fused path: bf16, K = V = 128, 16-byte aligned operands and strides.
bool chunk_fused_supported(const void *q, const void *k, const void *v, const gdn_shape &sh) {
  if (sh.dtype != GDN_BF16 || sh.K != KD || sh.V != VD) return false;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16)) return false;
  if ((sh.q_stride * 2) % 16 || (sh.k_stride * 2) % 16 || (sh.v_stride * 2) % 16) return false;
  const int64_t n_tok = sh.n_seqs > 0 && sh.B == 1 ? sh.T : (int64_t)sh.B * sh.T;
  return n_tok < (1LL << 31) && (int64_t)sh.n_seqs * sh.Hv < (1LL << 30);
}

// Grid and ring depth for `n_items` items inside `ws_bytes`; false when the device cannot
// hold every CTA at once or the workspace is too small for two records per chain.
static bool ff_plan(int n_items, size_t ws_bytes, int &grid, int &n_chain, int &R, FfLayout &L) {
  constexpr int kDev = 64;  // SM count and CTAs per SM of the fused kernel, per device
  static int sms[kDev] = {}, per_sm[kDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDev) return false;
  if (per_sm[dev] == 0) {
    int n = 0, b = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaFuncSetAttribute(chunk_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDynSmem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, chunk_fused_kernel, NT, kDynSmem) != cudaSuccess) {
      (void)cudaGetLastError();
      return false;
    }
    sms[dev] = n;
    per_sm[dev] = b > 0 ? b : -1;
  }
  if (per_sm[dev] < 1 || sms[dev] < 2) return false;
  grid = sms[dev];  // one CTA per SM: every CTA is resident at once
  n_chain = std::min(n_items, std::min(kMaxChains, grid - 1));
  for (R = kMaxRing; R >= 2; --R) {
    L = ff_layout(n_chain, R, n_items);
    if (L.total <= ws_bytes) return true;
  }
  return false;
}

size_t chunk_fused_workspace_bytes(const gdn_shape &sh) {
  const int n_items = sh.n_seqs * sh.Hv;
  const int n_chain = std::min(n_items, kMaxChains);
  return ff_layout(std::max(n_chain, 1), kMaxRing, n_items).total;
}

// Runs the fused path if it fits; returns GDN_ERR_UNSUPPORTED (before launching anything)
// when it cannot, so the caller can take another path.
gdn_status chunk_fwd_fused(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, const float *h0, const int32_t *cu,
                           const gdn_shape &sh, float scale, uint32_t flags, void *o, float *h_T,
                           void *workspace, size_t ws_bytes, cudaStream_t st) {
  const int64_t n_tok = cu ? sh.T : (int64_t)sh.B * sh.T;
  const int n_items = sh.n_seqs * sh.Hv;
  int grid = 0, n_chain = 0, R = 0;
  FfLayout L;
  if (n_items <= 0 || !ff_plan(n_items, ws_bytes, grid, n_chain, R, L)) return GDN_ERR_UNSUPPORTED;
  CUtensorMap mq, mk, mv;
  if (!make_tile_map(&mq, q, KD, sh.Hqk, n_tok, sh.q_stride) ||
      !make_tile_map(&mk, k, KD, sh.Hqk, n_tok, sh.k_stride) ||
      !make_tile_map(&mv, v, VD, sh.Hv, n_tok, sh.v_stride))
    return GDN_ERR_CUDA;
  uint8_t *ws = (uint8_t *)workspace;
  FfParams p{};
  p.g = g;
  p.beta = beta;
  p.h0 = h0;
  p.cu = cu;
  p.row_T = sh.T;
  p.n_tok = n_tok;
  p.n_seqs = sh.n_seqs;
  p.Hqk = sh.Hqk;
  p.Hv = sh.Hv;
  p.n_items = n_items;
  p.n_chain = n_chain;
  p.R = R;
  p.scale = scale;
  p.l2norm = (flags & GDN_FLAG_QK_L2NORM) ? 1 : 0;
  p.o_f32 = (flags & GDN_FLAG_O_F32) ? 1 : 0;
  p.o = o;
  p.hT = h_T;
  p.ctl = reinterpret_cast<FfCtl *>(ws + kHeader);
  p.consumed = reinterpret_cast<int32_t *>(ws + L.consumed);
  p.ready = reinterpret_cast<int32_t *>(ws + L.ready);
  p.P0 = reinterpret_cast<int32_t *>(ws + L.P0);
  p.nch = reinterpret_cast<int32_t *>(ws + L.nch);
  p.chainN = reinterpret_cast<int32_t *>(ws + L.chainN);
  p.ring = ws + L.ring;
  p.status = reinterpret_cast<int32_t *>(ws);
  p.spin = (flags & GDN_FLAG_TEST_NO_WAIT) ? 0u : kSpinDefault;
  chunk_fused_setup_kernel<<<1, 256, 0, st>>>(p);
  if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
  void *args[] = {(void *)&mq, (void *)&mk, (void *)&mv, (void *)&p};
  if (cudaLaunchCooperativeKernel((const void *)chunk_fused_kernel, dim3(grid), dim3(NT), args, kDynSmem, st) !=
      cudaSuccess) {
    // e.g. fewer SMs available than the device has: the set-up kernel only wrote the
    // control area, so another path can still run in this workspace
    (void)cudaGetLastError();
    return GDN_ERR_UNSUPPORTED;
  }
  return GDN_OK;
}

}  // namespace gdn
