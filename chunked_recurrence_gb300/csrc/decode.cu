// decode.cu -- one decode step of the gated delta rule layer core.
//
// After the prefill, decode continues from the final state on the standard recurrent
// path ("Qwen3.5 cp - #1", Architecture: the final ssm_state is what the non-CP decode
// path runs from).  Per sequence and token this is
//   - the causal conv1d over the new token with the last W-1 inputs carried per channel
//     (the conv of "[v1] support GDN Ulysses cp", Key decisions 5, at one position),
//   - q/k L2 norm,
//   - the delta-rule update S <- exp(g) S (I - beta k k^T) + beta v k^T and o = scale S q.
// The update is done as S <- a S + u k^T with a = exp(g) and u = beta (v - a S k), and
// o = scale (a S q + u (k^T q)): every row of S is read once and written once.
//
// The work is cut into units of (32 rows of S, v-head, sequence).  A unit computes its head's
// gates, forms the conv outputs of its head's q, k and v channels (q and k are shared by
// Hv / Hqk v-heads and by the V / 32 row blocks; each unit recomputes them from the same
// inputs), rounds them to the storage dtype as the prefill conv stores them, normalises q and
// k, then each of 4 warps takes 8 rows of S: lane l holds S[v][l + 32 j] (coalesced), the two
// dot products are warp reductions.  The conv state is double-buffered: the unit that owns a
// channel (its v channels; q and k channels by the first v-head of the group and row block 0)
// writes that channel's shifted inputs to the output buffer, so no unit overwrites what
// another still reads.  State traffic is 2 V K 4 bytes per (sequence, v-head).
//
// decode_kernel: one block per unit, one launch per step.  (Resident
// blocks walking the units with the next unit's rows staged into shared memory by cp.async
// measured slower, 72.9 against 59.6 us at B = 64 on the 4B layer: each unit's prologue then
// runs in series inside a block, with fewer blocks an SM.  So were units of 128 rows, one per
// head and sequence, the q/k conv done once (75.5 us), units of 16 rows (78.1 us), and the
// conv inputs held in registers across the rows' loads (80 registers, 6 blocks an SM: 52.0
// against 49.5 us).)
#include "common.cuh"
#include "gates.cuh"
#include "sm100.cuh"

using namespace gdn;
using namespace gdn::sm100;

namespace {

constexpr int kRowsPerWarp = 8;
constexpr int kDecWarps = 4;
constexpr int kDecThreads = 32 * kDecWarps;
constexpr int kDecRows = kRowsPerWarp * kDecWarps;  // rows of S per unit: 4 warps x 8

template <typename T>
__device__ __forceinline__ float round_to(float x) {
  return to_f32<T>(from_f32<T>(x));
}

struct DecArgs {
  const void *x, *cs_in;
  void *cs_out;
  const void *w, *bias;
  int act;
  const void *a, *b;
  const float *A_log, *dt_bias;
  float *state;
  int B, Hqk, Hv, V, l2norm, o_f32;
  float scale;
  void *o;
  int bulk;  // the conv inputs may come by bulk copies (bf16, W = 4, V % 32 == 0, 16-byte aligned)
};

// Per-unit values the rows need, after the prologue.
template <int KPL>
struct UnitIn {
  float kr[KPL], qr[KPL];  // this lane's unit-norm k and q features lane + 32 j
  float kq_n, a, bt;       // k.q of the normed vectors, exp(g), beta
};

// The first half of unit (vb, h, b)'s prologue: the gates; conv (+ SiLU) of the head's q and
// k channels and of the unit's v rows into qs, ks, vs; the shifted conv inputs of the
// channels the unit owns.  Ends with the block synced; qs, ks, vs stay in use until the rows
// are done.
template <typename T, int KPL, int W>
__device__ __forceinline__ void decode_conv(const DecArgs &d, int vb, int h, int b, float *qs, float *ks, float *vs,
                                            UnitIn<KPL> &u) {
  constexpr int K = KPL * 32;
  const T *x = (const T *)d.x, *cs = (const T *)d.cs_in, *w = (const T *)d.w, *bias = (const T *)d.bias;
  T *cs_out = (T *)d.cs_out;
  const int Hqk = d.Hqk, Hv = d.Hv, V = d.V, qh = h / (Hv / Hqk);
  const int C = 2 * Hqk * K + Hv * V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  {  // the gates first: their loads then overlap the conv's
    float gv;
    gdn_gates(to_f32<T>(((const T *)d.a)[(size_t)b * Hv + h]), to_f32<T>(((const T *)d.b)[(size_t)b * Hv + h]),
              d.A_log[h], d.dt_bias[h], gv, u.bt);
    u.a = __expf(gv);
  }
  // conv1d (+ SiLU) of channel c at the sequence's next token, in the prefill conv's order;
  // four bf16 taps, 8-byte aligned, come in one load
  const bool w8 = W == 4 && sizeof(T) == 2 && (reinterpret_cast<uintptr_t>(w) & 7) == 0;
  auto conv = [&](int c) -> float {
    float wt[W];
    if (w8) {
      const uint2 r = *reinterpret_cast<const uint2 *>(w + (size_t)c * W);
      const uint32_t h[2] = {r.x, r.y};
#pragma unroll
      for (int j = 0; j < W; ++j) wt[j] = __uint_as_float(j & 1 ? h[(j >> 1) & 1] & 0xffff0000u : h[(j >> 1) & 1] << 16);
    } else {
#pragma unroll
      for (int j = 0; j < W; ++j) wt[j] = to_f32<T>(w[(size_t)c * W + j]);
    }
    float acc = bias ? to_f32<T>(bias[c]) : 0.f;
#pragma unroll
    for (int j = 0; j < W - 1; ++j) acc = fmaf(wt[j], to_f32<T>(cs[((size_t)b * (W - 1) + j) * C + c]), acc);
    acc = fmaf(wt[W - 1], to_f32<T>(x[(size_t)b * C + c]), acc);
    if (d.act) acc = __fdividef(acc, 1.f + __expf(-acc));
    return round_to<T>(acc);
  };
  for (int i = tid; i < K; i += kDecThreads) {
    qs[i] = conv(qh * K + i);
    ks[i] = conv(Hqk * K + qh * K + i);
  }
  if (tid < kDecRows) {
    const int v = vb * kDecRows + tid;
    vs[tid] = v < V ? conv(2 * Hqk * K + h * V + v) : 0.f;
  }
  // shifted conv inputs of the channels this unit owns, into the output buffer
  if (W > 1) {
    auto shift = [&](int c) {
#pragma unroll
      for (int j = 0; j + 1 < W - 1; ++j)
        cs_out[((size_t)b * (W - 1) + j) * C + c] = cs[((size_t)b * (W - 1) + j + 1) * C + c];
      cs_out[((size_t)b * (W - 1) + W - 2) * C + c] = x[(size_t)b * C + c];
    };
    if (tid < kDecRows && vb * kDecRows + tid < V) shift(2 * Hqk * K + h * V + vb * kDecRows + tid);
    if (vb == 0 && h % (Hv / Hqk) == 0)
      for (int i = tid; i < K; i += kDecThreads) {
        shift(qh * K + i);
        shift(Hqk * K + qh * K + i);
      }
  }
  __syncthreads();
}

// The second half: the q/k norms from qs and ks, and this lane's normed features.
template <int KPL>
__device__ __forceinline__ void decode_norms(const DecArgs &d, const float *qs, const float *ks,
                                             float (*red)[kDecWarps], UnitIn<KPL> &u) {
  constexpr int K = KPL * 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // |q|^2, |k|^2 and k.q over the head's K features
  float sq = 0.f, sk = 0.f, kq = 0.f;
  for (int i = tid; i < K; i += kDecThreads) {
    sq = fmaf(qs[i], qs[i], sq);
    sk = fmaf(ks[i], ks[i], sk);
    kq = fmaf(qs[i], ks[i], kq);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    sq += __shfl_xor_sync(0xffffffffu, sq, off);
    sk += __shfl_xor_sync(0xffffffffu, sk, off);
    kq += __shfl_xor_sync(0xffffffffu, kq, off);
  }
  if (lane == 0) {
    red[0][warp] = sq;
    red[1][warp] = sk;
    red[2][warp] = kq;
  }
  __syncthreads();
  sq = sk = kq = 0.f;
#pragma unroll
  for (int i = 0; i < kDecWarps; ++i) {
    sq += red[0][i];
    sk += red[1][i];
    kq += red[2][i];
  }
  const float qn = d.l2norm ? 1.f / sqrtf(sq + kL2Eps) : 1.f;
  const float kn = d.l2norm ? 1.f / sqrtf(sk + kL2Eps) : 1.f;
  u.kq_n = kq * qn * kn;
#pragma unroll
  for (int j = 0; j < KPL; ++j) {
    u.kr[j] = ks[lane + 32 * j] * kn;
    u.qr[j] = qs[lane + 32 * j] * qn;
  }
}

// The 16 per-lane partial sums v[0..15] of a warp, each summed over the 32 lanes by one
// butterfly: at offsets 16, 8, 4, 2 a lane keeps the half of its values that its offset bit
// selects and adds its partner's copy of that half, then offset 1 adds the last pair.  Lanes
// 2 m and 2 m + 1 end with the total of value m.  16 shuffles instead of 5 a value, and the
// same additions, pair by pair, as one xor reduction per value (so the same sums bit for bit).
__device__ __forceinline__ float warp_sum16(float (&v)[16], int lane) {
#pragma unroll
  for (int o = 16, n = 16; o >= 2; o >>= 1, n >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float keep = up ? v[i + n / 2] : v[i], send = up ? v[i] : v[i + n / 2];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// The unit's rows of S: warp w takes rows 8 w .. 8 w + 7 of its 32, held in sr.  Writes the
// new rows to the state and their outputs to o.
template <typename T, int KPL>
__device__ __forceinline__ void decode_rows(const DecArgs &d, int vb, int h, int b, const float (&sr)[kRowsPerWarp][KPL],
                                            const float *vs, const UnitIn<KPL> &u) {
  static_assert(kRowsPerWarp == 8, "two dot products of 8 rows fill the 16-value butterfly");
  constexpr int K = KPL * 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float *Sh = d.state + ((size_t)b * d.Hv + h) * d.V * K;
  // this lane's parts of S k (values 0-7) and S q (values 8-15) of the warp's eight rows
  float part[16];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    float dk = 0.f, dq = 0.f;
#pragma unroll
    for (int j = 0; j < KPL; ++j) {
      dk = fmaf(sr[r][j], u.kr[j], dk);
      dq = fmaf(sr[r][j], u.qr[j], dq);
    }
    part[r] = dk;
    part[kRowsPerWarp + r] = dq;
  }
  // lanes 2 r, 2 r + 1 hold (S k)_r, lanes 16 + 2 r, 17 + 2 r hold (S q)_r
  const float tot = warp_sum16(part, lane);
  const int rl = (lane >> 1) & 7;  // the row whose sum this lane holds
  const int vr0 = warp * kRowsPerWarp;
  const float uu_l = u.bt * (vs[vr0 + rl] - u.a * tot);  // u of row rl (lanes 0-15)
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int vr = vr0 + r, v = vb * kDecRows + vr;
    const float uu = __shfl_sync(0xffffffffu, uu_l, 2 * r);
    if (v >= d.V) continue;
#pragma unroll
    for (int j = 0; j < KPL; ++j) Sh[(size_t)v * K + lane + 32 * j] = fmaf(u.a, sr[r][j], uu * u.kr[j]);
    if (lane == 16 + 2 * r) {  // holds (S q)_r
      const float ov = d.scale * fmaf(u.a, tot, uu * u.kq_n);
      const size_t oi = ((size_t)b * d.Hv + h) * d.V + v;
      if (d.o_f32) reinterpret_cast<float *>(d.o)[oi] = ov;
      else reinterpret_cast<T *>(d.o)[oi] = from_f32<T>(ov);
    }
  }
}

// one block per unit (vb, h, b) = (blockIdx.x, .y, .z).  The conv's few loads go first and
// the rows of S (16 KB a unit) after them: issued the other way round, the conv's loads, L2
// hits, waited behind the rows' HBM misses, and the conv took 5.4 of a block's 7.7 us
// (global-timer stamps at B = 64 on the 4B layer).  With bf16 inputs and W = 4 the conv's
// inputs come instead by bulk async copies (the unit's channels are three contiguous runs in
// the weights, the carried rows and x), which do not queue behind the rows' loads, so both
// are in flight at once.  The norms then overlap the rows' loads.
template <typename T, int KPL, int W>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(const DecArgs d) {
  constexpr int K = KPL * 32;
  constexpr bool kBulk = sizeof(T) == 2 && W == 4;
  constexpr int NCH = 2 * K + kDecRows;  // the unit's conv channels: q, k, then its v rows
  const int vb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ float qs[K], ks[K], vs[kDecRows];
  __shared__ float red[3][kDecWarps];
  __shared__ __align__(16) T cw[kBulk ? NCH * W : 1];   // the channels' taps
  __shared__ __align__(16) T cin[kBulk ? W * NCH : 1];  // the W - 1 carried rows, then x
  __shared__ __align__(8) uint64_t cbar;
  const bool bulk = kBulk && d.bulk;
  const int Hqk = d.Hqk, Hv = d.Hv, V = d.V, qh = h / (Hv / Hqk);
  const int C = 2 * Hqk * K + Hv * V;
  const int cq = qh * K, ck = Hqk * K + qh * K, cv = 2 * Hqk * K + h * V + vb * kDecRows;
  if (bulk) {
    if (tid == 0) {
      mbar_init(&cbar, 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
      const T *w = (const T *)d.w, *cs = (const T *)d.cs_in, *x = (const T *)d.x;
      constexpr uint32_t kb = sizeof(T);
      mbar_arrive_expect_tx(&cbar, (uint32_t)(2 * NCH * W) * kb);
      bulk_load(cw, w + (size_t)cq * W, K * W * kb, &cbar);
      bulk_load(cw + K * W, w + (size_t)ck * W, K * W * kb, &cbar);
      bulk_load(cw + 2 * K * W, w + (size_t)cv * W, kDecRows * W * kb, &cbar);
#pragma unroll
      for (int j = 0; j < W; ++j) {
        const T *row = j < W - 1 ? cs + ((size_t)b * (W - 1) + j) * C : x + (size_t)b * C;
        bulk_load(cin + j * NCH, row + cq, K * kb, &cbar);
        bulk_load(cin + j * NCH + K, row + ck, K * kb, &cbar);
        bulk_load(cin + j * NCH + 2 * K, row + cv, kDecRows * kb, &cbar);
      }
    }
  }
  UnitIn<KPL> u;
  float sr[kRowsPerWarp][KPL];
  const float *Sh = d.state + ((size_t)b * d.Hv + h) * d.V * K;
  auto load_rows = [&]() {
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int v = vb * kDecRows + warp * kRowsPerWarp + r;
#pragma unroll
      for (int j = 0; j < KPL; ++j) sr[r][j] = v < d.V ? Sh[(size_t)v * K + lane + 32 * j] : 0.f;
    }
  };
  bool staged = false;
  if (bulk) {
    float gv;
    gdn_gates(to_f32<T>(((const T *)d.a)[(size_t)b * Hv + h]), to_f32<T>(((const T *)d.b)[(size_t)b * Hv + h]),
              d.A_log[h], d.dt_bias[h], gv, u.bt);
    load_rows();
    u.a = __expf(gv);
    staged = mbar_wait(&cbar, 0, 1u << 20);
    if (!staged) (void)mbar_wait(&cbar, 0, 1u << 20);  // the copies land before the block moves on
  }
  if (staged) {
    // conv (+ SiLU) of local channel c from the staged inputs: the prefill conv's order
    const T *bias = (const T *)d.bias;
    auto conv_s = [&](int c, int ch) -> float {
      float acc = bias ? to_f32<T>(bias[ch]) : 0.f;
#pragma unroll
      for (int j = 0; j < W - 1; ++j) acc = fmaf(to_f32<T>(cw[c * W + j]), to_f32<T>(cin[j * NCH + c]), acc);
      acc = fmaf(to_f32<T>(cw[c * W + W - 1]), to_f32<T>(cin[(W - 1) * NCH + c]), acc);
      if (d.act) acc = __fdividef(acc, 1.f + __expf(-acc));
      return round_to<T>(acc);
    };
    T *cs_out = (T *)d.cs_out;
    auto shift = [&](int c, int ch) {
#pragma unroll
      for (int j = 0; j + 1 < W - 1; ++j) cs_out[((size_t)b * (W - 1) + j) * C + ch] = cin[(j + 1) * NCH + c];
      cs_out[((size_t)b * (W - 1) + W - 2) * C + ch] = cin[(W - 1) * NCH + c];
    };
    for (int i = tid; i < K; i += kDecThreads) {
      qs[i] = conv_s(i, cq + i);
      ks[i] = conv_s(K + i, ck + i);
    }
    if (tid < kDecRows) vs[tid] = conv_s(2 * K + tid, cv + tid);
    if (tid < kDecRows) shift(2 * K + tid, cv + tid);
    if (vb == 0 && h % (Hv / Hqk) == 0)
      for (int i = tid; i < K; i += kDecThreads) {
        shift(i, cq + i);
        shift(K + i, ck + i);
      }
    __syncthreads();
  } else if (bulk) {
    decode_conv<T, KPL, W>(d, vb, h, b, qs, ks, vs, u);  // (a copy that never landed)
  } else {
    decode_conv<T, KPL, W>(d, vb, h, b, qs, ks, vs, u);
    load_rows();
  }
  decode_norms<KPL>(d, qs, ks, red, u);
  decode_rows<T, KPL>(d, vb, h, b, sr, vs, u);
}

template <typename T, int KPL, int W>
gdn_status launch_decode(const DecArgs &d, cudaStream_t st) {
  const int nvb = (d.V + kDecRows - 1) / kDecRows;
  const dim3 grid((unsigned)nvb, (unsigned)d.Hv, (unsigned)d.B);
  decode_kernel<T, KPL, W><<<grid, kDecThreads, 0, st>>>(d);
  return launch_status();
}

template <typename T, int KPL>
gdn_status dispatch_w(int W, const DecArgs &d, cudaStream_t st) {
  switch (W) {
#define GDN_DEC_W(WW) \
  case WW:            \
    return launch_decode<T, KPL, WW>(d, st);
    GDN_DEC_W(1) GDN_DEC_W(2) GDN_DEC_W(3) GDN_DEC_W(4) GDN_DEC_W(5) GDN_DEC_W(6) GDN_DEC_W(7) GDN_DEC_W(8)
#undef GDN_DEC_W
    default: return GDN_ERR_UNSUPPORTED;
  }
}

template <typename T>
gdn_status dispatch_k(int K, int W, const DecArgs &d, cudaStream_t st) {
  switch (K / 32) {
#define GDN_DEC_K(KP) \
  case KP:            \
    return dispatch_w<T, KP>(W, d, st);
    GDN_DEC_K(1) GDN_DEC_K(2) GDN_DEC_K(3) GDN_DEC_K(4) GDN_DEC_K(5) GDN_DEC_K(6) GDN_DEC_K(7) GDN_DEC_K(8)
#undef GDN_DEC_K
    default: return GDN_ERR_UNSUPPORTED;
  }
}

}  // namespace

extern "C" gdn_status gdn_decode_step(const void *x, const void *conv_state_in, void *conv_state_out,
                                      const void *w, const void *bias, int32_t dtype, int32_t width, int32_t act,
                                      const void *a, const void *b, const float *A_log, const float *dt_bias,
                                      float *state, int32_t B, int32_t Hqk, int32_t Hv, int32_t K, int32_t V,
                                      float scale, uint32_t flags, void *o, void *stream) {
  if (dtype != GDN_F32 && dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (B < 0 || Hqk < 1 || Hv < 1 || Hv % Hqk != 0 || V < 1 || K < 32 || K > 256 || K % 32 != 0)
    return GDN_ERR_INVALID_ARG;
  if (width < 1 || width > 8 || (act != 0 && act != 1)) return GDN_ERR_INVALID_ARG;
  if (flags & ~(uint32_t)(GDN_FLAG_QK_L2NORM | GDN_FLAG_O_F32)) return GDN_ERR_INVALID_ARG;
  if (B == 0) return GDN_OK;
  if (!x || !w || !a || !b || !A_log || !dt_bias || !state || !o ||
      (width > 1 && (!conv_state_in || !conv_state_out || conv_state_in == conv_state_out)))
    return GDN_ERR_INVALID_ARG;
  if ((int64_t)2 * Hqk * K + (int64_t)Hv * V > 2147483647LL || B > 65535 || Hv > 65535)
    return GDN_ERR_UNSUPPORTED;
  const int bulk = dtype == GDN_BF16 && width == 4 && V % 32 == 0 && aligned(x, 16) && aligned(conv_state_in, 16) &&
                   aligned(w, 16);
  DecArgs d{x, conv_state_in, conv_state_out, w, bias, act, a, b, A_log, dt_bias, state, B, Hqk, Hv, V,
            (flags & GDN_FLAG_QK_L2NORM) ? 1 : 0, (flags & GDN_FLAG_O_F32) ? 1 : 0, scale, o, bulk};
  cudaStream_t st = (cudaStream_t)stream;
  if (dtype == GDN_BF16) return dispatch_k<__nv_bfloat16>(K, width, d, st);
  return dispatch_k<float>(K, width, d, st);
}
