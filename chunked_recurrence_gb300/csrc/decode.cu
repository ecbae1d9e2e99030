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
// decode_kernel: one block per (32 rows of S, v-head, sequence), one launch per step.  The
// block computes its head's gates, forms the conv outputs of its head's q, k and v channels
// (q and k are shared by Hv / Hqk v-heads and by the V / 32 row blocks; each block
// recomputes them from the same inputs), rounds them to the storage dtype as the prefill
// conv stores them, normalises q and k, then each warp streams 8 rows of S: lane l holds
// S[v][l + 32 j] (coalesced), the two dot products are warp reductions.  The conv state is
// double-buffered: the block that owns a channel (its v channels; q and k channels by the
// first v-head of the group and row block 0) writes that channel's shifted inputs to the
// output buffer, so no block overwrites what another still reads.  State traffic is
// 2 V K 4 bytes per (sequence, v-head).
#include "common.cuh"
#include "gates.cuh"

using namespace gdn;

namespace {

constexpr int kDecRows = 32;  // rows of S per block: 4 warps x 8

template <typename T>
__device__ __forceinline__ float round_to(float x) {
  return to_f32<T>(from_f32<T>(x));
}

template <typename T, int KPL, int W>
__global__ void __launch_bounds__(128) decode_kernel(const T *__restrict__ x, const T *__restrict__ conv_state,
                                                     T *__restrict__ conv_out, const T *__restrict__ w,
                                                     const T *__restrict__ bias, int act, const T *__restrict__ ga,
                                                     const T *__restrict__ gb, const float *__restrict__ A_log,
                                                     const float *__restrict__ dt_bias, float *__restrict__ S,
                                                     int Hqk, int Hv, int V, int l2norm, float scale,
                                                     int o_f32, void *__restrict__ o) {
  constexpr int K = KPL * 32;
  const int vb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int qh = h / (Hv / Hqk);
  const int C = 2 * Hqk * K + Hv * V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ float qs[K], ks[K], vs[kDecRows];
  __shared__ float red[3][4];
  // this warp's 8 rows of S, loaded first so that their latency overlaps the conv below
  constexpr int kRowsPerWarp = kDecRows / 4;
  float sr[kRowsPerWarp][KPL];
  float *Sh = S + ((size_t)b * Hv + h) * V * K;
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int v = vb * kDecRows + warp * kRowsPerWarp + r;
#pragma unroll
    for (int j = 0; j < KPL; ++j) sr[r][j] = v < V ? Sh[(size_t)v * K + lane + 32 * j] : 0.f;
  }

  // conv1d (+ SiLU) of channel c at the sequence's next token, in the prefill conv's order
  auto conv = [&](int c) -> float {
    float acc = bias ? to_f32<T>(bias[c]) : 0.f;
#pragma unroll
    for (int j = 0; j < W - 1; ++j)
      acc = fmaf(to_f32<T>(w[(size_t)c * W + j]), to_f32<T>(conv_state[((size_t)b * (W - 1) + j) * C + c]), acc);
    acc = fmaf(to_f32<T>(w[(size_t)c * W + W - 1]), to_f32<T>(x[(size_t)b * C + c]), acc);
    if (act) acc = __fdividef(acc, 1.f + __expf(-acc));
    return round_to<T>(acc);
  };
  for (int i = tid; i < K; i += 128) {
    qs[i] = conv(qh * K + i);
    ks[i] = conv(Hqk * K + qh * K + i);
  }
  if (tid < kDecRows) {
    const int v = vb * kDecRows + tid;
    vs[tid] = v < V ? conv(2 * Hqk * K + h * V + v) : 0.f;
  }
  // shifted conv inputs of the channels this block owns, into the output buffer
  if (W > 1) {
    auto shift = [&](int c) {
#pragma unroll
      for (int j = 0; j + 1 < W - 1; ++j)
        conv_out[((size_t)b * (W - 1) + j) * C + c] = conv_state[((size_t)b * (W - 1) + j + 1) * C + c];
      conv_out[((size_t)b * (W - 1) + W - 2) * C + c] = x[(size_t)b * C + c];
    };
    if (tid < kDecRows && vb * kDecRows + tid < V) shift(2 * Hqk * K + h * V + vb * kDecRows + tid);
    if (vb == 0 && h % (Hv / Hqk) == 0)
      for (int i = tid; i < K; i += 128) {
        shift(qh * K + i);
        shift(Hqk * K + qh * K + i);
      }
  }
  __syncthreads();
  // |q|^2, |k|^2 and k.q over the head's K features
  float sq = 0.f, sk = 0.f, kq = 0.f;
  for (int i = tid; i < K; i += 128) {
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
  sq = red[0][0] + red[0][1] + red[0][2] + red[0][3];
  sk = red[1][0] + red[1][1] + red[1][2] + red[1][3];
  kq = red[2][0] + red[2][1] + red[2][2] + red[2][3];
  const float qn = l2norm ? 1.f / sqrtf(sq + kL2Eps) : 1.f;
  const float kn = l2norm ? 1.f / sqrtf(sk + kL2Eps) : 1.f;
  const float kq_n = kq * qn * kn;
  float kr[KPL], qr[KPL];
#pragma unroll
  for (int j = 0; j < KPL; ++j) {
    kr[j] = ks[lane + 32 * j] * kn;
    qr[j] = qs[lane + 32 * j] * qn;
  }
  float gv, bt;
  gdn_gates(to_f32<T>(ga[(size_t)b * Hv + h]), to_f32<T>(gb[(size_t)b * Hv + h]), A_log[h], dt_bias[h], gv, bt);
  const float a = __expf(gv);
  // rows of S: warp w takes rows 8 w .. 8 w + 7 of this block's 32
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int vr = warp * kRowsPerWarp + r, v = vb * kDecRows + vr;
    float dk = 0.f, dq = 0.f;
#pragma unroll
    for (int j = 0; j < KPL; ++j) {
      dk = fmaf(sr[r][j], kr[j], dk);
      dq = fmaf(sr[r][j], qr[j], dq);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      dk += __shfl_xor_sync(0xffffffffu, dk, off);
      dq += __shfl_xor_sync(0xffffffffu, dq, off);
    }
    if (v >= V) continue;
    const float u = bt * (vs[vr] - a * dk);
#pragma unroll
    for (int j = 0; j < KPL; ++j) Sh[(size_t)v * K + lane + 32 * j] = fmaf(a, sr[r][j], u * kr[j]);
    if (lane == 0) {
      const float ov = scale * fmaf(a, dq, u * kq_n);
      const size_t oi = ((size_t)b * Hv + h) * V + v;
      if (o_f32) reinterpret_cast<float *>(o)[oi] = ov;
      else reinterpret_cast<T *>(o)[oi] = from_f32<T>(ov);
    }
  }
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
};

template <typename T, int KPL, int W>
void launch_decode(const DecArgs &d, cudaStream_t st) {
  const dim3 grid((unsigned)((d.V + kDecRows - 1) / kDecRows), (unsigned)d.Hv, (unsigned)d.B);
  decode_kernel<T, KPL, W><<<grid, 128, 0, st>>>((const T *)d.x, (const T *)d.cs_in, (T *)d.cs_out, (const T *)d.w,
                                                 (const T *)d.bias, d.act, (const T *)d.a, (const T *)d.b, d.A_log,
                                                 d.dt_bias, d.state, d.Hqk, d.Hv, d.V, d.l2norm, d.scale, d.o_f32,
                                                 d.o);
}

template <typename T, int KPL>
gdn_status dispatch_w(int W, const DecArgs &d, cudaStream_t st) {
  switch (W) {
#define GDN_DEC_W(WW)                   \
  case WW:                              \
    launch_decode<T, KPL, WW>(d, st);   \
    break;
    GDN_DEC_W(1) GDN_DEC_W(2) GDN_DEC_W(3) GDN_DEC_W(4) GDN_DEC_W(5) GDN_DEC_W(6) GDN_DEC_W(7) GDN_DEC_W(8)
#undef GDN_DEC_W
    default: return GDN_ERR_UNSUPPORTED;
  }
  return launch_status();
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
  DecArgs d{x, conv_state_in, conv_state_out, w, bias, act, a, b, A_log, dt_bias, state, B, Hqk, Hv, V,
            (flags & GDN_FLAG_QK_L2NORM) ? 1 : 0, (flags & GDN_FLAG_O_F32) ? 1 : 0, scale, o};
  cudaStream_t st = (cudaStream_t)stream;
  if (dtype == GDN_BF16) return dispatch_k<__nv_bfloat16>(K, width, d, st);
  return dispatch_k<float>(K, width, d, st);
}
