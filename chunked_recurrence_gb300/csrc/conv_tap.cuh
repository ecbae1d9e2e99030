// conv_tap.cuh -- the arithmetic of one token row of the bf16 causal conv1d (+ SiLU) over
// eight channels.  The staged conv kernel and the conv inside the chunk operand kernel's
// front end both call it, so the two give the same bf16 values for the same inputs
// ("[v1] support GDN Ulysses cp", What This PR Does: the layer's causal conv over the
// concatenated Q|K|V channels ahead of chunk_gated_delta_rule).
//
//   y[c] = act( bias[c] + sum_{j < W-1} w[c, j] hist[j][c] + w[c, W-1] cur[c] )
//
// with hist[0] the oldest of the W-1 previous rows.  Values travel as fp32 pairs (channels
// 2i and 2i+1 in one 64-bit register pair) so that the taps are packed fp32x2 FMAs in that
// order with no repacking.  SiLU(x) = x / (1 + e^-x) takes e^-x as 2^(-x log2 e) on the
// hardware base-2 exponential and the division as a hardware reciprocal (both flush to
// zero: the results round to bf16 right after).
#pragma once

#include <stdint.h>

namespace gdn {

__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float hw_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float hw_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// a bf16 pair (low half: the even channel) as an fp32 pair, exactly
__device__ __forceinline__ uint64_t f2_from_bf16x2(uint32_t w) {
  return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// an fp32 pair rounded (to nearest even) to a bf16 pair, the even channel in the low half
__device__ __forceinline__ uint32_t bf16x2_from_f2(uint64_t p) {
  float a, b;
  f2_unpack(p, a, b);
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}
// eight bf16 channels (16 bytes) as four fp32 pairs, and back
__device__ __forceinline__ void unpack8p(const uint4 &r, uint64_t (&p)[4]) {
  p[0] = f2_from_bf16x2(r.x);
  p[1] = f2_from_bf16x2(r.y);
  p[2] = f2_from_bf16x2(r.z);
  p[3] = f2_from_bf16x2(r.w);
}
__device__ __forceinline__ uint4 pack8p(const uint64_t (&p)[4]) {
  return make_uint4(bf16x2_from_f2(p[0]), bf16x2_from_f2(p[1]), bf16x2_from_f2(p[2]), bf16x2_from_f2(p[3]));
}

// One output row.  wt: [W][4] tap pairs; bs: bias pairs; hist: HW = max(W - 1, 1) previous
// rows (unused when W = 1); cur: this row.
template <int W, int HW>
__device__ __forceinline__ void conv_row8p(const uint64_t (&wt)[W][4], const uint64_t (&bs)[4],
                                           const uint64_t (&hist)[HW][4], const uint64_t (&cur)[4], bool act,
                                           uint64_t (&out)[4]) {
  constexpr float kLog2e = 1.4426950408889634f;
  const uint64_t neg_log2e = f2_pack(-kLog2e, -kLog2e), one = f2_pack(1.f, 1.f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint64_t acc = bs[i];
#pragma unroll
    for (int j = 0; j < W - 1; ++j) acc = f2_fma(wt[j][i], hist[j][i], acc);
    acc = f2_fma(wt[W - 1][i], cur[i], acc);
    if (act) {
      float e0, e1, d0, d1;
      f2_unpack(f2_mul(acc, neg_log2e), e0, e1);
      f2_unpack(f2_add(f2_pack(hw_exp2(e0), hw_exp2(e1)), one), d0, d1);
      acc = f2_mul(acc, f2_pack(hw_rcp(d0), hw_rcp(d1)));
    }
    out[i] = acc;
  }
}

// History shift: drop the oldest row, append cur.
template <int HW>
__device__ __forceinline__ void conv_shift8p(uint64_t (&hist)[HW][4], const uint64_t (&cur)[4]) {
#pragma unroll
  for (int j = 0; j + 1 < HW; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) hist[j][i] = hist[j + 1][i];
#pragma unroll
  for (int i = 0; i < 4; ++i) hist[HW - 1][i] = cur[i];
}

}  // namespace gdn
