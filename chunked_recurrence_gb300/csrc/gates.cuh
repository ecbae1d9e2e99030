// gates.cuh -- the Qwen3.5 gates of one (token, v-head), shared by gdn_gate_prep and the
// decode step so that both give the same values ("[v1] support GDN Ulysses cp", What This
// PR Does: A_log and dt_bias are per-v-head parameters, a and b per-token inputs):
//     g = -exp(A_log) softplus(a + dt_bias),  softplus(x) = max(x, 0) + log1p(exp(-|x|))
//     beta = sigmoid(b)
#pragma once

namespace gdn {

__device__ __forceinline__ void gdn_gates(float a, float b, float A_log, float dt_bias, float &g, float &beta) {
  const float x = a + dt_bias;
  const float softplus = fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
  g = -expf(A_log) * softplus;
  beta = 1.f / (1.f + expf(-b));
}

}  // namespace gdn
