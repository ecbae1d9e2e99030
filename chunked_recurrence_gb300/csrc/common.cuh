// common.cuh -- small helpers shared by the libgdn translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int kChunk = 64;          // tokens per chunk of the UT/WY form
constexpr float kL2Eps = 1e-6f;     // q/k L2 norm: x / sqrt(sum x^2 + eps)

// device status word written by kernels that detect a problem (first writer wins)
__device__ __forceinline__ void set_status(int32_t *status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// index of the sequence that holds token t: largest s with cu[s] <= t (n_seqs >= 1)
__device__ __forceinline__ int seq_of_token(const int32_t *cu, int n_seqs, int64_t t) {
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// 16-byte asynchronous global -> shared copies (both addresses 16-byte aligned), tracked in
// commit groups of the issuing thread; waiting on them is the hardware's own wait, no poll
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// every committed group has landed
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

inline gdn_status launch_status() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Inputs of the fused front end of gdn_layer_fwd: the conv over x's Q|K|V channels and the
// gates, computed inside the chunk operand kernel.
struct FrontArgs {
  const void *x, *w, *bias;
  int width;
  const void *a, *b;
  const float *A_log, *dt_bias;
};

// The gated RMS norm applied in the state scan's output epilogue (gdn_layer_fwd with z).
struct NormArgs {
  const void *z, *w;
  float eps;
};

// bytes of one conv'd q (or k) array [n_tok][Hqk][K] bf16 in the front end's workspace
inline size_t front_qk_bytes(const gdn_shape &sh, int64_t n_tok) {
  return ((size_t)n_tok * sh.Hqk * sh.K * 2 + 255) & ~(size_t)255;
}

}  // namespace gdn
