// chunk_common.cuh -- chunk slots, sequence ranges and bf16 packing shared by the
// tensor-core chunk kernels.
#pragma once

#include "common.cuh"

namespace gdn {

// Chunk c of sequence s (start token t_s) owns slot s + floor(t_s / 64) + c: unique over
// all chunks of all sequences and below n_seqs + ceil(n_tok / 64).
inline size_t n_slots(int64_t n_tok, int n_seqs) { return (size_t)n_seqs + (size_t)((n_tok + kChunk - 1) / kChunk); }

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
  return (int64_t)s + st / kChunk;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ float2 unpack_bf16(uint32_t u) {
  __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162 *>(&u);
  return __bfloat1622float2(h);
}

}  // namespace gdn
