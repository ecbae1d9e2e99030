// noalloc.cu -- gdn_chunk_fwd without a caller-provided workspace.
//
// Some callers cannot allocate device memory at all: a plugin inside a host
// application that owns the whole device memory pool (an inference server or
// engine with a fixed budget and its own allocator), or a latency-critical
// path where the implicit device-wide synchronisation of cudaMalloc/cudaFree
// is not allowed.  They still own their inputs and outputs, but have nowhere
// to put gdn_chunk_fwd's scratch (the status word and, on the tensor-core
// path, the per-chunk T matrices).  This entry point keeps that scratch in a
// file-scope device array of fixed size instead.
#include "common.cuh"

namespace {

// Scratch for gdn_chunk_fwd_noalloc: 16 MiB, held by every GPU that loads the
// library until the process exits.  On the tensor-core path (bf16, K = 128)
// this bounds the problem size: the compact workspace, 256 + 8320 * Hv *
// (n_seqs + ceil(tokens / 64)) bytes, must fit, e.g. 2048 tokens x 32 v-heads
// or 8192 tokens x 8 v-heads.  gdn_chunk_fwd then takes the path that fits in
// 16 MiB: the split operand/scan kernels for small shapes, else the compact pair.
constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device.  In host code the
// array's name is only a host-side stand-in; the kernels must be given this
// address.  It is looked up on every call (cudaGetSymbolAddress is cheap), so
// a device reset or a new primary context never leaves a stale address behind.
gdn_status scratch_for_current_device(void **out) {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GDN_ERR_CUDA;
  *out = p;
  return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_chunk_fwd_noalloc(const void *q, const void *k, const void *v,
                                            const float *g, const float *beta, const float *h0,
                                            const int32_t *cu_seqlens, const gdn_shape *shape,
                                            float scale, uint32_t flags, void *o, float *h_T,
                                            void *stream) {
  const size_t need = gdn_chunk_fwd_min_workspace_bytes(shape);
  if (need == 0) return GDN_ERR_INVALID_ARG;          // bad shape (same checks as gdn_chunk_fwd)
  if (need > kNoAllocScratchBytes) return GDN_ERR_WORKSPACE;  // beyond the fixed scratch
  void *scratch = nullptr;
  const gdn_status st = scratch_for_current_device(&scratch);
  if (st != GDN_OK) return st;
  // the array keeps the previous call's contents: the status word must start at zero
  const gdn_status rs = gdn_workspace_reset(scratch, kNoAllocScratchBytes, stream);
  if (rs != GDN_OK) return rs;
  return gdn_chunk_fwd(q, k, v, g, beta, h0, cu_seqlens, shape, scale, flags, o, h_T, scratch,
                       kNoAllocScratchBytes, stream);
}
