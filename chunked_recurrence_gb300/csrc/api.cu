// api.cu -- argument checking and dispatch of gdn_chunk_fwd, gdn_segment_summary and
// gdn_layer_fwd.
#include <algorithm>

#include "common.cuh"

namespace gdn {
gdn_status chunk_fwd_simt(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, const float *h0, const int32_t *cu,
                          const gdn_shape &sh, float scale, uint32_t flags, void *o, float *h_T,
                          int32_t *status, cudaStream_t st);
gdn_status segment_summary_simt(const void *k, const void *v, const float *g, const float *beta,
                                const int32_t *bounds, int n_seg, const gdn_shape &sh,
                                uint32_t flags, float *M, float *S_local, int32_t *status,
                                cudaStream_t st);
bool chunk_tc_supported(const void *q, const void *k, const void *v, const gdn_shape &sh);
size_t chunk_tc_workspace_bytes(const gdn_shape &sh, int64_t n_tok);
bool chunk_scan_supported(const void *q, const void *k, const void *v, const gdn_shape &sh);
size_t chunk_scan_workspace_bytes(const gdn_shape &sh, int64_t n_tok);
gdn_status chunk_fwd_scan(const void *q, const void *k, const void *v, const float *g,
                          const float *beta, const float *h0, const int32_t *cu,
                          const gdn_shape &sh, float scale, uint32_t flags, void *o, float *h_T,
                          void *workspace, size_t ws_bytes, cudaStream_t st, const NormArgs *nm);
bool chunk_norm_supported(const gdn_shape &sh, uint32_t flags, const NormArgs &nm);
gdn_status chunk_fwd_tc(const void *q, const void *k, const void *v, const float *g,
                        const float *beta, const float *h0, const int32_t *cu,
                        const gdn_shape &sh, float scale, uint32_t flags, void *o, float *h_T,
                        void *workspace, size_t ws_bytes, cudaStream_t st);
gdn_status summary_scan(const void *k, const void *v, const float *g, const float *beta,
                        const int32_t *bounds, int n_seg, const gdn_shape &sh, uint32_t flags,
                        float *M, float *S_local, void *workspace, size_t ws_bytes,
                        cudaStream_t st);
bool chunk_fused_supported(const void *q, const void *k, const void *v, const gdn_shape &sh);
size_t chunk_fused_workspace_bytes(const gdn_shape &sh);
gdn_status chunk_fwd_fused(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, const float *h0, const int32_t *cu,
                           const gdn_shape &sh, float scale, uint32_t flags, void *o, float *h_T,
                           void *workspace, size_t ws_bytes, cudaStream_t st);
bool chunk_front_supported(const void *x, const void *w, int width, const gdn_shape &sh);
gdn_status layer_conv_and_gates(const void *x, const void *w, const void *bias, int32_t dtype,
                                const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens, int32_t C,
                                int32_t width, void *y, const void *a, const void *b, const float *A_log,
                                const float *dt_bias, int32_t Hv, float *g, float *beta, void *stream);
size_t chunk_front_workspace_bytes(const gdn_shape &sh, int64_t n_tok);
gdn_status chunk_fwd_front(const FrontArgs &fr, const float *h0, const int32_t *cu, const gdn_shape &sh,
                           float scale, uint32_t flags, void *o, float *h_T, void *workspace,
                           size_t ws_bytes, cudaStream_t st, const NormArgs *nm);
gdn_status summary_tc(const void *k, const void *v, const float *g, const float *beta,
                      const int32_t *bounds, int n_seg, const gdn_shape &sh, uint32_t flags,
                      float *M, float *S_local, void *workspace, size_t ws_bytes, cudaStream_t st);
}  // namespace gdn

using namespace gdn;

namespace {

constexpr size_t kWorkspaceBase = 256;  // status word + padding to keep later regions aligned

// Fills dense strides and checks the shape.  Returns GDN_OK or the error.
gdn_status normalise_shape(const gdn_shape *in, gdn_shape *out) {
  if (!in) return GDN_ERR_INVALID_ARG;
  gdn_shape s = *in;
  if (s.dtype != GDN_F32 && s.dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
  if (s.B <= 0 || s.T < 0 || s.n_seqs < 0 || s.Hqk <= 0 || s.Hv <= 0 || s.K <= 0 || s.V <= 0)
    return GDN_ERR_INVALID_ARG;
  if (s.Hv % s.Hqk != 0) return GDN_ERR_INVALID_ARG;
  if (s.q_stride == 0) s.q_stride = (int64_t)s.Hqk * s.K;
  if (s.k_stride == 0) s.k_stride = (int64_t)s.Hqk * s.K;
  if (s.v_stride == 0) s.v_stride = (int64_t)s.Hv * s.V;
  if (s.q_stride < (int64_t)s.Hqk * s.K || s.k_stride < (int64_t)s.Hqk * s.K ||
      s.v_stride < (int64_t)s.Hv * s.V)
    return GDN_ERR_INVALID_ARG;
  if (!(s.K == 32 || s.K == 64 || s.K == 128)) return GDN_ERR_UNSUPPORTED;
  if (s.V % 32 != 0 || s.V > 256) return GDN_ERR_UNSUPPORTED;
  if (s.n_seqs > 65535 || s.Hv > 65535) return GDN_ERR_UNSUPPORTED;
  *out = s;
  return GDN_OK;
}

}  // namespace

// The tensor-core path (bf16, K = 128) keeps per-chunk operands in the workspace
// between its two kernels.  With room for every chunk's full operand record
// (gdn_chunk_fwd_workspace_bytes) the split operand/scan kernels run; with at
// least the compact size (gdn_chunk_fwd_min_workspace_bytes: only T of every
// chunk) the older kernel pair that rebuilds the operands inside the scan runs.
bool tc_shape(const gdn_shape &s) { return s.dtype == GDN_BF16 && s.K == 128 && s.V % 32 == 0; }
bool scan_shape(const gdn_shape &s) { return tc_shape(s) && s.V % 64 == 0 && s.V <= 256; }

bool fused_shape(const gdn_shape &s) { return s.dtype == GDN_BF16 && s.K == 128 && s.V == 128; }

extern "C" size_t gdn_chunk_fwd_workspace_bytes(const gdn_shape *shape) {
  gdn_shape s;
  if (normalise_shape(shape, &s) != GDN_OK) return 0;
  // the split path's records; they also hold the fused kernel's ring (GDN_FLAG_FUSED)
  if (scan_shape(s)) {
    const size_t split = chunk_scan_workspace_bytes(s, (int64_t)s.B * s.T);
    return fused_shape(s) ? std::max(split, chunk_fused_workspace_bytes(s)) : split;
  }
  if (tc_shape(s)) return chunk_tc_workspace_bytes(s, (int64_t)s.B * s.T);
  return kWorkspaceBase;
}

extern "C" size_t gdn_chunk_fwd_min_workspace_bytes(const gdn_shape *shape) {
  gdn_shape s;
  if (normalise_shape(shape, &s) != GDN_OK) return 0;
  if (tc_shape(s)) return chunk_tc_workspace_bytes(s, (int64_t)s.B * s.T);
  return kWorkspaceBase;
}

extern "C" size_t gdn_segment_summary_workspace_bytes(const gdn_shape *shape, int32_t n_seg) {
  gdn_shape s;
  if (n_seg < 0 || normalise_shape(shape, &s) != GDN_OK) return 0;
  if (tc_shape(s)) {  // the operand records (or T) of every chunk of every segment
    gdn_shape segs = s;
    segs.n_seqs = n_seg;
    return scan_shape(s) ? chunk_scan_workspace_bytes(segs, s.T) : chunk_tc_workspace_bytes(segs, s.T);
  }
  return kWorkspaceBase;
}

// gdn_chunk_fwd's dispatch.  With nm (gdn_layer_fwd's gated norm), the split scan applies the
// norm in its output epilogue where it can and sets *norm_done; other paths leave it false.
static gdn_status chunk_fwd_impl(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, const float *h0, const int32_t *cu_seqlens,
                                 const gdn_shape *shape, float scale, uint32_t flags, void *o,
                                 float *h_T, void *workspace, size_t workspace_bytes, void *stream,
                                 const NormArgs *nm, bool *norm_done) {
  if (norm_done) *norm_done = false;
  gdn_shape s;
  gdn_status st = normalise_shape(shape, &s);
  if (st != GDN_OK) return st;
  if (flags & ~(GDN_FLAG_QK_L2NORM | GDN_FLAG_SIMT | GDN_FLAG_O_F32 | GDN_FLAG_FUSED |
                GDN_FLAG_TEST_NO_WAIT))
    return GDN_ERR_INVALID_ARG;
  if (cu_seqlens) {
    if (s.B != 1 || s.n_seqs < 0) return GDN_ERR_INVALID_ARG;
  } else if (s.n_seqs != s.B) {
    return GDN_ERR_INVALID_ARG;
  }
  if (!workspace || workspace_bytes < kWorkspaceBase || !aligned(workspace, 256))
    return GDN_ERR_WORKSPACE;
  const int64_t n_tok = cu_seqlens ? s.T : (int64_t)s.B * s.T;
  if (s.n_seqs == 0) return GDN_OK;
  if (n_tok > 0 && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_INVALID_ARG;
  if (n_tok == 0 && !h_T) return GDN_OK;
  if ((flags & GDN_FLAG_FUSED) && !(flags & GDN_FLAG_SIMT) && n_tok > 0 && chunk_fused_supported(q, k, v, s)) {
    // the fused kernel; it declines (before launching anything) when the device cannot hold
    // its grid at once or the workspace is too small for its ring, and another path runs
    const gdn_status fs = chunk_fwd_fused(q, k, v, g, beta, h0, cu_seqlens, s, scale, flags, o, h_T,
                                          workspace, workspace_bytes, (cudaStream_t)stream);
    if (fs != GDN_ERR_UNSUPPORTED) return fs;
  }
  if (!(flags & GDN_FLAG_SIMT) && n_tok > 0 && tc_shape(s) && chunk_tc_supported(q, k, v, s)) {
    if (scan_shape(s) && chunk_scan_supported(q, k, v, s) &&
        workspace_bytes >= chunk_scan_workspace_bytes(s, n_tok)) {
      const bool fuse_norm = nm && chunk_norm_supported(s, flags, *nm);
      const gdn_status r = chunk_fwd_scan(q, k, v, g, beta, h0, cu_seqlens, s, scale, flags, o, h_T,
                                          workspace, workspace_bytes, (cudaStream_t)stream,
                                          fuse_norm ? nm : nullptr);
      if (norm_done) *norm_done = fuse_norm && r == GDN_OK;
      return r;
    }
    return chunk_fwd_tc(q, k, v, g, beta, h0, cu_seqlens, s, scale, flags, o, h_T, workspace,
                        workspace_bytes, (cudaStream_t)stream);
  }
  return chunk_fwd_simt(q, k, v, g, beta, h0, cu_seqlens, s, scale, flags, o, h_T,
                        (int32_t *)workspace, (cudaStream_t)stream);
}

extern "C" gdn_status gdn_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                                    const float *beta, const float *h0, const int32_t *cu_seqlens,
                                    const gdn_shape *shape, float scale, uint32_t flags, void *o,
                                    float *h_T, void *workspace, size_t workspace_bytes,
                                    void *stream) {
  return chunk_fwd_impl(q, k, v, g, beta, h0, cu_seqlens, shape, scale, flags, o, h_T, workspace,
                        workspace_bytes, stream, nullptr, nullptr);
}

extern "C" gdn_status gdn_segment_summary(const void *k, const void *v, const float *g,
                                          const float *beta, const int32_t *seg_bounds,
                                          int32_t n_seg, const gdn_shape *shape, uint32_t flags,
                                          float *M, float *S_local, void *workspace,
                                          size_t workspace_bytes, void *stream) {
  gdn_shape s;
  gdn_status st = normalise_shape(shape, &s);
  if (st != GDN_OK) return st;
  if (flags & ~(GDN_FLAG_QK_L2NORM | GDN_FLAG_SIMT)) return GDN_ERR_INVALID_ARG;
  if (s.B != 1 || n_seg < 0 || n_seg > 65535) return GDN_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < kWorkspaceBase || !aligned(workspace, 256))
    return GDN_ERR_WORKSPACE;
  if (n_seg == 0) return GDN_OK;
  if (!seg_bounds || !M || !S_local) return GDN_ERR_INVALID_ARG;
  if (s.T > 0 && (!k || !v || !g || !beta)) return GDN_ERR_INVALID_ARG;
  if (!(flags & GDN_FLAG_SIMT) && s.T > 0 && tc_shape(s) && chunk_tc_supported(k, k, v, s)) {
    gdn_shape segs = s;
    segs.n_seqs = n_seg;
    if (scan_shape(s) && chunk_scan_supported(k, k, v, s) &&
        workspace_bytes >= chunk_scan_workspace_bytes(segs, s.T))
      return summary_scan(k, v, g, beta, seg_bounds, n_seg, s, flags, M, S_local, workspace,
                          workspace_bytes, (cudaStream_t)stream);
    return summary_tc(k, v, g, beta, seg_bounds, n_seg, s, flags, M, S_local, workspace,
                      workspace_bytes, (cudaStream_t)stream);
  }
  return segment_summary_simt(k, v, g, beta, seg_bounds, n_seg, s, flags, M, S_local,
                              (int32_t *)workspace, (cudaStream_t)stream);
}

// ------------------------------------------------------------------ layer forward

namespace {

constexpr uint32_t kLayerFlags =
    GDN_FLAG_O_F32 | GDN_FLAG_SIMT | GDN_FLAG_LAYER_FRONT | GDN_FLAG_LAYER_NORM_EPILOGUE;

size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

bool front_applies(const gdn_shape &s, int width, uint32_t flags) {
  return (flags & GDN_FLAG_LAYER_FRONT) && !(flags & GDN_FLAG_SIMT) && s.dtype == GDN_BF16 && s.K == 128 &&
         s.V == 128 && width >= 1 && width <= 4;
}

// The chunk shape of the unfused sequence: q, k and v are views of the conv output y.
gdn_shape chunk_view(const gdn_shape &s) {
  gdn_shape c = s;
  const int64_t Cx = 2LL * s.Hqk * s.K + (int64_t)s.Hv * s.V;
  c.q_stride = c.k_stride = c.v_stride = Cx;
  return c;
}

// Unfused layout: [gdn_chunk_fwd's workspace][y][g][beta].
size_t unfused_bytes(const gdn_shape &s, int64_t n_tok) {
  const int64_t Cx = 2LL * s.Hqk * s.K + (int64_t)s.Hv * s.V;
  const size_t es = s.dtype == GDN_BF16 ? 2 : 4;
  gdn_shape c = chunk_view(s);
  return align256(gdn_chunk_fwd_workspace_bytes(&c)) + align256((size_t)n_tok * Cx * es) +
         2 * align256((size_t)n_tok * s.Hv * 4);
}

gdn_status layer_shape(const gdn_shape *shape, int32_t width, gdn_shape *s) {
  if (!shape || shape->q_stride || shape->k_stride || shape->v_stride) return GDN_ERR_INVALID_ARG;
  if (width < 1 || width > 8) return GDN_ERR_INVALID_ARG;
  return normalise_shape(shape, s);
}

}  // namespace

extern "C" size_t gdn_layer_fwd_workspace_bytes(const gdn_shape *shape, int32_t width, uint32_t flags) {
  gdn_shape s;
  if (layer_shape(shape, width, &s) != GDN_OK || (flags & ~kLayerFlags)) return 0;
  const int64_t n_tok = (int64_t)s.B * s.T;
  if (front_applies(s, width, flags)) return chunk_front_workspace_bytes(s, n_tok);
  return unfused_bytes(s, n_tok);
}

extern "C" gdn_status gdn_layer_fwd(const void *x, const void *conv_w, const void *conv_bias, int32_t width,
                                    const void *a, const void *b, const float *A_log, const float *dt_bias,
                                    const float *h0, const int32_t *cu_seqlens, const gdn_shape *shape,
                                    float scale, uint32_t flags, const void *z, const void *norm_w,
                                    float norm_eps, void *o, float *h_T, void *workspace,
                                    size_t workspace_bytes, void *stream) {
  gdn_shape s;
  gdn_status st = layer_shape(shape, width, &s);
  if (st != GDN_OK) return st;
  if (flags & ~kLayerFlags) return GDN_ERR_INVALID_ARG;
  if (cu_seqlens) {
    if (s.B != 1) return GDN_ERR_INVALID_ARG;
  } else if (s.n_seqs != s.B) {
    return GDN_ERR_INVALID_ARG;
  }
  if (z && ((flags & GDN_FLAG_O_F32) || !(norm_eps >= 0.f))) return GDN_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return GDN_ERR_WORKSPACE;
  const int64_t n_tok = cu_seqlens ? s.T : (int64_t)s.B * s.T;
  if (s.n_seqs == 0) return GDN_OK;
  if (n_tok > 0 && (!x || !conv_w || !a || !b || !A_log || !dt_bias || !o)) return GDN_ERR_INVALID_ARG;
  if (n_tok > 0 && !aligned(x, s.dtype == GDN_BF16 ? 16 : 4)) return GDN_ERR_INVALID_ARG;
  cudaStream_t cs = (cudaStream_t)stream;
  if (n_tok == 0) {  // only h_T = h0 (or 0) per sequence
    const gdn_shape c = chunk_view(s);
    return gdn_chunk_fwd(x, x, x, nullptr, nullptr, h0, cu_seqlens, &c, scale, GDN_FLAG_QK_L2NORM, o, h_T,
                         workspace, workspace_bytes, stream);
  }
  const NormArgs nm{z, norm_w, norm_eps};
  const bool want_epilogue = z && (flags & GDN_FLAG_LAYER_NORM_EPILOGUE);
  bool norm_done = false;
  if (front_applies(s, width, flags) && chunk_front_supported(x, conv_w, width, s)) {
    if (workspace_bytes < chunk_front_workspace_bytes(s, n_tok)) return GDN_ERR_WORKSPACE;
    const FrontArgs fr{x, conv_w, conv_bias, width, a, b, A_log, dt_bias};
    const bool fuse_norm = want_epilogue && chunk_norm_supported(s, flags, nm);
    st = chunk_fwd_front(fr, h0, cu_seqlens, s, scale, flags, o, h_T, workspace, workspace_bytes, cs,
                         fuse_norm ? &nm : nullptr);
    norm_done = fuse_norm;
  } else {
    if (workspace_bytes < unfused_bytes(s, n_tok)) return GDN_ERR_WORKSPACE;
    const gdn_shape c = chunk_view(s);
    const int64_t Cx = c.q_stride;
    const size_t es = s.dtype == GDN_BF16 ? 2 : 4;
    const size_t ws_chunk = align256(gdn_chunk_fwd_workspace_bytes(&c));
    uint8_t *ws = (uint8_t *)workspace;
    uint8_t *y = ws + ws_chunk;
    float *g = (float *)(y + align256((size_t)n_tok * Cx * es));
    float *beta = (float *)((uint8_t *)g + align256((size_t)n_tok * s.Hv * 4));
    st = layer_conv_and_gates(x, conv_w, conv_bias, s.dtype, cu_seqlens, s.n_seqs, n_tok, (int32_t)Cx, width, y,
                              a, b, A_log, dt_bias, s.Hv, g, beta, stream);
    if (st != GDN_OK) return st;
    st = chunk_fwd_impl(y, y + (size_t)s.Hqk * s.K * es, y + (size_t)2 * s.Hqk * s.K * es, g, beta, h0,
                        cu_seqlens, &c, scale, GDN_FLAG_QK_L2NORM | (flags & (GDN_FLAG_O_F32 | GDN_FLAG_SIMT)), o,
                        h_T, workspace, ws_chunk, stream, want_epilogue ? &nm : nullptr, &norm_done);
  }
  if (st != GDN_OK || !z || norm_done) return st;
  return gdn_gated_rmsnorm(o, z, norm_w, s.dtype, n_tok * s.Hv, s.V, norm_eps, o, stream);
}
