/*
 * gdn.h -- C ABI of libgdn: the chunked gated delta rule forward of a Qwen3.5
 * GatedDeltaNet layer and the steps around it, on one GB300 (sm_103a).
 *
 * The method (gated delta rule, Yang, Kautz, Hatamizadeh, "Gated Delta
 * Networks", ICLR 2025), per v-head h with state S in R^{V x K} kept in fp32:
 *     S_t = exp(g_t) * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = scale * S_t q_t
 * "feat: hybrid CP for Qwen3.5 MoE (DeltaNet + attention)", Summary: the layer
 * is recurrent in a compact per-head state matrix; Approach: a sequence split
 * only has to pass that state between pieces.
 *
 * Conventions shared by every call
 *  - Every pointer argument is a DEVICE pointer, allocated and owned by the
 *    caller, unless stated otherwise.  The library never allocates device
 *    memory, never synchronises the stream, and keeps no per-call state
 *    between calls beyond a cache of driver entry points.
 *  - Calls are asynchronous and ordered on `stream` (a cudaStream_t passed as
 *    void*; NULL is the legacy default stream).
 *  - Argument errors return GDN_ERR_INVALID_ARG / GDN_ERR_UNSUPPORTED before
 *    anything is launched.  A failed launch returns GDN_ERR_CUDA.  Errors that
 *    only the GPU can see (a bounded wait that gave up, a bad index) are
 *    written to the status word at the start of the workspace; read it with
 *    gdn_workspace_status() after the stream has been synchronised.
 *  - Layouts are token-major and row-major: a token's heads are contiguous,
 *    and a head's features are contiguous.  "Dense" strides mean the natural
 *    packed layout.
 *  - Sequences: with cu_seqlens == NULL the token axis holds B rows of T
 *    tokens each; with cu_seqlens (int32, n_seqs+1 increasing offsets, first
 *    0, last = total tokens) it holds n_seqs packed samples and B must be 1
 *    ("[v1] support GDN Ulysses cp", Key decisions 6: varlen only at batch 1).
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1, /* null required pointer, bad size, bad layout */
  GDN_ERR_UNSUPPORTED = 2, /* valid but not built: e.g. K > 128 */
  GDN_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
  GDN_ERR_TIMEOUT = 4,     /* device status: a bounded wait gave up */
  GDN_ERR_WORKSPACE = 5,   /* workspace missing or smaller than required */
  GDN_ERR_BOUNDS = 6       /* device status: an index check failed */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

/* flags of gdn_chunk_fwd / gdn_segment_summary */
#define GDN_FLAG_QK_L2NORM 1u  /* normalise q and k to unit L2 norm on load (eps 1e-6 inside the sqrt) */
#define GDN_FLAG_SIMT 2u       /* force the fp32 CUDA-core kernel (the tensor-core kernel is the default for bf16) */
#define GDN_FLAG_O_F32 4u      /* write o as fp32 whatever the input dtype (default: o has the input dtype) */
#define GDN_FLAG_FUSED 8u      /* gdn_chunk_fwd (bf16, K = V = 128): the fused persistent kernel instead of the two-kernel path */
#define GDN_FLAG_TEST_NO_WAIT 16u /* test only: every bounded wait of the tensor-core split kernels gives up
                                   * at its first missed poll (the state scan's after 32 polls), and with
                                   * GDN_FLAG_FUSED every wait of the fused kernel at its first check, so the
                                   * call ends with GDN_ERR_TIMEOUT in the status word; only the waits that let
                                   * copies and MMAs in flight land before memory is released keep their bound */
#define GDN_FLAG_LAYER_FRONT 32u /* gdn_layer_fwd: the fused front end (conv and gates inside the chunk operand
                                  * kernel) instead of separate launches, where the shape allows it */
#define GDN_FLAG_LAYER_NORM_EPILOGUE 64u /* gdn_layer_fwd with z: the gated norm in the state scan's output
                                          * epilogue instead of the standalone norm kernel, where it applies */

/* Problem shape of the recurrence. */
typedef struct {
  int32_t B;        /* batch rows; 1 when cu_seqlens is given */
  int64_t T;        /* tokens per batch row; total tokens when cu_seqlens is given */
  int32_t n_seqs;   /* number of sequences: B without cu_seqlens, else len(cu_seqlens) - 1 */
  int32_t Hqk;      /* q/k heads; v-head h reads q/k head h / (Hv / Hqk) */
  int32_t Hv;       /* v heads (state heads); a multiple of Hqk */
  int32_t K;        /* key / query width (32, 64 or 128) */
  int32_t V;        /* value width (a multiple of 32, at most 256) */
  int32_t dtype;    /* gdn_dtype of q, k, v and o */
  int64_t q_stride; /* elements between consecutive tokens of q; 0 = dense (Hqk * K) */
  int64_t k_stride; /* same for k; 0 = dense (Hqk * K) */
  int64_t v_stride; /* same for v; 0 = dense (Hv * V) */
} gdn_shape;

/* Human-readable name of a status code (static string). */
const char *gdn_status_string(int status);

/* ABI version: (major << 16) | minor. */
int32_t gdn_version(void);

/* Number of bytes of device workspace gdn_chunk_fwd needs for `shape` on its
 * fastest path (at least 256: the status word and padding).  0 on a bad shape.
 * On the tensor-core path (bf16, K = 128, V a multiple of 64 up to 256) this
 * holds one operand record per chunk and v-head: 256 + (n_seqs +
 * ceil(tokens / 64)) * Hv * (25600 + 256 V) bytes. */
size_t gdn_chunk_fwd_workspace_bytes(const gdn_shape *shape);

/* The smallest workspace gdn_chunk_fwd accepts for `shape`.  Between this and
 * gdn_chunk_fwd_workspace_bytes the tensor-core path keeps only T of every
 * chunk (256 + 8320 * Hv * (n_seqs + ceil(tokens / 64)) bytes) and rebuilds the
 * other operands inside its scan kernel: same results, slower.  0 on a bad
 * shape. */
size_t gdn_chunk_fwd_min_workspace_bytes(const gdn_shape *shape);

/* Zero the status word and the path word at the start of `workspace` (stream-ordered). */
gdn_status gdn_workspace_reset(void *workspace, size_t workspace_bytes, void *stream);

/* The second 32-bit word of a workspace records which kernel path the last
 * gdn_chunk_fwd or gdn_layer_fwd that ran in it took, when that path writes it:
 * GDN_PATH_FUSED for the fused persistent kernel (bf16, K = V = 128); the bits
 * GDN_PATH_FRONT and GDN_PATH_NORM for gdn_layer_fwd's fused front end and its norm
 * epilogue.  The other paths leave the word as they found it, and gdn_workspace_reset
 * clears it, so after a reset a value of 0 means another path ran. */
#define GDN_PATH_FUSED 1
#define GDN_PATH_FRONT 2 /* gdn_layer_fwd's fused front end (conv and gates inside the operand kernel) */
#define GDN_PATH_NORM 4  /* gdn_layer_fwd's gated norm applied in the state scan's output epilogue */

/* Copy the path word (see GDN_PATH_FUSED) of `workspace` to *path_out (host) and
 * synchronise `stream`. */
gdn_status gdn_workspace_path(const void *workspace, int32_t *path_out, void *stream);

/* Copy the status word at the start of `workspace` to *status_out (host) and
 * synchronise `stream`.  *status_out is a gdn_status: GDN_OK when no device
 * check failed since the last reset. */
gdn_status gdn_workspace_status(const void *workspace, int32_t *status_out, void *stream);

/* Gate prep of the Qwen3.5 GatedDeltaNet layer ("[v1] support GDN Ulysses
 * cp", What This PR Does: A_log and dt_bias are per-v-head parameters, a and
 * b per-token inputs):
 *     g    = -exp(A_log[h]) * softplus(a + dt_bias[h])
 *     beta = sigmoid(b)
 * a, b: [n_tokens, Hv] of ab_dtype; A_log, dt_bias: [Hv] fp32;
 * g, beta: [n_tokens, Hv] fp32 outputs.  n_tokens may be 0. */
gdn_status gdn_gate_prep(const void *a, const void *b, int32_t ab_dtype, const float *A_log,
                         const float *dt_bias, int64_t n_tokens, int32_t Hv, float *g, float *beta,
                         void *stream);

/* Depthwise causal conv1d over channels with per-sequence zero history
 * ("[v1] support GDN Ulysses cp", Key decisions 5: the conv is given
 * cu_seqlens so packed samples never read each other's tokens):
 *     y[t, c] = act( bias[c] + sum_{j<W} w[c, j] * x[t - W + 1 + j, c] )
 * where x before the start of t's sequence reads as 0 and act is identity
 * (act = 0) or SiLU (act = 1).  x, y: [n_tokens, C] (row stride C), w: [C, W],
 * bias: [C] or NULL, all of `dtype`; accumulation in fp32.  Sequences are
 * cu_seqlens (n_seqs+1 offsets) or, when cu_seqlens is NULL, n_seqs equal
 * rows of n_tokens / n_seqs tokens.  1 <= W <= 8.  x and y must not overlap.
 * bf16 with C a multiple of 8, W <= 6 and 16-byte aligned x, y stages token rows
 * through shared memory by bulk async copies; a copy wait that runs out (a failed
 * copy, never an input error) leaves NaN in the outputs it could not compute. */
gdn_status gdn_conv1d_varlen(const void *x, const void *w, const void *bias, int32_t dtype,
                             const int32_t *cu_seqlens, int32_t n_seqs, int64_t n_tokens, int32_t C,
                             int32_t width, int32_t act, void *y, void *stream);

/* The chunked gated delta rule forward (chunk size 64; UT/WY transform inside
 * each chunk, state passed from chunk to chunk in fp32).
 *   q, k: [tokens, Hqk, K] (token stride shape->q_stride / k_stride)
 *   v:    [tokens, Hv, V]  (token stride shape->v_stride)
 *   g, beta: [tokens, Hv] fp32 (log-decay and write strength, e.g. from gdn_gate_prep)
 *   h0:   [n_seqs, Hv, V, K] fp32 start states, or NULL for zero
 *   cu_seqlens: see the conventions above, or NULL
 *   scale: multiplies o (1/sqrt(K) in Qwen3.5)
 *   flags: GDN_FLAG_QK_L2NORM, GDN_FLAG_SIMT, GDN_FLAG_O_F32, GDN_FLAG_FUSED,
 *          GDN_FLAG_TEST_NO_WAIT
 *   o:    [tokens, Hv, V] (dense) of shape->dtype, or fp32 with GDN_FLAG_O_F32; every token written
 *   h_T:  [n_seqs, Hv, V, K] fp32 final states, or NULL
 *   workspace: at least gdn_chunk_fwd_workspace_bytes(shape) bytes, 256-byte aligned
 * A sequence of length 0 leaves h_T = h0 (or 0).  q, k, v, o must not overlap. */
gdn_status gdn_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                         const float *beta, const float *h0, const int32_t *cu_seqlens,
                         const gdn_shape *shape, float scale, uint32_t flags, void *o, float *h_T,
                         void *workspace, size_t workspace_bytes, void *stream);

/* gdn_chunk_fwd for callers that cannot allocate device memory.  The pages
 * have no counterpart of this call; it exists for users of this library whose
 * host application owns the whole device memory pool (an inference server or
 * engine plugin with a fixed budget and its own allocator), or whose code path
 * may not take the device-wide synchronisation of cudaMalloc/cudaFree.
 *
 * Arguments, layouts, results and error codes are those of gdn_chunk_fwd
 * without the workspace: the scratch lives in a 16 MiB file-scope device
 * array inside libgdn, held by every GPU that loads the library until the
 * process exits.  The call allocates nothing.
 *  - Size limit: gdn_chunk_fwd_min_workspace_bytes(shape) must fit in 16 MiB;
 *    larger shapes return GDN_ERR_WORKSPACE before anything runs (on the bf16,
 *    K = 128 path that is 256 + 8320 * Hv * (n_seqs + ceil(tokens/64)) bytes,
 *    e.g. 2048 tokens x 32 v-heads or 8192 tokens x 8 v-heads).  Shapes whose
 *    gdn_chunk_fwd_workspace_bytes also fits take the faster path.
 *  - Every call looks up the array's device address on the current device
 *    (cudaGetSymbolAddress), so it stays valid across device resets and new
 *    contexts; make the first call on a device before any stream capture.
 *  - Every call on a device shares the one array and clears its status word
 *    first; calls that overlap on the GPU (different streams, no ordering)
 *    race on it and must not be issued.  Device-side status (bad sequence
 *    ranges, timeouts) is not readable through this entry point. */
gdn_status gdn_chunk_fwd_noalloc(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, const float *h0, const int32_t *cu_seqlens,
                                 const gdn_shape *shape, float scale, uint32_t flags, void *o,
                                 float *h_T, void *stream);

/* Per-segment summary for the segment-parallel two-pass ("Qwen3.5 cp - #1",
 * Architecture and Patches: the pass that outputs each segment's total
 * transition M and local state b).  For segment i = [seg_bounds[i],
 * seg_bounds[i+1]) of the token axis and v-head h, for every start state S:
 *     S_end = S * M[i, h] + S_local[i, h]
 *   M:       [n_seg, Hv, K, K] fp32 = prod_t exp(g_t) (I - beta_t k_t k_t^T)
 *   S_local: [n_seg, Hv, V, K] fp32 = the state reached from 0
 * shape describes the whole token axis (B must be 1, cu_seqlens is not
 * taken: segments must lie inside one sequence).  seg_bounds: device int32
 * [n_seg+1], non-decreasing, inside [0, T]; empty segments give M = I and
 * S_local = 0.  flags: GDN_FLAG_QK_L2NORM.  workspace as for gdn_chunk_fwd. */
size_t gdn_segment_summary_workspace_bytes(const gdn_shape *shape, int32_t n_seg);
gdn_status gdn_segment_summary(const void *k, const void *v, const float *g, const float *beta,
                               const int32_t *seg_bounds, int32_t n_seg, const gdn_shape *shape,
                               uint32_t flags, float *M, float *S_local, void *workspace,
                               size_t workspace_bytes, void *stream);

/* Backward of gdn_chunk_fwd: the gradients that training takes through the layer
 * ("[v1] support GDN Ulysses cp", Testing: loss alignment over training steps;
 * "feat: hybrid CP for Qwen3.5 MoE (DeltaNet + attention)", Test plan:
 * forward/backward passes).  For upstream gradients d_o of o and dh_T of h_T it
 * writes the exact gradients of L = <d_o, o> + <dh_T, h_T> for the forward of
 * gdn_chunk_fwd with the same q, k, v, g, beta, h0, cu_seqlens, shape, scale and
 * flags (GDN_FLAG_QK_L2NORM only): dq, dk [tokens, Hqk, K] (summed over the v-heads
 * that share a q/k head, and taken back through the L2 norm when it is on), dv
 * [tokens, Hv, V], dg, dbeta [tokens, Hv], dh0 [n_seqs, Hv, V, K] (may be NULL).
 * d_o [tokens, Hv, V] and dh_T [n_seqs, Hv, V, K] (NULL: no loss on h_T) are fp32,
 * as are all outputs; q, k, v are of shape->dtype with the strides of gdn_shape.
 * K is 32, 64 or 128; V a multiple of 16 up to 256 (else GDN_ERR_UNSUPPORTED).
 * fp32 state and gradients, products on the tensor cores (TF32 with each fp32 operand split
 * in two, fp32-level accuracy); kernels, all on the stream: a chunk-parallel prep of each chunk's
 * state-independent matrices; a walk, one block per (32 or 16 state rows, v-head,
 * sequence), that recomputes its rows' chunk-start states and then walks the chunks
 * backward; a chunk-parallel pass for the gradients linear in the walk's per-chunk
 * sums; the L2-norm backward.  The workspace (gdn_chunk_bwd_workspace_bytes,
 * 256-byte aligned, caller-owned) holds the status word, the chunk-start states, the
 * walk's per-chunk tiles, the prep matrices, the per-chunk sums and the q/k gradient
 * accumulators; a bad cu_seqlens range sets GDN_ERR_BOUNDS in the status word
 * (gdn_workspace_status).  dq, dk and the per-chunk sums are added atomically, so
 * the last bits of dq, dk, dg and dbeta depend on the order. */
size_t gdn_chunk_bwd_workspace_bytes(const gdn_shape *shape);
gdn_status gdn_chunk_bwd(const void *q, const void *k, const void *v, const float *g, const float *beta,
                         const float *h0, const int32_t *cu_seqlens, const gdn_shape *shape, float scale,
                         uint32_t flags, const float *d_o, const float *dh_T, float *dq, float *dk, float *dv,
                         float *dg, float *dbeta, float *dh0, void *workspace, size_t workspace_bytes,
                         void *stream);

/* One decode step of the layer core for B sequences, continuing from their states
 * ("Qwen3.5 cp - #1", Architecture: after the prefill, decode runs the standard
 * recurrent path from the final ssm_state).  For each sequence b, with the new token's
 * Q|K|V projections x[b], its gate inputs a[b], b[b] and the last W-1 inputs in
 * conv_state_in[b]:
 *     g, beta = the gates of gdn_gate_prep (same arithmetic)
 *     y[c]  = act( bias[c] + sum_{j<W-1} w[c, j] conv_state_in[b, j, c] + w[c, W-1] x[b, c] )
 *             (the conv1d of gdn_conv1d_varlen at the sequence's next token; y rounded
 *             to `dtype` as gdn_conv1d_varlen stores it)
 *     q, k  = y's q and k channels of q/k head h / (Hv / Hqk), L2-normalised with
 *             GDN_FLAG_QK_L2NORM;  v = y's v channels of v-head h
 *     S    <- exp(g) S (I - beta k k^T) + beta v k^T,   o = scale S q
 *     conv_state_out[b] = rows 1 .. W-2 of conv_state_in[b], then x[b]
 *   x:              [B, C] of `dtype`, C = 2 Hqk K + Hv V (q | k | v channels)
 *   conv_state_in:  [B, W-1, C] of `dtype`;  conv_state_out: the same shape, a separate
 *                   buffer (swap the two between steps); both unused when W = 1
 *   w:              [C, W] of `dtype`;  bias: [C] of `dtype` or NULL;  act: 0 none, 1 SiLU
 *   a, b:           [B, Hv] of `dtype`;  A_log, dt_bias: [Hv] fp32
 *   state:          [B, Hv, V, K] fp32, in/out (the layout of gdn_chunk_fwd's h_T)
 *   flags:          GDN_FLAG_QK_L2NORM, GDN_FLAG_O_F32 (any other bit: GDN_ERR_INVALID_ARG)
 *   o:              [B, Hv, V] of `dtype`, or fp32 with GDN_FLAG_O_F32
 * K a multiple of 32 up to 256, V >= 1, 1 <= W <= 8, Hv a multiple of Hqk.  x, o and the
 * two conv-state buffers must not overlap.  One launch on `stream`. */
gdn_status gdn_decode_step(const void *x, const void *conv_state_in, void *conv_state_out, const void *w,
                           const void *bias, int32_t dtype, int32_t width, int32_t act, const void *a,
                           const void *b, const float *A_log, const float *dt_bias, float *state, int32_t B,
                           int32_t Hqk, int32_t Hv, int32_t K, int32_t V, float scale, uint32_t flags, void *o,
                           void *stream);

/* Gated RMS norm of the core's output: the layer's "+ norm" after chunk_gated_delta_rule
 * ("[v1] support GDN Ulysses cp", Design; z is one of the layer's per-token components).
 * The pages give no formula; the reading taken is, per row r of V values,
 *     y[r, v] = o[r, v] / sqrt(mean_v o[r, :]^2 + eps) * w[v] * silu(z[r, v])
 * with rows = tokens x v-heads of o [tokens, Hv, V].
 *   o, z, y: [n_rows, V] of dtype (dense rows); w: [V] of dtype, or NULL for ones
 *   eps >= 0 (1e-6 in Qwen3.5); accumulation in fp32.  y may be o (in place); z must not
 *   overlap y.  n_rows may be 0. */
gdn_status gdn_gated_rmsnorm(const void *o, const void *z, const void *w, int32_t dtype, int64_t n_rows,
                             int32_t V, float eps, void *y, void *stream);

/* The layer's forward in one call ("[v1] support GDN Ulysses cp", What This PR Does and
 * Key decisions 5: the causal conv over the concatenated Q|K|V projections, given cu_seqlens
 * so that packed samples never read each other's tokens, then chunk_gated_delta_rule, then
 * the norm):
 *   y     = SiLU(conv1d(x))            (gdn_conv1d_varlen with act = 1, y rounded to dtype)
 *   q, k, v = y's channels [0, Hqk K), [Hqk K, 2 Hqk K), [2 Hqk K, C); q and k L2-normalised
 *   g, beta = gdn_gate_prep(a, b, A_log, dt_bias)
 *   o, h_T  = gdn_chunk_fwd(q, k, v, g, beta, h0, cu_seqlens, scale)
 *   o      <- gdn_gated_rmsnorm(o, z, norm_w, norm_eps)  when z is not NULL (by default the
 *             standalone kernel on the stored o; with GDN_FLAG_LAYER_NORM_EPILOGUE, bf16 and
 *             V <= 128 a multiple of 64, the split scan's output epilogue on its fp32 o, the
 *             V / 32 scan blocks of a head exchanging each token's sum of squares as one
 *             thread-block cluster; the path word then has GDN_PATH_NORM)
 * Arguments:
 *   x:          [tokens, C] of shape->dtype, C = 2 Hqk K + Hv V, dense, 16-byte aligned
 *   conv_w:     [C, width] of shape->dtype, 1 <= width <= 8;  conv_bias: [C] or NULL
 *   a, b:       [tokens, Hv] of shape->dtype;  A_log, dt_bias: [Hv] fp32
 *   h0, cu_seqlens, scale, o, h_T: as for gdn_chunk_fwd (shape's strides must be 0)
 *   flags:      GDN_FLAG_O_F32, GDN_FLAG_SIMT, GDN_FLAG_LAYER_FRONT, GDN_FLAG_LAYER_NORM_EPILOGUE
 *   z:          [tokens, Hv, V] of shape->dtype or NULL (no norm);  norm_w: [V] or NULL
 *               (ones); norm_eps >= 0.  With z, GDN_FLAG_O_F32 is GDN_ERR_INVALID_ARG.
 *   workspace:  at least gdn_layer_fwd_workspace_bytes(shape, width, flags), 256-byte aligned
 * By default the four steps run as their own launches, with y, g and beta in the workspace.
 * GDN_FLAG_LAYER_FRONT with bf16, K = V = 128 and width <= 4 takes the fused front end
 * instead: the chunk operand kernel reads x's rows (a chunk and the 3 rows before it, zero
 * before the sample's start), applies the conv and SiLU in shared memory and computes the
 * gates, so neither y nor g and beta go to memory (only the conv'd q and k, which the state
 * scan reads again, sit in the workspace: about n_tok * C * 2 bytes less of it).  Its y
 * values are those of gdn_conv1d_varlen's staged bf16 kernel bit for bit, so the results
 * equal the default path's.  It sets the path word to GDN_PATH_FRONT.  (On a GB300 at the
 * Qwen3.5-4B layer's shape it measures a few percent slower than the separate launches: the
 * conv's arithmetic lengthens the latency-bound operand kernel by more than the separate
 * conv costs.)  x, o and z must not overlap; o may not alias the workspace. */
size_t gdn_layer_fwd_workspace_bytes(const gdn_shape *shape, int32_t width, uint32_t flags);
gdn_status gdn_layer_fwd(const void *x, const void *conv_w, const void *conv_bias, int32_t width,
                         const void *a, const void *b, const float *A_log, const float *dt_bias,
                         const float *h0, const int32_t *cu_seqlens, const gdn_shape *shape, float scale,
                         uint32_t flags, const void *z, const void *norm_w, float norm_eps, void *o,
                         float *h_T, void *workspace, size_t workspace_bytes, void *stream);

/* fp32 chain reduce of the segment summaries ("Qwen3.5 cp - #1",
 * Architecture: (b, M) chain reduce, fp32):
 *     S_start[0] = h0 (or 0);  S_start[i+1] = S_start[i] M[i] + S_local[i];  h_T = S_start[n_seg]
 * M: [n_seg, Hv, K, K], S_local: [n_seg, Hv, V, K], h0: [Hv, V, K] or NULL,
 * S_start: [n_seg, Hv, V, K] out, h_T: [Hv, V, K] out or NULL; all fp32, 16-byte aligned
 * (GDN_ERR_INVALID_ARG otherwise).  K a multiple of 4, at most 128 (else
 * GDN_ERR_UNSUPPORTED).  Pass 2 is gdn_chunk_fwd with cu_seqlens = seg_bounds and
 * h0 = S_start. */
gdn_status gdn_chain_reduce(const float *M, const float *S_local, const float *h0, int32_t n_seg,
                            int32_t Hv, int32_t K, int32_t V, float *S_start, float *h_T,
                            void *stream);

/* cu_seqlens from position_ids ("[v1] support GDN Ulysses cp", Key decisions
 * 4): a sample starts at token 0 and wherever position_ids is 0.
 * position_ids: [n_tokens] int64; cu_seqlens: [n_tokens + 1] int32 out, of
 * which the first n_seqs + 1 entries are written; n_seqs: one int32 out on
 * the device.  n_tokens may be 0 (then n_seqs = 0, cu_seqlens[0] = 0). */
gdn_status gdn_cu_seqlens_from_position_ids(const int64_t *position_ids, int64_t n_tokens,
                                            int32_t *cu_seqlens, int32_t *n_seqs, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* GDN_H_ */
