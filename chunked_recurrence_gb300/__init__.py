"""Python binding of libgdn: the chunked gated delta rule forward on one GB300.

Argument marshalling only.  Every function here has the name of the C entry
point it calls (include/gdn.h), checks tensor dtypes, devices and layouts,
allocates outputs with torch when the caller passes none, and passes raw
device pointers and the current CUDA stream through ctypes.  All arithmetic
runs in the library's CUDA kernels; there is no CPU or PyTorch fallback, and
every call raises if libgdn.so is missing or returns an error.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

GDN_OK = 0
GDN_ERR_TIMEOUT, GDN_ERR_BOUNDS = 4, 6  # device-side statuses read from a workspace
GDN_PATH_FUSED = 1                      # path word of a workspace after the fused kernel ran
GDN_PATH_FRONT = 2                      # bit: gdn_layer_fwd's fused front end ran
GDN_PATH_NORM = 4                       # bit: gdn_layer_fwd's norm ran in the scan's epilogue
GDN_F32, GDN_BF16 = 0, 1
GDN_FLAG_QK_L2NORM = 1
GDN_FLAG_SIMT = 2
GDN_FLAG_O_F32 = 4
GDN_FLAG_FUSED = 8
GDN_FLAG_TEST_NO_WAIT = 16
GDN_FLAG_LAYER_FRONT = 32
GDN_FLAG_LAYER_NORM_EPILOGUE = 64
CHUNK = 64

_lib = None
_lock = threading.Lock()


class GdnError(RuntimeError):
    """A libgdn entry point returned a status other than GDN_OK."""


class GdnShape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int64), ("n_seqs", ctypes.c_int32),
                ("Hqk", ctypes.c_int32), ("Hv", ctypes.c_int32), ("K", ctypes.c_int32),
                ("V", ctypes.c_int32), ("dtype", ctypes.c_int32), ("q_stride", ctypes.c_int64),
                ("k_stride", ctypes.c_int64), ("v_stride", ctypes.c_int64)]


_P, _I32, _I64, _U32, _F32, _SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                   ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t)
_SIGS = {
    "gdn_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "gdn_version": ([], _I32),
    "gdn_chunk_fwd_workspace_bytes": ([ctypes.POINTER(GdnShape)], _SZ),
    "gdn_chunk_fwd_min_workspace_bytes": ([ctypes.POINTER(GdnShape)], _SZ),
    "gdn_segment_summary_workspace_bytes": ([ctypes.POINTER(GdnShape), _I32], _SZ),
    "gdn_workspace_reset": ([_P, _SZ, _P], ctypes.c_int),
    "gdn_workspace_status": ([_P, ctypes.POINTER(_I32), _P], ctypes.c_int),
    "gdn_workspace_path": ([_P, ctypes.POINTER(_I32), _P], ctypes.c_int),
    "gdn_gate_prep": ([_P, _P, _I32, _P, _P, _I64, _I32, _P, _P, _P], ctypes.c_int),
    "gdn_conv1d_varlen": ([_P, _P, _P, _I32, _P, _I32, _I64, _I32, _I32, _I32, _P, _P],
                          ctypes.c_int),
    "gdn_chunk_fwd": ([_P, _P, _P, _P, _P, _P, _P, ctypes.POINTER(GdnShape), _F32, _U32, _P, _P,
                       _P, _SZ, _P], ctypes.c_int),
    "gdn_chunk_fwd_noalloc": ([_P, _P, _P, _P, _P, _P, _P, ctypes.POINTER(GdnShape), _F32, _U32,
                               _P, _P, _P], ctypes.c_int),
    "gdn_segment_summary": ([_P, _P, _P, _P, _P, _I32, ctypes.POINTER(GdnShape), _U32, _P, _P,
                             _P, _SZ, _P], ctypes.c_int),
    "gdn_chain_reduce": ([_P, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P], ctypes.c_int),
    "gdn_gated_rmsnorm": ([_P, _P, _P, _I32, _I64, _I32, _F32, _P, _P], ctypes.c_int),
    "gdn_decode_step": ([_P, _P, _P, _P, _P, _I32, _I32, _I32, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32,
                         _I32, _F32, _U32, _P, _P], ctypes.c_int),
    "gdn_cu_seqlens_from_position_ids": ([_P, _I64, _P, _P, _P], ctypes.c_int),
    "gdn_layer_fwd_workspace_bytes": ([ctypes.POINTER(GdnShape), _I32, _U32], _SZ),
    "gdn_layer_fwd": ([_P, _P, _P, _I32, _P, _P, _P, _P, _P, _P, ctypes.POINTER(GdnShape), _F32, _U32, _P, _P,
                       _F32, _P, _P, _P, _SZ, _P], ctypes.c_int),
    "gdn_chunk_bwd_workspace_bytes": ([ctypes.POINTER(GdnShape)], _SZ),
    "gdn_chunk_bwd": ([_P, _P, _P, _P, _P, _P, _P, ctypes.POINTER(GdnShape), _F32, _U32, _P, _P, _P, _P, _P,
                       _P, _P, _P, _P, _SZ, _P], ctypes.c_int),
}


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libgdn.so (optionally building it first) and declare the signatures."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_missing:
            _build.build()
        if not os.path.exists(_build.LIB):
            raise RuntimeError(
                f"libgdn.so not found at {_build.LIB}: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` (no fallback exists)")
        lib = ctypes.CDLL(_build.LIB)
        for name, (args, res) in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def exported_symbols():
    return sorted(_SIGS)


def _check(status: int, what: str):
    if status != GDN_OK:
        msg = load().gdn_status_string(status).decode()
        raise GdnError(f"{what} failed: {msg} ({status})")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor, stream=None):
    if stream is not None:
        return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _dtype_code(dt) -> int:
    if dt == torch.bfloat16:
        return GDN_BF16
    if dt == torch.float32:
        return GDN_F32
    raise TypeError(f"unsupported dtype {dt}: bf16 or fp32")


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("libgdn takes CUDA tensors only (no CPU path exists)")


def _contig(name, t):
    if t is not None and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# --------------------------------------------------------------- front end

def gdn_gate_prep(a, b, A_log, dt_bias, g=None, beta=None, stream=None):
    """g = -exp(A_log) softplus(a + dt_bias), beta = sigmoid(b); a, b [n_tok, Hv]."""
    _need_cuda(a, b, A_log, dt_bias)
    for n, t in (("a", a), ("b", b), ("A_log", A_log), ("dt_bias", dt_bias)):
        _contig(n, t)
    assert a.shape == b.shape and a.dtype == b.dtype and a.dim() == 2
    assert A_log.dtype == torch.float32 and dt_bias.dtype == torch.float32
    n_tok, Hv = a.shape
    g = torch.empty((n_tok, Hv), device=a.device, dtype=torch.float32) if g is None else g
    beta = torch.empty((n_tok, Hv), device=a.device, dtype=torch.float32) if beta is None else beta
    _check(load().gdn_gate_prep(_ptr(a), _ptr(b), _dtype_code(a.dtype), _ptr(A_log),
                                _ptr(dt_bias), n_tok, Hv, _ptr(g), _ptr(beta), _stream(a, stream)),
           "gdn_gate_prep")
    return g, beta


def gdn_decode_step(x, conv_state, w, a, b, A_log, dt_bias, state, Hqk, Hv, K, V, bias=None, act=1,
                    scale=None, l2norm_qk=True, o=None, o_f32=False, conv_state_out=None, stream=None):
    """One decode step for B sequences: the token's gates from a, b [B, Hv], conv1d (+SiLU) of the
    new token x [B, C] with the carried inputs conv_state [B, W-1, C], q/k L2 norm and the
    recurrence on state [B, Hv, V, K] fp32 (updated in place).  Returns (o [B, Hv, V],
    conv_state_out): the carried inputs for the next step, in conv_state_out if given (a
    buffer other than conv_state), else in a new tensor."""
    _need_cuda(x, conv_state, w, a, b, A_log, dt_bias, state, bias)
    for n, t in (("x", x), ("w", w), ("a", a), ("b", b), ("state", state)):
        _contig(n, t)
    B, C = x.shape
    width = w.shape[1]
    assert C == 2 * Hqk * K + Hv * V and w.shape[0] == C and w.dtype == x.dtype
    assert a.dtype == x.dtype == b.dtype and tuple(a.shape) == (B, Hv) == tuple(b.shape)
    assert A_log.dtype == torch.float32 and dt_bias.dtype == torch.float32 and state.dtype == torch.float32
    assert tuple(state.shape) == (B, Hv, V, K)
    _contig("conv_state", conv_state)
    assert tuple(conv_state.shape) == (B, width - 1, C) and conv_state.dtype == x.dtype
    if conv_state_out is None:
        conv_state_out = torch.empty_like(conv_state)
    assert conv_state_out.shape == conv_state.shape and conv_state_out.is_contiguous()
    assert width == 1 or conv_state.numel() == 0 or conv_state_out.data_ptr() != conv_state.data_ptr()
    if scale is None:
        scale = K ** -0.5
    o_dtype = torch.float32 if o_f32 else x.dtype
    if o is None:
        o = torch.empty((B, Hv, V), device=x.device, dtype=o_dtype)
    assert o.dtype == o_dtype and o.is_contiguous()
    flags = (GDN_FLAG_QK_L2NORM if l2norm_qk else 0) | (GDN_FLAG_O_F32 if o_f32 else 0)
    wide = width > 1
    _check(load().gdn_decode_step(_ptr(x), _ptr(conv_state) if wide else None,
                                  _ptr(conv_state_out) if wide else None, _ptr(w), _ptr(bias),
                                  _dtype_code(x.dtype), width, int(act), _ptr(a), _ptr(b), _ptr(A_log),
                                  _ptr(dt_bias), _ptr(state), B, Hqk, Hv, K, V, float(scale), flags, _ptr(o),
                                  _stream(x, stream)), "gdn_decode_step")
    return o, conv_state_out


def gdn_gated_rmsnorm(o, z, w=None, eps=1e-6, y=None, stream=None):
    """y = o / sqrt(mean(o^2) + eps) * w * silu(z) over the last axis (V) of o [..., V]; y may be o."""
    _need_cuda(o, z, w)
    _contig("o", o)
    _contig("z", z)
    assert z.shape == o.shape and z.dtype == o.dtype
    V = o.shape[-1]
    if w is not None:
        assert w.shape == (V,) and w.dtype == o.dtype
    y = torch.empty_like(o) if y is None else y
    assert y.shape == o.shape and y.dtype == o.dtype and y.is_contiguous()
    rows = o.numel() // V if V else 0
    _check(load().gdn_gated_rmsnorm(_ptr(o), _ptr(z), _ptr(w), _dtype_code(o.dtype), rows, V, float(eps),
                                    _ptr(y), _stream(o, stream)), "gdn_gated_rmsnorm")
    return y


def gdn_conv1d_varlen(x, w, bias=None, cu_seqlens=None, n_seqs=None, act=1, y=None, stream=None):
    """Causal depthwise conv1d (+SiLU) per sequence; x [n_tok, C], w [C, W]."""
    _need_cuda(x, w, bias, cu_seqlens)
    _contig("x", x)
    _contig("w", w)
    n_tok, C = x.shape
    width = w.shape[1]
    assert w.shape[0] == C and w.dtype == x.dtype
    if cu_seqlens is not None:
        assert cu_seqlens.dtype == torch.int32
        n_seqs = cu_seqlens.numel() - 1
    elif n_seqs is None:
        n_seqs = 1
    y = torch.empty_like(x) if y is None else y
    _check(load().gdn_conv1d_varlen(_ptr(x), _ptr(w), _ptr(bias), _dtype_code(x.dtype),
                                    _ptr(cu_seqlens), n_seqs, n_tok, C, width, int(act), _ptr(y),
                                    _stream(x, stream)), "gdn_conv1d_varlen")
    return y


def gdn_cu_seqlens_from_position_ids(position_ids, stream=None):
    """Device cu_seqlens (int32 [n_tokens + 1]) and the device count n_seqs (int32 [1])."""
    _need_cuda(position_ids)
    assert position_ids.dtype == torch.int64 and position_ids.dim() == 1
    n = position_ids.numel()
    cu = torch.empty(n + 1, device=position_ids.device, dtype=torch.int32)
    cnt = torch.empty(1, device=position_ids.device, dtype=torch.int32)
    _check(load().gdn_cu_seqlens_from_position_ids(_ptr(position_ids), n, _ptr(cu), _ptr(cnt),
                                                   _stream(position_ids, stream)),
           "gdn_cu_seqlens_from_position_ids")
    return cu, cnt


# -------------------------------------------------------------- recurrence

def make_shape(q, k, v, cu_seqlens=None, B=None, n_seqs=None) -> GdnShape:
    """Shape of a call.  q, k: [n_tok, Hqk, K] (token stride may exceed Hqk*K, e.g. a
    view into the conv output); v: [n_tok, Hv, V]."""
    n_tok, Hqk, K = k.shape
    Hv, V = v.shape[1], v.shape[2]
    for n, t, inner in (("q", q, K), ("k", k, K), ("v", v, V)):
        if t.stride(2) != 1 or t.stride(1) != inner:
            raise ValueError(f"{n}: heads and features must be contiguous within a token")
    if cu_seqlens is not None:
        Bv, T, ns = 1, n_tok, (cu_seqlens.numel() - 1 if n_seqs is None else n_seqs)
    else:
        Bv = 1 if B is None else B
        assert n_tok % Bv == 0
        T, ns = n_tok // Bv, Bv
    return GdnShape(Bv, T, ns, Hqk, Hv, K, V, _dtype_code(k.dtype), q.stride(0), k.stride(0),
                    v.stride(0))


class Workspace:
    """Caller-owned device workspace (torch allocation) for gdn_chunk_fwd / gdn_segment_summary."""

    def __init__(self, nbytes: int, device):
        self.nbytes = max(256, int(nbytes))
        self.buf = torch.zeros(self.nbytes, device=device, dtype=torch.uint8)

    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())

    def status(self, stream=None) -> int:
        out = ctypes.c_int32(0)
        _check(load().gdn_workspace_status(self.ptr(), ctypes.byref(out), _stream(self.buf, stream)),
               "gdn_workspace_status")
        return out.value

    def path(self, stream=None) -> int:
        """The path word: GDN_PATH_FUSED after the fused kernel ran in this workspace."""
        out = ctypes.c_int32(0)
        _check(load().gdn_workspace_path(self.ptr(), ctypes.byref(out), _stream(self.buf, stream)),
               "gdn_workspace_path")
        return out.value

    def reset(self, stream=None):
        _check(load().gdn_workspace_reset(self.ptr(), self.nbytes, _stream(self.buf, stream)),
               "gdn_workspace_reset")


_ws_cache = {}


def _workspace_for(nbytes, device):
    key = (str(device), nbytes)
    ws = _ws_cache.get(key)
    if ws is None:
        ws = _ws_cache[key] = Workspace(nbytes, device)
    return ws


def gdn_chunk_fwd_workspace_bytes(shape: GdnShape) -> int:
    return int(load().gdn_chunk_fwd_workspace_bytes(ctypes.byref(shape)))


def gdn_chunk_fwd_min_workspace_bytes(shape: GdnShape) -> int:
    return int(load().gdn_chunk_fwd_min_workspace_bytes(ctypes.byref(shape)))


def gdn_chunk_fwd(q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None, l2norm_qk=True,
                  B=None, simt=False, o=None, h_T=None, want_h_T=True, workspace=None,
                  stream=None, o_f32=False, fused=False, _test_no_wait=False):
    """Chunked gated delta rule forward; returns (o [n_tok, Hv, V], h_T [n_seqs, Hv, V, K] or None).

    fused=True (bf16, K = V = 128) runs the fused persistent kernel instead of the two-kernel
    split path.  _test_no_wait (tests only) makes every bounded wait of the tensor-core kernels
    (split, or fused) give up at once, so the call ends with GDN_ERR_TIMEOUT in the workspace
    status."""
    _need_cuda(q, k, v, g, beta, h0, cu_seqlens)
    for n, t in (("g", g), ("beta", beta), ("h0", h0)):
        _contig(n, t)
    assert g.dtype == torch.float32 and beta.dtype == torch.float32
    assert q.dtype == k.dtype == v.dtype
    sh = make_shape(q, k, v, cu_seqlens, B)
    n_tok = k.shape[0]
    if scale is None:
        scale = sh.K ** -0.5
    flags = ((GDN_FLAG_QK_L2NORM if l2norm_qk else 0) | (GDN_FLAG_SIMT if simt else 0)
             | (GDN_FLAG_O_F32 if o_f32 else 0) | (GDN_FLAG_FUSED if fused else 0)
             | (GDN_FLAG_TEST_NO_WAIT if _test_no_wait else 0))
    o_dtype = torch.float32 if o_f32 else v.dtype
    if o is None:
        o = torch.empty((n_tok, sh.Hv, sh.V), device=v.device, dtype=o_dtype)
    assert o.dtype == o_dtype and o.is_contiguous()
    if h_T is None and want_h_T:
        h_T = torch.empty((sh.n_seqs, sh.Hv, sh.V, sh.K), device=v.device, dtype=torch.float32)
    if h0 is not None:
        assert h0.dtype == torch.float32 and tuple(h0.shape) == (sh.n_seqs, sh.Hv, sh.V, sh.K)
    if workspace is None:
        workspace = _workspace_for(gdn_chunk_fwd_workspace_bytes(sh), v.device)
    ws = workspace
    _check(load().gdn_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                _ptr(cu_seqlens), ctypes.byref(sh), float(scale), flags, _ptr(o),
                                _ptr(h_T), ws.ptr(), ws.nbytes, _stream(v, stream)),
           "gdn_chunk_fwd")
    return o, h_T


def gdn_chunk_bwd_workspace_bytes(shape: GdnShape) -> int:
    return int(load().gdn_chunk_bwd_workspace_bytes(ctypes.byref(shape)))


def gdn_chunk_bwd(q, k, v, g, beta, d_o, dh_T=None, h0=None, cu_seqlens=None, scale=None, l2norm_qk=True,
                  B=None, want_dh0=True, workspace=None, stream=None):
    """Gradients of <d_o, o> + <dh_T, h_T> for gdn_chunk_fwd's forward with the same inputs.

    d_o [n_tok, Hv, V] and dh_T [n_seqs, Hv, V, K] (or None) are fp32.  Returns
    (dq, dk, dv, dg, dbeta, dh0), all fp32; dh0 is None when want_dh0 is False.
    """
    _need_cuda(q, k, v, g, beta, d_o, dh_T, h0, cu_seqlens)
    for n, t in (("g", g), ("beta", beta), ("d_o", d_o), ("dh_T", dh_T), ("h0", h0)):
        _contig(n, t)
        assert t is None or t.dtype == torch.float32, f"{n} must be fp32"
    assert q.dtype == k.dtype == v.dtype
    sh = make_shape(q, k, v, cu_seqlens, B)
    n_tok = k.shape[0]
    if scale is None:
        scale = sh.K ** -0.5
    dev = v.device
    dq = torch.empty((n_tok, sh.Hqk, sh.K), device=dev, dtype=torch.float32)
    dk = torch.empty_like(dq)
    dv = torch.empty((n_tok, sh.Hv, sh.V), device=dev, dtype=torch.float32)
    dg = torch.empty((n_tok, sh.Hv), device=dev, dtype=torch.float32)
    dbeta = torch.empty_like(dg)
    dh0 = torch.empty((sh.n_seqs, sh.Hv, sh.V, sh.K), device=dev, dtype=torch.float32) if want_dh0 else None
    nbytes = gdn_chunk_bwd_workspace_bytes(sh)
    if nbytes == 0:
        raise GdnError("gdn_chunk_bwd: shape not supported (K 32/64/128, V a multiple of 16 up to 256)")
    ws = workspace or _workspace_for(nbytes, dev)
    flags = GDN_FLAG_QK_L2NORM if l2norm_qk else 0
    _check(load().gdn_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(cu_seqlens),
                                ctypes.byref(sh), float(scale), flags, _ptr(d_o), _ptr(dh_T), _ptr(dq), _ptr(dk),
                                _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(dh0), ws.ptr(), ws.nbytes,
                                _stream(v, stream)),
           "gdn_chunk_bwd")
    return dq, dk, dv, dg, dbeta, dh0


def gdn_chunk_fwd_noalloc(q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None, l2norm_qk=True,
                          B=None, o=None, h_T=None, stream=None):
    """gdn_chunk_fwd without a workspace, for callers that cannot allocate device
    memory: the library's fixed 16 MiB device scratch array is used instead.
    Outputs must then be passed in (o, h_T); shapes whose scratch does not fit
    raise GdnError (GDN_ERR_WORKSPACE)."""
    _need_cuda(q, k, v, g, beta, h0, cu_seqlens)
    sh = make_shape(q, k, v, cu_seqlens, B)
    if scale is None:
        scale = sh.K ** -0.5
    flags = GDN_FLAG_QK_L2NORM if l2norm_qk else 0
    assert o is not None, "gdn_chunk_fwd_noalloc writes into caller-provided o"
    _check(load().gdn_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0),
                                        _ptr(cu_seqlens), ctypes.byref(sh), float(scale), flags,
                                        _ptr(o), _ptr(h_T), _stream(v, stream)),
           "gdn_chunk_fwd_noalloc")
    return o, h_T


def gdn_segment_summary(k, v, g, beta, seg_bounds, l2norm_qk=True, simt=False, M=None,
                        S_local=None, workspace=None, stream=None):
    """Per-segment transition M [n_seg, Hv, K, K] and local state S_local [n_seg, Hv, V, K]."""
    _need_cuda(k, v, g, beta, seg_bounds)
    assert seg_bounds.dtype == torch.int32
    sh = make_shape(k, k, v, None, 1)
    n_seg = seg_bounds.numel() - 1
    flags = (GDN_FLAG_QK_L2NORM if l2norm_qk else 0) | (GDN_FLAG_SIMT if simt else 0)
    if M is None:
        M = torch.empty((n_seg, sh.Hv, sh.K, sh.K), device=v.device, dtype=torch.float32)
    if S_local is None:
        S_local = torch.empty((n_seg, sh.Hv, sh.V, sh.K), device=v.device, dtype=torch.float32)
    nbytes = int(load().gdn_segment_summary_workspace_bytes(ctypes.byref(sh), n_seg))
    ws = workspace or _workspace_for(nbytes, v.device)
    _check(load().gdn_segment_summary(_ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(seg_bounds),
                                      n_seg, ctypes.byref(sh), flags, _ptr(M), _ptr(S_local),
                                      ws.ptr(), ws.nbytes, _stream(v, stream)),
           "gdn_segment_summary")
    return M, S_local


def gdn_chain_reduce(M, S_local, h0=None, S_start=None, h_T=None, stream=None):
    """fp32 chain S_start[i+1] = S_start[i] M_i + S_local_i; returns (S_start, h_T)."""
    _need_cuda(M, S_local, h0)
    _contig("M", M)
    _contig("S_local", S_local)
    n_seg, Hv, V, K = S_local.shape
    S_start = torch.empty_like(S_local) if S_start is None else S_start
    h_T = torch.empty((Hv, V, K), device=S_local.device, dtype=torch.float32) if h_T is None else h_T
    _check(load().gdn_chain_reduce(_ptr(M), _ptr(S_local), _ptr(h0), n_seg, Hv, K, V,
                                   _ptr(S_start), _ptr(h_T), _stream(S_local, stream)),
           "gdn_chain_reduce")
    return S_start, h_T


# -------------------------------------------------------------- composites

def split_qkv(y, Hqk, Hv, K, V):
    """Views of q, k, v inside the conv output y [n_tok, 2*Hqk*K + Hv*V] (Q|K|V channel order)."""
    n_tok, base = y.shape[0], y.storage_offset()
    assert y.stride(1) == 1 and y.shape[1] == 2 * Hqk * K + Hv * V
    q = y.as_strided((n_tok, Hqk, K), (y.stride(0), K, 1), base)
    k = y.as_strided((n_tok, Hqk, K), (y.stride(0), K, 1), base + Hqk * K)
    v = y.as_strided((n_tok, Hv, V), (y.stride(0), V, 1), base + 2 * Hqk * K)
    return q, k, v


def layer_fwd(x, conv_w, a, b, A_log, dt_bias, Hqk, Hv, K, V, h0=None, cu_seqlens=None, B=1,
              scale=None, stream=None, bufs=None, front=False):
    """The GDN layer forward hot path through gdn_layer_fwd: conv1d+SiLU over Q|K|V, gates,
    then the chunked rule with q/k L2 norm (front=True: the fused front end).
    Returns dict(o, h_T)."""
    bufs = bufs if bufs is not None else {}
    o, h_T = gdn_layer_fwd(x, conv_w, a, b, A_log, dt_bias, Hqk, Hv, K, V, h0, cu_seqlens, B, scale,
                           o=bufs.get("o"), h_T=bufs.get("h_T"), front=front,
                           workspace=bufs.get("workspace"), stream=stream)
    return dict(o=o, h_T=h_T)


def layer_shape(x, Hqk, Hv, K, V, cu_seqlens=None, B=1, n_seqs=None) -> GdnShape:
    """Shape of a gdn_layer_fwd call on x [n_tok, 2*Hqk*K + Hv*V] (dense)."""
    n_tok = x.shape[0]
    if x.dim() != 2 or x.shape[1] != 2 * Hqk * K + Hv * V:
        raise ValueError("x must be [n_tok, 2*Hqk*K + Hv*V]")
    if cu_seqlens is not None:
        Bv, T, ns = 1, n_tok, (cu_seqlens.numel() - 1 if n_seqs is None else n_seqs)
    else:
        assert n_tok % B == 0
        Bv, T, ns = B, n_tok // B, B
    return GdnShape(Bv, T, ns, Hqk, Hv, K, V, _dtype_code(x.dtype), 0, 0, 0)


def gdn_layer_fwd_workspace_bytes(shape: GdnShape, width: int, flags: int = 0) -> int:
    return int(load().gdn_layer_fwd_workspace_bytes(ctypes.byref(shape), int(width), int(flags)))


def gdn_layer_fwd(x, conv_w, a, b, A_log, dt_bias, Hqk, Hv, K, V, h0=None, cu_seqlens=None, B=1,
                  scale=None, conv_bias=None, z=None, norm_w=None, norm_eps=1e-6, o=None, h_T=None,
                  want_h_T=True, o_f32=False, simt=False, front=False, norm_epilogue=False, workspace=None,
                  stream=None):
    """The layer's forward in one call: conv1d+SiLU over x's Q|K|V channels, gates, the
    chunked rule with q/k L2 norm and, with z, the gated RMS norm of o.  Returns (o, h_T).

    By default gate prep, conv and gdn_chunk_fwd run as separate launches; front=True (bf16,
    K = V = 128, conv width <= 4) runs the fused front end instead (conv and gates inside the
    chunk operand kernel, same results bit for bit).  With z the gated norm runs as the
    standalone kernel, or with norm_epilogue=True in the state scan's output epilogue."""
    _need_cuda(x, conv_w, a, b, A_log, dt_bias, h0, cu_seqlens, z, norm_w, conv_bias)
    for n, t in (("x", x), ("conv_w", conv_w), ("a", a), ("b", b), ("A_log", A_log),
                 ("dt_bias", dt_bias), ("h0", h0), ("z", z), ("norm_w", norm_w), ("conv_bias", conv_bias)):
        _contig(n, t)
    sh = layer_shape(x, Hqk, Hv, K, V, cu_seqlens, B)
    n_tok = x.shape[0]
    width = conv_w.shape[1]
    assert conv_w.dtype == a.dtype == b.dtype == x.dtype
    assert A_log.dtype == dt_bias.dtype == torch.float32
    if scale is None:
        scale = K ** -0.5
    flags = ((GDN_FLAG_O_F32 if o_f32 else 0) | (GDN_FLAG_SIMT if simt else 0)
             | (GDN_FLAG_LAYER_FRONT if front else 0)
             | (GDN_FLAG_LAYER_NORM_EPILOGUE if norm_epilogue else 0))
    o_dtype = torch.float32 if o_f32 else x.dtype
    if o is None:
        o = torch.empty((n_tok, Hv, V), device=x.device, dtype=o_dtype)
    assert o.dtype == o_dtype and o.is_contiguous()
    if h_T is None and want_h_T:
        h_T = torch.empty((sh.n_seqs, Hv, V, K), device=x.device, dtype=torch.float32)
    if h0 is not None:
        assert h0.dtype == torch.float32 and tuple(h0.shape) == (sh.n_seqs, Hv, V, K)
    if z is not None:
        assert z.dtype == x.dtype and tuple(z.shape) == (n_tok, Hv, V)
    if workspace is None:
        workspace = _workspace_for(gdn_layer_fwd_workspace_bytes(sh, width, flags), x.device)
    ws = workspace
    _check(load().gdn_layer_fwd(_ptr(x), _ptr(conv_w), _ptr(conv_bias), int(width), _ptr(a), _ptr(b),
                                _ptr(A_log), _ptr(dt_bias), _ptr(h0), _ptr(cu_seqlens), ctypes.byref(sh),
                                float(scale), flags, _ptr(z), _ptr(norm_w), float(norm_eps), _ptr(o),
                                _ptr(h_T), ws.ptr(), ws.nbytes, _stream(x, stream)),
           "gdn_layer_fwd")
    return o, h_T


def segment_parallel_fwd(q, k, v, g, beta, seg_bounds, h0=None, scale=None, l2norm_qk=True,
                         stream=None):
    """Two-pass segment-parallel forward of one sequence: per-segment (M, S_local),
    fp32 chain reduce, then every segment from its true start state.  Returns (o, h_T)."""
    M, S_loc = gdn_segment_summary(k, v, g, beta, seg_bounds, l2norm_qk, stream=stream)
    S_start, h_T = gdn_chain_reduce(M, S_loc, h0, stream=stream)
    o, _ = gdn_chunk_fwd(q, k, v, g, beta, S_start, seg_bounds, scale, l2norm_qk,
                         want_h_T=False, stream=stream)
    return o, h_T
