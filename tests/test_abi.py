"""The C-ABI library builds, loads and exports what include/gdn.h declares;
host-side argument checks return errors before anything is launched (CPU only)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from chunked_recurrence_gb300 import build as b
    b.build()
    import chunked_recurrence_gb300 as crg
    return crg.load()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(gdn_\w+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_boundary():
    names = _declared()
    for must in ["gdn_gate_prep", "gdn_conv1d_varlen", "gdn_chunk_fwd", "gdn_segment_summary",
                 "gdn_chain_reduce", "gdn_cu_seqlens_from_position_ids"]:
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    from chunked_recurrence_gb300 import build as b
    out = subprocess.run(["nm", "-D", "--defined-only", b.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (gdn_\w+)", out))
    for name in _declared():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_binding_covers_every_symbol(lib):
    import chunked_recurrence_gb300 as crg
    assert set(_declared()) == set(crg.exported_symbols())


def test_status_strings_and_version(lib):
    assert lib.gdn_status_string(0) == b"GDN_OK"
    assert lib.gdn_status_string(4) == b"GDN_ERR_TIMEOUT"
    assert lib.gdn_status_string(99) == b"GDN_ERR_UNKNOWN"
    assert lib.gdn_version() >> 16 == 1


def _shape(**kw):
    import chunked_recurrence_gb300 as crg
    d = dict(B=1, T=128, n_seqs=1, Hqk=2, Hv=4, K=128, V=128, dtype=1, q_stride=0, k_stride=0,
             v_stride=0)
    d.update(kw)
    return crg.GdnShape(**d)


def test_workspace_bytes(lib):
    assert lib.gdn_chunk_fwd_workspace_bytes(ctypes.byref(_shape())) >= 256
    assert lib.gdn_chunk_fwd_workspace_bytes(ctypes.byref(_shape(Hv=3))) == 0  # Hv % Hqk
    assert lib.gdn_chunk_fwd_workspace_bytes(ctypes.byref(_shape(K=96))) == 0
    assert lib.gdn_segment_summary_workspace_bytes(ctypes.byref(_shape()), 4) >= 256


def test_argument_errors_return_before_launch(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)  # never dereferenced: every call below fails validation first
    ws = P(0x20000)    # 256-byte aligned
    sh = _shape()
    # missing workspace
    assert lib.gdn_chunk_fwd(fake, fake, fake, fake, fake, None, None, ctypes.byref(sh), 1.0, 0,
                             fake, None, None, 0, None) == 5
    # misaligned workspace
    assert lib.gdn_chunk_fwd(fake, fake, fake, fake, fake, None, None, ctypes.byref(sh), 1.0, 0,
                             fake, None, P(0x20004), 256, None) == 5
    # null q
    assert lib.gdn_chunk_fwd(None, fake, fake, fake, fake, None, None, ctypes.byref(sh), 1.0, 0,
                             fake, None, ws, 256, None) == 1
    # unknown flag bit
    assert lib.gdn_chunk_fwd(fake, fake, fake, fake, fake, None, None, ctypes.byref(sh), 1.0, 64,
                             fake, None, ws, 256, None) == 1
    # varlen needs B == 1
    sh2 = _shape(B=2, n_seqs=2)
    assert lib.gdn_chunk_fwd(fake, fake, fake, fake, fake, None, fake, ctypes.byref(sh2), 1.0, 0,
                             fake, None, ws, 256, None) == 1
    # unsupported widths
    assert lib.gdn_chunk_fwd(fake, fake, fake, fake, fake, None, None,
                             ctypes.byref(_shape(K=256)), 1.0, 0, fake, None, ws, 256, None) == 2
    assert lib.gdn_chunk_fwd(fake, fake, fake, fake, fake, None, None,
                             ctypes.byref(_shape(V=48)), 1.0, 0, fake, None, ws, 256, None) == 2
    # q stride smaller than a token
    assert lib.gdn_chunk_fwd(fake, fake, fake, fake, fake, None, None,
                             ctypes.byref(_shape(q_stride=100)), 1.0, 0, fake, None, ws, 256,
                             None) == 1
    # zero sequences is a no-op
    assert lib.gdn_chunk_fwd(None, None, None, None, None, None, fake,
                             ctypes.byref(_shape(n_seqs=0, T=0)), 1.0, 0, None, None, ws, 256,
                             None) == 0
    # gate prep / conv / chain reduce / cu_seqlens checks
    assert lib.gdn_gate_prep(fake, fake, 7, fake, fake, 10, 4, fake, fake, None) == 1
    assert lib.gdn_gate_prep(None, None, 1, None, None, 0, 4, None, None, None) == 0
    assert lib.gdn_gate_prep(None, fake, 1, fake, fake, 10, 4, fake, fake, None) == 1
    assert lib.gdn_conv1d_varlen(fake, fake, None, 1, None, 1, 10, 8, 9, 1, fake, None) == 1
    assert lib.gdn_conv1d_varlen(fake, fake, None, 1, None, 3, 10, 8, 4, 1, fake, None) == 1
    assert lib.gdn_conv1d_varlen(fake, fake, None, 1, None, 1, 10, 8, 4, 2, fake, None) == 1
    assert lib.gdn_chain_reduce(None, None, None, 2, 4, 128, 128, None, None, None) == 1
    assert lib.gdn_chain_reduce(fake, fake, None, 2, 4, 256, 128, fake, None, None) == 2
    assert lib.gdn_cu_seqlens_from_position_ids(fake, -1, fake, fake, None) == 1
    assert lib.gdn_segment_summary(fake, fake, fake, fake, fake, 2, ctypes.byref(_shape(B=2)), 0,
                                   fake, fake, ws, 256, None) == 1
    # decode step: x, cs_in, cs_out, w, bias, dtype, width, act, a, b, A_log, dt_bias, state,
    #              B, Hqk, Hv, K, V, scale, flags, o
    dec = lib.gdn_decode_step
    def d(**kw):
        args = dict(x=fake, ci=fake, co=P(0x30000), w=fake, bias=None, dt=1, W=4, act=1, a=fake, b=fake, al=fake,
                    db=fake, st=fake, B=2, Hqk=2, Hv=4, K=128, V=128, scale=1.0, flags=1, o=fake)
        args.update(kw)
        return dec(*args.values(), None)
    assert d(dt=7) == 1
    assert d(K=48) == 1
    assert d(Hqk=3) == 1
    assert d(W=9) == 1
    assert d(act=2) == 1
    assert d(flags=2) == 1
    assert d(x=None) == 1
    assert d(ci=None) == 1
    assert d(co=fake) == 1      # the conv state may not be updated in place
    assert d(a=None) == 1
    assert d(B=0, x=None, ci=None, co=None, w=None, a=None, b=None, al=None, db=None, st=None, o=None) == 0
    # gated rms norm: o, z, w, dtype, n_rows, V, eps, y
    assert lib.gdn_gated_rmsnorm(fake, fake, None, 7, 10, 128, 1e-6, fake, None) == 1
    assert lib.gdn_gated_rmsnorm(fake, fake, None, 1, 10, 0, 1e-6, fake, None) == 1
    assert lib.gdn_gated_rmsnorm(fake, fake, None, 1, 10, 128, -1.0, fake, None) == 1
    assert lib.gdn_gated_rmsnorm(None, fake, None, 1, 10, 128, 1e-6, fake, None) == 1
    assert lib.gdn_gated_rmsnorm(None, None, None, 1, 0, 128, 1e-6, None, None) == 0
    assert lib.gdn_workspace_reset(None, 0, None) == 5
    assert lib.gdn_workspace_status(None, None, None) == 1


def test_noalloc_refuses_shapes_beyond_its_scratch(lib):
    """gdn_chunk_fwd_noalloc checks the scratch it needs against its fixed 16 MiB
    array before any CUDA call: a million tokens x 4 v-heads (~545 MB) is refused."""
    P = ctypes.c_void_p
    fake = P(0x10000)  # never dereferenced
    big = _shape(T=1 << 20)
    assert lib.gdn_chunk_fwd_noalloc(fake, fake, fake, fake, fake, None, None, ctypes.byref(big),
                                     1.0, 1, fake, None, None) == 5  # GDN_ERR_WORKSPACE
    assert lib.gdn_chunk_fwd_noalloc(fake, fake, fake, fake, fake, None, None,
                                     ctypes.byref(_shape(Hv=3)), 1.0, 1, fake, None, None) == 1


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "chunked_recurrence_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in src and "from oracle" not in src, fn
                assert "gdn_oracle" not in src, fn


def test_chunk_bwd_argument_errors_return_before_launch(lib):
    """gdn_chunk_bwd's host checks: shape, flags, workspace, pointers; nothing is launched."""
    P = ctypes.c_void_p
    fake = P(0x10000)  # never dereferenced
    ws = P(0x20000)    # 256-byte aligned
    sh = _shape()
    need = lib.gdn_chunk_bwd_workspace_bytes(ctypes.byref(sh))
    # over (1 + 2) chunk slots x 4 heads: states of 128 x 128 fp32, the forward sweep's three
    # 64 x 128 fp32 tiles, prep's Z, KG and QG (3 x 64 x 64 fp32) and five 64-vectors, the
    # walk's sums dP, dT (2 x 64 x 64) and dd, db (2 x 64); then two q/k accumulators of
    # 128 x 2 x 128 (each part rounded up to 256 bytes)
    slots_h = 3 * 4
    r256 = lambda b: (b + 255) // 256 * 256
    assert need == (256 + slots_h * 128 * 128 * 4 + slots_h * 3 * 64 * 128 * 4
                    + r256(slots_h * (3 * 64 * 64 + 5 * 64) * 4)
                    + slots_h * (2 * 64 * 64 + 2 * 64) * 4 + 2 * 128 * 2 * 128 * 4)
    assert lib.gdn_chunk_bwd_workspace_bytes(ctypes.byref(_shape(K=96))) == 0
    assert lib.gdn_chunk_bwd_workspace_bytes(ctypes.byref(_shape(V=40))) == 0
    assert lib.gdn_chunk_bwd_workspace_bytes(ctypes.byref(_shape(V=48))) > 0

    def call(q=fake, shape=sh, flags=1, cu=None, w=ws, nbytes=need, dq=fake):
        return lib.gdn_chunk_bwd(q, fake, fake, fake, fake, None, cu, shape if shape is None else ctypes.byref(shape),
                                 1.0, flags, fake, None, dq, fake, fake, fake, fake, None, w, nbytes, None)
    assert call(shape=None) == 1
    assert call(shape=_shape(K=256)) == 2
    assert call(shape=_shape(Hv=3)) == 1
    assert call(flags=2) == 1              # only the L2-norm flag
    assert call(w=None) == 5
    assert call(w=P(0x20004)) == 5
    assert call(nbytes=need - 1) == 5
    assert call(q=None) == 1
    assert call(dq=None) == 1
    assert call(shape=_shape(B=2, n_seqs=2), cu=fake) == 1
    assert call(q=None, shape=_shape(T=0, n_seqs=0), cu=fake, nbytes=256) == 0  # no sequences: no-op


def test_flag_values_match_header_and_test_mode_is_off_by_default():
    """The binding's flag constants are the header's, and no call sets the test-only
    GDN_FLAG_TEST_NO_WAIT unless asked to."""
    import inspect
    import re
    import chunked_recurrence_gb300 as crg
    hdr = open(os.path.join(ROOT, "include", "gdn.h")).read()
    defs = {k: int(v) for k, v in re.findall(r"#define (GDN_FLAG_\w+) (\d+)u", hdr)}
    defs.update({k: int(v) for k, v in re.findall(r"#define (GDN_PATH_\w+) (\d+)", hdr)})
    assert "GDN_FLAG_LAYER_FRONT" in defs and "GDN_PATH_FRONT" in defs
    for name, val in defs.items():
        assert getattr(crg, name) == val, name
    assert inspect.signature(crg.gdn_chunk_fwd).parameters["_test_no_wait"].default is False
    src = inspect.getsource(crg)
    assert src.count("GDN_FLAG_TEST_NO_WAIT if _test_no_wait") == 1


def test_layer_fwd_argument_errors_return_before_launch(lib):
    """gdn_layer_fwd checks the conv width, the flags, dense strides, the norm's arguments, the
    alignment of x and the workspace before anything runs."""
    P = ctypes.c_void_p
    fake, ws = P(0x10000), P(0x20000)  # never dereferenced
    sh = _shape()
    sz = lambda s, w, f: lib.gdn_layer_fwd_workspace_bytes(ctypes.byref(s), w, f)
    assert sz(sh, 4, 0) > 0 and sz(sh, 4, 32) > 0
    assert sz(sh, 0, 0) == 0 and sz(sh, 9, 0) == 0       # width 1..8
    assert sz(sh, 4, 1) == 0 and sz(sh, 4, 8) == 0       # flags the layer call does not take
    assert sz(_shape(q_stride=512), 4, 0) == 0           # x is dense: strides must be 0
    # the fused front end needs no room for y, g and beta
    assert sz(sh, 4, 32) < sz(sh, 4, 0)

    def call(x=fake, w=fake, width=4, shape=sh, flags=0, z=None, eps=1e-6, o_ptr=fake, ws_ptr=ws, nbytes=1 << 30):
        return lib.gdn_layer_fwd(x, w, None, width, fake, fake, fake, fake, None, None, ctypes.byref(shape),
                                 1.0, flags, z, None, eps, o_ptr, None, ws_ptr, nbytes, None)
    assert call(width=9) == 1
    assert call(flags=8) == 1
    assert call(z=fake, flags=4) == 1                    # the norm writes o in the input dtype
    assert call(z=fake, eps=-1.0) == 1
    assert call(x=P(0x10008)) == 1                       # x not 16-byte aligned
    assert call(x=None) == 1
    assert call(ws_ptr=None) == 5
    assert call(ws_ptr=P(0x20040)) == 5                  # workspace not 256-byte aligned
    assert call(nbytes=256) == 5                         # too small
    assert call(nbytes=256, flags=32) == 5              # too small for the front end
    # zero sequences (cu_seqlens of one entry) is a no-op
    assert lib.gdn_layer_fwd(None, None, None, 4, None, None, None, None, None, fake,
                             ctypes.byref(_shape(n_seqs=0, T=0)), 1.0, 0, None, None, 1e-6, None, None, ws,
                             256, None) == 0
