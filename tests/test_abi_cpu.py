"""C-ABI library checks that need no GPU: it loads, exports every declared symbol,
sizes its buffers as documented, and rejects invalid arguments before launching."""
import ctypes

import numpy as np
import pytest

import __graft_entry__
from mxfp4_precision_gemms_gb300 import binding as mx


@pytest.fixture(scope="module")
def L():
    __graft_entry__.build()
    return mx.lib()


def test_exports_every_declared_symbol(L):
    names = mx.declared_symbols()
    assert len(names) >= 13
    for n in names:
        assert hasattr(L, n), n


def test_buffer_sizes(L):
    assert L.mxfp4_codes_bytes(256, 512) == 256 * 256
    assert L.mxfp4_scales_bytes(256, 512, mx.LAYOUT_ROW, mx.SF_PLAIN) == 256 * 16
    # MMA order pads rows to 128 and 32-blocks to a multiple of 8
    assert L.mxfp4_scales_bytes(200, 96, mx.LAYOUT_ROW, mx.SF_MMA) == 256 * 8
    assert L.mxfp4_scales_bytes(8192, 4096, mx.LAYOUT_COLT, mx.SF_MMA) == 8192 * 128
    assert L.mxfp4_scales_bytes(64, 64, mx.LAYOUT_2D, mx.SF_PLAIN) == 4
    assert L.mxfp4_scales_bytes(64, 64, mx.LAYOUT_2D, mx.SF_MMA) == 0
    assert L.mxfp4_scales_bytes(64, 48, mx.LAYOUT_ROW, mx.SF_PLAIN) == 0  # cols % 32 != 0
    q = L.mxfp4_quantized_bytes(8192, 4096, mx.LAYOUT_ROW, mx.SF_MMA)
    assert q == 8192 * 2048 + 8192 * 128
    cfg = mx.Config()
    assert mx.workspace_bytes(mx.OP_FPROP, 8192, 6144, 4096, cfg) == (
        L.mxfp4_quantized_bytes(8192, 4096, 1, 1) + L.mxfp4_quantized_bytes(6144, 4096, 1, 1))
    assert mx.workspace_bytes(mx.OP_DGRAD, 8192, 6144, 4096, cfg) == L.mxfp4_quantized_bytes(8192, 6144, 1, 1)
    assert mx.workspace_bytes(mx.OP_WGRAD, 8192, 6144, 4096, cfg) == 0


def _tensor(codes=0x1000, scales=0x2000, rows=128, cols=256, layout=1, sf=1, had=16, mode=0):
    return mx.MxTensorC(codes, scales, rows, cols, layout, sf, had, mode)


# With no GPU in this process, any call that gets past validation reaches its first CUDA
# call (the device check) and returns MXFP4_ERR_CUDA.  A validation status therefore
# shows that the call returned before touching CUDA, i.e. before any launch.
PASSED_VALIDATION = 5


def _rq(L, x=0x1000, rows=64, cols=64, ld=64, had=16, mode=0, layouts=1, row=None, colT=None, twoD=None):
    return L.mxfp4_rotate_quantize(ctypes.c_void_p(x), rows, cols, ld, had, mode, layouts,
                                   ctypes.byref(row) if row else None, ctypes.byref(colT) if colT else None,
                                   ctypes.byref(twoD) if twoD else None, None)


def test_rotate_quantize_rejects_bad_arguments(L):
    """Every case fails validation before any CUDA call (the pointers are never touched)."""
    t = _tensor()
    assert _rq(L, x=0, row=t) == 1                       # NULL input
    assert _rq(L, x=0, rows=0, row=t) == 0               # empty: nothing is touched
    assert _rq(L, had=8, row=t) == 1                     # bad Hadamard size
    assert _rq(L, mode=2, row=t) == 1                    # bad scale mode
    assert _rq(L, layouts=0, row=t) == 1                 # nothing requested
    assert _rq(L, layouts=5, row=t, twoD=t) == 1         # 2D mixed with row
    assert _rq(L, cols=48, ld=48, row=t) == 2            # cols % 32
    assert _rq(L, rows=40, layouts=2, colT=t) == 2       # rows % 32 for the column copy
    assert _rq(L, ld=60, row=t) == 3                     # ld % 8
    assert b"ld" in L.mxfp4_last_error()
    assert _rq(L, x=0x1008, row=t) == 3                  # misaligned x
    assert _rq(L, row=None) == 1                         # missing output
    assert _rq(L, row=_tensor(codes=0x1004)) == 3        # misaligned codes
    assert _rq(L, layouts=4, twoD=_tensor(sf=1)) == 1    # 2D has plain scales only


def test_quantiser_row_limit(L):
    t = _tensor()
    assert _rq(L, rows=65535 * 64 + 1, row=t) == 2        # grid limit of the 64-row tiles
    assert b"rows" in L.mxfp4_last_error()


def test_quantiser_fixes_reject_bad_arguments(L):
    P = ctypes.c_void_p
    t1, t2 = _tensor(), _tensor()
    of = lambda x=0x1000, rows=64, cols=256, ld=256, had=16, mode=0, a=-1, q1=t1, q2=t2: L.mxfp4_rotate_quantize_of(
        P(x), rows, cols, ld, had, mode, a, ctypes.byref(q1) if q1 else None, ctypes.byref(q2) if q2 else None, None)
    assert of(a=1) == 1 and of(a=-9) == 1                 # alpha = 2^a with a in [-8, 0]
    assert of(had=8) == 1 and of(mode=3) == 1
    assert of(cols=48, ld=48) == 2                        # cols % 32
    assert of(q2=None) == 1                               # missing output
    assert of(x=0) == 1                                   # NULL input
    assert of(rows=0) == 0                                # empty: nothing touched
    assert of(ld=100) == 3 and of(x=0x1008) == 3          # ld % 8, misaligned x
    assert of(q1=_tensor(codes=0x1004)) == 3              # misaligned codes
    mbs = lambda cols=256, ld=256, m=0x5000, q=t1: L.mxfp4_rotate_quantize_mbs(
        P(0x1000), 64, cols, ld, 16, 0, ctypes.byref(q) if q else None, P(m) if m else None, None)
    assert mbs(cols=96, ld=96) == 2                       # cols % 128
    assert mbs(m=0) == 1                                  # mbs bytes missing
    assert mbs(q=None) == 1


def test_randomised_options_reject_bad_arguments(L):
    P = ctypes.c_void_p
    t1, t2 = _tensor(), _tensor()

    def ex(layouts=3, cs=0, rs=0, srr=0, src=0, rows=64, cols=256, twoD=None):
        o = mx.QuantOptsC(cs or None, rs or None, srr or None, src or None)
        return L.mxfp4_rotate_quantize_ex(P(0x1000), rows, cols, cols, 16, 0, layouts, ctypes.byref(o),
                                          ctypes.byref(t1), ctypes.byref(t2), ctypes.byref(twoD) if twoD else None,
                                          None)
    assert ex(srr=0x8000) == 1                            # stochastic rounding for one of two copies
    assert ex(layouts=4, cs=0x8000, twoD=_tensor(layout=4, sf=0)) == 2  # 2D with an option
    assert ex(cs=0x8008) == 3                             # option arrays 16-byte aligned
    assert ex(rows=40, cs=0x8000) == 2                    # rows % 32 for the column copy
    assert ex(rows=0, srr=0x8000, src=0x9000) == 0        # empty: nothing touched


def test_gemm_rejects_bad_arguments(L):
    a, b = _tensor(), _tensor()
    c = ctypes.c_void_p(0x4000)
    g = lambda A, B, C=c, ldc=128, out=0, acc=0: L.mxfp4_gemm(ctypes.byref(A), ctypes.byref(B), C, ldc, out, acc,
                                                                  None, 0, None)
    assert g(a, _tensor(cols=512)) == 2                  # contraction mismatch
    assert g(a, _tensor(sf=0)) == 1                      # plain scales cannot feed the GEMM
    assert g(a, b, C=ctypes.c_void_p(0)) == 1            # NULL output
    assert g(a, b, out=1, acc=1) == 1                    # accumulate needs fp32
    assert g(a, b, ldc=100) == 3                         # ldc % 8
    assert g(a, b, ldc=64) == 3                          # ldc < N
    assert g(a, _tensor(layout=4)) == 1                  # 2D operand
    assert g(_tensor(cols=48), _tensor(cols=48)) == 2    # cols % 32
    assert g(a, b) == PASSED_VALIDATION


def test_gemm_rejects_operands_of_different_provenance(L):
    """The rotations cancel only when both operands carry the same Hadamard (and scale
    rule); a transposed copy on the A side needs a transposed B (Wgrad)."""
    c = ctypes.c_void_p(0x4000)
    g = lambda A, B: L.mxfp4_gemm(ctypes.byref(A), ctypes.byref(B), c, 128, 0, 0, None, 0, None)
    row, colT = dict(layout=mx.LAYOUT_ROW), dict(layout=mx.LAYOUT_COLT)
    assert g(_tensor(had=16), _tensor(had=32)) == 1      # H16 against H32: no cancellation
    assert g(_tensor(had=16), _tensor(had=0)) == 1
    assert g(_tensor(mode=0), _tensor(mode=1)) == 1      # floor against ceiling scales
    assert b"quantised differently" in L.mxfp4_last_error()
    assert g(_tensor(had=8), _tensor(had=8)) == 1        # not a rotation this library makes
    assert g(_tensor(mode=5), _tensor(mode=5)) == 1
    assert g(_tensor(layout=3), _tensor(layout=3)) == 1  # not one layout
    assert g(_tensor(**colT), _tensor(**row)) == 1       # transposed A with a row-copy B
    for A, B in ((row, row), (row, colT), (colT, colT)):  # Fprop, Dgrad, Wgrad pairs
        assert g(_tensor(**A), _tensor(**B)) == PASSED_VALIDATION


def test_linear_rejects_bad_arguments(L):
    cfg = mx.MxConfigC(16, 0, 0, 0)
    bad = mx.MxConfigC(7, 0, 0, 0)
    P = ctypes.c_void_p
    f = lambda M, N, K, c=cfg, ws=P(0x10000), nb=1 << 40: L.mxfp4_linear_fprop(
        P(0x1000), P(0x2000), M, N, K, ctypes.byref(c), P(0x3000), None, None, ws, nb, None)
    assert f(64, 64, 64, c=bad) == 1
    assert f(64, 64, 48) == 2
    assert f(0, 64, 64) == 2
    assert f(64, 64, 64, ws=P(0), nb=0) == 4             # workspace missing
    assert f(64, 64, 64, nb=10) == 4                     # workspace too small
    assert f(64, 64, 64, ws=P(0x10010)) == 3             # workspace not 256-aligned
    wT = _tensor(rows=64, cols=96)
    assert L.mxfp4_linear_dgrad(P(0x1000), ctypes.byref(wT), 64, 64, 64, ctypes.byref(cfg), P(0x3000), None,
                                P(0x10000), 1 << 40, None) == 2  # wT shape mismatch


def test_fprop_validates_both_operands_before_any_launch(L):
    """Fprop quantises X, then W, then multiplies: a bad W, saved copy or output must be
    rejected before X's pass is queued (the old order launched it first)."""
    P = ctypes.c_void_p
    cfg, bf16_acc = mx.MxConfigC(16, 0, 0, 0), mx.MxConfigC(16, 0, 1, 1)

    def f(M=128, N=256, K=256, x=0x1000, w=0x2000, y=0x3000, c=cfg, xT=None, wT=None):
        return L.mxfp4_linear_fprop(P(x), P(w), M, N, K, ctypes.byref(c), P(y), ctypes.byref(xT) if xT else None,
                                    ctypes.byref(wT) if wT else None, P(0x100000), 1 << 40, None)
    xT, wT = _tensor(rows=256, cols=128, layout=2), _tensor(rows=256, cols=256, layout=2)
    assert f(xT=xT, wT=wT) == PASSED_VALIDATION
    assert f(w=0x2008) == 3                              # misaligned W
    assert f(y=0x3004) == 3                              # misaligned Y
    assert f(N=100) == 3                                 # ldc = N not a multiple of 8
    assert f(N=200, wT=wT) == 2                          # W^T copy needs N % 32 == 0
    assert f(M=100, xT=xT) == 2                          # X^T copy needs M % 32 == 0
    assert f(wT=_tensor(codes=0x5004, layout=2)) == 3    # misaligned saved copy
    assert f(xT=_tensor(scales=0, layout=2)) == 1        # saved copy without scales
    assert f(c=bf16_acc) == 1                            # accumulate needs fp32 output


def test_dgrad_and_wgrad_check_operand_roles(L):
    """W^T must be the transposed copy under the layer's rotation and scale rule, and
    Wgrad takes two transposed copies under it: a row copy of a square W, or an H32 copy
    in an H16 layer, would give a silently wrong product."""
    P = ctypes.c_void_p
    cfg = mx.MxConfigC(16, 0, 1, 0)

    def d(wT, M=256, dy=0x1000, dx=0x3000, dyT=None):
        return L.mxfp4_linear_dgrad(P(dy), ctypes.byref(wT), M, 256, 256, ctypes.byref(cfg), P(dx),
                                    ctypes.byref(dyT) if dyT else None, P(0x100000), 1 << 40, None)
    good = dict(rows=256, cols=256, layout=mx.LAYOUT_COLT)
    assert d(_tensor(**good)) == PASSED_VALIDATION
    assert d(_tensor(**{**good, "layout": mx.LAYOUT_ROW})) == 1   # W's row copy (square W)
    assert d(_tensor(**good, had=32)) == 1                       # H32 copy in an H16 layer
    assert d(_tensor(**good, mode=1)) == 1
    assert d(_tensor(**good), dy=0x1008) == 3                    # misaligned dY
    assert d(_tensor(**good), dx=0x3004) == 3                    # misaligned dX
    assert d(_tensor(**good), M=100, dyT=_tensor(rows=256, cols=100, layout=2)) == 2  # dY^T needs M % 32

    wcfg = mx.MxConfigC(16, 0, 0, 0)
    w = lambda a, b, c=wcfg: L.mxfp4_linear_wgrad(ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), P(0x3000),
                                                  None, 0, None)
    colT = dict(rows=256, cols=512, layout=mx.LAYOUT_COLT)
    assert w(_tensor(**colT), _tensor(**colT)) == PASSED_VALIDATION
    assert w(_tensor(**{**colT, "layout": mx.LAYOUT_ROW}), _tensor(**colT)) == 1
    assert w(_tensor(**colT), _tensor(**{**colT, "layout": mx.LAYOUT_ROW})) == 1
    assert w(_tensor(**colT, had=0), _tensor(**colT, had=0)) == 1  # both H-less in an H16 layer
    assert w(_tensor(**colT), _tensor(**colT), c=mx.MxConfigC(32, 0, 0, 0)) == 1


def test_status_strings(L):
    for s in range(8):
        assert L.mxfp4_status_string(s)
    assert L.mxfp4_status_string(99) == b"unknown status"


@pytest.mark.parametrize("rows,cols", [(128, 256), (200, 96), (33, 32), (256, 4096)])
def test_mma_scale_order_roundtrip(rows, cols):
    """Host-side MMA scale order: a bijection onto the non-padding bytes, matching the
    documented formula at hand-computed positions."""
    g = np.random.default_rng(0)
    plain = g.integers(0, 254, size=(rows, cols // 32), dtype=np.uint8)
    buf = mx.sf_plain_to_mma(plain, rows, cols)
    assert buf.size == ((rows + 127) // 128) * 128 * ((cols // 32 + 7) // 8) * 8
    assert np.array_equal(mx.sf_mma_to_plain(buf, rows, cols), plain)
    idx = mx._mma_index(rows, cols)
    assert len(np.unique(idx)) == idx.size
    assert idx[0, 0] == 0
    if rows > 33 and cols // 32 > 5:
        # row 33 = (r%32 = 1, (r/32)%4 = 1); block 5 = (k/4 = 1, k%4 = 1)
        kb_pad = ((cols // 32 + 7) // 8) * 8
        assert idx[33, 5] == 1 * 512 + 1 * 16 + 1 * 4 + 1
        if rows > 130:
            assert idx[130, 0] == (kb_pad // 4) * 512 + 2 * 16


def test_pair_quantiser_rejects_bad_arguments(L):
    """mxfp4_rotate_quantize_pair validates both matrices and every output before its
    one launch."""
    P = ctypes.c_void_p
    t = [_tensor() for _ in range(4)]

    def pq(a=0x1000, ra=64, lda=256, b=0x9000, rb=64, ldb=256, cols=256, layouts=3, outs=t):
        r = [ctypes.byref(o) if o is not None else None for o in outs]
        return L.mxfp4_rotate_quantize_pair(P(a), ra, lda, P(b), rb, ldb, cols, 16, 0, layouts, *r, None)
    assert pq() == PASSED_VALIDATION
    assert pq(layouts=4) == 1                              # no 2D
    assert pq(b=0x9008) == 3                               # misaligned second matrix
    assert pq(ldb=100) == 3                                # its leading dimension
    assert pq(rb=40) == 2                                  # its transposed copy needs rows % 32
    assert pq(cols=48, lda=48, ldb=48) == 2                # shared cols % 32
    assert pq(outs=[t[0], t[1], t[2], None]) == 1          # a requested output missing
    assert pq(outs=[t[0], t[1], _tensor(codes=0x1004), t[3]]) == 3
    assert pq(ra=0, rb=0) == 0                             # both empty: nothing touched


def test_gemm_group_rejects_bad_arguments(L):
    """Every problem is checked (its index named), at most 8 problems, and no two outputs
    may share a byte -- all before any launch."""
    tensors = []

    def desc(C=0x40000, ldc=128, out=0, acc=0, **kw):
        a, b = _tensor(), _tensor(**kw)
        tensors.extend([a, b])
        return mx.GemmDescC(ctypes.addressof(a), ctypes.addressof(b), C, ldc, out, acc)

    def g(*ds, n=None):
        arr = (mx.GemmDescC * len(ds))(*ds)
        return L.mxfp4_gemm_group(arr, len(ds) if n is None else n, None)
    ok1, ok2 = desc(C=0x40000), desc(C=0x80000)
    assert g(ok1, ok2) == PASSED_VALIDATION
    assert g(ok1, ok2, n=0) == 1 and g(*[desc(C=0x40000 * (i + 1)) for i in range(9)]) == 1
    assert g(ok1, desc(C=0x80000, had=32)) == 1          # problem 1: operands of two rotations
    assert b"problem 1" in L.mxfp4_last_error()
    assert g(ok1, desc(C=0x80000, ldc=100)) == 3         # problem 1: ldc % 8
    assert g(ok1, desc(C=0x40000 + 128 * 127 * 4)) == 1  # overlaps problem 0's last row
    assert b"overlap" in L.mxfp4_last_error()
    assert g(ok1, desc(C=0x40000 + 128 * 128 * 4)) == PASSED_VALIDATION  # right after it


def test_linear_backward_checks_roles_and_workspace(L):
    P = ctypes.c_void_p
    cfg = mx.MxConfigC(16, 0, 1, 0)
    colT = dict(layout=mx.LAYOUT_COLT)

    def b(wT, xT, M=256, N=256, K=256, dx=0x3000, dw=0x80000, ws=P(0x100000), nb=1 << 40):
        return L.mxfp4_linear_backward(P(0x1000), ctypes.byref(wT), ctypes.byref(xT), M, N, K, ctypes.byref(cfg),
                                       P(dx), P(dw), ws, nb, None)
    wT, xT = _tensor(rows=256, cols=256, **colT), _tensor(rows=256, cols=256, **colT)
    assert b(wT, xT) == PASSED_VALIDATION
    assert b(_tensor(rows=256, cols=256), xT) == 1                      # W's row copy in W^T's place
    assert b(wT, _tensor(rows=256, cols=256, had=32, **colT)) == 1      # X^T under another rotation
    assert b(wT, _tensor(rows=256, cols=512, **colT)) == 2              # X^T must be [K, M]
    assert b(wT, xT, ws=P(0), nb=0) == 4                                # workspace missing
    assert b(wT, xT, dx=0x3004) == 3
    assert mx.workspace_bytes(mx.OP_BACKWARD, 8192, 4096, 4096, mx.Config()) == (
        L.mxfp4_quantized_bytes(8192, 4096, 1, 1) + L.mxfp4_quantized_bytes(4096, 8192, 2, 1))


def test_philox_quantiser_rejects_bad_arguments(L):
    P = ctypes.c_void_p
    t1, t2 = _tensor(), _tensor()

    def ph(layouts=3, reserved=0, opts=True, rows=64, x=0x1000):
        o = mx.PhiloxOptsC(1, 2, 3, 1, 1, 1, reserved)
        return L.mxfp4_rotate_quantize_philox(P(x), rows, 256, 256, 16, 0, layouts,
                                              ctypes.byref(o) if opts else None, ctypes.byref(t1), ctypes.byref(t2),
                                              None)
    assert ph() == PASSED_VALIDATION
    assert ph(opts=False) == 1
    assert ph(reserved=1) == 1
    assert ph(layouts=4) == 1                             # no 2D
    assert ph(rows=40) == 2                               # the transposed copy needs rows % 32
    assert ph(x=0x1008) == 3
    assert ph(rows=0) == 0                                # empty: nothing touched


def test_gemm_mbs_rejects_bad_arguments(L):
    P = ctypes.c_void_p
    g = lambda A, B, C=0x40000, ldc=128: L.mxfp4_gemm_mbs(ctypes.byref(A), P(0x9000), ctypes.byref(B), None, P(C),
                                                           ldc, 0, 0, None)
    assert g(_tensor(cols=256), _tensor(cols=256)) == PASSED_VALIDATION
    assert g(_tensor(cols=160), _tensor(cols=160)) == 2            # K % 128
    assert g(_tensor(cols=16512), _tensor(cols=16512)) == 2        # K above 16384
    assert g(_tensor(cols=256, had=16), _tensor(cols=256, had=32)) == 1
    assert g(_tensor(cols=256), _tensor(cols=256), ldc=100) == 3


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c", "c11"), ("c++", "c++11"), ("c++", "c++17")])
def test_header_compiles_standalone(lang, std):
    """include/mxfp4.h is a plain C ABI: it compiles on its own, without CUDA or torch
    headers, as C and as C++, warning-free under -Wall -Wextra -pedantic (the translation
    unit comes on standard input; nothing is written)."""
    import os
    import shutil
    import subprocess

    cc = "gcc" if lang == "c" else "g++"
    if shutil.which(cc) is None:
        pytest.skip(f"{cc} not found")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = '#include "mxfp4.h"\nint main(void) { return mxfp4_status_string(MXFP4_OK) == 0; }\n'
    r = subprocess.run([cc, "-fsyntax-only", f"-std={std}", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.join(root, "include"), "-x", lang, "-"], input=src, capture_output=True,
                       text=True)
    assert r.returncode == 0, r.stderr
