"""ctypes binding of libmxfp4.so (include/mxfp4.h).

Argument marshalling only: every step of the path (rotation, scale, quantisation,
GEMM) runs in the library's CUDA kernels.  torch supplies device memory, streams
and events.  If the library is missing, every call raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from dataclasses import dataclass

import numpy as np
import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmxfp4.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "mxfp4.h")

HAD_NONE, HAD_16, HAD_32 = 0, 16, 32
SCALE_FLOOR, SCALE_CEIL = 0, 1
LAYOUT_ROW, LAYOUT_COLT, LAYOUT_2D = 1, 2, 4
OUT_F32, OUT_BF16 = 0, 1
SF_PLAIN, SF_MMA = 0, 1
OP_FPROP, OP_DGRAD, OP_WGRAD, OP_BACKWARD = 0, 1, 2, 3

STATUS = {0: "MXFP4_OK", 1: "MXFP4_ERR_INVALID_ARG", 2: "MXFP4_ERR_UNSUPPORTED_SHAPE", 3: "MXFP4_ERR_MISALIGNED",
          4: "MXFP4_ERR_WORKSPACE", 5: "MXFP4_ERR_CUDA", 6: "MXFP4_ERR_TIMEOUT", 7: "MXFP4_ERR_UNSUPPORTED_DEVICE"}


class MxTensorC(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("layout", ctypes.c_int32), ("sf_layout", ctypes.c_int32),
                ("had", ctypes.c_int32), ("mode", ctypes.c_int32)]


class QuantOptsC(ctypes.Structure):
    """mxfp4_quant_opts: sign bitmasks and random integers (device pointers or NULL)."""
    _fields_ = [("col_signs", ctypes.c_void_p), ("row_signs", ctypes.c_void_p), ("sr_row", ctypes.c_void_p),
                ("sr_colT", ctypes.c_void_p)]


class GemmDescC(ctypes.Structure):
    """mxfp4_gemm_desc: one problem of a grouped GEMM launch."""
    _fields_ = [("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("C", ctypes.c_void_p), ("ldc", ctypes.c_int64),
                ("out_dtype", ctypes.c_int32), ("accumulate", ctypes.c_int32)]


class PhiloxOptsC(ctypes.Structure):
    """mxfp4_philox_opts: seeds and switches of the in-kernel Philox4x32-10 numbers."""
    _fields_ = [("col_sign_seed", ctypes.c_uint64), ("row_sign_seed", ctypes.c_uint64), ("sr_seed", ctypes.c_uint64),
                ("col_signs", ctypes.c_int32), ("row_signs", ctypes.c_int32),
                ("stochastic_rounding", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class MxConfigC(ctypes.Structure):
    _fields_ = [("had", ctypes.c_int32), ("mode", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("accumulate", ctypes.c_int32)]


class Mxfp4Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def lib():
    """Loads libmxfp4.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                                   "g.build()'` (there is no CPU fallback)")
            L = ctypes.CDLL(LIB_PATH)
            P, I64, I, U, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
            T = ctypes.POINTER(MxTensorC)
            CF = ctypes.POINTER(MxConfigC)
            sig = {
                "mxfp4_codes_bytes": ([I64, I64], S),
                "mxfp4_scales_bytes": ([I64, I64, I, I], S),
                "mxfp4_quantized_bytes": ([I64, I64, I, I], S),
                "mxfp4_rotate_quantize": ([P, I64, I64, I64, I, I, U, T, T, T, P], I),
                "mxfp4_rotate_quantize_pair": ([P, I64, I64, P, I64, I64, I64, I, I, U, T, T, T, T, P], I),
                "mxfp4_rotate_quantize_of": ([P, I64, I64, I64, I, I, I, T, T, P], I),
                "mxfp4_rotate_quantize_ex": ([P, I64, I64, I64, I, I, U, ctypes.POINTER(QuantOptsC), T, T, T, P], I),
                "mxfp4_rotate_quantize_mbs": ([P, I64, I64, I64, I, I, T, P, P], I),
                "mxfp4_rotate_quantize_philox": ([P, I64, I64, I64, I, I, U, ctypes.POINTER(PhiloxOptsC), T, T, P],
                                                 I),
                "mxfp4_gemm": ([T, T, P, I64, I, I, P, S, P], I),
                "mxfp4_gemm_group": ([ctypes.POINTER(GemmDescC), I, P], I),
                "mxfp4_gemm_mbs": ([T, P, T, P, P, I64, I, I, P], I),
                "mxfp4_workspace_bytes": ([I, I64, I64, I64, CF], S),
                "mxfp4_linear_fprop": ([P, P, I64, I64, I64, CF, P, T, T, P, S, P], I),
                "mxfp4_linear_dgrad": ([P, T, I64, I64, I64, CF, P, T, P, S, P], I),
                "mxfp4_linear_wgrad": ([T, T, CF, P, P, S, P], I),
                "mxfp4_linear_backward": ([P, T, T, I64, I64, I64, CF, P, P, P, S, P], I),
                "mxfp4_linear_fprop_noalloc": ([P, P, I64, I64, I64, CF, P, T, T, P], I),
                "mxfp4_noalloc_scratch_bytes": ([], S),
                "mxfp4_error_decomposition": ([P, I64, I64, I64, I, I, P, P], I),
                "mxfp4_mma_peak_probe": ([I, I64, ctypes.POINTER(ctypes.c_double)], I),
                "mxfp4_device_status": ([P], I),
                "mxfp4_set_wait_limit_ns": ([ctypes.c_uint64], None),
                "mxfp4_test_inject_gemm_fault": ([I], None),
                "mxfp4_status_string": ([I], ctypes.c_char_p),
                "mxfp4_last_error": ([], ctypes.c_char_p),
            }
            for name, (args, res) in sig.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
    return _lib


def declared_symbols() -> list[str]:
    """Function names declared in include/mxfp4.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(mxfp4_[a-z0-9_]+)\s*\(", text)))


def _check(status: int):
    if status != 0:
        raise Mxfp4Error(status, lib().mxfp4_last_error().decode())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr())


# ----------------------------------------------------------------- quantised tensors
@dataclass
class QTensor:
    """A quantised matrix [rows, cols] (blocks of 32 along cols) held in torch memory."""
    codes: torch.Tensor   # uint8 [rows, cols/2]
    scales: torch.Tensor  # uint8: plain [rows, cols/32] / [rows/32, cols/32], or flat MMA order
    rows: int
    cols: int
    layout: int
    sf_layout: int
    had: int = 0
    mode: int = 0

    def c(self) -> MxTensorC:
        return MxTensorC(self.codes.data_ptr(), self.scales.data_ptr(), self.rows, self.cols, self.layout,
                         self.sf_layout, self.had, self.mode)

    def plain_scales(self) -> np.ndarray:
        s = self.scales.cpu().numpy()
        if self.sf_layout == SF_PLAIN:
            return s
        return sf_mma_to_plain(s, self.rows, self.cols)

    @property
    def nbytes(self) -> int:
        return self.codes.numel() + self.scales.numel()


def codes_bytes(rows: int, cols: int) -> int:
    return lib().mxfp4_codes_bytes(rows, cols)


def scales_bytes(rows: int, cols: int, layout: int, sf_layout: int) -> int:
    return lib().mxfp4_scales_bytes(rows, cols, layout, sf_layout)


def empty_qtensor(rows: int, cols: int, layout: int, sf_layout: int, device="cuda") -> QTensor:
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=device)
    if layout == LAYOUT_2D:
        scales = torch.empty((rows // 32, cols // 32), dtype=torch.uint8, device=device)
    elif sf_layout == SF_PLAIN:
        scales = torch.empty((rows, cols // 32), dtype=torch.uint8, device=device)
    else:
        scales = torch.empty(scales_bytes(rows, cols, layout, sf_layout), dtype=torch.uint8, device=device)
    return QTensor(codes, scales, rows, cols, layout, sf_layout)


# ----------------------------------------------------------------- MMA scale order (host marshalling)
def _mma_index(rows: int, cols: int) -> np.ndarray:
    kb = cols // 32
    kb_pad = ((kb + 7) // 8) * 8
    r = np.arange(rows, dtype=np.int64)[:, None]
    k = np.arange(kb, dtype=np.int64)[None, :]
    return ((r // 128) * (kb_pad // 4) + k // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (k % 4)


def sf_mma_bytes(rows: int, cols: int) -> int:
    return ((rows + 127) // 128) * 128 * (((cols // 32 + 7) // 8) * 8)


def sf_mma_to_plain(buf: np.ndarray, rows: int, cols: int) -> np.ndarray:
    return np.asarray(buf).reshape(-1)[_mma_index(rows, cols)]


def sf_plain_to_mma(plain: np.ndarray, rows: int, cols: int) -> np.ndarray:
    out = np.zeros(sf_mma_bytes(rows, cols), np.uint8)
    out[_mma_index(rows, cols)] = plain
    return out


def qtensor_from_host(codes: np.ndarray, plain_scales: np.ndarray, layout: int = LAYOUT_ROW,
                      device="cuda", had: int = HAD_NONE, mode: int = SCALE_FLOOR) -> QTensor:
    """Uploads host codes [rows, cols/2] and plain scales [rows, cols/32] as an MMA-order
    QTensor; had / mode record how they were produced (the GEMM requires both operands
    to agree)."""
    rows, cols = codes.shape[0], codes.shape[1] * 2
    c = torch.from_numpy(np.ascontiguousarray(codes)).to(device)
    s = torch.from_numpy(sf_plain_to_mma(plain_scales, rows, cols)).to(device)
    return QTensor(c, s, rows, cols, layout, SF_MMA, had, mode)


# ----------------------------------------------------------------- entry points
def rotate_quantize(x: torch.Tensor, had: int = HAD_16, mode: int = SCALE_FLOOR, layouts: int = LAYOUT_ROW,
                    sf_layout: int = SF_MMA, outs: dict | None = None, stream=None) -> dict:
    """mxfp4_rotate_quantize on a bf16 CUDA matrix [rows, cols] (row-major, ld = stride(0)).
    Returns {'row': QTensor, 'colT': QTensor, '2d': QTensor} for the requested layouts."""
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 2 or (x.numel() and x.stride(1) != 1):
        raise ValueError("x must be a CUDA bf16 matrix with unit column stride")
    R, C = x.shape
    outs = dict(outs or {})
    if layouts & LAYOUT_ROW and "row" not in outs:
        outs["row"] = empty_qtensor(R, C, LAYOUT_ROW, sf_layout, x.device)
    if layouts & LAYOUT_COLT and "colT" not in outs:
        outs["colT"] = empty_qtensor(C, R, LAYOUT_COLT, sf_layout, x.device)
    if layouts & LAYOUT_2D and "2d" not in outs:
        outs["2d"] = empty_qtensor(R, C, LAYOUT_2D, SF_PLAIN, x.device)
    cs = {k: v.c() for k, v in outs.items()}
    ref = lambda k: ctypes.byref(cs[k]) if (k in cs) else None
    _check(lib().mxfp4_rotate_quantize(_ptr(x), R, C, x.stride(0), had, mode, layouts, ref("row"), ref("colT"),
                                       ref("2d"), _stream(stream)))
    for v in outs.values():
        v.had, v.mode = had, mode
    return outs


def rotate_quantize_pair(a: torch.Tensor, b: torch.Tensor, had: int = HAD_16, mode: int = SCALE_FLOOR,
                         layouts: int = LAYOUT_ROW | LAYOUT_COLT, sf_layout: int = SF_MMA,
                         outs_a: dict | None = None, outs_b: dict | None = None, stream=None) -> tuple[dict, dict]:
    """mxfp4_rotate_quantize_pair: two bf16 CUDA matrices with the same number of columns
    (a GEMM's operands) rotated and quantised in one launch.  Returns two dicts like
    rotate_quantize's ({'row': QTensor, 'colT': QTensor} for the requested layouts)."""
    for x in (a, b):
        _check_bf16_matrix(x)
    if a.shape[1] != b.shape[1]:
        raise ValueError("a and b must have the same number of columns")
    C = a.shape[1]
    res = []
    for x, outs in ((a, outs_a), (b, outs_b)):
        outs = dict(outs or {})
        R = x.shape[0]
        if layouts & LAYOUT_ROW and "row" not in outs:
            outs["row"] = empty_qtensor(R, C, LAYOUT_ROW, sf_layout, x.device)
        if layouts & LAYOUT_COLT and "colT" not in outs:
            outs["colT"] = empty_qtensor(C, R, LAYOUT_COLT, sf_layout, x.device)
        res.append(outs)
    cs = [{k: v.c() for k, v in o.items()} for o in res]
    ref = lambda i, k: ctypes.byref(cs[i][k]) if k in cs[i] else None
    _check(lib().mxfp4_rotate_quantize_pair(_ptr(a), a.shape[0], a.stride(0), _ptr(b), b.shape[0], b.stride(0), C,
                                            had, mode, layouts, ref(0, "row"), ref(0, "colT"), ref(1, "row"),
                                            ref(1, "colT"), _stream(stream)))
    for o in res:
        for v in o.values():
            v.had, v.mode = had, mode
    return res[0], res[1]


def _check_bf16_matrix(x: torch.Tensor):
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 2 or (x.numel() and x.stride(1) != 1):
        raise ValueError("x must be a CUDA bf16 matrix with unit column stride")


def rotate_quantize_of(x: torch.Tensor, had: int = HAD_16, mode: int = SCALE_FLOOR, alpha_log2: int = -1,
                       sf_layout: int = SF_MMA, stream=None) -> tuple[QTensor, QTensor]:
    """mxfp4_rotate_quantize_of: outlier fallback, row layout.  Returns (q1, q2) with
    the OF value dq(q1) + dq(q2) (alpha = 2^alpha_log2 carried by q2's scales)."""
    _check_bf16_matrix(x)
    R, C = x.shape
    q1 = empty_qtensor(R, C, LAYOUT_ROW, sf_layout, x.device)
    q2 = empty_qtensor(R, C, LAYOUT_ROW, sf_layout, x.device)
    c1, c2 = q1.c(), q2.c()
    _check(lib().mxfp4_rotate_quantize_of(_ptr(x), R, C, x.stride(0), had, mode, alpha_log2, ctypes.byref(c1),
                                          ctypes.byref(c2), _stream(stream)))
    for q in (q1, q2):
        q.had, q.mode = had, mode
    return q1, q2


def rotate_quantize_rand(x: torch.Tensor, had: int = HAD_16, mode: int = SCALE_FLOOR, layouts: int = LAYOUT_ROW,
                         col_signs: torch.Tensor | None = None, row_signs: torch.Tensor | None = None,
                         sr_row: torch.Tensor | None = None, sr_colT: torch.Tensor | None = None,
                         sf_layout: int = SF_MMA, stream=None) -> dict:
    """mxfp4_rotate_quantize_ex: random sign flips (uint8 bitmask tensors) and stochastic
    rounding (int16/uint16 tensors of uniform 16-bit integers, [rows, cols] for the row
    copy and [cols, rows] for the transposed copy).  Returns {'row': ..., 'colT': ...}."""
    _check_bf16_matrix(x)
    R, C = x.shape
    outs = {}
    if layouts & LAYOUT_ROW:
        outs["row"] = empty_qtensor(R, C, LAYOUT_ROW, sf_layout, x.device)
    if layouts & LAYOUT_COLT:
        outs["colT"] = empty_qtensor(C, R, LAYOUT_COLT, sf_layout, x.device)
    ptr = lambda t: None if t is None else t.data_ptr()
    opts = QuantOptsC(ptr(col_signs), ptr(row_signs), ptr(sr_row), ptr(sr_colT))
    cs = {k: v.c() for k, v in outs.items()}
    ref = lambda k: ctypes.byref(cs[k]) if (k in cs) else None
    _check(lib().mxfp4_rotate_quantize_ex(_ptr(x), R, C, x.stride(0), had, mode, layouts, ctypes.byref(opts),
                                          ref("row"), ref("colT"), None, _stream(stream)))
    for v in outs.values():
        v.had, v.mode = had, mode
    return outs


def rotate_quantize_philox(x: torch.Tensor, had: int = HAD_16, mode: int = SCALE_FLOOR, layouts: int = LAYOUT_ROW,
                           col_sign_seed: int | None = None, row_sign_seed: int | None = None,
                           sr_seed: int | None = None, sf_layout: int = SF_MMA, stream=None) -> dict:
    """mxfp4_rotate_quantize_philox: random signs (a seed per dimension) and stochastic
    rounding (sr_seed) drawn in the kernel from Philox4x32-10; None turns an option off.
    Returns {'row': ..., 'colT': ...} for the requested layouts."""
    _check_bf16_matrix(x)
    R, C = x.shape
    outs = {}
    if layouts & LAYOUT_ROW:
        outs["row"] = empty_qtensor(R, C, LAYOUT_ROW, sf_layout, x.device)
    if layouts & LAYOUT_COLT:
        outs["colT"] = empty_qtensor(C, R, LAYOUT_COLT, sf_layout, x.device)
    opts = PhiloxOptsC(col_sign_seed or 0, row_sign_seed or 0, sr_seed or 0, int(col_sign_seed is not None),
                       int(row_sign_seed is not None), int(sr_seed is not None), 0)
    cs = {k: v.c() for k, v in outs.items()}
    ref = lambda k: ctypes.byref(cs[k]) if (k in cs) else None
    _check(lib().mxfp4_rotate_quantize_philox(_ptr(x), R, C, x.stride(0), had, mode, layouts, ctypes.byref(opts),
                                              ref("row"), ref("colT"), _stream(stream)))
    for v in outs.values():
        v.had, v.mode = had, mode
    return outs


def rotate_quantize_mbs(x: torch.Tensor, had: int = HAD_16, mode: int = SCALE_FLOOR, sf_layout: int = SF_MMA,
                        stream=None) -> tuple[QTensor, torch.Tensor]:
    """mxfp4_rotate_quantize_mbs: macro-block scaling, row layout.  Returns (q, mbs) with
    mbs [rows, cols/128] uint8; the reconstruction is dq(q) / (1 + mbs/256)."""
    _check_bf16_matrix(x)
    R, C = x.shape
    q = empty_qtensor(R, C, LAYOUT_ROW, sf_layout, x.device)
    mbs = torch.empty((R, max(C // 128, 0)), dtype=torch.uint8, device=x.device)
    c = q.c()
    _check(lib().mxfp4_rotate_quantize_mbs(_ptr(x), R, C, x.stride(0), had, mode, ctypes.byref(c), _ptr(mbs),
                                           _stream(stream)))
    q.had, q.mode = had, mode
    return q, mbs


def gemm(A: QTensor, B: QTensor, out_dtype: int = OUT_F32, accumulate: bool = False,
         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """C[M,N] = A . B^T (block-scaled MXFP4, fp32 accumulation)."""
    if out is None:
        dt = torch.float32 if out_dtype == OUT_F32 else torch.bfloat16
        out = (torch.zeros if accumulate else torch.empty)((A.rows, B.rows), dtype=dt, device=A.codes.device)
    a, b = A.c(), B.c()
    _check(lib().mxfp4_gemm(ctypes.byref(a), ctypes.byref(b), _ptr(out), out.stride(0), out_dtype, int(accumulate),
                            None, 0, _stream(stream)))
    return out


def gemm_mbs(A: QTensor, mbs_a: torch.Tensor | None, B: QTensor, mbs_b: torch.Tensor | None,
             out_dtype: int = OUT_F32, accumulate: bool = False, out: torch.Tensor | None = None,
             stream=None) -> torch.Tensor:
    """mxfp4_gemm_mbs: C = x_hat_A . x_hat_B^T over macro-block-scaled operands (mbs_a /
    mbs_b: uint8 [rows, K/128] device tensors from rotate_quantize_mbs, or None)."""
    if out is None:
        dt = torch.float32 if out_dtype == OUT_F32 else torch.bfloat16
        out = (torch.zeros if accumulate else torch.empty)((A.rows, B.rows), dtype=dt, device=A.codes.device)
    a, b = A.c(), B.c()
    _check(lib().mxfp4_gemm_mbs(ctypes.byref(a), None if mbs_a is None else _ptr(mbs_a), ctypes.byref(b),
                                None if mbs_b is None else _ptr(mbs_b), _ptr(out), out.stride(0), out_dtype,
                                int(accumulate), _stream(stream)))
    return out


def gemm_group(problems, stream=None) -> list:
    """mxfp4_gemm_group: several C = A . B^T in one launch.  `problems` is a list of
    (A, B, out_dtype, accumulate, out) tuples (out may be None: allocated here).
    Returns the outputs in order."""
    outs, cs, descs = [], [], []
    for A, B, out_dtype, accumulate, out in problems:
        if out is None:
            dt = torch.float32 if out_dtype == OUT_F32 else torch.bfloat16
            out = (torch.zeros if accumulate else torch.empty)((A.rows, B.rows), dtype=dt, device=A.codes.device)
        a, b = A.c(), B.c()
        cs += [a, b]
        outs.append(out)
        descs.append(GemmDescC(ctypes.addressof(a), ctypes.addressof(b), out.data_ptr(), out.stride(0), out_dtype,
                               int(accumulate)))
    arr = (GemmDescC * len(descs))(*descs)
    _check(lib().mxfp4_gemm_group(arr, len(descs), _stream(stream)))
    return outs


@dataclass
class Config:
    had: int = HAD_16
    mode: int = SCALE_FLOOR
    out_dtype: int = OUT_F32
    accumulate: int = 0

    def c(self) -> MxConfigC:
        return MxConfigC(self.had, self.mode, self.out_dtype, self.accumulate)


class Workspace:
    """Caller-owned scratch (torch memory), grown on demand, 256-byte aligned."""

    def __init__(self):
        self.buf = None

    def get(self, nbytes: int, device) -> torch.Tensor | None:
        if nbytes == 0:
            return None
        if self.buf is None or self.buf.numel() < nbytes + 256 or self.buf.device != torch.device(device):
            self.buf = torch.empty(nbytes + 256, dtype=torch.uint8, device=device)
        off = (-self.buf.data_ptr()) % 256
        return self.buf[off:off + nbytes]


_default_ws = Workspace()


def workspace_bytes(op: int, M: int, N: int, K: int, cfg: Config) -> int:
    c = cfg.c()
    return lib().mxfp4_workspace_bytes(op, M, N, K, ctypes.byref(c))


def _out(shape, cfg: Config, device, out):
    if out is not None:
        return out
    dt = torch.float32 if cfg.out_dtype == OUT_F32 else torch.bfloat16
    return (torch.zeros if cfg.accumulate else torch.empty)(shape, dtype=dt, device=device)


def _ref(c):
    return ctypes.byref(c) if c is not None else None


def linear_fprop(x: torch.Tensor, w: torch.Tensor, cfg: Config, save_xT: bool = True, save_wT: bool = True,
                 y: torch.Tensor | None = None, xT: QTensor | None = None, wT: QTensor | None = None,
                 ws: Workspace | None = None, stream=None):
    """Y = X W^T with X [M,K], W [N,K] bf16; returns (Y, X^T quantised along M, W^T quantised along N)."""
    M, K = x.shape
    N = w.shape[0]
    y = _out((M, N), cfg, x.device, y)
    if save_xT and xT is None:
        xT = empty_qtensor(K, M, LAYOUT_COLT, SF_MMA, x.device)
    if save_wT and wT is None:
        wT = empty_qtensor(K, N, LAYOUT_COLT, SF_MMA, x.device)
    c = cfg.c()
    nb = workspace_bytes(OP_FPROP, M, N, K, cfg)
    buf = (ws or _default_ws).get(nb, x.device)
    cx = xT.c() if save_xT else None
    cw = wT.c() if save_wT else None
    _check(lib().mxfp4_linear_fprop(_ptr(x), _ptr(w), M, N, K, ctypes.byref(c), _ptr(y), _ref(cx), _ref(cw),
                                    _ptr(buf) if buf is not None else None, nb, _stream(stream)))
    for q, cq in ((xT, cx), (wT, cw)):
        if cq is not None:
            q.had, q.mode = cfg.had, cfg.mode
    return y, (xT if save_xT else None), (wT if save_wT else None)


def linear_dgrad(dy: torch.Tensor, wT: QTensor, cfg: Config, save_dyT: bool = True,
                 dx: torch.Tensor | None = None, dyT: QTensor | None = None, ws: Workspace | None = None,
                 stream=None):
    """dX = dY W with dY [M,N] bf16 and W^T [K,N] quantised along N; returns (dX, dY^T quantised along M)."""
    M, N = dy.shape
    K = wT.rows
    dx = _out((M, K), cfg, dy.device, dx)
    if save_dyT and dyT is None:
        dyT = empty_qtensor(N, M, LAYOUT_COLT, SF_MMA, dy.device)
    c = cfg.c()
    nb = workspace_bytes(OP_DGRAD, M, N, K, cfg)
    buf = (ws or _default_ws).get(nb, dy.device)
    cw = wT.c()
    cd = dyT.c() if save_dyT else None
    _check(lib().mxfp4_linear_dgrad(_ptr(dy), ctypes.byref(cw), M, N, K, ctypes.byref(c), _ptr(dx), _ref(cd),
                                    _ptr(buf) if buf is not None else None, nb, _stream(stream)))
    if cd is not None:
        dyT.had, dyT.mode = cfg.had, cfg.mode
    return dx, (dyT if save_dyT else None)


def linear_wgrad(dyT: QTensor, xT: QTensor, cfg: Config, dw: torch.Tensor | None = None, stream=None):
    """dW = dY^T X from dY^T [N,M] and X^T [K,M] (both quantised along M)."""
    dw = _out((dyT.rows, xT.rows), cfg, dyT.codes.device, dw)
    c, a, b = cfg.c(), dyT.c(), xT.c()
    _check(lib().mxfp4_linear_wgrad(ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), _ptr(dw), None, 0,
                                    _stream(stream)))
    return dw


def linear_backward(dy: torch.Tensor, wT: QTensor, xT: QTensor, cfg: Config, dx: torch.Tensor | None = None,
                    dw: torch.Tensor | None = None, ws: Workspace | None = None, stream=None):
    """dX = dY W (cfg.out_dtype) and dW = dY^T X (fp32; added to dw when cfg.accumulate)
    from dY [M,N] bf16 and the saved W^T [K,N], X^T [K,M]: one dY quantisation and one
    grouped GEMM launch.  Returns (dX, dW)."""
    M, N = dy.shape
    K = wT.rows
    if dx is None:
        dx = torch.empty((M, K), dtype=torch.float32 if cfg.out_dtype == OUT_F32 else torch.bfloat16,
                         device=dy.device)
    if dw is None:
        dw = (torch.zeros if cfg.accumulate else torch.empty)((N, K), dtype=torch.float32, device=dy.device)
    c, cw, cx = cfg.c(), wT.c(), xT.c()
    nb = workspace_bytes(OP_BACKWARD, M, N, K, cfg)
    buf = (ws or _default_ws).get(nb, dy.device)
    _check(lib().mxfp4_linear_backward(_ptr(dy), ctypes.byref(cw), ctypes.byref(cx), M, N, K, ctypes.byref(c),
                                       _ptr(dx), _ptr(dw), _ptr(buf), nb, _stream(stream)))
    return dx, dw


DECOMP_KEYS = ("e2", "scale2", "dz2", "grid2", "scale_grid", "n_deadzone", "n")


def error_decomposition(x: torch.Tensor, had: int = HAD_16, mode: int = SCALE_CEIL, stream=None) -> dict:
    """Tensor-wide sums of the MXFP4 error components of a row-quantised bf16 matrix
    (mxfp4_error_decomposition); returns a dict keyed by DECOMP_KEYS."""
    if x.dtype != torch.bfloat16 or not x.is_cuda or x.dim() != 2 or (x.numel() and x.stride(1) != 1):
        raise ValueError("x must be a CUDA bf16 matrix with unit column stride")
    out = torch.empty(7, dtype=torch.float64, device=x.device)
    _check(lib().mxfp4_error_decomposition(_ptr(x), x.shape[0], x.shape[1], x.stride(0), had, mode, _ptr(out),
                                           _stream(stream)))
    return dict(zip(DECOMP_KEYS, out.cpu().tolist()))


def mma_peak_tflops(kind: int = 0, iters: int = 1 << 16) -> float:
    """Dense tensor-core rate from mxfp4_mma_peak_probe (0: kind::mxf4, 1: kind::mxf4nvf4
    2X, 2: bf16 kind::f16, 3: kind::mxf4nvf4 4X with UE4M3 scales, 4: kind::mxf4 on CTA pairs),
    in TFLOP/s."""
    out = ctypes.c_double(0.0)
    _check(lib().mxfp4_mma_peak_probe(kind, iters, ctypes.byref(out)))
    return out.value


def device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status (0 = ok)."""
    return lib().mxfp4_device_status(_stream(stream))


def set_wait_limit_ns(ns: int) -> None:
    lib().mxfp4_set_wait_limit_ns(int(ns))


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """bf16 bit patterns (numpy uint16) -> bf16 torch tensor on `device`."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)
