"""CPU oracle for H16/H32 + MXFP4 linear-layer GEMMs (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It shares no code with the CUDA path: the arithmetic
lives in ``mxfp4_oracle.c`` (plain C, fp64/integer), and this module only marshals
numpy arrays through ctypes and composes the primitives the way the pages state
the three linear-layer GEMMs.

Sources (cited by page title and section):
  "Pretraining Large Language Models with MXFP4 on Native FP4 Hardware":
      A.1 (MXFP4 reconstruction), A.2 (tiled deterministic Hadamard),
      C.1-C.3 (Fprop / Dgrad / Wgrad cancellation), D (1x32, 32x1, 32x32 layouts).
  "Decomposing MXFP4 quantization error for LLM reinforcement learning":
      E2M1 grid and E8M0 scale ("pain point"), ideal-scale quantiser and the
      error decomposition ("core insight", property 1), QDQ equivalence
      ("experiments").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxfp4_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

HAD_NONE, HAD_16, HAD_32 = 1, 16, 32
SCALE_FLOOR, SCALE_CEIL = 0, 1


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (IEEE arithmetic, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            L.oracle_e2m1_code.argtypes = [ctypes.c_double]
            L.oracle_e2m1_code.restype = I
            L.oracle_e2m1_value.argtypes = [I]
            L.oracle_e2m1_value.restype = ctypes.c_double
            L.oracle_shared_exponent.argtypes = [ctypes.c_float, I]
            L.oracle_shared_exponent.restype = I
            L.oracle_scale_byte.argtypes = [ctypes.c_float, I]
            L.oracle_scale_byte.restype = I
            L.oracle_hadamard_pm1.argtypes = [I, P]
            L.oracle_rotate_f32.argtypes = [P, I64, I, P]
            L.oracle_rotate_f64.argtypes = [P, I64, I, P]
            L.oracle_quantize_vec.argtypes = [P, I64, I64, I, I, P, P]
            for name in ("oracle_quantize_row", "oracle_quantize_colT", "oracle_quantize_2d"):
                getattr(L, name).argtypes = [P, I64, I64, I64, I, I, P, P]
            L.oracle_dequant_row.argtypes = [P, P, I64, I64, P]
            L.oracle_gemm.argtypes = [P, P, P, P, I64, I64, I64, P, P]
            L.oracle_dot_pairs.argtypes = [P, P, P, P, I64, I64, P, P]
            L.oracle_error_decomposition.argtypes = [P, I64, I64, I64, I, I, P]
            L.oracle_quantize_f32_rows.argtypes = [P, I64, I64, I, P, P]
            L.oracle_quantize_of_row.argtypes = [P, I64, I64, I64, I, I, I, P, P, P, P]
            L.oracle_quantize_of_row.restype = I64
            L.oracle_mbs_byte.argtypes = [ctypes.c_float]
            L.oracle_mbs_byte.restype = I
            L.oracle_quantize_mbs_row.argtypes = [P, I64, I64, I64, I, I, P, P, P]
            L.oracle_dequant_mbs_row.argtypes = [P, P, P, I64, I64, P]
            L.oracle_gemm_mbs.argtypes = [P, P, P, P, P, P, I64, I64, I64, P, P]
            L.oracle_e2m1_code_sr.argtypes = [ctypes.c_float, ctypes.c_uint16]
            L.oracle_e2m1_code_sr.restype = I
            L.oracle_quantize_row_rand.argtypes = [P, I64, I64, I64, I, I, P, P, P, P]
            L.oracle_quantize_colT_rand.argtypes = [P, I64, I64, I64, I, I, P, P, P, P]
            L.oracle_rotation_divergence.argtypes = [P, I64, I64, I64, I, I, P]
            L.oracle_philox4x32_10.argtypes = [P, P, P]
            L.oracle_philox_signs.argtypes = [ctypes.c_uint64, I64, P]
            L.oracle_philox_sr.argtypes = [ctypes.c_uint64, I64, I64, ctypes.c_uint32, P]
            L.oracle_num_threads.restype = I
            L.oracle_set_num_threads.argtypes = [I]
            _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check_rotation(had: int, mode: int | None = None) -> None:
    """The oracle's rotation argument is the Hadamard block size (1: none, 16, 32), not
    the library's 0 / 16 / 32; its scale rule is 0 (OCP floor) or 1 (ceiling).  Anything
    else is refused here, before it reaches the C code."""
    if had not in (1, 16, 32):
        raise ValueError(f"oracle rotation block must be 1, 16 or 32 (got {had})")
    if mode is not None and mode not in (0, 1):
        raise ValueError(f"oracle scale rule must be 0 or 1 (got {mode})")


def _u16(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (numpy uint16)")
    return x


# --------------------------------------------------------------------------- scalars
def e2m1_code(u: float) -> int:
    return lib().oracle_e2m1_code(float(u))


def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(int(code))


def shared_exponent(amax: float, mode: int) -> int:
    return lib().oracle_shared_exponent(float(amax), int(mode))


def scale_byte(amax: float, mode: int) -> int:
    return lib().oracle_scale_byte(float(amax), int(mode))


def num_threads() -> int:
    return lib().oracle_num_threads()


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))


# --------------------------------------------------------------------------- rotation
def hadamard_pm1(n: int) -> np.ndarray:
    h = np.zeros((n, n), dtype=np.int8)
    lib().oracle_hadamard_pm1(n, _p(h))
    return h


def rotate_f32(x: np.ndarray, had: int) -> np.ndarray:
    """Canonical fp32 rotation of the last axis (blocks of ``had``)."""
    _check_rotation(had)
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    flat_in, flat_out = x.reshape(-1), out.reshape(-1)
    lib().oracle_rotate_f32(_p(flat_in), flat_in.size, had, _p(flat_out))
    return out


def rotate_f64(x: np.ndarray, had: int) -> np.ndarray:
    """Exact (fp64) rotation of the last axis by block-diagonal H_n / sqrt(n)."""
    _check_rotation(had)
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty_like(x)
    lib().oracle_rotate_f64(_p(x.reshape(-1)), x.size, had, _p(out.reshape(-1)))
    return out


# --------------------------------------------------------------------------- quantiser
def quantize(x_bf16: np.ndarray, had: int, mode: int, layout: str):
    """Quantise a [R, C] bf16 (uint16 bit patterns) matrix.

    layout 'row'  -> codes [R, C/2],  scales [R, C/32]   (rotation along C)
    layout 'colT' -> codes [C, R/2],  scales [C, R/32]   (rotation along R)
    layout '2d'   -> codes [R, C/2],  scales [R/32, C/32] (rotation along C)
    """
    _check_rotation(had, mode)
    x = _u16(x_bf16)
    R, C = x.shape
    L = lib()
    if layout == "row":
        assert C % 32 == 0
        codes = np.zeros((R, C // 2), np.uint8)
        scales = np.zeros((R, C // 32), np.uint8)
        L.oracle_quantize_row(_p(x), R, C, C, had, mode, _p(codes), _p(scales))
    elif layout == "colT":
        assert R % 32 == 0
        codes = np.zeros((C, R // 2), np.uint8)
        scales = np.zeros((C, R // 32), np.uint8)
        L.oracle_quantize_colT(_p(x), R, C, C, had, mode, _p(codes), _p(scales))
    elif layout == "2d":
        assert R % 32 == 0 and C % 32 == 0
        codes = np.zeros((R, C // 2), np.uint8)
        scales = np.zeros((R // 32, C // 32), np.uint8)
        L.oracle_quantize_2d(_p(x), R, C, C, had, mode, _p(codes), _p(scales))
    else:
        raise ValueError(layout)
    return codes, scales


def quantize_vec(x_bf16: np.ndarray, had: int, mode: int):
    """Quantise one contiguous vector (length % 32 == 0) along itself."""
    _check_rotation(had, mode)
    x = _u16(x_bf16).reshape(-1)
    n = x.size
    codes = np.zeros(n // 2, np.uint8)
    scales = np.zeros(n // 32, np.uint8)
    lib().oracle_quantize_vec(_p(x), 1, n, had, mode, _p(codes), _p(scales))
    return codes, scales


def unpack_codes(codes: np.ndarray) -> np.ndarray:
    """Packed nibbles [..., n/2] -> one code per element [..., n] (element 2i low)."""
    lo = codes & 0xF
    hi = codes >> 4
    return np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)


def dequant_row(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales)
    R, C = codes.shape[0], codes.shape[1] * 2
    out = np.empty((R, C), np.float64)
    lib().oracle_dequant_row(_p(codes), _p(scales), R, C, _p(out))
    return out


# --------------------------------------------------------------------------- GEMM
def gemm(ca, sa, cb, sb):
    """C = dq(A) dq(B)^T for row-layout operands A [M,K], B [N,K]; returns (C, S)
    with S[m][n] = sum_k |dq a_k| |dq b_k| (both fp64)."""
    ca, sa, cb, sb = (np.ascontiguousarray(a) for a in (ca, sa, cb, sb))
    M, K = ca.shape[0], ca.shape[1] * 2
    N = cb.shape[0]
    assert cb.shape[1] * 2 == K and sa.shape == (M, K // 32) and sb.shape == (N, K // 32)
    C = np.empty((M, N), np.float64)
    S = np.empty((M, N), np.float64)
    lib().oracle_gemm(_p(ca), _p(sa), _p(cb), _p(sb), M, N, K, _p(C), _p(S))
    return C, S


def dot_pairs(ca, sa, cb, sb):
    """Row-wise dots of P (row of A, row of B) pairs; returns (C[P], S[P])."""
    ca, sa, cb, sb = (np.ascontiguousarray(a) for a in (ca, sa, cb, sb))
    P, K = ca.shape[0], ca.shape[1] * 2
    C = np.empty(P, np.float64)
    S = np.empty(P, np.float64)
    lib().oracle_dot_pairs(_p(ca), _p(sa), _p(cb), _p(sb), P, K, _p(C), _p(S))
    return C, S


# --------------------------------------------------------------------------- linear layer
# The three GEMMs of a linear layer with the rotation along each contraction
# ("Pretraining ... Native FP4 Hardware", C.1-C.3).  X [M,K], W [N,K], dY [M,N].
def fprop(x, w, had, mode):
    """Y = X W^T: X and W each rotated and quantised along K (row layout)."""
    return gemm(*quantize(x, had, mode, "row"), *quantize(w, had, mode, "row"))


def dgrad(dy, w, had, mode):
    """dX = dY W: dY along N (row layout), W^T along N (column layout of W)."""
    return gemm(*quantize(dy, had, mode, "row"), *quantize(w, had, mode, "colT"))


def wgrad(dy, x, had, mode):
    """dW = dY^T X: dY^T and X^T along the tokens M (column layouts)."""
    return gemm(*quantize(dy, had, mode, "colT"), *quantize(x, had, mode, "colT"))


def fprop_sample(x, w, had, mode, rows, cols):
    """Y[m][n] for the listed (m, n) pairs, quantising only the rows involved."""
    qa = [quantize_vec(x[m], had, mode) for m in rows]
    qb = [quantize_vec(w[n], had, mode) for n in cols]
    return dot_pairs(np.stack([q[0] for q in qa]), np.stack([q[1] for q in qa]),
                     np.stack([q[0] for q in qb]), np.stack([q[1] for q in qb]))


def dgrad_sample(dy, w, had, mode, rows, cols):
    """dX[m][k] for the listed (m, k) pairs: row m of dY, column k of W."""
    qa = [quantize_vec(dy[m], had, mode) for m in rows]
    qb = [quantize_vec(np.ascontiguousarray(w[:, k]), had, mode) for k in cols]
    return dot_pairs(np.stack([q[0] for q in qa]), np.stack([q[1] for q in qa]),
                     np.stack([q[0] for q in qb]), np.stack([q[1] for q in qb]))


def wgrad_sample(dy, x, had, mode, rows, cols):
    """dW[n][k] for the listed (n, k) pairs: column n of dY, column k of X."""
    qa = [quantize_vec(np.ascontiguousarray(dy[:, n]), had, mode) for n in rows]
    qb = [quantize_vec(np.ascontiguousarray(x[:, k]), had, mode) for k in cols]
    return dot_pairs(np.stack([q[0] for q in qa]), np.stack([q[1] for q in qa]),
                     np.stack([q[0] for q in qb]), np.stack([q[1] for q in qb]))


# --------------------------------------------------------------------------- error decomposition
def error_decomposition(x_bf16, had, mode):
    """Sums over a row-quantised [R, C] tensor of the three error components of the
    MXFP4 error ("Decomposing MXFP4 quantization error ...", core insight):
    dict with e2, scale2, dz2, grid2, scale_grid, n_deadzone, n (fp64 sums)."""
    _check_rotation(had, mode)
    x = _u16(x_bf16)
    R, C = x.shape
    out = np.zeros(7, np.float64)
    lib().oracle_error_decomposition(_p(x), R, C, C, had, mode, _p(out))
    keys = ("e2", "scale2", "dz2", "grid2", "scale_grid", "n_deadzone", "n")
    return dict(zip(keys, out.tolist()))


def rotation_divergence(x_bf16: np.ndarray, had: int, mode: int) -> dict:
    """Diagnostic of the canonical fp32 rotation ("Pretraining Large Language Models with
    MXFP4 on Native FP4 Hardware", A.2, which defines the rotation exactly): among the
    32-blocks of the row layout of x [R, C], how many would get other codes or another
    E8M0 byte if the exact fp64 rotation were quantised instead.  Not a failure."""
    _check_rotation(had, mode)
    x = _u16(x_bf16)
    R, C = x.shape
    out = np.zeros(3, np.int64)
    lib().oracle_rotation_divergence(_p(x), R, C, C, had, mode, _p(out))
    return {"blocks_differ": int(out[0]), "bytes_differ": int(out[1]), "blocks": int(out[2])}


# --------------------------------------------------------------------------- quantiser fixes
# "Decomposing MXFP4 quantization error ...", the MBS and OF fixes (row layout).
def quantize_f32_rows(v: np.ndarray, mode: int):
    """Quantise fp32 values [R, C] in 32-blocks along C, without rotation."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    R, C = v.shape
    codes = np.zeros((R, C // 2), np.uint8)
    scales = np.zeros((R, C // 32), np.uint8)
    lib().oracle_quantize_f32_rows(_p(v), R, C, mode, _p(codes), _p(scales))
    return codes, scales


def quantize_of(x_bf16: np.ndarray, had: int, mode: int, alpha_log2: int = -1):
    """Outlier fallback: q1 = Q(x), q2 = Q(x - dq(q1)) with alpha = 2^alpha_log2 folded
    into q2's scale bytes, so x_OF = dq(q1) + dq(q2).  Returns (c1, s1, c2, s2,
    number of residuals that were not exact in fp32)."""
    _check_rotation(had, mode)
    x = _u16(x_bf16)
    R, C = x.shape
    c1 = np.zeros((R, C // 2), np.uint8)
    s1 = np.zeros((R, C // 32), np.uint8)
    c2 = np.zeros((R, C // 2), np.uint8)
    s2 = np.zeros((R, C // 32), np.uint8)
    bad = lib().oracle_quantize_of_row(_p(x), R, C, C, had, mode, int(alpha_log2), _p(c1), _p(s1), _p(c2), _p(s2))
    return c1, s1, c2, s2, int(bad)


def mbs_byte(amax: float) -> int:
    return lib().oracle_mbs_byte(float(amax))


def quantize_mbs(x_bf16: np.ndarray, had: int, mode: int):
    """Macro-block scaling: returns (codes [R, C/2], scales [R, C/32], mbs [R, C/128])."""
    _check_rotation(had, mode)
    x = _u16(x_bf16)
    R, C = x.shape
    assert C % 128 == 0
    codes = np.zeros((R, C // 2), np.uint8)
    scales = np.zeros((R, C // 32), np.uint8)
    mbs = np.zeros((R, C // 128), np.uint8)
    lib().oracle_quantize_mbs_row(_p(x), R, C, C, had, mode, _p(codes), _p(scales), _p(mbs))
    return codes, scales, mbs


def dequant_mbs(codes, scales, mbs) -> np.ndarray:
    codes, scales, mbs = (np.ascontiguousarray(a) for a in (codes, scales, mbs))
    R, C = codes.shape[0], codes.shape[1] * 2
    out = np.empty((R, C), np.float64)
    lib().oracle_dequant_mbs_row(_p(codes), _p(scales), _p(mbs), R, C, _p(out))
    return out


def gemm_mbs(ca, sa, mbs_a, cb, sb, mbs_b):
    """C = x_hat_A x_hat_B^T over MBS operands (mbs_a / mbs_b [rows, K/128] bytes, or
    None for a plain MXFP4 operand): each 128-element macro block's partial product
    scaled by its two postscale factors 1 / (1 + byte/256).  Returns (C, S), fp64."""
    ca, sa, cb, sb = (np.ascontiguousarray(a) for a in (ca, sa, cb, sb))
    M, K = ca.shape[0], ca.shape[1] * 2
    N = cb.shape[0]
    assert K % 128 == 0 and cb.shape[1] * 2 == K
    ma = None if mbs_a is None else np.ascontiguousarray(mbs_a, np.uint8)
    mb = None if mbs_b is None else np.ascontiguousarray(mbs_b, np.uint8)
    assert ma is None or ma.shape == (M, K // 128)
    assert mb is None or mb.shape == (N, K // 128)
    C = np.empty((M, N), np.float64)
    S = np.empty((M, N), np.float64)
    lib().oracle_gemm_mbs(_p(ca), _p(sa), None if ma is None else _p(ma), _p(cb), _p(sb),
                          None if mb is None else _p(mb), M, N, K, _p(C), _p(S))
    return C, S


# --------------------------------------------------------------------------- randomised baselines
# "Pretraining ... Native FP4 Hardware", A.2 (random sign flips before the Hadamard)
# and the ablation of table 1 (stochastic rounding): the random numbers are inputs.
def e2m1_code_sr(u: float, r: int) -> int:
    return lib().oracle_e2m1_code_sr(float(np.float32(u)), int(r))


def pack_signs(neg: np.ndarray) -> np.ndarray:
    """Boolean vector (True = negate) -> bitmask bytes, bit i of byte i // 8."""
    return np.packbits(np.asarray(neg, bool), bitorder="little")


def quantize_rand(x_bf16: np.ndarray, had: int, mode: int, layout: str, signs=None, sr=None):
    """Like quantize() for 'row' ([R, C], signs over C, sr [R, C] uint16) and 'colT'
    ([C, R] output, signs over R, sr [C, R] uint16); signs is a bitmask (pack_signs)."""
    _check_rotation(had, mode)
    x = _u16(x_bf16)
    R, C = x.shape
    sg = None if signs is None else np.ascontiguousarray(signs, np.uint8)
    rr = None if sr is None else np.ascontiguousarray(sr, np.uint16)
    ps = _p(sg) if sg is not None else None
    pr = _p(rr) if rr is not None else None
    if layout == "row":
        if rr is not None:
            assert rr.shape == (R, C)
        codes = np.zeros((R, C // 2), np.uint8)
        scales = np.zeros((R, C // 32), np.uint8)
        lib().oracle_quantize_row_rand(_p(x), R, C, C, had, mode, ps, pr, _p(codes), _p(scales))
    elif layout == "colT":
        if rr is not None:
            assert rr.shape == (C, R)
        codes = np.zeros((C, R // 2), np.uint8)
        scales = np.zeros((C, R // 32), np.uint8)
        lib().oracle_quantize_colT_rand(_p(x), R, C, C, had, mode, ps, pr, _p(codes), _p(scales))
    else:
        raise ValueError(layout)
    return codes, scales


# --------------------------------------------------------------------------- counter-based generator
# The randomised baselines with their random numbers drawn from Philox4x32-10 (Salmon et
# al., SC'11) instead of passed in: the sign vectors and the stochastic-rounding integers
# are generated with the counter layout of oracle_philox_signs / oracle_philox_sr, then
# the quantiser above runs on them unchanged.
def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, np.uint32)
    k = np.ascontiguousarray(key, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().oracle_philox4x32_10(_p(c), _p(k), _p(out))
    return out


def philox_signs(seed: int, n: int) -> np.ndarray:
    bits = np.zeros((n + 7) // 8, np.uint8)
    lib().oracle_philox_signs(int(seed), n, _p(bits))
    return bits


def philox_sr(seed: int, lines: int, length: int, copy: int) -> np.ndarray:
    out = np.zeros((lines, length), np.uint16)
    lib().oracle_philox_sr(int(seed), lines, length, int(copy), _p(out))
    return out


def quantize_philox(x_bf16: np.ndarray, had: int, mode: int, layout: str, col_sign_seed=None, row_sign_seed=None,
                    sr_seed=None):
    """quantize_rand with generated numbers: 'row' uses the column-sign vector (seed
    col_sign_seed, over C) and the SR integers of copy 0 ([R, C]); 'colT' the row-sign
    vector (row_sign_seed, over R) and copy 1 ([C, R]).  A seed of None turns that
    option off."""
    x = _u16(x_bf16)
    R, C = x.shape
    if layout == "row":
        signs = None if col_sign_seed is None else philox_signs(col_sign_seed, C)
        sr = None if sr_seed is None else philox_sr(sr_seed, R, C, 0)
    elif layout == "colT":
        signs = None if row_sign_seed is None else philox_signs(row_sign_seed, R)
        sr = None if sr_seed is None else philox_sr(sr_seed, C, R, 1)
    else:
        raise ValueError(layout)
    return quantize_rand(x, had, mode, layout, signs=signs, sr=sr)
