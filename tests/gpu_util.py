"""Helpers shared by the GPU parity tests (no method arithmetic here)."""
import numpy as np
import pytest

ORACLE_HAD = {0: 1, 16: 16, 32: 32}  # ABI hadamard value -> oracle block size


def gpu_ready():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch


def assert_within(got: np.ndarray, want: np.ndarray, S: np.ndarray, bf16: bool = False, what: str = ""):
    """|got - want| <= 1e-5 * S (+ 2^-8 |want| for bf16 output), element by element."""
    tol = 1e-5 * S + (2.0 ** -8 * np.abs(want) if bf16 else 0.0)
    err = np.abs(got.astype(np.float64) - want)
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[:5]
        detail = ", ".join(f"{tuple(j)}: got {got[tuple(j)]:.6e} want {want[tuple(j)]:.6e} S {S[tuple(j)]:.3e}"
                           for j in i)
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outside tolerance; {detail}")


def sample_pairs(M, N, n_random, seed, edge=8):
    """Random (row, col) pairs plus the first/last `edge` rows and cols (tile edges)."""
    g = np.random.default_rng(seed)
    rows = list(g.integers(0, M, n_random))
    cols = list(g.integers(0, N, n_random))
    for r in list(range(min(edge, M))) + list(range(max(0, M - edge), M)):
        rows.append(r)
        cols.append(int(g.integers(0, N)))
    for c in list(range(min(edge, N))) + list(range(max(0, N - edge), N)):
        rows.append(int(g.integers(0, M)))
        cols.append(c)
    return np.array(rows), np.array(cols)
