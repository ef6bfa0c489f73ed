"""CPU oracle for the W8A8 block-FP8 matmul -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The product
path (``block_scaled_fp8_w8a8_gb300``) never imports it; the two share no code
besides the seeded input generator ``block_scaled_fp8_w8a8_gb300.synth``, which
holds none of the matmul's arithmetic.

The operator ("feat: optimize w8a8 block fp8 matmul for Hopper", FlagGems-vllm
PR #693, Description: E4M3 activations scaled per token and K block, E4M3
weights scaled per [block_n, block_k] block; Numerical safety: the sums are
kept in fp32 and the result is cast to bf16, fp16 or fp32):

    C[m,n] = cast_out( sum_g a_s[m,g] * b_s[n // block_n, g] * sum_{k in g} A[m,k] * B[n,k] )

Two independent implementations live here and are checked against each other
and against closed forms in ``tests/test_oracle.py``:

* ``reference_numpy``: the definition with numpy, one float64 matmul per K
  group (each group sum is exact, see ``w8a8_oracle.c``), scales applied and
  groups summed in ascending order.
* ``reference_c`` / ``reference_c_sampled``: plain C loops (``w8a8_oracle.c``),
  multithreaded over rows, for full-size shapes and sampled elements.

Both return double; ``cast_out`` rounds once to the output dtype (round to
nearest, ties to even), with the rounding written out in ``round_to_format``.

Every function here is pinned by a ``-m "not gpu"`` test; nothing is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "w8a8_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libw8a8_oracle.so")
_lib = None


def e4m3fn_value(code: int) -> float:
    """Decode one OCP E4M3FN byte: sign, 4-bit exponent (bias 7), 3-bit mantissa;
    exponent 0 is subnormal (f * 2^-9); S.1111.111 is NaN; no infinities."""
    s, e, f = (code >> 7) & 1, (code >> 3) & 0xF, code & 0x7
    if e == 0xF and f == 0x7:
        return math.nan
    mag = f * 2.0 ** -9 if e == 0 else (1.0 + f / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


def e4m3fn_table() -> np.ndarray:
    """All 256 E4M3FN codes decoded exactly to float64."""
    return np.array([e4m3fn_value(c) for c in range(256)], dtype=np.float64)


_TABLE = e4m3fn_table()


def _np(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x)


def reference_numpy(A, a_s, B, b_s, block_n: int = 128, block_k: int = 128) -> np.ndarray:
    """The definition in float64, one exact matmul per K group, groups in order."""
    A, B = _np(A).astype(np.uint8), _np(B).astype(np.uint8)
    a_s, b_s = _np(a_s).astype(np.float32), _np(b_s).astype(np.float32)
    M, K = A.shape
    N, Kb = B.shape
    assert K == Kb
    G = -(-K // block_k)
    assert a_s.shape == (M, G) and b_s.shape == (-(-N // block_n), G)
    Ad, Bd = _TABLE[A], _TABLE[B]
    nb = np.arange(N) // block_n
    C = np.zeros((M, N), dtype=np.float64)
    for g in range(G):
        k0, k1 = g * block_k, min((g + 1) * block_k, K)
        p = Ad[:, k0:k1] @ Bd[:, k0:k1].T                      # exact group sums
        s = a_s[:, g].astype(np.float64)[:, None] * b_s[nb, g].astype(np.float64)[None, :]
        C = C + s * p
    return C


def build(force: bool = False) -> str:
    """Compile the C oracle into oracle/_build/ (gcc, no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_LIB), exist_ok=True)
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_w8a8_block_fp8.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, ctypes.c_int]
        lib.oracle_w8a8_block_fp8.restype = ctypes.c_int
        lib.oracle_w8a8_block_fp8_sampled.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64,
                                                      p, i64, ctypes.c_int]
        lib.oracle_w8a8_block_fp8_sampled.restype = ctypes.c_int
        lib.oracle_e4m3fn_table.argtypes = [p]
        lib.oracle_e4m3fn_table.restype = None
        _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def c_table() -> np.ndarray:
    out = np.zeros(256, dtype=np.float64)
    _load().oracle_e4m3fn_table(out.ctypes.data)
    return out


def _prep(A, a_s, B, b_s, block_n, block_k):
    A, B = _np(A).astype(np.uint8), _np(B).astype(np.uint8)
    a_s, b_s = _np(a_s).astype(np.float32), _np(b_s).astype(np.float32)
    M, K = A.shape
    N = B.shape[0]
    G = -(-K // block_k) if K else 0
    assert B.shape[1] == K and a_s.shape == (M, G) and b_s.shape == (-(-N // block_n), G)
    return A, a_s, B, b_s, M, N, K


def reference_c(A, a_s, B, b_s, block_n: int = 128, block_k: int = 128,
                threads: int | None = None) -> np.ndarray:
    """Full [M, N] float64 product with the C oracle."""
    A, a_s, B, b_s, M, N, K = _prep(A, a_s, B, b_s, block_n, block_k)
    C = np.zeros((M, N), dtype=np.float64)
    rc = _load().oracle_w8a8_block_fp8(A.ctypes.data, a_s.ctypes.data, B.ctypes.data,
                                       b_s.ctypes.data, C.ctypes.data, M, N, K, block_n,
                                       block_k, threads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return C


def reference_c_sampled(A, a_s, B, b_s, rows, cols, block_n: int = 128, block_k: int = 128,
                        threads: int | None = None) -> np.ndarray:
    """C[rows[i], cols[i]] in float64 for each i, with the C oracle."""
    A, a_s, B, b_s, M, N, K = _prep(A, a_s, B, b_s, block_n, block_k)
    pairs = np.ascontiguousarray(np.stack([np.asarray(rows, dtype=np.int64),
                                           np.asarray(cols, dtype=np.int64)], axis=1))
    out = np.zeros(pairs.shape[0], dtype=np.float64)
    rc = _load().oracle_w8a8_block_fp8_sampled(A.ctypes.data, a_s.ctypes.data, B.ctypes.data,
                                               b_s.ctypes.data, out.ctypes.data, M, N, K,
                                               block_n, block_k, pairs.ctypes.data,
                                               pairs.shape[0], threads or default_threads())
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out


# (significand bits incl. the hidden one, exponent of the smallest subnormal,
#  largest finite value) of each output format, IEEE 754 binary16 / binary32
#  and bfloat16 (binary32 with a 7-bit fraction).
_FORMATS = {
    "bf16": (8, -133, (2.0 - 2.0 ** -7) * 2.0 ** 127),
    "fp16": (11, -24, 65504.0),
    "fp32": (24, -149, (2.0 - 2.0 ** -23) * 2.0 ** 127),
}


def round_to_format(C: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values once, to nearest with ties to even, onto the grid of
    ``dtype`` ('bf16', 'fp16' or 'fp32'); overflow goes to +-inf, NaN stays NaN.
    The result is float64 holding values exactly representable in ``dtype``."""
    p, emin_sub, vmax = _FORMATS[dtype]
    x = np.asarray(C, dtype=np.float64)
    _, e = np.frexp(x)                       # |x| = m * 2^e with 0.5 <= m < 1
    q = np.maximum(e - p, emin_sub)          # exponent of one unit in the last place
    with np.errstate(invalid="ignore", over="ignore"):
        r = np.ldexp(np.rint(np.ldexp(x, -q)), q)   # np.rint: ties to even
        r = np.where(np.abs(r) > vmax, np.copysign(np.inf, x), r)
    return r


def cast_out(C: np.ndarray, dtype: str):
    """``cast_out`` of the definition: round-to-nearest-even into the output
    dtype; returns a torch CPU tensor of that dtype (the conversion from the
    already-rounded float64 values is exact)."""
    import torch
    r = torch.from_numpy(np.ascontiguousarray(round_to_format(C, dtype)))
    return r.to({"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[dtype])


if __name__ == "__main__":  # pragma: no cover - manual build helper
    print(build(force="--force" in sys.argv))


# --------------------------------------------------------------------------- quantiser
#
# The operator's activation input is FP8 E4M3 with one fp32 scale per token per
# 128-wide K group ("feat: optimize w8a8 block fp8 matmul for Hopper", FlagGems-vllm
# PR #693, Description); the workloads fix the scale as amax / 448.  Reading of the
# steps (the page gives only "scale = amax/448"): in fp32, scale = amax / 448, set
# to 1 where that quotient is 0 (an all-zero group, or a max below 448 times the
# smallest fp32 subnormal, whose quotient underflows), then each code is the E4M3FN
# value nearest to x / scale (true fp32 division), ties to the even code, after
# clamping to +-448.

_POS_VALUES = _TABLE[:127]          # codes 0x00..0x7E, increasing, 0 .. 448


def e4m3fn_encode(v: np.ndarray) -> np.ndarray:
    """Round float64 values (already within [-448, 448], no NaN) to the nearest
    E4M3FN code, ties to the code with an even mantissa; returns uint8 codes.
    Written from the format: search the 127 non-negative codes for the nearest
    value, then attach the sign."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    hi = np.clip(np.searchsorted(_POS_VALUES, a, side="left"), 0, 126)   # first value >= a
    lo = np.clip(hi - 1, 0, 126)
    d_hi = _POS_VALUES[hi] - a
    d_lo = a - _POS_VALUES[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    neg = np.signbit(v)
    return np.where(neg, code | 0x80, code).astype(np.uint8)


def quantize_per_token_group(X, group: int = 128):
    """Per-token-group quantisation of a [M, K] activation matrix.

    Returns (codes uint8 [M, K], scales float32 [M, ceil(K/group)]).  All
    arithmetic that decides a code is fp32, as on the GPU: amax is exact, the
    scale is the fp32 quotient amax / 448, each element is divided by the scale
    in fp32 and then rounded to E4M3FN."""
    X = _np(X)
    X = X.astype(np.float32)
    M, K = X.shape
    G = -(-K // group) if K else 0
    codes = np.zeros((M, K), dtype=np.uint8)
    scales = np.ones((M, G), dtype=np.float32)
    for g in range(G):
        k0, k1 = g * group, min((g + 1) * group, K)
        blk = X[:, k0:k1]
        amax = np.max(np.abs(blk), axis=1)
        s = (amax / np.float32(448.0)).astype(np.float32)
        s = np.where(s == 0, np.float32(1.0), s).astype(np.float32)
        q = (blk / s[:, None]).astype(np.float32)
        q = np.clip(q, np.float32(-448.0), np.float32(448.0))
        codes[:, k0:k1] = e4m3fn_encode(q.astype(np.float64))
        scales[:, g] = s
    return codes, scales


# --------------------------------------------------------------------------- grouped (MoE)
#
# The grouped form of the same matmul: E experts, each with its own weights B[e]
# [N, K] and block scales b_s[e] [ceil(N/128), ceil(K/128)]; every token row is
# multiplied by the weights of the expert it is routed to.  The MoE pages run
# this per-expert GEMM with the decode swap-AB mapping ("[SM90] Optimize FP8
# MegaMoE across L2 epilogue, 4WG launch heuristic and decode swap-AB",
# sgl-project/DeepGEMM PR #69, Summary).  Reading: two layouts, both with the
# definition above applied per expert and nothing else changed.
#  * masked: A [E, max_m, K], a_s [E, max_m, G]; expert e owns rows
#    0 .. masked_m[e]-1 of its slab; C [E, max_m, N]; rows at or past
#    masked_m[e] are unspecified (NaN here).
#  * contiguous: A [M, K], a_s [M, G]; m_indices[m] is row m's expert, -1 for a
#    padding row; C [M, N]; padding rows are unspecified (NaN here).
# Each expert's rows go through reference_c with that expert's B and b_s.

def reference_grouped_masked(A, a_s, B, b_s, masked_m, block_n: int = 128, block_k: int = 128):
    A, a_s, B, b_s = _np(A), _np(a_s), _np(B), _np(b_s)
    masked_m = np.asarray(_np(masked_m), dtype=np.int64)
    E, max_m, _ = A.shape
    N = B.shape[1]
    C = np.full((E, max_m, N), np.nan, dtype=np.float64)
    for e in range(E):
        m = int(masked_m[e])
        if not 0 <= m <= max_m:
            raise ValueError("masked_m out of range")
        if m:
            C[e, :m] = reference_c(A[e, :m], a_s[e, :m], B[e], b_s[e], block_n, block_k)
    return C


def reference_grouped_contiguous(A, a_s, B, b_s, m_indices, block_n: int = 128,
                                 block_k: int = 128):
    A, a_s, B, b_s = _np(A), _np(a_s), _np(B), _np(b_s)
    idx = np.asarray(_np(m_indices), dtype=np.int64)
    M = A.shape[0]
    E, N = B.shape[0], B.shape[1]
    C = np.full((M, N), np.nan, dtype=np.float64)
    for e in range(E):
        rows = np.flatnonzero(idx == e)
        if rows.size:
            C[rows] = reference_c(A[rows], a_s[rows], B[e], b_s[e], block_n, block_k)
    if np.any((idx < -1) | (idx >= E)):
        raise ValueError("m_indices out of range")
    return C
