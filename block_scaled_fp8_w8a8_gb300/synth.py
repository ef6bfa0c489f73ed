"""Seeded synthetic inputs for the W8A8 block-FP8 matmul.

This module is shared by the CPU oracle (under ``oracle/``) and by the CUDA
path's tests and benchmark.  It holds none of the matmul's arithmetic: it only
draws Gaussian data and block-quantises it to FP8 E4M3 (OCP "FN" variant,
max finite 448) with fp32 de-quantisation scales, which is how the operator's
inputs are described in "feat: optimize w8a8 block fp8 matmul for Hopper"
(FlagGems-vllm PR #693, Description: E4M3 activations scaled per token and K
block, E4M3 weights scaled per [block_n, block_k] block).

Recipe (the plainest reading of the workload descriptions; every choice is
stated so that the two sides of a parity test see identical bytes):

* ``torch.Generator('cpu').manual_seed(seed)``; draw ``A`` ~ N(0,1) of shape
  [M, K], then ``B`` ~ N(0,1) of shape [N, K], both fp32.
* optional outliers: for each element independently, with probability
  ``outlier_p`` (drawn after A and B from the same generator, A's mask first),
  multiply it by ``outlier_scale``.  Applied before quantisation.
* activations: one scale per (row, 128-wide K group); weights: one scale per
  128x128 block.  ``scale = amax / 448`` in fp32 over the group or block
  (``scale = 1`` where the block is all zero); codes are
  ``e4m3fn_RNE(clamp(x / scale, -448, 448))`` with true division.
* scales are stored row-major: ``a_s[M, ceil(K/block_k)]`` and
  ``b_s[ceil(N/block_n), ceil(K/block_k)]``.

FP8 codes are returned as ``torch.uint8`` tensors holding the raw E4M3 bytes.
"""
from __future__ import annotations

import dataclasses
import math

import torch

E4M3_MAX = 448.0


@dataclasses.dataclass
class W8A8Inputs:
    A: torch.Tensor      # uint8 [M, K]   E4M3FN codes, row-major
    a_s: torch.Tensor    # float32 [M, ceil(K/block_k)]
    B: torch.Tensor      # uint8 [N, K]   E4M3FN codes, row-major
    b_s: torch.Tensor    # float32 [ceil(N/block_n), ceil(K/block_k)]
    block_n: int = 128
    block_k: int = 128

    @property
    def shape(self):
        return self.A.shape[0], self.B.shape[0], self.A.shape[1]


def _cdiv(a: int, b: int) -> int:
    return (a + b - 1) // b


def _to_e4m3_codes(x: torch.Tensor) -> torch.Tensor:
    """fp32 -> E4M3FN (round to nearest even, saturating input) -> raw bytes."""
    x = x.clamp(-E4M3_MAX, E4M3_MAX)
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def quantize_blocks(x: torch.Tensor, block_rows: int, block_cols: int):
    """Block-quantise a 2-D fp32 tensor with one scale per [block_rows, block_cols].

    Returns (codes uint8 [R, C], scales fp32 [ceil(R/block_rows), ceil(C/block_cols)]).
    Ragged edge blocks are quantised over the elements they hold.
    """
    assert x.dim() == 2 and x.dtype == torch.float32
    R, C = x.shape
    nr, nc = _cdiv(R, block_rows), _cdiv(C, block_cols)
    pr, pc = nr * block_rows - R, nc * block_cols - C
    xp = torch.nn.functional.pad(x, (0, pc, 0, pr)) if (pr or pc) else x
    blocks = xp.reshape(nr, block_rows, nc, block_cols)
    amax = blocks.abs().amax(dim=(1, 3))                        # [nr, nc]
    scale = (amax / E4M3_MAX).to(torch.float32)
    scale = torch.where(amax == 0, torch.ones_like(scale), scale)
    q = blocks / scale[:, None, :, None]
    codes = _to_e4m3_codes(q).reshape(nr * block_rows, nc * block_cols)[:R, :C]
    return codes.contiguous(), scale.contiguous()


def make_inputs(M: int, N: int, K: int, *, seed: int = 0, block_n: int = 128,
                block_k: int = 128, outlier_p: float = 0.0,
                outlier_scale: float = 20.0) -> W8A8Inputs:
    """Seeded N(0,1) inputs block-quantised as described in the module docstring."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    A = torch.randn(M, K, generator=g, dtype=torch.float32)
    B = torch.randn(N, K, generator=g, dtype=torch.float32)
    if outlier_p > 0.0:
        ma = torch.rand(M, K, generator=g) < outlier_p
        mb = torch.rand(N, K, generator=g) < outlier_p
        A = torch.where(ma, A * outlier_scale, A)
        B = torch.where(mb, B * outlier_scale, B)
    Aq, a_s = quantize_blocks(A, 1, block_k)        # per token, per K group
    Bq, b_s = quantize_blocks(B, block_n, block_k)  # per [block_n, block_k] block
    return W8A8Inputs(Aq, a_s, Bq, b_s, block_n, block_k)


def activations(M: int, K: int, *, seed: int = 0, dtype: torch.dtype = torch.float32,
                outlier_p: float = 0.0, outlier_scale: float = 20.0) -> torch.Tensor:
    """Seeded unquantised activations [M, K]: N(0,1) fp32 draws (a fraction
    ``outlier_p`` of them times ``outlier_scale``), rounded once to ``dtype``."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    X = torch.randn(M, K, generator=g, dtype=torch.float32)
    if outlier_p > 0.0:
        X = torch.where(torch.rand(M, K, generator=g) < outlier_p, X * outlier_scale, X)
    return X.to(dtype)


def make_grouped_masked(E: int, max_m: int, N: int, K: int, *, seed: int = 0, counts=None,
                        outlier_p: float = 0.0):
    """Masked-layout MoE inputs: per expert, N(0,1) activations [max_m, K] and
    weights [N, K] block-quantised as in make_inputs, and a token count (drawn
    uniformly from 0..max_m unless ``counts`` is given).  Returns (A [E,max_m,K],
    a_s [E,max_m,G], B [E,N,K], b_s [E,NB,G], masked_m int32 [E])."""
    parts = [make_inputs(max_m, N, K, seed=seed * 1000 + e, outlier_p=outlier_p) for e in range(E)]
    if counts is None:
        g = torch.Generator(device="cpu").manual_seed(seed)
        counts = torch.randint(0, max_m + 1, (E,), generator=g)
    masked_m = torch.as_tensor(counts, dtype=torch.int32)
    return (torch.stack([x.A for x in parts]), torch.stack([x.a_s for x in parts]),
            torch.stack([x.B for x in parts]), torch.stack([x.b_s for x in parts]), masked_m)


def make_grouped_contiguous(counts, N: int, K: int, *, seed: int = 0, align: int = 128):
    """Contiguous-layout MoE inputs: expert e's ``counts[e]`` token rows form one
    segment padded with -1 rows to a multiple of ``align``; padding rows hold
    zero codes and unit scales.  Returns (A [M,K], a_s [M,G], B [E,N,K],
    b_s [E,NB,G], m_indices int32 [M])."""
    E = len(counts)
    rows, idx = [], []
    for e, c in enumerate(counts):
        c = int(c)
        padded = _cdiv(c, align) * align
        x = make_inputs(max(c, 1), 8, K, seed=seed * 1000 + e)
        if c:
            rows.append((x.A[:c], x.a_s[:c]))
        if padded > c:
            rows.append((torch.zeros(padded - c, K, dtype=torch.uint8),
                         torch.ones(padded - c, _cdiv(K, 128), dtype=torch.float32)))
        idx += [e] * c + [-1] * (padded - c)
    A = torch.cat([r[0] for r in rows]) if rows else torch.zeros(0, K, dtype=torch.uint8)
    a_s = torch.cat([r[1] for r in rows]) if rows else torch.zeros(0, _cdiv(K, 128))
    w = [make_inputs(1, N, K, seed=seed * 1000 + 500 + e) for e in range(E)]
    return (A.contiguous(), a_s.contiguous(), torch.stack([x.B for x in w]),
            torch.stack([x.b_s for x in w]), torch.tensor(idx, dtype=torch.int32))


def random_codes(rows: int, cols: int, *, seed: int, allow_nan: bool = False) -> torch.Tensor:
    """Uniformly random E4M3FN bytes (all codes, including subnormals and -0).

    NaN codes (0x7F, 0xFF) are replaced by 0x00 unless ``allow_nan``.
    """
    g = torch.Generator(device="cpu").manual_seed(seed)
    c = torch.randint(0, 256, (rows, cols), generator=g, dtype=torch.int32).to(torch.uint8)
    if not allow_nan:
        c = torch.where((c & 0x7F) == 0x7F, torch.zeros_like(c), c)
    return c


def random_scales(rows: int, cols: int, *, seed: int, lo: float = 2.0 ** -12,
                  hi: float = 2.0 ** -4) -> torch.Tensor:
    """Log-uniform positive fp32 scales in [lo, hi), the range amax/448 takes for
    N(0,1) data with outliers."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    u = torch.rand(rows, cols, generator=g, dtype=torch.float64)
    return torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))).to(torch.float32)


# The workloads of the operator's shape sweep, by name.  Shapes follow the
# DeepSeek-V4-Flash trace grid (N in {512,1536,4096,8192}, K in {256,1024,4096},
# M in [1,16384]) of the PR #693 Performance section.
WORKLOADS = {
    "pr1_64x512x256": dict(shapes=[(64, 512, 256)], outlier_p=0.0),
    "decode_n4096_k256": dict(shapes=[(m, 4096, 256) for m in (1, 16, 100, 184, 214)],
                              outlier_p=0.0),
    "skinny_n512_k4096": dict(shapes=[(m, 512, 4096) for m in (16, 64, 158)],
                              outlier_p=1e-3),
    "widen_n8192_k1024": dict(shapes=[(m, 8192, 1024) for m in (1, 32, 128, 264)],
                              outlier_p=0.0),
    "prefill_k4096": dict(shapes=[(4096, 4096, 4096), (16384, 4096, 4096),
                                  (4096, 1536, 4096), (16384, 1536, 4096)],
                          outlier_p=0.0),
}


def algorithmic_bytes(M: int, N: int, K: int, out_bytes: int = 2, block: int = 128) -> int:
    """A + a_s + B + b_s + C, each moved once."""
    G = _cdiv(K, block)
    return M * K + 4 * M * G + N * K + 4 * _cdiv(N, block) * G + out_bytes * M * N


def algorithmic_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K
