"""Seeded synthetic inputs for the GEMM C = A . B^T.

This module only draws numbers: it holds no part of the matrix product and no
conversion the product path performs.  Both the CUDA path's tests and the CPU
oracle's tests take their operands from here, so that the two sides see the
same bits.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used counter-style.  Stream ``(seed, s)``
starts from ``base = ((seed << 8) | s) * GAMMA`` and element ``i`` is the
SplitMix64 finaliser applied to ``base + (i + 1) * GAMMA`` (mod 2**64).
Operand A is stream 0 and operand B is stream 1 of a workload's seed.

Distributions (the workloads of the tiled-GEMM tutorial pages use uniform and
normal fp16/bf16 matrices; the recipe is fixed here):

* ``uniform``: ``u = (x >> 11) * 2**-53`` in [0, 1), value ``lo + (hi - lo) * u``.
* ``normal``: Box-Muller on two consecutive draws,
  ``sqrt(-2 ln(1 - u1)) * cos(2 pi u2)``, times ``scale``.
* ``int``: ``(x mod (hi - lo + 1)) + lo``, small integers exactly representable
  in fp16 and bf16.

Values are produced in float64 and rounded once to the operand dtype
(round-to-nearest-even, numpy for fp16, torch for bf16).  The result is
returned as raw 16-bit patterns (``numpy.uint16``) together with a torch
tensor view of the same bits.
"""

from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

_CHUNK = 1 << 22


def splitmix64(seed: int, stream: int, n: int) -> np.ndarray:
    """``n`` SplitMix64 outputs of stream ``(seed, stream)`` as uint64."""
    if n < 0:
        raise ValueError("n must be >= 0")
    base = np.uint64((((seed << 8) | (stream & 0xFF)) * int(GAMMA)) & 0xFFFFFFFFFFFFFFFF)
    out = np.empty(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        for lo in range(0, n, _CHUNK):
            hi = min(n, lo + _CHUNK)
            z = np.arange(lo + 1, hi + 1, dtype=np.uint64) * GAMMA + base
            z = (z ^ (z >> np.uint64(30))) * _M1
            z = (z ^ (z >> np.uint64(27))) * _M2
            out[lo:hi] = z ^ (z >> np.uint64(31))
    return out


def _unit(x: np.ndarray) -> np.ndarray:
    return (x >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def draw(seed: int, stream: int, n: int, dist: str, **kw) -> np.ndarray:
    """``n`` float64 values of distribution ``dist`` from stream ``(seed, stream)``."""
    if dist == "uniform":
        lo, hi = kw.get("lo", -1.0), kw.get("hi", 1.0)
        return lo + (hi - lo) * _unit(splitmix64(seed, stream, n))
    if dist == "normal":
        scale = kw.get("scale", 1.0)
        x = splitmix64(seed, stream, 2 * n)
        u1 = _unit(x[0::2])
        u2 = _unit(x[1::2])
        return scale * np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * np.pi * u2)
    if dist == "int":
        lo, hi = int(kw.get("lo", -4)), int(kw.get("hi", 4))
        span = np.uint64(hi - lo + 1)
        return (splitmix64(seed, stream, n) % span).astype(np.int64).astype(np.float64) + lo
    raise ValueError(f"unknown distribution {dist!r}")


def to_bits(values: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values once to ``dtype`` ('f16' or 'bf16'); return uint16 bits."""
    if dtype == "f16":
        return values.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        import torch

        t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float64)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16)
    raise ValueError(f"unknown dtype {dtype!r}")


def matrix_bits(seed: int, stream: int, rows: int, cols: int, dtype: str, dist: str, **kw) -> np.ndarray:
    """A ``rows x cols`` row-major operand as uint16 bit patterns."""
    return to_bits(draw(seed, stream, rows * cols, dist, **kw), dtype).reshape(rows, cols)


def bits_to_torch(bits: np.ndarray, dtype: str):
    """A torch CPU tensor of ``dtype`` sharing the given uint16 bit patterns."""
    import torch

    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(tdt)


def operands(seed: int, M: int, N: int, K: int, dtype: str, dist: str, **kw):
    """Operands ``A[M,K]`` (stream 0) and ``B[N,K]`` (stream 1) as uint16 bits."""
    a = matrix_bits(seed, 0, M, K, dtype, dist, **kw)
    b = matrix_bits(seed, 1, N, K, dtype, dist, **kw)
    return a, b


# The workloads of the tutorial pages, one per line: shape, operand dtype,
# output dtype, distribution and seed.  Tile and depth are the pages' or the
# tuned defaults.
WORKLOADS = {
    "gemm_128_f16_uniform": dict(M=128, N=128, K=128, dtype="f16", out="f32",
                                 dist="uniform", seed=1, tile=(128, 128, 32), stages=3),
    "gemm_4096_f16_normal": dict(M=4096, N=4096, K=4096, dtype="f16", out="f16",
                                 dist="normal", seed=2, tile=None, stages=None),
    "gemm_8192_bf16_normal": dict(M=8192, N=8192, K=8192, dtype="bf16", out="bf16",
                                  dist="normal", kw=dict(scale=0.5), seed=3, tile=None, stages=None),
    "gemm_512x512x32768_f16_uniform": dict(M=512, N=512, K=32768, dtype="f16", out="f32",
                                           dist="uniform", seed=4, tile=None, stages=None),
    "gemm_512x512x32768_f16_int": dict(M=512, N=512, K=32768, dtype="f16", out="f32",
                                       dist="int", kw=dict(lo=-4, hi=4), seed=40, tile=None, stages=None),
    "gemm_4000x3000x5000_f16_uniform": dict(M=4000, N=3000, K=5000, dtype="f16", out="f32",
                                            dist="uniform", seed=5, tile=None, stages=None),
}


def workload_operands(name: str):
    """Operands of a named workload, as uint16 bits."""
    w = WORKLOADS[name]
    return operands(w["seed"], w["M"], w["N"], w["K"], w["dtype"], w["dist"], **w.get("kw", {}))
