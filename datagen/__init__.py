"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

This module only draws numbers; it holds none of the arithmetic of the GEMM,
the convolution or the copy. Both sides receive the same bf16 bit arrays
(numpy ``uint16``) and decode them on their own.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), used in its counter form. Draw ``i``
(0-based) of stream ``seed`` is the SplitMix64 finaliser applied to
``seed + (i + 1) * 0x9E3779B97F4A7C15`` (mod 2**64), so any slice of a stream
can be produced independently and in parallel.

Distributions (every element consumes draws in row-major order of the array
as stored, operands drawn one after another from one stream):

* ``uniform``: ``u = (r >> 40) * 2**-24``, ``v = 2u - 1`` (exact in fp32),
  rounded to bf16 with round-to-nearest-even. One draw per element.
* ``normal``: Box-Muller on two draws (fp64), times ``scale``, to fp32, then
  bf16 RNE. Two draws per element.
* ``bits``: the low 16 bits of one draw (every pattern, NaNs included).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Pad elements of a strided buffer (ld > logical width) hold a bf16 NaN, so a
# kernel that reads padding produces NaNs that no tolerance check accepts.
BF16_POISON = np.uint16(0x7FC1)

_CHUNK = 1 << 22


def _splitmix_block(seed: int, start: int, count: int) -> np.ndarray:
    idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of stream ``seed`` as uint64."""
    if count <= _CHUNK:
        return _splitmix_block(seed, start, count)
    out = np.empty(count, dtype=np.uint64)

    def work(off: int) -> None:
        n = min(_CHUNK, count - off)
        out[off:off + n] = _splitmix_block(seed, start + off, n)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, range(0, count, _CHUNK)))
    return out


def f32_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


class Stream:
    """Sequential consumer of one SplitMix64 stream."""

    def __init__(self, seed: int):
        self.seed = int(seed)
        self.pos = 0

    def _take(self, n: int) -> np.ndarray:
        r = splitmix64(self.seed, self.pos, n)
        self.pos += n
        return r

    def uniform_bf16(self, shape) -> np.ndarray:
        n = int(np.prod(shape))
        r = self._take(n)
        u = (r >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)
        v = np.float32(2.0) * u - np.float32(1.0)
        return f32_to_bf16_rne(v).reshape(shape)

    def normal_bf16(self, shape, scale: float = 0.02) -> np.ndarray:
        n = int(np.prod(shape))
        r = self._take(2 * n).reshape(n, 2)
        u1 = ((r[:, 0] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (r[:, 1] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        return f32_to_bf16_rne((z * scale).astype(np.float32)).reshape(shape)

    def bits16(self, shape) -> np.ndarray:
        n = int(np.prod(shape))
        r = self._take(n)
        return (r & np.uint64(0xFFFF)).astype(np.uint16).reshape(shape)


def pad_rows(a: np.ndarray, ld: int, fill=BF16_POISON) -> np.ndarray:
    """Embed a rows x cols uint16 matrix into a rows x ld buffer (pad = fill)."""
    rows, cols = a.shape
    if ld == cols:
        return np.ascontiguousarray(a)
    out = np.full((rows, ld), fill, dtype=np.uint16)
    out[:, :cols] = a
    return out


# ---------------------------------------------------------------------------
# Workloads. Each returns plain uint16 arrays plus sizes; nothing is computed.
# ---------------------------------------------------------------------------

def gemm_operands(M: int, N: int, K: int, seed: int, dist: str = "uniform",
                  lda: int | None = None, ldb: int | None = None,
                  stream: Stream | None = None):
    """A (M x K row-major, pitch lda) then B (stored N x K, i.e. K x N
    column-major, pitch ldb), drawn in that order from one stream."""
    lda = K if lda is None else lda
    ldb = K if ldb is None else ldb
    s = Stream(seed) if stream is None else stream
    draw = s.uniform_bf16 if dist == "uniform" else s.normal_bf16
    a = draw((M, K))
    b = draw((N, K))
    return pad_rows(a, lda), pad_rows(b, ldb)


def conv_operands(N: int, H: int, W: int, C: int, K: int, R: int, S: int,
                  seed: int, dist: str = "uniform"):
    """x (NHWC) then w (KRSC), drawn in that order from one stream."""
    s = Stream(seed)
    draw = s.uniform_bf16 if dist == "uniform" else s.normal_bf16
    x = draw((N, H, W, C))
    w = draw((K, R, S, C))
    return x, w


def copy_source(rows: int, cols: int, seed: int, ld: int | None = None) -> np.ndarray:
    """rows x cols random 16-bit patterns (pitch ld, pad = 0)."""
    ld = cols if ld is None else ld
    a = Stream(seed).bits16((rows, cols))
    return pad_rows(a, ld, fill=np.uint16(0))


# The workloads the benchmarks and the full-size parity tests run, with the
# seeds that make them reproducible.
SKINNY_SHAPES = ((128, 8192, 16384), (4096, 4096, 512), (1000, 1000, 1000))


def skinny_operands():
    """The three skinny/deep-K GEMMs, drawn one after another from seed 3."""
    s = Stream(3)
    return [gemm_operands(M, N, K, 3, "uniform", stream=s) for (M, N, K) in SKINNY_SHAPES]
