"""Seeded synthetic SGEMM workloads: shapes, scalars and input matrices.

This module only *draws* inputs.  It holds none of the GEMM arithmetic, so both
the CUDA library's tests/bench and the CPU oracle can take their operands from
here without sharing any of the method's code.

Generator (counter-based, portable, defined here):

* ``key = mix64(seed XOR stream * 0xD1B54A32D192ED03)`` per (seed, stream);
  streams are 1 = A, 2 = B, 3 = C.
* ``x_i = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)`` for element ``i`` of the
  stream, where ``mix64`` is the SplitMix64 finaliser (Steele, Lea, Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014).
* uniform[-1, 1): ``j = x_i >> 40`` (24 bits), value ``(j - 2**23) / 2**23``;
  every value is an exact float32 and the interval is half-open (the T4 page's
  generator draws from a closed [-1, 1] with libc ``rand``; that generator is
  not portable, so only its distribution is kept).
* normal(mu, sigma): Box-Muller on consecutive pairs, ``u1 = (j0 + 1) / 2**24``
  in (0, 1], ``u2 = j1 / 2**24``; element ``2p`` takes ``r cos(2 pi u2)``, element
  ``2p + 1`` takes ``r sin(2 pi u2)``, computed in float64 and rounded to float32.

All matrices are row-major float32.  ``ld`` values default to the row width.
"""
from __future__ import annotations

import concurrent.futures
import dataclasses
import math
import os
from typing import Dict, Optional, Tuple

import numpy as np

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_STREAM_MUL = 0xD1B54A32D192ED03
STREAM_A, STREAM_B, STREAM_C = 1, 2, 3
_CHUNK = 1 << 22


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    return z


def stream_key(seed: int, stream: int) -> np.uint64:
    base = (int(seed) ^ (int(stream) * _STREAM_MUL)) & 0xFFFFFFFFFFFFFFFF
    return _mix64(np.array([base], dtype=np.uint64))[0]


def _bits(key: np.uint64, start: int, count: int) -> np.ndarray:
    """The 24-bit draws ``x_i >> 40`` of stream key ``key`` for i in
    [start, start + count), as uint32 (one chunk, one thread)."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = key + idx * _GAMMA
    return (_mix64(z) >> np.uint64(40)).astype(np.uint32)


def _chunked(count: int, step: int, fill) -> None:
    """Call fill(lo, hi) over [0, count) in chunks of ``step``.  Element i of a
    stream depends only on i (the generator is counter-based), so the chunks
    run on a thread pool (numpy releases the interpreter lock in its array
    loops) and the values do not depend on the chunking.  The pool lives only
    for this call, so a process forked later inherits no worker threads."""
    spans = [(lo, min(count, lo + step)) for lo in range(0, count, step)]
    if len(spans) <= 1:
        for lo, hi in spans:
            fill(lo, hi)
        return
    workers = max(1, min(len(spans), os.cpu_count() or 1, 32))
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        for f in [ex.submit(fill, lo, hi) for lo, hi in spans]:
            f.result()


def raw_bits(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """The 24-bit draws ``x_i >> 40`` for i in [start, start + count) as uint32."""
    key = stream_key(seed, stream)
    out = np.empty(count, dtype=np.uint32)

    def fill(lo, hi):
        out[lo:hi] = _bits(key, start + lo, hi - lo)

    _chunked(count, _CHUNK, fill)
    return out


def uniform_pm1(seed: int, stream: int, count: int) -> np.ndarray:
    """``count`` float32 values in [-1, 1), each an exact multiple of 2**-23."""
    key = stream_key(seed, stream)
    out = np.empty(count, dtype=np.float32)

    def fill(lo, hi):
        j = _bits(key, lo, hi - lo).astype(np.int64) - (1 << 23)
        out[lo:hi] = (j.astype(np.float64) * 2.0 ** -23).astype(np.float32)

    _chunked(count, _CHUNK, fill)
    return out


def normal(seed: int, stream: int, count: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """``count`` float32 normal(mean, std) draws by Box-Muller on draw pairs."""
    key = stream_key(seed, stream)
    pairs = (count + 1) // 2
    out = np.empty(2 * pairs, dtype=np.float32)

    def fill(lo, hi):  # pairs lo .. hi-1, draws 2*lo .. 2*hi-1
        bits = _bits(key, 2 * lo, 2 * (hi - lo)).astype(np.float64)
        u1 = (bits[0::2] + 1.0) * 2.0 ** -24
        u2 = bits[1::2] * 2.0 ** -24
        r = np.sqrt(-2.0 * np.log(u1))
        t = 2.0 * math.pi * u2
        blk = np.empty(2 * (hi - lo), dtype=np.float64)
        blk[0::2] = r * np.cos(t)
        blk[1::2] = r * np.sin(t)
        out[2 * lo:2 * hi] = (mean + std * blk).astype(np.float32)

    _chunked(pairs, _CHUNK, fill)
    return out[:count]


def draw(dist: str, seed: int, stream: int, count: int) -> np.ndarray:
    """One flat float32 stream for a distribution tag."""
    if dist == "u11":
        return uniform_pm1(seed, stream, count)
    if dist == "n01":
        return normal(seed, stream, count, 0.0, 1.0)
    if dist == "n002":
        return normal(seed, stream, count, 0.0, 0.02)
    if dist == "zero":
        return np.zeros(count, dtype=np.float32)
    raise ValueError(f"unknown distribution tag {dist!r}")


@dataclasses.dataclass(frozen=True)
class Workload:
    """One SGEMM problem ``C = alpha * A @ B + beta * C`` with its input recipe."""

    name: str
    M: int
    N: int
    K: int
    alpha: float
    beta: float
    seed: int
    dist_ab: str
    dist_c: str
    lda: Optional[int] = None
    ldb: Optional[int] = None
    ldc: Optional[int] = None

    @property
    def lds(self) -> Tuple[int, int, int]:
        return (self.lda or self.K, self.ldb or self.N, self.ldc or self.N)

    def flops(self) -> float:
        """2*M*N*K: one multiply and one add per (i, j, k) term."""
        return 2.0 * self.M * self.N * self.K

    def min_bytes(self) -> float:
        """Each operand read once, C written once and read only when beta != 0."""
        c_reads = 1 if self.beta != 0.0 else 0
        return 4.0 * (self.M * self.K + self.K * self.N + self.M * self.N * (1 + c_reads))

    def make(self) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
        """Host float32 arrays (A, B, C) shaped (M, lda), (K, ldb), (M, ldc).

        Padding columns beyond K / N (when ld is larger) are drawn from the same
        stream, so they hold finite garbage that a correct GEMM never reads.
        """
        lda, ldb, ldc = self.lds
        A = draw(self.dist_ab, self.seed, STREAM_A, self.M * lda).reshape(self.M, lda)
        B = draw(self.dist_ab, self.seed, STREAM_B, self.K * ldb).reshape(self.K, ldb)
        C = draw(self.dist_c, self.seed, STREAM_C, self.M * ldc).reshape(self.M, ldc)
        return A, B, C


SWEEP_SIZES = (128, 256, 512, 1024, 2048, 4096, 8192)


def _build() -> Dict[str, Workload]:
    w = {}
    w["square512"] = Workload("square512", 512, 512, 512, 1.0, 0.0, 0, "u11", "zero")
    w["square4096"] = Workload("square4096", 4096, 4096, 4096, 1.0, 0.5, 1, "u11", "u11")
    w["ragged1000x1025x777"] = Workload("ragged1000x1025x777", 1000, 1025, 777, 0.75, -1.25, 2,
                                        "n01", "n01", lda=777, ldb=1025, ldc=1025)
    for n in SWEEP_SIZES:
        w[f"sweep{n}"] = Workload(f"sweep{n}", n, n, n, 1.0, 0.0, 3, "u11", "zero")
    w["mlp8192x11008x4096"] = Workload("mlp8192x11008x4096", 8192, 11008, 4096, 1.0, 1.0, 4,
                                       "n002", "u11")
    w["skinny16x4096x4096"] = Workload("skinny16x4096x4096", 16, 4096, 4096, 1.0, 1.0, 4,
                                       "n002", "u11")
    return w


WORKLOADS: Dict[str, Workload] = _build()
HEADLINE = "square4096"
