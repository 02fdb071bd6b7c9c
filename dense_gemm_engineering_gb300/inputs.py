"""Seeded synthetic operands for the GEMM workloads.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It holds no GEMM arithmetic: it only draws numbers and rounds
them once to the 16-bit storage type, so that the GPU kernel and the oracle
consume the very same bit patterns.

Generator (counter-based SplitMix64, Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014; the 64-bit finaliser is the one
published with Vigna's reference implementation):

    gamma  = 0x9E3779B97F4A7C15
    mix(z) = z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
             z ^= z >> 27; z *= 0x94D049BB133111EB; z ^ (z >> 31)   (mod 2^64)
    key(seed, stream) = mix((seed * 2^16 + stream + 1) * gamma)
    draw i            = mix(key + (i + 1) * gamma)          i = 0, 1, 2, ...

Distributions (element i of a row-major matrix, i = row * cols + col):
    uniform U[-1, 1):  u = (draw_i >> 40) * 2^-24;  v = 2u - 1     (exact in fp32)
    normal  N(0, s^2): Box-Muller on draws 2i and 2i+1:
                       u1 = ((d_2i >> 11) + 1) * 2^-53,  u2 = (d_2i+1 >> 11) * 2^-53
                       v  = fp32(s * sqrt(-2 ln u1) * cos(2 pi u2))
Then v is rounded once (nearest, ties to even) to binary16 or bfloat16, or to
the 8-bit E4M3 / E5M2 formats (OCP 8-bit floating point; magnitudes beyond the
largest finite value saturate to it, which the drawn values never reach).

Stream 0 draws A, stream 1 draws B.  Padding columns (row stride > cols) are
filled with a quiet NaN so that any read of padding poisons the result.

Block scales (MX): one UE8M0 byte per 32 K elements of each row of A (stream 2)
and of B (stream 3), row-major with ceil(K/32) bytes per row; byte i of a
stream is lo + (draw_i >> 11) mod (hi - lo + 1), a power-of-two scale
2^(byte - 127).  Padding bytes hold 255, the UE8M0 NaN.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0, "e4m3": 0x7F, "e5m2": 0x7E}
FP8 = ("e4m3", "e5m2")


def _fp8_positive_table(fmt: str):
    """(values, codes) of the finite non-negative codes of an FP8 format, in
    increasing order (the codes are monotonic in value)."""
    if fmt == "e4m3":  # 1.4.3, bias 7, no infinities, 0x7F is NaN
        codes = np.arange(0x7F)
        e, f = codes >> 3, codes & 7
        vals = np.where(e == 0, f * 2.0 ** -9, (8 + f) * np.exp2(e - 10.0))
    elif fmt == "e5m2":  # 1.5.2, bias 15, 0x7C is inf
        codes = np.arange(0x7C)
        e, f = codes >> 2, codes & 3
        vals = np.where(e == 0, f * 2.0 ** -16, (4 + f) * np.exp2(e - 17.0))
    else:
        raise ValueError(f"unknown FP8 format {fmt!r}")
    return vals.astype(np.float64), codes.astype(np.uint8)


_FP8_TABLES = {f: _fp8_positive_table(f) for f in FP8}


def f32_to_fp8_bits(x: np.ndarray, fmt: str) -> np.ndarray:
    """binary32 -> FP8 pattern, nearest with ties to the even code; finite
    magnitudes above the largest finite value saturate to it."""
    vals, codes = _FP8_TABLES[fmt]
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    a = np.minimum(np.abs(x), vals[-1])
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, len(vals) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - vals[lo], vals[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((codes[hi] & 1) == 0))
    c = np.where(pick_hi, codes[hi], codes[lo]).astype(np.uint8)
    return c | np.where(np.signbit(x), np.uint8(0x80), np.uint8(0)).astype(np.uint8)


def _mix(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _C1
    z = z ^ (z >> np.uint64(27))
    z = z * _C2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        base = np.array([(int(seed) * 65536 + int(stream) + 1) & ((1 << 64) - 1)],
                        dtype=np.uint64)
        return _mix(base * GAMMA)[0]


def draws(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Draws start .. start+count-1 of stream (seed, stream) as uint64."""
    key = stream_key(seed, stream)
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix(key + idx * GAMMA)


def splitmix64_sequence(state: int, count: int) -> np.ndarray:
    """Plain SplitMix64 outputs from an initial state (used to pin the mixer)."""
    with np.errstate(over="ignore"):
        idx = np.arange(1, count + 1, dtype=np.uint64)
        return _mix(np.uint64(state) + idx * GAMMA)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """binary32 -> bfloat16 pattern, nearest with ties to even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def _to_bits(v32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype in FP8:
        return f32_to_fp8_bits(v32, dtype)
    if dtype == "f16":
        return v32.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        return f32_to_bf16_bits(v32)
    raise ValueError(f"unknown dtype {dtype!r}")


def values_f32(seed: int, stream: int, start: int, count: int, dist: str,
               sigma: float = 0.02) -> np.ndarray:
    """Elements start .. start+count-1 of a stream, as binary32 before rounding."""
    if dist == "uniform":
        d = draws(seed, stream, start, count)
        u = (d >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)
        return np.float32(2.0) * u - np.float32(1.0)
    if dist == "normal":
        d = draws(seed, stream, 2 * start, 2 * count)
        u1 = ((d[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (d[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        return (sigma * z).astype(np.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def bits(seed: int, stream: int, count: int, dtype: str, dist: str,
         sigma: float = 0.02) -> np.ndarray:
    """First `count` elements of a stream as storage patterns (uint16, or
    uint8 for the FP8 formats).

    Chunks are independent (the generator is counter-based), so they are drawn
    on a thread pool; the result does not depend on the chunking.
    """
    out = np.empty(count, dtype=np.uint8 if dtype in FP8 else np.uint16)

    def fill(s):
        n = min(_CHUNK, count - s)
        out[s:s + n] = _to_bits(values_f32(seed, stream, s, n, dist, sigma), dtype)

    starts = range(0, count, _CHUNK)
    if len(starts) <= 1:
        for s in starts:
            fill(s)
    else:
        workers = min(len(starts), os.cpu_count() or 1, 16)
        with ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(fill, starts))
    return out


def matrix(seed: int, stream: int, rows: int, cols: int, dtype: str, dist: str,
           ld: int | None = None, sigma: float = 0.02) -> np.ndarray:
    """A rows x cols operand of 16-bit patterns, row-major with row stride ld.

    Returns the (rows, cols) view of a (rows, ld) buffer; padding is NaN.
    """
    ld = cols if ld is None else ld
    if ld < cols:
        raise ValueError("ld < cols")
    flat = bits(seed, stream, rows * cols, dtype, dist, sigma)
    if ld == cols:
        return flat.reshape(rows, cols)
    buf = np.full((rows, ld), NAN_BITS[dtype], dtype=flat.dtype)
    buf[:, :cols] = flat.reshape(rows, cols)
    return buf[:, :cols]


def mx_scales(seed: int, stream: int, rows: int, K: int, lo: int = 124, hi: int = 130,
              ld: int | None = None) -> np.ndarray:
    """UE8M0 scale bytes of a rows x K block-scaled operand: (rows, ceil(K/32))
    uint8, uniform integers in [lo, hi]; row stride ld (padding is 255)."""
    if not (0 <= lo <= hi <= 254):
        raise ValueError("scale bytes must lie in [0, 254]")
    groups = -(-K // 32)
    ld = groups if ld is None else ld
    if ld < groups:
        raise ValueError("ld < ceil(K / 32)")
    d = draws(seed, stream, 0, rows * groups)
    x = (np.uint64(lo) + (d >> np.uint64(11)) % np.uint64(hi - lo + 1)).astype(np.uint8)
    if ld == groups:
        return x.reshape(rows, groups)
    buf = np.full((rows, ld), 255, dtype=np.uint8)
    buf[:, :groups] = x.reshape(rows, groups)
    return buf[:, :groups]


def mx_operands(M: int, N: int, K: int, fmt: str, dist: str, seed: int, lda: int | None = None,
                ldb: int | None = None, lo: int = 124, hi: int = 130):
    """(A, B, SA, SB) of a block-scaled FP8 D = A.Bt: FP8 patterns as operands()
    draws them, and the scale bytes of mx_scales() (streams 2 and 3)."""
    A, B = operands(M, N, K, "abt", fmt, dist, seed, lda=lda, ldb=ldb)
    return A, B, mx_scales(seed, 2, M, K, lo, hi), mx_scales(seed, 3, N, K, lo, hi)


def operands(M: int, N: int, K: int, layout: str, dtype: str, dist: str, seed: int,
             lda: int | None = None, ldb: int | None = None):
    """(A, B) for D = A.Bt (layout 'abt', B is N x K) or D = A.B ('ab', B is K x N).
    FP8 operands ('e4m3', 'e5m2') exist for the A.Bt layout only."""
    if dtype in FP8 and layout != "abt":
        raise ValueError("FP8 operands are K-major: layout 'abt' only")
    A = matrix(seed, 0, M, K, dtype, dist, lda)
    if layout == "abt":
        B = matrix(seed, 1, N, K, dtype, dist, ldb)
    elif layout == "ab":
        B = matrix(seed, 1, K, N, dtype, dist, ldb)
    else:
        raise ValueError(f"unknown layout {layout!r}")
    return A, B
