"""Helpers for the GPU parity tests: device copies of 16-bit patterns, the
tolerance check, and the seeded tile sampler for large shapes."""
from __future__ import annotations

import numpy as np
import torch

TORCH_DTYPE = {"f16": torch.float16, "bf16": torch.bfloat16}
ATOL = 1e-2
RTOL = {"f16": 1e-3, "bf16": 8e-3}


def to_device(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """uint16 patterns (any 2-D view with unit inner stride) -> device tensor view.

    The whole underlying row buffer (padding included) is copied, so a padded
    host view becomes a padded device view with the same row stride.
    """
    rows, cols = bits.shape
    ld = bits.strides[0] // 2 if rows > 1 else cols
    base = np.lib.stride_tricks.as_strided(bits, shape=(rows, ld), strides=(ld * 2, 2)) \
        if ld != cols else bits
    host = torch.from_numpy(np.ascontiguousarray(base).view(np.int16))
    dev = host.to(device).view(TORCH_DTYPE[dtype])
    return dev[:, :cols]


def from_device(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return b.view(np.float16).astype(np.float64)
    return torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


def check_close(got_bits, ref_bits, dtype, what="", ref_f64=None):
    """|got - ref| <= 1e-2 + rtol * |ref| element by element (ref = oracle output).

    Returns a dict of diagnostics: the max abs error, the worst ratio to the
    bound, and (when the unrounded binary64 sums are given) the max error in
    output ulps against them.
    """
    got = decode(got_bits, dtype)
    ref = decode(ref_bits, dtype)
    err = np.abs(got - ref)
    bound = ATOL + RTOL[dtype] * np.abs(ref)
    bad = ~(err <= bound)  # NaN counts as bad
    if bad.any():
        idx = np.argwhere(bad)
        i, j = idx[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first at {tuple(idx[0])}: "
            f"got {got[i, j]!r} ref {ref[i, j]!r}")
    out = {"max_abs_err": float(err.max()) if err.size else 0.0,
           "worst_ratio": float((err / bound).max()) if err.size else 0.0}
    if ref_f64 is not None and err.size:
        ulp_bits = 10 if dtype == "f16" else 7
        mag = np.maximum(np.abs(ref_f64), 2.0 ** (-14 if dtype == "f16" else -126))
        ulp = 2.0 ** (np.floor(np.log2(mag)) - ulp_bits)
        out["max_ulp"] = float((np.abs(got - ref_f64) / ulp).max())
    return out


def ulp_of(x64: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the 16-bit output format at |x| (IEEE binary16, or bfloat16)."""
    emin, p = (-14, 10) if dtype == "f16" else (-126, 7)
    mag = np.maximum(np.abs(x64), 2.0 ** emin)
    return 2.0 ** (np.floor(np.log2(mag)) - p)


STRICT_REL = 2.0 ** -16


def check_strict(got_bits, ref_f64, sum_abs_f64, dtype, what=""):
    """|got - ref64| <= ulp(ref64) + 2^-16 * sum_k |A[i,k] B'[j,k]|, element by
    element, against the oracle's unrounded binary64 sums.

    The method's arithmetic is fixed ("TIRx GEMM on Blackwell", Take away 1:
    FP32 accumulation, only the order of additions changes) and the output is
    rounded once: FP32 sums of any order stay within a few 2^-24 of
    sum |terms| of the exact sum, and the rounding adds at most half an ulp.
    A K = 16 slice lost or counted twice moves an output by about
    sqrt(16) * E|term|, far outside the bound.  Returns the largest error in
    output ulps and the worst ratio to the bound.
    """
    got = decode(got_bits, dtype)
    ref = np.asarray(ref_f64, dtype=np.float64)
    ulp = ulp_of(ref, dtype)
    bound = ulp + STRICT_REL * np.asarray(sum_abs_f64, dtype=np.float64)
    err = np.abs(got - ref)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)
        i, j = idx[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} outside 1 ulp + 2^-16 sum|terms|; first at "
            f"{tuple(idx[0])}: got {got[i, j]!r} exact {ref[i, j]!r} bound {bound[i, j]!r}")
    if not err.size:
        return {"max_ulp": 0.0, "worst_strict_ratio": 0.0}
    return {"max_ulp": float((err / ulp).max()), "worst_strict_ratio": float((err / bound).max())}


def abs_bits(bits: np.ndarray) -> np.ndarray:
    """16-bit patterns with the sign bit cleared (|x| for FP16 and BF16)."""
    return np.asarray(bits, dtype=np.uint16) & np.uint16(0x7FFF)


def oracle_with_bound(orc, A, B, layout, dtype, rows=None, cols=None):
    """The oracle's rounded D, its unrounded binary64 sums, and the binary64
    sums of |terms| (the oracle run on |A| and |B|) for the strict check."""
    kw = {"layout": layout, "dtype": dtype, "want_f64": True}
    if rows is not None:
        kw["rows"] = rows
    if cols is not None:
        kw["cols"] = cols
    ref, ref64 = orc.gemm(A, B, **kw)
    _, sum_abs = orc.gemm(abs_bits(A), abs_bits(B), **kw)
    return ref, ref64, sum_abs


def sample_tiles(M, N, K, block_m, block_n, group, num_clusters, stages, tile_origin,
                 seed=0, extra_random=16, block_k=64):
    """Seeded sample of whole output tiles that covers every value of
    (cluster, iteration, ring stage at tile start, ring phase at tile start,
    TMEM accumulator buffer) at least once, plus `extra_random` random tiles and
    every tile on the last tile row and the last tile column.

    `tile_origin(task) -> (m0, n0)` is the scheduler's map; cluster c takes
    tasks c, c + C, c + 2C, ...
    """
    m_tiles = -(-M // block_m)
    n_tiles = -(-N // block_n)
    tiles = m_tiles * n_tiles
    kb = -(-K // block_k)  # k-blocks per tile (64 for 16-bit, 128 for FP8 inputs)
    feats = []
    for t in range(tiles):
        c, it = t % num_clusters, t // num_clusters
        start = it * kb
        feats.append((c, it, start % stages, (start // stages) % 2, it % 2))
    need = [set(f[i] for f in feats) for i in range(5)]
    chosen = []
    rng = np.random.default_rng(seed)
    order = rng.permutation(tiles)
    # greedy cover: take a tile whenever it shows a value not yet seen
    for t in order:
        f = feats[t]
        if any(f[i] in need[i] for i in range(5)):
            chosen.append(int(t))
            for i in range(5):
                need[i].discard(f[i])
        if not any(need):
            break
    chosen += [int(t) for t in rng.choice(tiles, size=min(extra_random, tiles), replace=False)]
    origins = {tile_origin(t) for t in chosen}
    last_m = (m_tiles - 1) * block_m
    last_n = (n_tiles - 1) * block_n
    origins.add((last_m, last_n))
    if M % block_m:  # ragged last tile row: check all of it
        origins |= {(last_m, n) for n in range(0, N, block_n)}
    if N % block_n:
        origins |= {(m, last_n) for m in range(0, M, block_m)}
    return sorted(origins)
