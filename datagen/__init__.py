"""Seeded synthetic inputs for dense GEMM, shared by the oracle side and the CUDA side.

This module only draws numbers and lays them out in memory. It holds none of the
GEMM arithmetic: no products, no sums, no rounding of results. Both the CPU
oracle (``oracle/``) and the CUDA library (``dense_gemm_06_gb300``) consume the
host buffers made here, so a parity test compares the two on byte-identical
inputs.

Generator: a counter-based SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014). Draw ``i`` of stream ``(seed,
stream)`` is ``mix64(key + (i + 1) * GOLDEN)`` with ``key = mix64(seed * GOLDEN
^ stream * STREAM_MUL)``, all modulo 2**64. Being counter-based, any element can
be regenerated without drawing the ones before it, and the result does not
depend on chunking.

Distributions (the workloads of the pages):

* ``int``: integers uniform in ``[lo, hi]`` (inclusive). The CuTe Ampere SGEMM
  example (``run()``, ``create_and_permute_tensor``) and the CK Tile practice
  GEMM ("Host Matrix Creation") both fill operands with small integers in
  [-5, 5]; integer-valued inputs make every partial sum exact in fp32. The
  draw takes the top 32 bits ``u`` and returns ``lo + (u * (hi - lo + 1)) >>
  32`` (multiply-shift; bias below 2**-28 for the ranges used here).
* ``pm1``: uniform on [-1, 1): ``(x >> 40) * 2**-23 - 1``, exact in fp32.
* ``normal``: N(0, 1) by the Box-Muller transform in float64 from two draws
  ``u1 = ((x0 >> 11) + 1) * 2**-53`` (in (0, 1]) and ``u2 = (x1 >> 11) * 2**-53``,
  ``z = sqrt(-2 ln u1) * cos(2 pi u2)``, then rounded to the storage type.

Storage rounding: f32 by IEEE round-to-nearest-even from float64 (numpy cast);
f16 by numpy's float64 -> float16 cast (round-to-nearest-even); bf16 by
float64 -> float32 (RNE) and then float32 -> bf16 round-to-nearest-even on the
bit pattern. Integer-valued draws are exact in every storage type used.

Layout (the element addressing of the C ABI, matching the CuTe SGEMM example's
``a_major``/``b_major`` options): a logical ``rows x kdim`` operand (A is M x K,
B is N x K) is stored either K-major (element (r, k) at ``r * ld + k``) or
MN-major (element (r, k) at ``k * ld + r``). Values are always drawn in the
logical order ``r * kdim + k``, so the same seed gives the same logical matrix
for every major and every leading dimension; padding elements (``ld`` beyond
the extent) hold ``pad`` (NaN by default, so a kernel that reads padding is
caught).
"""

from __future__ import annotations

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
STREAM_MUL = 0xD1B54A32D192ED03
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1

# Storage codes, matching the oracle's and the C ABI's element types.
F32, F16, BF16 = "f32", "f16", "bf16"
MAJOR_K, MAJOR_MN = 0, 1

_CHUNK = 1 << 22  # elements per vectorised block (bounds temporary memory)


def _mix64_scalar(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> int:
    return _mix64_scalar(((seed * GOLDEN) ^ (stream * STREAM_MUL)) & _MASK64)


def draws(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of stream (seed, stream) as uint64."""
    key = np.uint64(stream_key(seed, stream))
    z = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    t = np.empty_like(z)
    with np.errstate(over="ignore"):  # in place: same values as _mix64
        z *= np.uint64(GOLDEN)
        z += key
        np.right_shift(z, np.uint64(30), out=t)
        z ^= t
        z *= np.uint64(_M1)
        np.right_shift(z, np.uint64(27), out=t)
        z ^= t
        z *= np.uint64(_M2)
        np.right_shift(z, np.uint64(31), out=t)
        z ^= t
    return z


def _values(dist: str, seed: int, stream: int, start: int, count: int,
            lo: int, hi: int) -> np.ndarray:
    """float64 values of logical elements start..start+count-1."""
    if dist == "int":
        if hi < lo:
            raise ValueError("empty integer range")
        u = draws(seed, stream, start, count) >> np.uint64(32)
        span = np.uint64(hi - lo + 1)
        with np.errstate(over="ignore"):
            v = (u * span) >> np.uint64(32)
        return v.astype(np.int64).astype(np.float64) + float(lo)
    if dist == "pm1":
        u = draws(seed, stream, start, count) >> np.uint64(40)
        return u.astype(np.float64) * 2.0 ** -23 - 1.0
    if dist == "normal":
        x = draws(seed, stream, 2 * start, 2 * count)
        u1 = ((x[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (x[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    raise ValueError(f"unknown distribution {dist!r}")


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest-even) and return the bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    with np.errstate(over="ignore"):
        return ((b + bias) >> np.uint32(16)).astype(np.uint16)


def to_storage(v: np.ndarray, dtype: str) -> np.ndarray:
    """float64 -> storage array (float32, or uint16 bit patterns for f16/bf16)."""
    if dtype == F32:
        return v.astype(np.float32)
    if dtype == F16:
        return v.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        return f32_to_bf16_bits(v.astype(np.float32))
    raise ValueError(f"unknown dtype {dtype!r}")


def _pad_bits(dtype: str, pad: float) -> np.ndarray:
    return to_storage(np.array([pad], dtype=np.float64), dtype)


def storage_dtype(dtype: str):
    return np.float32 if dtype == F32 else np.uint16


def storage_elems(rows: int, kdim: int, major: int, ld: int) -> int:
    """Number of elements a (rows x kdim) operand occupies with this layout."""
    if rows == 0 or kdim == 0:
        return 0
    outer, inner = (rows, kdim) if major == MAJOR_K else (kdim, rows)
    if ld < inner:
        raise ValueError("leading dimension below the contiguous extent")
    return (outer - 1) * ld + inner


def operand(rows: int, kdim: int, *, major: int = MAJOR_K, ld: int | None = None,
            dtype: str = F32, dist: str = "int", lo: int = -5, hi: int = 5,
            seed: int = 0, stream: int = 0, pad: float = float("nan")) -> np.ndarray:
    """A seeded (rows x kdim) operand in the requested storage layout.

    Returns a flat storage array of ``storage_elems(rows, kdim, major, ld)``
    elements (float32, or uint16 bit patterns for f16/bf16).
    """
    inner = kdim if major == MAJOR_K else rows
    if ld is None:
        ld = inner
    n = storage_elems(rows, kdim, major, ld)
    if n == 0:
        return np.empty(0, dtype=storage_dtype(dtype))
    outer = rows if major == MAJOR_K else kdim
    full = np.full(outer * ld, _pad_bits(dtype, pad)[0], dtype=storage_dtype(dtype))
    grid = full.reshape(outer, ld)
    lg = logical(rows, kdim, dtype=dtype, dist=dist, lo=lo, hi=hi, seed=seed,
                 stream=stream)
    if major == MAJOR_K:
        grid[:, :kdim] = lg
    else:
        grid[:, :rows] = lg.T
    return np.ascontiguousarray(full[:n])


def logical(rows: int, kdim: int, *, dtype: str = F32, dist: str = "int",
            lo: int = -5, hi: int = 5, seed: int = 0, stream: int = 0) -> np.ndarray:
    """The same draws as ``operand`` as a (rows, kdim) storage array (row = r)."""
    total = rows * kdim
    out = np.empty(total, dtype=storage_dtype(dtype))
    for start in range(0, total, _CHUNK):
        cnt = min(_CHUNK, total - start)
        out[start:start + cnt] = to_storage(
            _values(dist, seed, stream, start, cnt, lo, hi), dtype)
    return out.reshape(rows, kdim)


def sample_indices(n: int, count: int, seed: int, stream: int = 99,
                   always=(0, -1)) -> np.ndarray:
    """``count`` distinct indices in [0, n) drawn without replacement, plus the
    ``always`` ones (0 and n-1 by default, which cover the ragged tail), sorted."""
    if n <= 0:
        return np.zeros(0, dtype=np.int64)
    chosen = {a % n for a in always}
    want = min(n, count + len(chosen))
    i = 0
    while len(chosen) < want:
        batch = draws(seed, stream, i, 4096)
        for x in batch:
            chosen.add(int(x % np.uint64(n)))
            if len(chosen) >= want:
                break
        i += 4096
    return np.array(sorted(chosen), dtype=np.int64)
