"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no convolution arithmetic. It only draws numbers:

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014) in its counter form: element k of a stream is
  ``mix64(base + (k + 1) * GAMMA)``, with ``base = mix64(seed + (stream + 1) * GAMMA)``.
* uniforms on [0, 1) from the top 53 bits;
* normals by the Box-Muller transform (Box and Muller, 1958) on consecutive
  pairs of uniforms (u1, u2): ``r = sqrt(-2 ln(1 - u1))``, ``r cos(2 pi u2)``,
  ``r sin(2 pi u2)``.

Values are drawn in float64, rounded to float32 (round to nearest even), and
for half-precision tensors rounded once more from float32 to float16 or
bfloat16 (round to nearest even). The same bytes go to the GPU and to the
oracle, which widens them exactly to float64, so quantisation of the inputs is
never counted as error.

Stream ids (per tensor, so shapes can change without reshuffling others):
x = 0, w = 1, bias = 2, gy = 3, epilogue scale = 4, epilogue shift = 5,
pointwise weights / scale / shift = 6 / 7 / 8; branch i > 0 of a
multi-branch op uses w = 1 + 16 i and bias = 2 + 16 i.
"""
from __future__ import annotations

import os

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

STREAM_X, STREAM_W, STREAM_B, STREAM_GY = 0, 1, 2, 3
STREAM_SCALE, STREAM_SHIFT = 4, 5
STREAM_PW, STREAM_PW_SCALE, STREAM_PW_SHIFT = 6, 7, 8

_CHUNK = 1 << 22


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _base(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([seed & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        s = s + np.uint64(stream + 1) * GAMMA
        return _mix64(s)[0]


def raw_u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Elements [start, start+count) of stream ``stream`` as uint64."""
    base = _base(seed, stream)
    k = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(base + k * GAMMA)


def _parallel(count: int, step: int, fill) -> None:
    """Run ``fill(start, n)`` over [0, count) in pieces of ``step``. Large
    tensors are filled by a few threads at once (numpy releases the GIL on
    these array operations); the values do not depend on the split, because
    every element is a function of its own counter."""
    pieces = [(s, min(step, count - s)) for s in range(0, count, step)]
    if len(pieces) <= 2:
        for s, n in pieces:
            fill(s, n)
        return
    from concurrent.futures import ThreadPoolExecutor
    workers = max(1, min(len(pieces), (os.cpu_count() or 2), 16))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        for f in [ex.submit(fill, s, n) for s, n in pieces]:
            f.result()


def uniform(seed: int, stream: int, count: int) -> np.ndarray:
    """``count`` float64 uniforms on [0, 1)."""
    out = np.empty(count, dtype=np.float64)

    def fill(s, n):
        out[s:s + n] = (raw_u64(seed, stream, s, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)

    _parallel(count, _CHUNK, fill)
    return out


def normal(seed: int, stream: int, count: int) -> np.ndarray:
    """``count`` float64 standard normals (Box-Muller on uniform pairs)."""
    out = np.empty(count, dtype=np.float64)
    pairs = (count + 1) // 2

    def fill(p0, np_):
        u = (raw_u64(seed, stream, 2 * p0, 2 * np_) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log1p(-u1))
        t = 2.0 * np.pi * u2
        z = np.empty(2 * np_, dtype=np.float64)
        z[0::2] = r * np.cos(t)
        z[1::2] = r * np.sin(t)
        n = min(2 * np_, count - 2 * p0)
        out[2 * p0:2 * p0 + n] = z[:n]

    _parallel(pairs, _CHUNK // 2, fill)
    return out


def round_bf16_bits(a32: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even."""
    b = np.ascontiguousarray(a32, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    return ((b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


class Tensor:
    """A synthetic tensor in its storage dtype plus its exact float64 widening.

    ``dtype`` is one of "f32", "f16", "bf16". ``store`` holds the bytes the GPU
    sees (float32, float16, or uint16 bit patterns for bfloat16); ``f64`` is
    the same values widened exactly.
    """

    def __init__(self, values64: np.ndarray, shape, dtype: str):
        v32 = values64.astype(np.float32).reshape(shape)
        self.dtype = dtype
        self.shape = tuple(shape)
        self._f64 = None
        if dtype == "f32":
            self.store = v32
        elif dtype == "f16":
            self.store = v32.astype(np.float16)
        elif dtype == "bf16":
            self.store = round_bf16_bits(v32).reshape(shape)
        else:
            raise ValueError(f"unknown dtype {dtype!r}")

    @property
    def f64(self) -> np.ndarray:
        """The stored values widened exactly to float64 (computed on first use)."""
        if self._f64 is None:
            if self.dtype == "bf16":
                self._f64 = bf16_bits_to_f64(self.store).reshape(self.shape)
            else:
                self._f64 = self.store.astype(np.float64)
        return self._f64

    @property
    def nbytes(self) -> int:
        return self.store.nbytes


def _count(shape) -> int:
    n = 1
    for s in shape:
        n *= int(s)
    return n


def uniform_tensor(shape, dtype: str, seed: int, stream: int, lo=-1.0, hi=1.0) -> Tensor:
    u = uniform(seed, stream, _count(shape))
    return Tensor(lo + (hi - lo) * u, shape, dtype)


def normal_tensor(shape, dtype: str, seed: int, stream: int, std=1.0) -> Tensor:
    return Tensor(std * normal(seed, stream, _count(shape)), shape, dtype)
