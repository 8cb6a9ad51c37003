"""Seeded synthetic inputs for the int4-weight linear layer workloads.

This module is shared by the tests, ``bench.py`` and the smoke check. It holds
none of the layer's arithmetic: it only draws random bits and values with the
shapes, dtypes and distributions of the workloads, and hands them out as numpy
arrays (bf16 tensors travel as their raw ``uint16`` bit patterns).

Random numbers come from one counter-based generator, SplitMix64 (Steele, Lea
and Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014), keyed
by ``(seed, tag)`` and indexed by the element's flat position, so any element
can be regenerated on its own and the stream is the same on every host.

Seeds follow one convention: activations 0, weight codes 1, weight scales 2,
zeros 3, outlier channels 4, MoE router logits 5.
"""
from __future__ import annotations

import numpy as np
import torch

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_GOLDEN = np.uint64(0x9E3779B97F4A7C15)


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser (the generator's output function)."""
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= np.uint64(0xBF58476D1CE4E5B9)
        z ^= z >> np.uint64(27)
        z *= np.uint64(0x94D049BB133111EB)
        z ^= z >> np.uint64(31)
    return z


def raw_u64(seed: int, tag: int, n: int, offset: int = 0) -> np.ndarray:
    """``n`` 64-bit words of stream ``(seed, tag)``, counters ``offset..offset+n-1``."""
    key = _mix(np.array([(seed & 0xFFFFFFFF) << 32 | (tag & 0xFFFFFFFF)], dtype=np.uint64))[0]
    ctr = np.arange(offset, offset + n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = key + (ctr + np.uint64(1)) * _GOLDEN
    return _mix(state)


def uniform(seed: int, tag: int, n: int) -> np.ndarray:
    """Uniform float64 in [0, 1) with 53 random bits."""
    return (raw_u64(seed, tag, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, tag: int, n: int) -> np.ndarray:
    """Standard normal float64 by the Box-Muller transform on two uniform streams."""
    u1 = 1.0 - uniform(seed, tag * 2 + 0, n)  # (0, 1]
    u2 = uniform(seed, tag * 2 + 1, n)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float values to bf16 (torch's round-to-nearest-even cast); return uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (for building inputs only)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------------
# workload tensors
# ---------------------------------------------------------------------------

def activations_bf16(M: int, K: int, seed: int = 0, outlier_frac: float = 0.0,
                     outlier_gain: float = 20.0, std: float = 1.0) -> np.ndarray:
    """x ~ N(0, std^2) as bf16 bits ``[M, K]``; optionally a fraction of the K
    channels (picked by seed 4) multiplied by ``outlier_gain`` before rounding."""
    x = normal(seed, 10, M * K).reshape(M, K) * std
    if outlier_frac > 0.0:
        x[:, outlier_channels(K, outlier_frac)] *= outlier_gain
    return to_bf16_bits(x)


def outlier_channels(K: int, frac: float, seed: int = 4) -> np.ndarray:
    """Sorted indices of round(frac*K) distinct channels."""
    n = int(round(frac * K))
    order = np.argsort(raw_u64(seed, 11, K), kind="stable")
    return np.sort(order[:n])


def random_words(shape, seed: int = 1, tag: int = 20) -> np.ndarray:
    """Uniform random 32-bit words as int32. Every 4-bit field of a uniform word
    is a uniform code in 0..15, so these are uniform int4 codes in any packing."""
    n = int(np.prod(shape))
    return (raw_u64(seed, tag, n) >> np.uint64(32)).astype(np.uint32).view(np.int32).reshape(shape)


def scales_f16(shape, lo: float = 0.005, hi: float = 0.02, seed: int = 2, tag: int = 30) -> np.ndarray:
    """Scales ~ U[lo, hi] rounded to fp16."""
    n = int(np.prod(shape))
    return (lo + (hi - lo) * uniform(seed, tag, n)).astype(np.float16).reshape(shape)


def scales_bf16(shape, lo: float = 0.005, hi: float = 0.02, seed: int = 2, tag: int = 31) -> np.ndarray:
    """Scales ~ U[lo, hi] rounded to bf16 (uint16 bits)."""
    n = int(np.prod(shape))
    return to_bf16_bits((lo + (hi - lo) * uniform(seed, tag, n)).reshape(shape))


def zeros_bf16(shape, std: float = 0.01, seed: int = 3) -> np.ndarray:
    """Per-group additive zeros ~ N(0, std^2) as bf16 bits."""
    n = int(np.prod(shape))
    return to_bf16_bits((normal(seed, 40, n) * std).reshape(shape))


def bias_bf16(N: int, std: float = 0.1, seed: int = 6) -> np.ndarray:
    return to_bf16_bits(normal(seed, 50, N) * std)


def fp8_codes(shape, seed: int = 0, tag: int = 60) -> np.ndarray:
    """Random finite e4m3fn codes (uint8, never 0x7F/0xFF) for direct GEMM tests."""
    n = int(np.prod(shape))
    c = (raw_u64(seed, tag, n) >> np.uint64(56)).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] &= 0xFE
    return c.reshape(shape)


def router_logits(tokens: int, experts: int, seed: int = 5) -> np.ndarray:
    """MoE router logits ``[tokens, experts]``: N(0,1) rounded to float32."""
    return normal(seed, 70, tokens * experts).reshape(tokens, experts).astype(np.float32)


def offsets_from_counts(counts) -> np.ndarray:
    counts = np.asarray(counts, dtype=np.int64)
    off = np.zeros(len(counts) + 1, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    return off
