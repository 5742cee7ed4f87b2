"""Seeded synthetic inputs for attention workloads.

This module is the one place where the CUDA path and the float64 oracle meet:
both receive the exact same input bits from here.  It holds no attention
arithmetic, only random draws, rounding to the storage dtype, and the
bookkeeping of workload shapes (sequence lengths, cu_seqlens, page tables).

Values are i.i.d. N(0, 1), drawn in float32 from numpy's PCG64 stream and
rounded to fp16 or bf16 with round-to-nearest-even, which is how the
FlashAttention FAQ (Inference Cookbook, "常见问题" Q2, Q16) and the
Flash-Attention 2.8.3 sm_86 verification note build their test tensors
(``torch.randn`` in fp16/bf16).

Layouts follow the (batch, seqlen, heads, head_dim) convention of the
Inference Cookbook FAQ Q5.
"""
from __future__ import annotations

import numpy as np

F16 = "f16"
BF16 = "bf16"
DTYPE_CODES = {F16: 0, BF16: 1}


def round_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to fp16/bf16 (RNE) and return the uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == F16:
        return x.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        u = x.view(np.uint32).astype(np.uint64)
        u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
        return u.astype(np.uint16)
    raise ValueError(f"unknown dtype {dtype!r}")


def bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of fp16/bf16 bit patterns to float64."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == F16:
        return bits.view(np.float16).astype(np.float64)
    if dtype == BF16:
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


E4M3 = "e4m3"  # OCP FP8 E4M3 ("fn": no infinities, 0x7F/0xFF are NaN, max 448)


def e4m3_values() -> np.ndarray:
    """The float64 value of every E4M3 bit pattern 0..255 (NaN for 0x7F, 0xFF):
    sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 is
    subnormal (m/8 * 2^-6)."""
    b = np.arange(256)
    e = (b >> 3) & 0xF
    m = (b & 7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    val = np.where(b & 0x80, -mag, mag)
    val[(b & 0x7F) == 0x7F] = np.nan
    return val


def e4m3_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of E4M3 bit patterns (uint8) to float64."""
    return e4m3_values()[np.asarray(bits, dtype=np.uint8)]


def round_e4m3(x: np.ndarray) -> np.ndarray:
    """Round to the nearest E4M3 value (ties to the even pattern), saturating
    magnitudes above 448 to 448; returns uint8 bit patterns."""
    x = np.asarray(x, dtype=np.float64)
    pos = e4m3_values()[:0x7F]                      # 0x00..0x7E, increasing
    a = np.minimum(np.abs(x), pos[-1])
    i = np.clip(np.searchsorted(pos, a), 1, len(pos) - 1)
    lo, hi = pos[i - 1], pos[i]
    take_hi = (a - lo > hi - a) | ((a - lo == hi - a) & ((i & 1) == 0))
    code = np.where(take_hi, i, i - 1).astype(np.uint8)
    code = np.where(a == 0, 0, code).astype(np.uint8)
    return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)


def normal_e4m3(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) draws rounded to E4M3; returns uint8 bits."""
    return round_e4m3(rng.standard_normal(size=shape, dtype=np.float32))


def normal_bits(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """N(0,1) float32 draws rounded to ``dtype``; returns uint16 bits."""
    return round_bits(rng.standard_normal(size=shape, dtype=np.float32), dtype)


def dense_case(seed: int, b: int, sq: int, sk: int, hq: int, hkv: int, d: int,
               dtype: str, with_dout: bool = False) -> dict:
    """Q (b,sq,hq,d), K/V (b,sk,hkv,d) and optionally dO (b,sq,hq,d) as uint16 bits."""
    rng = np.random.default_rng(seed)
    out = {
        "q": normal_bits(rng, (b, sq, hq, d), dtype),
        "k": normal_bits(rng, (b, sk, hkv, d), dtype),
        "v": normal_bits(rng, (b, sk, hkv, d), dtype),
    }
    if with_dout:
        out["dout"] = normal_bits(rng, (b, sq, hq, d), dtype)
    return out


def varlen_lengths(seed: int, nseq: int = 64, lo: int = 100, hi: int = 4096) -> np.ndarray:
    """Sequence lengths uniform in [lo, hi] (inclusive), int64."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=nseq)


def cu_seqlens(lengths) -> np.ndarray:
    """[0, cumsum(lengths)] as int32, the packing of the Inference Cookbook FAQ Q8."""
    lengths = np.asarray(lengths, dtype=np.int64)
    out = np.zeros(len(lengths) + 1, dtype=np.int64)
    np.cumsum(lengths, out=out[1:])
    if out[-1] > np.iinfo(np.int32).max:
        raise ValueError("total length does not fit int32")
    return out.astype(np.int32)


def varlen_case(seed: int, lengths_q, lengths_k, hq: int, hkv: int, d: int,
                dtype: str, with_dout: bool = False) -> dict:
    """Packed Q (Tq,hq,d), K/V (Tk,hkv,d) with their cu_seqlens."""
    rng = np.random.default_rng(seed + 1_000_003)
    cq, ck = cu_seqlens(lengths_q), cu_seqlens(lengths_k)
    tq, tk = int(cq[-1]), int(ck[-1])
    out = {
        "q": normal_bits(rng, (tq, hq, d), dtype),
        "k": normal_bits(rng, (tk, hkv, d), dtype),
        "v": normal_bits(rng, (tk, hkv, d), dtype),
        "cu_seqlens_q": cq,
        "cu_seqlens_k": ck,
    }
    if with_dout:
        out["dout"] = normal_bits(rng, (tq, hq, d), dtype)
    return out


def decode_layout(seed: int, b: int, max_len: int, page_size: int, s_new: int):
    """cache_seqlens uniform in [1, max_len] and a random page placement.

    Returns (cache_seqlens int32 (b,), block_table int32 (b, pages_per_seq),
    num_pages).  Each sequence gets enough pages for max_len + s_new tokens
    and the pool is a random permutation of all pages, so logically adjacent
    pages are scattered through the pool.
    """
    rng = np.random.default_rng(seed)
    cache_seqlens = rng.integers(1, max_len + 1, size=b).astype(np.int32)
    pages_per_seq = -(-(max_len + s_new) // page_size)
    num_pages = b * pages_per_seq
    block_table = rng.permutation(num_pages).astype(np.int32).reshape(b, pages_per_seq)
    return cache_seqlens, block_table, num_pages


def decode_case(seed: int, b: int, sq: int, s_new: int, hq: int, hkv: int, d: int,
                max_len: int, page_size: int, dtype: str) -> dict:
    """Host-side paged decode inputs (small pools only; the pool is generated here)."""
    cache_seqlens, block_table, num_pages = decode_layout(seed, b, max_len, page_size, s_new)
    rng = np.random.default_rng(seed + 7_919)
    out = {
        "cache_seqlens": cache_seqlens,
        "block_table": block_table,
        "k_cache": normal_bits(rng, (num_pages, page_size, hkv, d), dtype),
        "v_cache": normal_bits(rng, (num_pages, page_size, hkv, d), dtype),
        "q": normal_bits(rng, (b, sq, hq, d), dtype),
    }
    if s_new > 0:
        out["k_new"] = normal_bits(rng, (b, s_new, hkv, d), dtype)
        out["v_new"] = normal_bits(rng, (b, s_new, hkv, d), dtype)
    return out


def device_normal(shape, dtype: str, seed: int, device="cuda"):
    """Seeded N(0,1) tensor generated on the device with torch's generator.

    Used for pools too large to draw on the host (the 8256-page decode pool).
    The float32 draw is rounded to the storage dtype by torch (RNE).
    """
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return t.to(torch.float16 if dtype == F16 else torch.bfloat16)
