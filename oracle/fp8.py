"""fp8 (e4m3) KV-pool oracle -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this module.  It shares no code with the CUDA library.

The pages do not have an fp8 pool; it is the bandwidth-halving variant of
the cache write and the decode gather that follows from decode being bound
by reading the whole cache every step ("Prefill/Decode" of the
inference-engine talk write-up).  Readings taken where the pages are silent:

- e4m3 is the OCP 8-bit format with 4 exponent bits (bias 7) and 3 mantissa
  bits, subnormals, no infinities, one NaN pattern per sign (S.1111.111);
  its largest finite value is 448.
- A pool stores code(x * inv_scale), one scale per pool (K and V have their
  own); inv_scale is the fp32 reciprocal of the scale, the product is taken
  in fp32, and the code is the nearest e4m3 value (ties to even), with
  values beyond 448 saturated to +-448 (NaN stays NaN).
- Attention reads value(code) * scale for every key and value.

Parity status: pinned by ``tests/test_oracle_fp8.py`` (every code decoded
from the format's definition and checked against torch.float8_e4m3fn,
rounding against brute force over all codes, and attention equal to the C
oracle on pools whose dequantised values are bf16-exact).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def decode_codes() -> np.ndarray:
    """float64 value of each of the 256 codes (NaN for the two NaN codes)."""
    out = np.empty(256, dtype=np.float64)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            out[c] = np.nan
        elif e == 0:
            out[c] = s * (m / 8.0) * 2.0 ** -6
        else:
            out[c] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


_VALUES = decode_codes()
_FINITE = np.array([c for c in range(128) if not np.isnan(_VALUES[c])], dtype=np.int64)  # non-negative codes


def encode(x) -> np.ndarray:
    """Nearest e4m3 code of each float (ties to the even code), saturating to
    +-448; NaN gives the NaN code of its sign."""
    x = np.asarray(x, dtype=np.float64)
    mag = np.abs(x)
    vals = _VALUES[_FINITE]                                  # 0, 2^-9, ..., 448, increasing
    i = np.searchsorted(vals, np.minimum(mag, E4M3_MAX))
    i = np.clip(i, 1, len(vals) - 1)
    lo, hi = vals[i - 1], vals[i]
    m = np.minimum(mag, E4M3_MAX)
    pick_hi = (m - lo > hi - m) | ((m - lo == hi - m) & (_FINITE[i] % 2 == 0))
    code = np.where(pick_hi, _FINITE[i], _FINITE[i - 1])
    code = np.where(m <= 0.0, 0, code)
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F | np.where(np.signbit(x), 0x80, 0), code)
    return code.astype(np.uint8)


def value(codes) -> np.ndarray:
    return _VALUES[np.asarray(codes, dtype=np.int64)]


def quantize_bf16_rows(bits_u16, inv_scale: float) -> np.ndarray:
    """Codes of bf16 values (uint16 bit patterns) times the fp32 inv_scale,
    the product rounded to fp32 first."""
    f = (np.asarray(bits_u16, dtype=np.uint32) << 16).view(np.float32)
    prod = (f * np.float32(inv_scale)).astype(np.float32)
    return encode(prod.astype(np.float64))


def cache_write(k_pool, v_pool, k_new, v_new, slot_mapping, k_inv_scale, v_inv_scale):
    """In place on uint8 pools [num_blocks][Hkv][16][d]: row t of k_new/v_new
    (bf16 bits [T][Hkv][d]) goes to slot slot_mapping[t] (negative = skip)."""
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        b, r = divmod(slot, 16)
        k_pool[b, :, r, :] = quantize_bf16_rows(k_new[t], k_inv_scale)
        v_pool[b, :, r, :] = quantize_bf16_rows(v_new[t], v_inv_scale)


def decode_attention(k_pool, v_pool, q_bits, context_lens, block_tables, scale, k_scale, v_scale):
    """fp64 decode attention over dequantised fp8 pools: one query row per
    sequence ([B][Hq][d] bf16 bits), out [B][Hq][d] float64."""
    q = (np.asarray(q_bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)
    B, hq, d = q.shape
    hkv = k_pool.shape[1]
    G = hq // hkv
    out = np.zeros((B, hq, d), dtype=np.float64)
    for s in range(B):
        n = int(context_lens[s])
        if n == 0:
            continue
        pos = np.arange(n)
        blocks = np.asarray(block_tables[s])[pos // 16]
        K = value(k_pool[blocks, :, pos % 16, :]) * k_scale       # [n][Hkv][d]
        V = value(v_pool[blocks, :, pos % 16, :]) * v_scale
        for h in range(hq):
            x = scale * (K[:, h // G, :] @ q[s, h])
            w = np.exp(x - x.max())
            out[s, h] = (w @ V[:, h // G, :]) / w.sum()
    return out
