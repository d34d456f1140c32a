"""Pins for the fp8 (e4m3) pool oracle (no GPU): the code table against the
format's definition in torch (float8_e4m3fn), rounding against brute force,
saturation, and attention over dequantised pools against the C oracle where
the dequantised values are exactly bf16."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
import pkv_workloads as W


def test_every_code_matches_torch_float8_e4m3fn():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = fp8.decode_codes()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[~np.isnan(got)], ref[~np.isnan(ref)])
    assert fp8.value([0x7E])[0] == 448.0 and fp8.value([0x01])[0] == 2.0 ** -9


def test_rounding_is_nearest_even_against_brute_force_and_torch():
    rng = np.random.default_rng(0)
    vals = fp8.decode_codes()[:127]                            # non-negative finite, increasing
    mids = (vals[:-1] + vals[1:]) / 2                          # every tie
    x = np.concatenate([rng.uniform(-460, 460, 4000), rng.normal(0, 0.01, 2000), mids, -mids, vals, -vals])
    got = fp8.encode(x)
    m = np.minimum(np.abs(x), 448.0)
    dist = np.abs(m[:, None] - vals[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = np.where(dist == best, np.arange(127)[None, :], 1 << 20)
    even = np.where(cand % 2 == 0, cand, 1 << 20).min(axis=1)
    brute = np.where(even < (1 << 20), even, cand.min(axis=1)) | np.where(np.signbit(x), 0x80, 0)
    assert np.array_equal(got, brute.astype(np.uint8))
    ok = np.abs(x) <= 448
    t = torch.tensor(x[ok], dtype=torch.float64).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got[ok], t)


def test_saturation_and_nan():
    assert fp8.encode([1000.0, -1e6, 448.1])[:].tolist() == [0x7E, 0xFE, 0x7E]
    assert fp8.encode([np.nan])[0] & 0x7F == 0x7F


def test_quantize_rounds_the_fp32_product_first():
    rng = np.random.default_rng(1)
    bits = W.normal_bf16(3, 1, 512)
    inv = np.float32(1 / 0.037)
    f = (bits.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(fp8.quantize_bf16_rows(bits, inv), fp8.encode((f * inv).astype(np.float32)))


def test_fp32_product_decides_a_tie():
    """x = 1.0078125 (bf16 0x3F81) times inv_scale = 1.0542635917663574 (an
    fp32 value) is 1.0625 + 2.6e-8 exactly, but rounds in fp32 to 1.0625, the
    midpoint of the e4m3 values 1.0 (code 0x38, even mantissa) and 1.125
    (0x39).  Rounding the fp32 product gives the even code; rounding the exact
    product would give 0x39.  The same with the sign bit set."""
    inv = np.float32(1.0542635917663574)
    x = np.float32(1.0078125)
    assert np.float32(x * inv) == np.float32(1.0625) and float(x) * float(inv) > 1.0625   # the premise
    codes = fp8.quantize_bf16_rows(np.array([0x3F81, 0xBF81], dtype=np.uint16), inv)
    assert codes.tolist() == [0x38, 0xB8]


@pytest.mark.parametrize("hq,hkv,d", [(16, 8, 128), (32, 8, 64)])
def test_fp8_attention_equals_the_c_oracle_on_bf16_exact_values(hq, hkv, d):
    """With power-of-two scales every dequantised value is exactly bf16, so
    attention over the fp8 pools must equal the C oracle over those bf16
    pools."""
    rng = np.random.default_rng(hq + d)
    NB, B = 24, 3
    k8 = rng.integers(0, 256, size=(NB, hkv, 16, d)).astype(np.uint8)
    v8 = rng.integers(0, 256, size=(NB, hkv, 16, d)).astype(np.uint8)
    k8[(k8 & 0x7F) == 0x7F] = 0x11                           # no NaN codes
    v8[(v8 & 0x7F) == 0x7F] = 0x22
    ks, vs = 2.0 ** -5, 2.0 ** -3
    ctx = np.array([37, 1, 100], np.int32)
    tables = rng.permutation(NB)[:3 * 8].reshape(B, 8).astype(np.int32)
    q = W.normal_bf16(5, 2, B * hq * d).reshape(B, hq, d)
    got = fp8.decode_attention(k8, v8, q, ctx, tables, 1 / np.sqrt(d), ks, vs)

    def to_bf16(codes, s):
        f = (fp8.value(codes) * s).astype(np.float32)
        return (f.view(np.uint32) >> 16).astype(np.uint16)   # exact: 3 mantissa bits
    kb, vb = to_bf16(k8, ks), to_bf16(v8, vs)
    assert np.array_equal((kb.astype(np.uint32) << 16).view(np.float32), (fp8.value(k8) * ks).astype(np.float32))
    ref = oracle.decode_attention(kb, vb, q, ctx, tables, 1 / np.sqrt(d))
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
