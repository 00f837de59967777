"""Pins of the oracle's element codecs against independent implementations.

The fp16/bf16 decoders are checked on all 65,536 bit patterns against NumPy's
float16 and PyTorch's bfloat16; the e4m3 decoder on all 256 codes against
PyTorch's float8_e4m3fn; the encoder against PyTorch's cast on in-range
values (including every tie between neighbouring codes) and against
hand-worked saturation, subnormal and tie cases.  The pages name the format
only ("KV Cache 완전 정리 — PagedAttention vs RadixAttention, SGLang이 빠른
이유", section "FP8 KV 캐시": --kv-cache-dtype fp8_e4m3).
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _same(a, b):
    return (math.isnan(a) and math.isnan(b)) or a == b


def test_f16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    for i in range(0, 65536, 1):
        assert _same(oracle.f16_to_double(int(bits[i])), float(ref[i])), hex(i)


def test_bf16_decode_exhaustive():
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    for i in range(65536):
        assert _same(oracle.bf16_to_double(i), float(ref[i])), hex(i)


def test_e4m3_decode_exhaustive():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        assert _same(oracle.e4m3_to_double(c), float(ref[c])), hex(c)
    # the format's landmarks
    assert oracle.e4m3_to_double(0x7E) == 448.0
    assert oracle.e4m3_to_double(0x08) == 2.0 ** -6
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9
    assert oracle.e4m3_to_double(0x38) == 1.0
    assert math.isnan(oracle.e4m3_to_double(0x7F)) and math.isnan(oracle.e4m3_to_double(0xFF))


def test_e4m3_encode_matches_torch_in_range():
    finite = [oracle.e4m3_to_double(c) for c in range(256) if not math.isnan(oracle.e4m3_to_double(c))]
    finite = sorted(set(finite))
    mids = [(a + b) / 2 for a, b in zip(finite[:-1], finite[1:])]
    rng = np.random.default_rng(0)
    rand = list(rng.uniform(-448, 448, 4000)) + list(rng.normal(0, 1, 4000)) + \
        list(rng.normal(0, 0.01, 2000))
    vals = np.array(finite + mids + rand, dtype=np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for x, r in zip(vals, ref):
        got = oracle.e4m3_from_float(float(x))
        if x == 0.0:  # sign of zero is kept
            assert got == (0x80 if math.copysign(1.0, float(x)) < 0 else 0x00)
            continue
        assert got == int(r), (float(x), hex(got), hex(int(r)))


@pytest.mark.parametrize("x,code", [
    (1.0, 0x38), (-1.0, 0xB8), (0.0, 0x00), (-0.0, 0x80),
    (448.0, 0x7E), (449.0, 0x7E), (464.0, 0x7E), (480.0, 0x7E), (1e30, 0x7E),
    (float("inf"), 0x7E), (float("-inf"), 0xFE), (-1000.0, 0xFE),
    (2.0 ** -9, 0x01), (2.0 ** -10, 0x00),          # tie 0 | 2^-9 -> even 0
    (3 * 2.0 ** -10, 0x02),                          # tie 2^-9 | 2^-8 -> even (m=2)
    (7 * 2.0 ** -9, 0x07), (2.0 ** -6, 0x08),         # largest subnormal, smallest normal
    (1.0625, 0x38), (1.1875, 0x3A),                  # ties within a binade go to even mantissa
    (2.0 ** -20, 0x00), (float("nan"), 0x7F),
])
def test_e4m3_encode_hand_cases(x, code):
    assert oracle.e4m3_from_float(x) == code


def test_div_f32_is_correctly_rounded():
    rng = np.random.default_rng(1)
    x = rng.normal(0, 10, 5000).astype(np.float32)
    s = np.abs(rng.normal(0, 1, 5000)).astype(np.float32) + np.float32(1e-3)
    ref = (x / s).astype(np.float32)  # NumPy float32 division is IEEE round-to-nearest
    for a, b, r in zip(x, s, ref):
        assert oracle.div_f32(float(a), float(b)) == float(r)
