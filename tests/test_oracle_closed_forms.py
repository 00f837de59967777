"""Closed-form pins of both fp64 oracles (C and NumPy).

Each case has an answer worked by hand from softmax(QK^T/sqrt(d_k))V
("KV Cache에 대해 알아보자 (Feat. Attention)", §1), chosen so that a dropped
scale, a swapped K/V, a wrong GQA head mapping, a wrong block-table index or a
causal off-by-one gives a different number.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import ref_numpy
from tests.pkv_testlib import BF16, E4M3, F16, bits_of, empty_pool, put_sequence


def run_decode(impl, k, v, cdt, ks, vs, q, qdt, tables, lens, hq, scale):
    if impl == "c":
        out, lse, st = oracle.paged_decode(k, v, cdt, ks, vs, q, qdt, tables, lens, hq, scale)
        assert st == 0
        return out, lse
    return ref_numpy.paged_decode(k, v, cdt, ks, vs, q, qdt, tables, lens, hq, scale)


def run_extend(impl, k, v, cdt, ks, vs, q, qdt, indptr, prefix, tables, hq, scale):
    if impl == "c":
        out, lse, st = oracle.paged_extend(k, v, cdt, ks, vs, q, qdt, indptr, prefix, tables, hq,
                                           scale)
        assert st == 0
        return out, lse
    return ref_numpy.paged_extend(k, v, cdt, ks, vs, q, qdt, indptr, prefix, tables, hq, scale)


IMPLS = ["c", "numpy"]


@pytest.mark.parametrize("impl", IMPLS)
def test_single_token_returns_its_value(impl):
    # one cached token: softmax weight 1, out = v, lse = the one score
    d = 64
    k = empty_pool(4, 1, 16, d, F16)
    v = empty_pool(4, 1, 16, d, F16)
    kv = np.linspace(-1, 1, d)
    vv = np.linspace(2, -3, d)
    table = np.array([[2, -1]], np.int32)
    put_sequence(k, table[0], 0, bits_of(kv[None, :], F16))
    put_sequence(v, table[0], 0, bits_of(vv[None, :], F16))
    qv = np.full((1, 1, d), 0.5)
    q = bits_of(qv, F16)
    out, lse = run_decode(impl, k, v, F16, 1, 1, q, F16, table, [1], 1, 0.125)
    vexp = np.float16(vv).astype(np.float64)
    np.testing.assert_array_equal(out[0, 0], vexp)
    s = 0.125 * float(np.dot(np.float16(qv[0, 0]).astype(np.float64), np.float16(kv).astype(np.float64)))
    assert lse[0, 0] == pytest.approx(s, abs=1e-12)


@pytest.mark.parametrize("impl", IMPLS)
def test_zero_query_is_mean_of_values(impl):
    # q = 0: all scores equal, weights 1/n, out = mean of V, lse = ln n
    rng = np.random.default_rng(3)
    n, d = 37, 64
    k = empty_pool(8, 1, 16, d, BF16)
    v = empty_pool(8, 1, 16, d, BF16)
    table = np.array([[5, 0, 3, -1]], np.int32)
    vals = rng.normal(size=(n, d))
    put_sequence(k, table[0], 0, bits_of(rng.normal(size=(n, d)), BF16))
    vb = bits_of(vals, BF16)
    put_sequence(v, table[0], 0, vb)
    q = bits_of(np.zeros((1, 2, d)), BF16)
    out, lse = run_decode(impl, k, v, BF16, 1, 1, q, BF16, table, [n], 2, 0.125)
    vdec = ref_numpy.decode_storage(vb, BF16)
    np.testing.assert_allclose(out[0, 0], vdec.mean(axis=0), rtol=0, atol=1e-13)
    np.testing.assert_allclose(out[0, 1], vdec.mean(axis=0), rtol=0, atol=1e-13)
    assert lse[0, 0] == pytest.approx(math.log(n), abs=1e-12)


@pytest.mark.parametrize("impl", IMPLS)
def test_two_keys_sigmoid(impl):
    # two keys: out = sig(s1-s0) v1 + sig(s0-s1) v0, s_i = scale * q.k_i
    d = 64
    k = empty_pool(4, 1, 16, d, F16)
    v = empty_pool(4, 1, 16, d, F16)
    table = np.array([[1]], np.int32)
    k0 = np.zeros(d); k0[0] = 1.0
    k1 = np.zeros(d); k1[1] = 2.0
    v0 = np.zeros(d); v0[3] = 4.0
    v1 = np.zeros(d); v1[3] = -2.0; v1[5] = 1.0
    put_sequence(k, table[0], 0, bits_of(np.stack([k0, k1]), F16))
    put_sequence(v, table[0], 0, bits_of(np.stack([v0, v1]), F16))
    qv = np.zeros((1, 1, d)); qv[0, 0, 0] = 3.0; qv[0, 0, 1] = 0.5
    scale = 0.5
    out, lse = run_decode(impl, k, v, F16, 1, 1, bits_of(qv, F16), F16, table, [2], 1, scale)
    s0, s1 = scale * 3.0, scale * 1.0          # q.k0 = 3, q.k1 = 1
    w1 = 1.0 / (1.0 + math.exp(s0 - s1))
    expect = w1 * v1 + (1 - w1) * v0
    np.testing.assert_allclose(out[0, 0], expect, rtol=0, atol=1e-14)
    assert lse[0, 0] == pytest.approx(math.log(math.exp(s0) + math.exp(s1)), abs=1e-13)


@pytest.mark.parametrize("impl", IMPLS)
def test_dominant_key(impl):
    # a score gap of 80: the weight of every other key is below e^-80
    d = 64
    rng = np.random.default_rng(5)
    n = 20
    keys = np.zeros((n, d))
    keys[7, 0] = 8.0
    vals = rng.normal(size=(n, d))
    k = empty_pool(4, 1, 16, d, F16)
    v = empty_pool(4, 1, 16, d, F16)
    table = np.array([[3, 0]], np.int32)
    put_sequence(k, table[0], 0, bits_of(keys, F16))
    vb = bits_of(vals, F16)
    put_sequence(v, table[0], 0, vb)
    qv = np.zeros((1, 1, d)); qv[0, 0, 0] = 10.0
    out, _ = run_decode(impl, k, v, F16, 1, 1, bits_of(qv, F16), F16, table, [n], 1, 1.0)
    np.testing.assert_allclose(out[0, 0], ref_numpy.decode_storage(vb[7], F16), atol=1e-25)


@pytest.mark.parametrize("impl", IMPLS)
def test_gqa_head_mapping(impl):
    # V of kv head g is the constant c_g everywhere, so out[h] = c_{h // (Hq/Hkv)}
    # for any q and K: 8 q heads over 2 kv heads -> heads 0-3 read kv 0, 4-7 read kv 1.
    rng = np.random.default_rng(7)
    d, n, hkv, hq = 64, 23, 2, 8
    k = empty_pool(6, hkv, 16, d, F16)
    v = empty_pool(6, hkv, 16, d, F16)
    table = np.array([[4, 1]], np.int32)
    consts = [0.25, -1.5]
    for g in range(hkv):
        put_sequence(k, table[0], g, bits_of(rng.normal(size=(n, d)), F16))
        put_sequence(v, table[0], g, bits_of(np.full((n, d), consts[g]), F16))
    q = bits_of(rng.normal(size=(1, hq, d)), F16)
    out, _ = run_decode(impl, k, v, F16, 1, 1, q, F16, table, [n], hq, 0.125)
    for h in range(hq):
        np.testing.assert_allclose(out[0, h], consts[h // 4], rtol=0, atol=1e-14)


@pytest.mark.parametrize("impl", IMPLS)
def test_fp8_codes_times_scale(impl):
    # every K code 0x38 (1.0), V code 0x40 (2.0): keys equal -> out = 2 * v_scale
    d = 64
    k = np.full((2, 1, 16, d), 0x38, np.uint8)
    v = np.full((2, 1, 16, d), 0x40, np.uint8)
    table = np.array([[1, 0]], np.int32)
    q = bits_of(np.ones((1, 1, d)), BF16)
    out, lse = run_decode(impl, k, v, E4M3, 0.5, 0.25, q, BF16, table, [20], 1, 0.125)
    np.testing.assert_allclose(out[0, 0], 0.5, rtol=0, atol=1e-15)
    # every score is 0.125 * 64 * 0.5 = 4, so lse = 4 + ln 20
    assert lse[0, 0] == pytest.approx(4.0 + math.log(20), abs=1e-12)


@pytest.mark.parametrize("impl", IMPLS)
def test_block_table_order_matters(impl):
    # tokens are read in LOGICAL order through the table: with q = 0 the output
    # is the mean, so use a decreasing causal case instead: extend row i sees
    # tokens 0..P+i; token values are their logical index.
    d = 64
    k = empty_pool(8, 1, 16, d, F16)
    v = empty_pool(8, 1, 16, d, F16)
    table = np.array([[7, 1, 3]], np.int32)
    n = 40
    vals = np.repeat(np.arange(n, dtype=np.float64)[:, None], d, axis=1)
    put_sequence(k, table[0], 0, bits_of(np.zeros((n, d)), F16))
    put_sequence(v, table[0], 0, bits_of(vals, F16))
    q = bits_of(np.zeros((3, 1, d)), F16)
    # prefix 17 (ends one token into physical block 1), suffix rows at positions 17, 18, 19
    out, _ = run_extend(impl, k, v, F16, 1, 1, q, F16, np.array([0, 3], np.int32),
                        np.array([17], np.int32), table, 1, 0.125)
    for i in range(3):
        npos = 17 + i + 1
        np.testing.assert_allclose(out[i, 0], (npos - 1) / 2.0, rtol=0, atol=1e-13)


@pytest.mark.parametrize("impl", IMPLS)
def test_causal_first_rows(impl):
    # prefill of 2 tokens (prefix 0): row 0 sees only token 0 -> v0;
    # row 1 sees both -> the two-key sigmoid.
    d = 64
    k = empty_pool(2, 1, 16, d, F16)
    v = empty_pool(2, 1, 16, d, F16)
    table = np.array([[1]], np.int32)
    k0 = np.zeros(d); k0[2] = 1.0
    k1 = np.zeros(d); k1[2] = -1.0
    v0 = np.full(d, 1.0)
    v1 = np.full(d, -1.0)
    put_sequence(k, table[0], 0, bits_of(np.stack([k0, k1]), F16))
    put_sequence(v, table[0], 0, bits_of(np.stack([v0, v1]), F16))
    qv = np.zeros((2, 1, d)); qv[:, 0, 2] = 2.0
    out, _ = run_extend(impl, k, v, F16, 1, 1, bits_of(qv, F16), F16, np.array([0, 2], np.int32),
                        np.array([0], np.int32), table, 1, 1.0)
    np.testing.assert_allclose(out[0, 0], v0, atol=1e-15)
    w1 = 1.0 / (1.0 + math.exp(2.0 - (-2.0)))
    np.testing.assert_allclose(out[1, 0], w1 * v1 + (1 - w1) * v0, atol=1e-14)


@pytest.mark.parametrize("impl", IMPLS)
def test_empty_sequence(impl):
    d = 64
    k = empty_pool(2, 1, 16, d, F16)
    v = empty_pool(2, 1, 16, d, F16)
    table = np.array([[0], [1]], np.int32)
    q = bits_of(np.ones((2, 1, d)), F16)
    out, lse = run_decode(impl, k, v, F16, 1, 1, q, F16, table, [0, 0], 1, 1.0)
    assert np.all(out == 0)
    assert np.all(np.isneginf(lse))
