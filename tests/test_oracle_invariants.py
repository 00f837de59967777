"""Invariants the pages fix, checked on the fp64 oracle, plus a cross-check of
the C oracle against its independent NumPy twin.

* Reusing a prefix does not change model outputs ("PagedAttention과
  RadixAttention으로 LLM KV 캐시 최적화", section 05: both chain hashing and
  radix lookup skip the repeated prefill without changing outputs).  Hence:
  permuting physical blocks, sharing prefix blocks vs duplicating them, and
  reading a paged vs a contiguous cache all give identical results; extend over
  a 1,900-token cached prefix + 100-token suffix equals the last 100 rows of a
  full 2,000-token prefill (same page, section 03); and Request II, which reuses
  4 tokens of Request I and computes 1, matches row 5 of prefilling all five
  (same page, section 03, the "What day is it" figure).
"""
import numpy as np
import pytest

import oracle
from oracle import ref_numpy
from paged_kv_cache_285_gb300 import workloads as W
from tests.pkv_testlib import BF16, E4M3, F16


def np_case(case):
    s = W.to_numpy_storage
    return dict(k=s(case.k_cache), v=s(case.v_cache), q=s(case.q),
                tables=case.block_tables.cpu().numpy(), cdt=case.cache_dtype,
                adt=case.act_dtype, ks=case.k_scale, vs=case.v_scale, hq=case.num_q_heads,
                scale=case.sm_scale)


def decode_c(c, tables=None, k=None, v=None, lens=None):
    out, lse, st = oracle.paged_decode(c["k"] if k is None else k, c["v"] if v is None else v,
                                       c["cdt"], c["ks"], c["vs"], c["q"], c["adt"],
                                       c["tables"] if tables is None else tables, lens, c["hq"],
                                       c["scale"])
    assert st == 0
    return out, lse


@pytest.mark.parametrize("cdt,adt", [(F16, F16), (BF16, BF16), (E4M3, BF16)])
def test_block_permutation_invariance(cdt, adt):
    case = W.decode_case([37, 60, 16, 1, 45], 8, 2, 64, 16, cdt, adt, seed=11, pool_blocks=40)
    c = np_case(case)
    lens = case.seq_lens.numpy()
    out0, lse0 = decode_c(c, lens=lens)
    rng = np.random.default_rng(0)
    nb = c["k"].shape[0]
    perm = rng.permutation(nb)            # new block j holds old block perm[j]
    inv = np.empty_like(perm)
    inv[perm] = np.arange(nb)
    k2, v2 = c["k"][perm].copy(), c["v"][perm].copy()
    t2 = np.where(c["tables"] >= 0, inv[np.maximum(c["tables"], 0)], -1).astype(np.int32)
    out1, lse1 = decode_c(c, tables=t2, k=k2, v=v2, lens=lens)
    np.testing.assert_array_equal(out0, out1)
    np.testing.assert_array_equal(lse0, lse1)


def test_shared_prefix_equals_duplicated():
    # 6 requests share a 40-token prefix (2 full shared blocks + 8-token tail copied)
    case = W.decode_case([55, 70, 41, 90, 48, 64], 4, 1, 64, 16, F16, F16, seed=12,
                         shared_prefix=40)
    c = np_case(case)
    lens = case.seq_lens.numpy()
    t = c["tables"]
    assert np.all(t[:, :2] == t[0, :2]), "prefix blocks are shared"
    out0, _ = decode_c(c, lens=lens)
    # give every request private copies of the shared blocks
    k, v = list(c["k"]), list(c["v"])
    t2 = t.copy()
    for b in range(1, t.shape[0]):
        for j in range(2):
            k.append(c["k"][t[b, j]].copy())
            v.append(c["v"][t[b, j]].copy())
            t2[b, j] = len(k) - 1
    out1, _ = decode_c(c, tables=t2, k=np.stack(k), v=np.stack(v), lens=lens)
    np.testing.assert_array_equal(out0, out1)


def test_paged_equals_contiguous():
    case = W.decode_case([37, 60, 16, 1], 4, 1, 64, 16, F16, F16, seed=13, pool_blocks=64)
    c = np_case(case)
    lens = case.seq_lens.numpy()
    out0, lse0 = decode_c(c, lens=lens)
    # one block per request, block_size = the longest length: table = [b]
    bs = int(lens.max())
    n_b = len(lens)
    kc = np.zeros((n_b, 1, bs, 64), np.uint16)
    vc = np.zeros_like(kc)
    for b in range(n_b):
        for t in range(int(lens[b])):
            blk, off = c["tables"][b, t // 16], t % 16
            kc[b, 0, t] = c["k"][blk, 0, off]
            vc[b, 0, t] = c["v"][blk, 0, off]
    out1, lse1 = decode_c(c, tables=np.arange(n_b, dtype=np.int32)[:, None], k=kc, v=vc, lens=lens)
    np.testing.assert_array_equal(out0, out1)
    np.testing.assert_array_equal(lse0, lse1)


def test_extend_1900_plus_100_equals_full_prefill():
    # one request, 2,000 tokens: extend rows (prefix 1900) vs full prefill rows 1900..1999
    case = W.extend_case([1900], [100], 4, 1, 64, 16, BF16, BF16, seed=14)
    s = W.to_numpy_storage
    k, v = s(case.k_cache), s(case.v_cache)
    tables = case.block_tables.numpy()
    q_suffix = s(case.q)                                  # [100, 4, 64]
    out_ext, lse_ext, st = oracle.paged_extend(k, v, BF16, 1, 1, q_suffix, BF16,
                                               np.array([0, 100], np.int32),
                                               np.array([1900], np.int32), tables, 4, 0.125)
    assert st == 0
    # full prefill: 2,000 query rows, prefix 0; only rows 1900..1999 are evaluated
    q_full = np.zeros((2000, 4, 64), np.uint16)
    q_full[1900:] = q_suffix
    rows = np.array([(1900 + i, h) for i in range(100) for h in range(4)], np.int32)
    out_full, lse_full, st = oracle.paged_extend(k, v, BF16, 1, 1, q_full, BF16,
                                                 np.array([0, 2000], np.int32),
                                                 np.array([0], np.int32), tables, 4, 0.125,
                                                 rows=rows)
    assert st == 0
    np.testing.assert_array_equal(out_ext.reshape(-1, 64), out_full)
    np.testing.assert_array_equal(lse_ext.reshape(-1), lse_full)


def test_request_ii_reuses_four_tokens():
    # Request I computes 5 tokens; Request II reuses 4 and computes 1 (prefix 4, suffix 1)
    case = W.extend_case([0], [5], 2, 1, 64, 16, F16, F16, seed=15)
    s = W.to_numpy_storage
    k, v, q = s(case.k_cache), s(case.v_cache), s(case.q)
    tables = case.block_tables.numpy()
    out_i, _, st = oracle.paged_extend(k, v, F16, 1, 1, q, F16, np.array([0, 5], np.int32),
                                       np.array([0], np.int32), tables, 2, 0.125)
    assert st == 0
    out_ii, _, st = oracle.paged_extend(k, v, F16, 1, 1, q[4:5].copy(), F16,
                                        np.array([0, 1], np.int32), np.array([4], np.int32),
                                        tables, 2, 0.125)
    assert st == 0
    np.testing.assert_array_equal(out_i[4], out_ii[0])
    # and the last extend row equals a decode over all 5 tokens with the same query
    out_d, _, st = oracle.paged_decode(k, v, F16, 1, 1, q[4:5].copy(), F16, tables,
                                       np.array([5], np.int32), 2, 0.125)
    assert st == 0
    np.testing.assert_array_equal(out_i[4], out_d[0])


@pytest.mark.parametrize("cdt,adt,d,bs,hq,hkv", [
    (F16, F16, 64, 16, 4, 1), (BF16, BF16, 128, 16, 8, 2), (F16, F16, 128, 32, 4, 4),
    (E4M3, BF16, 128, 16, 8, 1), (E4M3, F16, 64, 32, 2, 1), (BF16, BF16, 64, 32, 8, 8),
])
def test_c_oracle_matches_numpy_twin(cdt, adt, d, bs, hq, hkv):
    lens = [1, 17, 40, 33, 16, 64]
    case = W.decode_case(lens, hq, hkv, d, bs, cdt, adt, seed=20 + d + bs + hq)
    c = np_case(case)
    out_c, lse_c = decode_c(c, lens=np.array(lens, np.int32))
    out_n, lse_n = ref_numpy.paged_decode(c["k"], c["v"], cdt, c["ks"], c["vs"], c["q"], adt,
                                          c["tables"], lens, hq, c["scale"])
    np.testing.assert_allclose(out_c, out_n, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_c, lse_n, rtol=0, atol=1e-12)
    ext = W.extend_case([0, 13, 30], [5, 19, 16], hq, hkv, d, bs, cdt, adt, seed=30 + d)
    s = W.to_numpy_storage
    args = (s(ext.k_cache), s(ext.v_cache), cdt, ext.k_scale, ext.v_scale, s(ext.q), adt,
            ext.q_indptr.numpy(), ext.prefix_lens.numpy(), ext.block_tables.numpy(), hq,
            ext.sm_scale)
    out_c, lse_c, st = oracle.paged_extend(*args)
    assert st == 0
    out_n, lse_n = ref_numpy.paged_extend(*args)
    np.testing.assert_allclose(out_c, out_n, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_c, lse_n, rtol=0, atol=1e-12)


def test_bad_block_id_is_reported():
    case = W.decode_case([20], 1, 1, 64, 16, F16, F16, seed=40, pool_blocks=4)
    c = np_case(case)
    t = c["tables"].copy()
    t[0, 1] = 99
    _, _, st = oracle.paged_decode(c["k"], c["v"], F16, 1, 1, c["q"], F16, t, np.array([20]), 1, 1.0)
    assert st == 1
