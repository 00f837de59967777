"""Pins from figures the pages print: KV sizing arithmetic and the block-table
diagram, plus hand-worked append (slot scatter and fp8 store) cases."""
import os

import numpy as np
import pytest

import oracle
from paged_kv_cache_285_gb300 import workloads as W
from tests.pkv_testlib import BF16, E4M3, F16, bits_of, empty_pool

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
UNITS = {"B": 1.0, "KiB": 1024.0, "kB": 1000.0, "GB": 1e9, "GiB": 2.0 ** 30,
         "MIXED": 1024.0 * 1e6}


def _sizing_rows():
    rows = []
    with open(os.path.join(GOLDEN, "kv_sizing.txt"), encoding="utf-8") as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            parts = [p.strip() for p in line.split("|")]
            rows.append(parts)
    return rows


@pytest.mark.parametrize("row", _sizing_rows(), ids=lambda r: r[0])
def test_printed_kv_sizes(row):
    name, layers, heads, hd, elem, tokens, printed, unit, decimals, _src = row
    per_tok = oracle.kv_bytes_per_token(int(layers), int(heads), int(hd), int(elem))
    total = per_tok * int(tokens)
    value = total / UNITS[unit]
    assert round(value, int(decimals)) == pytest.approx(float(printed), abs=1e-9), (name, value)


def test_fp8_halves_the_cache():
    # "KV 캐시를 FP16 대신 FP8로 저장하면 메모리를 절반으로" -- section "FP8 KV 캐시"
    assert oracle.kv_bytes_per_token(80, 8, 128, 1) * 2 == oracle.kv_bytes_per_token(80, 8, 128, 2)


def test_only_needed_blocks_are_allocated():
    # a 60-token request gets only the blocks it needs (first page, section 02)
    tables, nb = W._alloc_tables([60], 16, None, __import__("torch").Generator().manual_seed(0))
    assert nb == 4 and int((tables >= 0).sum()) == 4
    tables, nb = W._alloc_tables([60], 32, None, __import__("torch").Generator().manual_seed(0))
    assert nb == 2


def _block_figure():
    with open(os.path.join(GOLDEN, "block_table_7_1_3.txt"), encoding="utf-8") as f:
        lines = [l.split() for l in f if l.strip() and not l.startswith("#")]
    bs = int(lines[0][1])
    table = [int(x) for x in lines[1][1:]]
    rows = [tuple(int(x) for x in l) for l in lines[2:]]
    return bs, table, rows


def test_block_figure_gather_and_append():
    bs, table, rows = _block_figure()
    d = 64
    # append: write token t (value t+1 in every lane) at its hand-worked slot
    k = empty_pool(8, 1, bs, d, F16, fill=-7.0)
    v = empty_pool(8, 1, bs, d, F16, fill=-7.0)
    toks = [r[0] for r in rows]
    new = bits_of(np.repeat(np.array(toks, np.float64)[:, None] + 1, d, axis=1)[:, None, :], F16)
    slots = np.array([r[3] for r in rows], np.int64)
    k2, v2, st = oracle.kv_append(k, v, F16, 1, 1, new, new, F16, slots)
    assert st == 0
    expect = k.copy()
    for (t, blk, off, _slot), val in zip(rows, new[:, 0, :]):
        expect[blk, 0, off] = val
    np.testing.assert_array_equal(k2, expect)   # nothing else touched
    np.testing.assert_array_equal(v2, expect)
    # gather: decode over 48 tokens with q = 0 returns the mean of the values that
    # the table maps, in logical order -- place value t at (table[t//16], t%16)
    vals = np.zeros((8, 1, bs, d))
    for t in range(48):
        vals[table[t // bs], 0, t % bs] = t
    vb = bits_of(vals, F16)
    q = bits_of(np.zeros((1, 1, d)), F16)
    tab = np.array([table], np.int32)
    for n in (1, 16, 17, 40, 48):
        out, _, st = oracle.paged_decode(vb, vb, F16, 1, 1, q, F16, tab, np.array([n]), 1, 1.0)
        assert st == 0
        np.testing.assert_allclose(out[0, 0], (n - 1) / 2.0, atol=1e-13)


def test_append_skips_negative_and_reports_out_of_pool():
    d = 64
    k = empty_pool(2, 2, 16, d, BF16, fill=3.0)
    v = empty_pool(2, 2, 16, d, BF16, fill=3.0)
    new = bits_of(np.ones((3, 2, d)), BF16)
    k2, v2, st = oracle.kv_append(k, v, BF16, 1, 1, new, new, BF16,
                                  np.array([-1, 5 * 16, 17], np.int64))
    assert st == 1
    expect = k.copy()
    expect[1, :, 1, :] = new[2]
    np.testing.assert_array_equal(k2, expect)


@pytest.mark.parametrize("act", [F16, BF16])
def test_fp8_append_hand_codes(act):
    d = 64
    k = empty_pool(1, 1, 16, d, E4M3)
    v = empty_pool(1, 1, 16, d, E4M3)
    # x / scale:  1.0/0.5 = 2 -> 0x40;  -3.0/0.5 = -6 -> 0xCC;  300/0.5 = 600 -> 448 (0x7E);
    #             0.03125/0.5 = 2^-4 -> 0x18;  2^-12/0.5 = 2^-11, below half of 2^-9 -> 0
    xs = np.zeros((1, 1, d))
    xs[0, 0, :5] = [1.0, -3.0, 300.0, 0.03125, 2.0 ** -12]
    new = bits_of(xs, act)
    k2, v2, st = oracle.kv_append(k, v, E4M3, 0.5, 2.0, new, new, act, np.array([0], np.int64))
    assert st == 0
    assert list(k2[0, 0, 0, :5]) == [0x40, 0xCC, 0x7E, 0x18, 0x00]
    # v_scale 2: 1/2 = 0.5 -> 0x30; -3/2 = -1.5 -> 0xBC; 300/2 = 150 lies between
    # 144 = 1.125*2^7 and 160 = 1.25*2^7, nearer 144: exponent field 7+7 = 14, mantissa 1 -> 0x71;
    # 0.03125/2 = 2^-6 -> 0x08
    assert list(v2[0, 0, 0, :4]) == [0x30, 0xBC, 0x71, 0x08]
