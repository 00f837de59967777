"""GPU parity of pkv_paged_extend_attn (suffix prefill over cached prefix
blocks) against the fp64 oracle: ragged suffixes spanning several 128-row
tiles, prefixes that end mid-block, GQA groups from 1 to 32 (powers of two and
others), head_dim 64 and 128, both block sizes, 16-bit and fp8 caches; the
1,900 + 100 case of the first page; the 256-request shared-prefix workload the
benchmark times (sampled rows); and the device-side length checks."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_285_gb300 as pkv
from paged_kv_cache_285_gb300 import workloads as W
from tests.pkv_testlib import BF16, E4M3, F16, assert_attention_close, to_f64

pytestmark = pytest.mark.gpu
S = W.to_numpy_storage


def gpu_extend(case, workspace="auto"):
    out = torch.full_like(case.q, float("nan"))
    rows, hq, _ = case.q.shape
    lse = torch.full((rows, hq), float("nan"), dtype=torch.float32, device="cuda")
    suf = (case.q_indptr[1:] - case.q_indptr[:-1]).cpu()
    tot = case.prefix_lens.cpu() + suf
    if isinstance(workspace, str):
        nbytes = pkv.extend_workspace_bytes(case.k_cache, int(suf.numel()), hq, rows, int(tot.max()),
                                            k_scale=case.k_scale, v_scale=case.v_scale)
        # filled with garbage: the call may not rely on its contents
        workspace = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda") if nbytes else None
    pkv.paged_extend_attn(case.k_cache, case.v_cache, case.q, out, case.q_indptr,
                          case.prefix_lens, case.block_tables, case.sm_scale,
                          int(suf.max()), int(tot.max()), k_scale=case.k_scale,
                          v_scale=case.v_scale, lse_out=lse, workspace=workspace)
    torch.cuda.synchronize()
    return out, lse


def check(case, out, lse, what, rows=None, fp8=False):
    args = (S(case.k_cache), S(case.v_cache), case.cache_dtype, case.k_scale, case.v_scale,
            S(case.q), case.act_dtype, case.q_indptr.cpu().numpy(), case.prefix_lens.cpu().numpy(),
            case.block_tables.cpu().numpy(), case.num_q_heads, case.sm_scale)
    ref, ref_lse, st = oracle.paged_extend(*args, rows=rows)
    assert st == 0
    got, gl = to_f64(out), lse.cpu().double().numpy()
    if rows is not None:
        got = np.stack([got[r, h] for r, h in rows])
        gl = np.array([gl[r, h] for r, h in rows])
    assert_attention_close(got, ref, case.act_dtype, fp8=fp8, what=what)
    assert np.max(np.abs(gl - ref_lse)) <= (3e-2 if fp8 else 1e-3), what


CASES = [
    # (prefix_lens, suffix_lens, hq, hkv, bs, dtype, head_dim)
    ([0], [5], 4, 1, 16, F16, 128),
    ([4], [1], 4, 1, 16, F16, 128),
    ([1900], [100], 32, 8, 16, BF16, 128),
    ([0, 13, 30, 200], [37, 19, 130, 1], 8, 2, 16, BF16, 128),
    ([100, 0], [300, 129], 8, 8, 32, F16, 128),
    ([17, 250], [64, 33], 16, 2, 16, BF16, 128),
    ([129, 64, 1], [200, 17, 256], 64, 8, 16, BF16, 128),
    ([500], [40], 4, 2, 32, BF16, 128),
    # requests with no suffix rows between others (equal q_indptr entries)
    ([40, 7, 0, 300, 0], [0, 50, 0, 3, 0], 8, 2, 16, BF16, 128),
    # GQA groups that are not powers of two (3, 6: tiles of 42 / 21 tokens) and above 8
    ([33, 0, 90], [70, 45, 130], 12, 4, 16, BF16, 128),
    ([200, 16], [50, 77], 24, 4, 32, F16, 128),
    ([64, 301], [40, 19], 64, 4, 16, BF16, 128),
    ([10], [37], 32, 1, 16, F16, 128),
    # the largest groups a 128-row tile takes: 2 tokens x 64 heads, 1 token x 128 heads
    ([40, 3], [9, 5], 128, 2, 16, BF16, 128),
    ([17, 0], [6, 3], 128, 1, 32, F16, 64),
    # head_dim 64: ragged, mid-block prefixes, groups 1 / 4 / 8, both block sizes
    ([0], [5], 4, 1, 16, F16, 64),
    ([4], [1], 4, 1, 16, F16, 64),
    ([1900], [100], 32, 8, 16, BF16, 64),
    ([0, 13, 30, 200], [37, 19, 130, 1], 8, 2, 16, BF16, 64),
    ([100, 0], [300, 129], 8, 8, 32, F16, 64),
    ([129, 64, 1], [200, 17, 256], 64, 8, 16, BF16, 64),
    ([37, 60, 16, 1], [20, 3, 64, 9], 4, 1, 16, F16, 64),
    ([500, 7], [40, 250], 24, 4, 32, BF16, 64),
]


@pytest.mark.parametrize("cfg", CASES,
                         ids=lambda c: f"P{c[0]}-S{c[1]}-h{c[2]}x{c[3]}-bs{c[4]}-d{c[5]}-hd{c[6]}")
def test_extend_small(cfg):
    P, Sx, hq, hkv, bs, dt, hd = cfg
    case = W.extend_case(P, Sx, hq, hkv, hd, bs, dt, dt, seed=sum(P) + sum(Sx) + hq + hd,
                         device="cuda")
    out, lse = gpu_extend(case)
    check(case, out, lse, str(cfg))
    assert pkv.get_device_error() == 0


def test_extend_with_no_suffix_rows_is_a_no_op():
    # every request fully cached: nothing to compute, nothing written, no error
    case = W.extend_case([33, 0, 200], [0, 0, 0], 8, 2, 128, 16, BF16, BF16, seed=9, device="cuda")
    assert case.q.shape[0] == 0
    out, lse = gpu_extend(case)
    assert out.shape[0] == 0 and lse.shape[0] == 0
    assert pkv.get_device_error() == 0


def test_extend_matches_full_prefill_rows():
    # 1,900 cached + 100 suffix == rows 1,900..1,999 of prefilling all 2,000 tokens
    ext = W.extend_case([1900], [100], 32, 8, 128, 16, BF16, BF16, seed=70, device="cuda")
    out_e, lse_e = gpu_extend(ext)
    full = W.PagedBatch  # same pool and table, prefix 0, 2,000 query rows
    q_full = torch.zeros((2000, 32, 128), dtype=torch.bfloat16, device="cuda")
    q_full[1900:] = ext.q
    pre = W.ExtendCase(k_cache=ext.k_cache, v_cache=ext.v_cache, cache_dtype=BF16, act_dtype=BF16,
                       k_scale=1.0, v_scale=1.0, block_tables=ext.block_tables, num_q_heads=32,
                       sm_scale=ext.sm_scale,
                       q_indptr=torch.tensor([0, 2000], dtype=torch.int32, device="cuda"),
                       prefix_lens=torch.tensor([0], dtype=torch.int32, device="cuda"), q=q_full)
    out_p, lse_p = gpu_extend(pre)
    del full
    a = to_f64(out_e)
    b = to_f64(out_p[1900:])
    assert np.max(np.abs(a - b)) <= 2e-3
    check(ext, out_e, lse_e, "1900+100")


def test_shared_prefix_extend_workload_sampled():
    # the benchmark's launch: 256 requests x 100 suffix rows over a shared 1,900-token prefix;
    # 2,048 (row, head) outputs: for 8 requests spread over the batch, every head (so every kv
    # head) of the first and last token of each 32-token row tile (both tiles of both pairs,
    # the 4-token tail tile included) against the oracle
    case = W.shared_prefix_extend(device="cuda")
    out, lse = gpu_extend(case)
    reqs = [0, 37, 64, 101, 128, 170, 211, 255]
    toks = [0, 31, 32, 63, 64, 95, 96, 99]
    rows = [(r * 100 + i, h) for r in reqs for i in toks for h in range(32)]
    assert len(rows) == 2048
    check(case, out, lse, "shared-prefix extend", rows=rows)
    assert pkv.get_device_error() == 0


@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8)], ids=["gqa4", "mha"])
def test_extend_many_items_mixed_lengths(hq, hkv):
    # Many more (request, kv head, row-tile pair) items than SMs, with key-tile
    # counts from 1 to dozens per item and many empty row tiles (short
    # suffixes next to long ones), so the persistent pipeline crosses item
    # boundaries of every kind; rows are sampled against the oracle.
    rng = np.random.default_rng(11)
    B = 40
    P = [int(x) for x in rng.integers(0, 3000, B)]
    P[0], P[1] = 0, 0
    Sx = [int(x) for x in rng.integers(1, 300, B)]
    Sx[2], Sx[3] = 1, 2
    case = W.extend_case(P, Sx, hq, hkv, 128, 16, BF16, BF16, seed=81 + hq, device="cuda")
    out, lse = gpu_extend(case)
    total_rows = case.q.shape[0]
    rows = [(int(r), int(h)) for r, h in zip(rng.integers(0, total_rows, 300), rng.integers(0, hq, 300))]
    # every request's first and last suffix row, too
    starts = case.q_indptr.cpu().numpy()
    for b in range(B):
        rows.append((int(starts[b]), int(rng.integers(0, hq))))
        rows.append((int(starts[b + 1]) - 1, int(rng.integers(0, hq))))
    check(case, out, lse, f"many items {hq}x{hkv}", rows=rows)
    assert pkv.get_device_error() == 0


def test_extend_after_bulk_append():
    # the step the benchmark times: append the suffix K/V, then extend over the pool
    case = W.extend_case([1900] * 4, [100] * 4, 32, 8, 128, 16, BF16, BF16, seed=71,
                         device="cuda", shared_prefix=1900)
    k0, v0 = S(case.k_cache), S(case.v_cache)
    pkv.kv_append(case.k_cache, case.v_cache, case.suffix_k, case.suffix_v, case.suffix_slots)
    out, lse = gpu_extend(case)
    kr, vr, st = oracle.kv_append(k0, v0, BF16, 1, 1, S(case.suffix_k), S(case.suffix_v), BF16,
                                  case.suffix_slots.cpu().numpy())
    assert st == 0
    ref, _, st = oracle.paged_extend(kr, vr, BF16, 1, 1, S(case.q), BF16, case.q_indptr.cpu().numpy(),
                                     case.prefix_lens.cpu().numpy(), case.block_tables.cpu().numpy(),
                                     32, case.sm_scale)
    assert st == 0
    assert_attention_close(to_f64(out), ref, BF16, what="append+extend")


def test_extend_garbage_past_end_is_ignored():
    case = W.extend_case([30], [20], 8, 2, 128, 16, BF16, BF16, seed=72, device="cuda")
    total = 50
    blk = int(case.block_tables[0, (total - 1) // 16])
    case.k_cache[blk, :, total % 16:] = float("inf")
    case.v_cache[blk, :, total % 16:] = float("nan")
    out, lse = gpu_extend(case)
    check(case, out, lse, "garbage tail")


FP8_CASES = [
    # (prefix_lens, suffix_lens, hq, hkv, bs, act dtype, head_dim)
    ([0, 13, 30, 200], [37, 19, 130, 1], 8, 2, 16, BF16, 128),
    ([1900], [100], 32, 8, 16, BF16, 128),
    ([100, 0], [300, 129], 8, 8, 32, F16, 128),
    ([129, 64, 1], [200, 17, 256], 64, 8, 16, BF16, 128),
    ([33, 0, 90], [70, 45, 130], 12, 4, 16, F16, 128),
    ([0, 13, 30, 200], [37, 19, 130, 1], 8, 2, 16, BF16, 64),
    ([1900], [100], 32, 8, 16, F16, 64),
    ([100, 0], [300, 129], 8, 8, 32, BF16, 64),
    ([129, 64, 1], [200, 17, 256], 64, 8, 16, F16, 64),
]


@pytest.mark.parametrize("cfg", FP8_CASES,
                         ids=lambda c: f"fp8-P{c[0]}-S{c[1]}-h{c[2]}x{c[3]}-bs{c[4]}-a{c[5]}-hd{c[6]}")
def test_extend_fp8_cache(cfg):
    # e4m3 pages with per-tensor scales, read as codes and widened inside the
    # kernel; vs the oracle on the same dequantised values, fp8 bound
    P, Sx, hq, hkv, bs, act, hd = cfg
    case = W.extend_case(P, Sx, hq, hkv, hd, bs, E4M3, act, seed=90 + sum(Sx) + hd, device="cuda")
    out, lse = gpu_extend(case)
    check(case, out, lse, "fp8 " + str(cfg), fp8=True)
    assert pkv.get_device_error() == 0


def test_extend_fp8_shared_prefix_many_requests():
    # 64 requests over one shared 1,900-token prefix in an fp8 pool; sampled rows
    case = W.extend_case([1900] * 64, [100] * 64, 32, 8, 128, 16, E4M3, BF16, seed=95,
                         device="cuda", shared_prefix=1900)
    out, lse = gpu_extend(case)
    rng = np.random.default_rng(5)
    rows = [(int(r), int(h)) for r, h in zip(rng.integers(0, case.q.shape[0], 256), rng.integers(0, 32, 256))]
    check(case, out, lse, "fp8 shared prefix", rows=rows, fp8=True)
    assert pkv.get_device_error() == 0


@pytest.mark.parametrize("hd", [128, 64])
def test_extend_fp8_garbage_past_end_is_ignored(hd):
    case = W.extend_case([30], [20], 8, 2, hd, 16, E4M3, BF16, seed=96, device="cuda")
    total = 50
    blk = int(case.block_tables[0, (total - 1) // 16])
    case.k_cache[blk, :, total % 16:] = 0x7F  # e4m3 NaN codes
    case.v_cache[blk, :, total % 16:] = 0xFF
    out, lse = gpu_extend(case)
    check(case, out, lse, "fp8 garbage tail", fp8=True)


def test_extend_needs_no_workspace():
    # every cache dtype is read in place: the workspace size is 0 and none is passed
    for dt, act in ((F16, F16), (BF16, BF16), (E4M3, BF16)):
        case = W.extend_case([16], [8], 8, 2, 128, 16, dt, act, seed=97, device="cuda")
        assert pkv.extend_workspace_bytes(case.k_cache, 1, 8, 8, 24, k_scale=case.k_scale,
                                          v_scale=case.v_scale) == 0
        out, lse = gpu_extend(case, workspace=None)
        check(case, out, lse, f"no workspace {dt}", fp8=(dt == E4M3))


def test_extend_unsupported_combinations_raise():
    case = W.extend_case([4], [4], 4, 1, 128, 16, BF16, BF16, seed=73, device="cuda")
    with pytest.raises(pkv.PkvError):  # f16 queries over a bf16 cache
        pkv.paged_extend_attn(case.k_cache, case.v_cache, case.q.half(), case.q.half(),
                              case.q_indptr, case.prefix_lens, case.block_tables, case.sm_scale,
                              4, 8)


def test_extend_rows_beyond_the_call_are_reported_not_written():
    # q_indptr[batch] larger than the call's rows: the request is not computed, the length
    # error is recorded and nothing past `out` is written (guard rows keep their value)
    case = W.extend_case([20, 30], [10, 12], 8, 2, 128, 16, BF16, BF16, seed=74, device="cuda")
    rows = case.q.shape[0]
    big = torch.full((rows + 16, 8, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    out = big[:rows]
    bad_indptr = case.q_indptr.clone()
    bad_indptr[2] = rows + 9
    pkv.get_device_error()  # clear
    pkv.paged_extend_attn(case.k_cache, case.v_cache, case.q, out, bad_indptr, case.prefix_lens,
                          case.block_tables, case.sm_scale, 21, 60)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 3
    assert bool(torch.all(big[rows:] == 7.0))
    # request 0 is intact and still computed
    ref, _, st = oracle.paged_extend(S(case.k_cache), S(case.v_cache), BF16, 1, 1, S(case.q), BF16,
                                     case.q_indptr.cpu().numpy(), case.prefix_lens.cpu().numpy(),
                                     case.block_tables.cpu().numpy(), 8, case.sm_scale,
                                     rows=[(r, h) for r in range(10) for h in range(8)])
    assert st == 0
    got = to_f64(out[:10]).reshape(80, 128)
    assert_attention_close(got, ref, BF16, what="request 0 beside a bad one")


def test_extend_suffix_longer_than_hint_is_reported():
    # max_suffix_len below the real suffix: the rows past the hint's tiles are not computed
    # and the device error word says so
    case = W.extend_case([40], [300], 8, 2, 128, 16, BF16, BF16, seed=75, device="cuda")
    out = torch.zeros_like(case.q)
    pkv.get_device_error()  # clear
    pkv.paged_extend_attn(case.k_cache, case.v_cache, case.q, out, case.q_indptr, case.prefix_lens,
                          case.block_tables, case.sm_scale, 100, 340)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 3
