"""GPU tests of pkv_paged_extend_attn_append (the suffix's K/V written into the
cache by the same call, slots derived from the extend layout): the same
output bits and the same cache bytes as pkv_kv_append of the suffix followed
by pkv_paged_extend_attn, with the suffix slots holding NaN (16-bit) or
NaN codes (fp8) before the call (every row read must have been written); and
parity with the oracle, for head_dim 64 and 128 and fp8 caches.  "KV Cache에 대해 알아보자 (Feat.
Attention)", §3; "PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화",
section 03."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_285_gb300 as pkv
from paged_kv_cache_285_gb300 import workloads as W
from tests.pkv_testlib import BF16, E4M3, F16, assert_attention_close, to_f64

pytestmark = pytest.mark.gpu
S = W.to_numpy_storage


def poison_suffix(case):
    slots = case.suffix_slots.to(torch.int64)
    bs = case.block_size
    blk, off = slots // bs, slots % bs
    for pool in (case.k_cache, case.v_cache):
        pool[blk, :, off, :] = 0x7F if pool.dtype == torch.uint8 else float("nan")


def run(case, fused):
    suf = (case.q_indptr[1:] - case.q_indptr[:-1]).cpu()
    tot = suf + case.prefix_lens.cpu()
    out = torch.full_like(case.q, float("nan"))
    lse = torch.full(case.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    sc = dict(k_scale=case.k_scale, v_scale=case.v_scale)
    if fused:
        pkv.paged_extend_attn_append(case.k_cache, case.v_cache, case.suffix_k, case.suffix_v,
                                     case.q, out, case.q_indptr, case.prefix_lens,
                                     case.block_tables, case.sm_scale, int(suf.max()),
                                     int(tot.max()), lse_out=lse, **sc)
    else:
        pkv.kv_append(case.k_cache, case.v_cache, case.suffix_k, case.suffix_v, case.suffix_slots,
                      **sc)
        pkv.paged_extend_attn(case.k_cache, case.v_cache, case.q, out, case.q_indptr,
                              case.prefix_lens, case.block_tables, case.sm_scale, int(suf.max()),
                              int(tot.max()), lse_out=lse, **sc)
    torch.cuda.synchronize()
    return out, lse


CASES = [
    # (prefix_lens, suffix_lens, hq, hkv, bs, cache dtype, act dtype, head_dim)
    ([0], [5], 4, 1, 16, F16, F16, 128),
    ([1900], [100], 32, 8, 16, BF16, BF16, 128),
    ([0, 13, 30, 200], [37, 19, 130, 1], 8, 2, 16, BF16, BF16, 128),
    ([100, 0], [300, 129], 8, 8, 32, F16, F16, 128),
    ([129, 64, 1], [200, 17, 256], 64, 8, 16, BF16, BF16, 128),
    ([511, 7], [700, 64], 16, 4, 32, BF16, BF16, 128),
    # requests with no suffix rows: the slot search must skip them
    ([40, 7, 0, 300, 0], [0, 50, 0, 3, 0], 8, 2, 16, BF16, BF16, 128),
    # head_dim 64
    ([0, 13, 30, 200], [37, 19, 130, 1], 8, 2, 16, BF16, BF16, 64),
    ([100, 0], [300, 129], 4, 1, 32, F16, F16, 64),
    # fp8 caches: the suffix is stored as e4m3(x / scale), then read as codes
    ([1900], [100], 32, 8, 16, E4M3, BF16, 128),
    ([0, 13, 30, 200], [37, 19, 130, 1], 8, 2, 16, E4M3, F16, 128),
    ([129, 64, 1], [200, 17, 256], 64, 8, 32, E4M3, BF16, 64),
]


@pytest.mark.parametrize("cfg", CASES,
                         ids=lambda c: f"p{c[0]}-s{c[1]}-h{c[2]}x{c[3]}-bs{c[4]}-c{c[5]}a{c[6]}-hd{c[7]}")
def test_fused_append_equals_append_then_extend(cfg):
    pre, suf, hq, hkv, bs, dt, act, hd = cfg
    seed = sum(pre) + sum(suf) + hq + hd
    ref = W.extend_case(pre, suf, hq, hkv, hd, bs, dt, act, seed=seed, device="cuda")
    fus = W.extend_case(pre, suf, hq, hkv, hd, bs, dt, act, seed=seed, device="cuda")
    poison_suffix(ref)
    poison_suffix(fus)
    out_r, lse_r = run(ref, False)
    out_f, lse_f = run(fus, True)
    assert np.array_equal(S(ref.k_cache), S(fus.k_cache))
    assert np.array_equal(S(ref.v_cache), S(fus.v_cache))
    assert torch.equal(out_r.view(torch.int16), out_f.view(torch.int16))
    assert torch.equal(lse_r.view(torch.int32), lse_f.view(torch.int32))
    # and the oracle on the written pool
    r, rl, st = oracle.paged_extend(S(fus.k_cache), S(fus.v_cache), dt, fus.k_scale, fus.v_scale,
                                    S(fus.q), act, fus.q_indptr.cpu().numpy(),
                                    fus.prefix_lens.cpu().numpy(), fus.block_tables.cpu().numpy(),
                                    hq, fus.sm_scale)
    assert st == 0
    assert_attention_close(to_f64(out_f), r, act, fp8=(dt == E4M3), what=str(cfg))
    assert pkv.get_device_error() == 0


def test_fused_append_shared_prefix_extend_workload():
    # the benchmark's workload: 256 requests x 100 suffix tokens over a shared 1,900-token prefix
    a = W.shared_prefix_extend(device="cuda")
    b = W.shared_prefix_extend(device="cuda")
    poison_suffix(a)
    poison_suffix(b)
    out_r, _ = run(a, False)
    out_f, _ = run(b, True)
    assert torch.equal(out_r.view(torch.int16), out_f.view(torch.int16))
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(a.v_cache.view(torch.int16), b.v_cache.view(torch.int16))
    assert pkv.get_device_error() == 0


def test_fp8_suffix_matches_the_oracle_store():
    # the fused call's fp8 stores are the oracle's e4m3(fp32(x) / scale) codes, bit for bit
    c = W.extend_case([32, 7], [16, 40], 8, 2, 128, 16, E4M3, BF16, seed=3, device="cuda")
    k0, v0 = S(c.k_cache), S(c.v_cache)
    run(c, True)
    kr, vr, st = oracle.kv_append(k0, v0, E4M3, c.k_scale, c.v_scale, S(c.suffix_k),
                                  S(c.suffix_v), BF16, c.suffix_slots.cpu().numpy())
    assert st == 0
    assert np.array_equal(kr, S(c.k_cache)) and np.array_equal(vr, S(c.v_cache))
    assert pkv.get_device_error() == 0
