"""GPU tests of pkv_paged_extend_attn_append (the suffix's K/V written into the
cache by the same call, slots derived from the extend layout): the same
output bits and the same cache bytes as pkv_kv_append of the suffix followed
by pkv_paged_extend_attn, with the suffix slots holding NaN before the call
(every row read must have been written); and parity with the oracle.  "KV Cache에 대해 알아보자 (Feat.
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
        pool[blk, :, off, :] = float("nan")


def run(case, fused):
    suf = (case.q_indptr[1:] - case.q_indptr[:-1]).cpu()
    tot = suf + case.prefix_lens.cpu()
    out = torch.full_like(case.q, float("nan"))
    lse = torch.full(case.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    if fused:
        pkv.paged_extend_attn_append(case.k_cache, case.v_cache, case.suffix_k, case.suffix_v,
                                     case.q, out, case.q_indptr, case.prefix_lens,
                                     case.block_tables, case.sm_scale, int(suf.max()),
                                     int(tot.max()), lse_out=lse)
    else:
        pkv.kv_append(case.k_cache, case.v_cache, case.suffix_k, case.suffix_v, case.suffix_slots)
        pkv.paged_extend_attn(case.k_cache, case.v_cache, case.q, out, case.q_indptr,
                              case.prefix_lens, case.block_tables, case.sm_scale, int(suf.max()),
                              int(tot.max()), lse_out=lse)
    torch.cuda.synchronize()
    return out, lse


CASES = [
    # (prefix_lens, suffix_lens, hq, hkv, bs, dtype)
    ([0], [5], 4, 1, 16, F16),
    ([1900], [100], 32, 8, 16, BF16),
    ([0, 13, 30, 200], [37, 19, 130, 1], 8, 2, 16, BF16),
    ([100, 0], [300, 129], 8, 8, 32, F16),
    ([129, 64, 1], [200, 17, 256], 64, 8, 16, BF16),
    ([511, 7], [700, 64], 16, 4, 32, BF16),
    # requests with no suffix rows: the slot search must skip them
    ([40, 7, 0, 300, 0], [0, 50, 0, 3, 0], 8, 2, 16, BF16),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: f"p{c[0]}-s{c[1]}-h{c[2]}x{c[3]}-bs{c[4]}-d{c[5]}")
def test_fused_append_equals_append_then_extend(cfg):
    pre, suf, hq, hkv, bs, dt = cfg
    seed = sum(pre) + sum(suf) + hq
    ref = W.extend_case(pre, suf, hq, hkv, 128, bs, dt, dt, seed=seed, device="cuda")
    fus = W.extend_case(pre, suf, hq, hkv, 128, bs, dt, dt, seed=seed, device="cuda")
    poison_suffix(ref)
    poison_suffix(fus)
    out_r, lse_r = run(ref, False)
    out_f, lse_f = run(fus, True)
    assert np.array_equal(S(ref.k_cache), S(fus.k_cache))
    assert np.array_equal(S(ref.v_cache), S(fus.v_cache))
    assert torch.equal(out_r.view(torch.int16), out_f.view(torch.int16))
    assert torch.equal(lse_r.view(torch.int32), lse_f.view(torch.int32))
    # and the oracle on the written pool
    r, rl, st = oracle.paged_extend(S(fus.k_cache), S(fus.v_cache), dt, 1, 1, S(fus.q), dt,
                                    fus.q_indptr.cpu().numpy(), fus.prefix_lens.cpu().numpy(),
                                    fus.block_tables.cpu().numpy(), hq, fus.sm_scale)
    assert st == 0
    assert_attention_close(to_f64(out_f), r, dt, what=str(cfg))
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


def test_fp8_cache_is_refused():
    c = W.extend_case([32], [16], 8, 2, 128, 16, E4M3, BF16, seed=3, device="cuda")
    kn = torch.zeros((16, 2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_extend_attn_append(c.k_cache, c.v_cache, kn, kn, c.q, torch.empty_like(c.q),
                                     c.q_indptr, c.prefix_lens, c.block_tables, c.sm_scale, 16, 48)
    assert e.value.status == 2
