"""Prefix reuse end to end: requests sharing a system prompt go through the
host prefix index (match, allocate, append the suffix only, extend over the
matched prefix, insert, release), and every output row equals the oracle's
full causal prefill of the whole request on contiguous K/V -- reusing cached
KV does not change outputs ("PagedAttention과 RadixAttention으로 LLM KV 캐시
최적화", sections 03 and 05)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_285_gb300 as pkv
from paged_kv_cache_285_gb300 import workloads as W
from tests.pkv_testlib import BF16, assert_attention_close, to_f64

pytestmark = pytest.mark.gpu
S = W.to_numpy_storage


def kv_of(tokens, hkv, d, table_k, table_v):
    """Synthetic K/V rows of a token sequence: a fixed function of (token,
    position), so equal prefixes have equal K/V."""
    pos = np.arange(len(tokens))
    idx = (np.asarray(tokens) * 131 + pos * 7) % table_k.shape[0]
    return table_k[idx], table_v[idx]


def test_requests_through_the_prefix_index_match_full_prefill():
    rng = np.random.default_rng(21)
    hq, hkv, d, bs = 32, 8, 128, 16
    nb = 512
    gen = torch.Generator().manual_seed(21)
    table_k = torch.randn((997, hkv, d), generator=gen).to(torch.bfloat16)
    table_v = torch.randn((997, hkv, d), generator=gen).to(torch.bfloat16)
    k_cache = torch.zeros((nb, hkv, bs, d), dtype=torch.bfloat16, device="cuda")
    v_cache = torch.zeros_like(k_cache)
    index = pkv.RadixIndex(bs, nb)
    system = rng.integers(0, 5000, 300).tolist()
    sm_scale = 1.0 / np.sqrt(d)
    for r in range(8):
        q_tokens = rng.integers(0, 5000, int(rng.integers(1, 90))).tolist()
        tokens = system + q_tokens if r != 5 else system[:150] + q_tokens  # one diverges early
        L = len(tokens)
        m, blk = index.match(np.array(tokens, np.int32))
        new = index.alloc(-(-L // bs) - len(blk))
        table = np.concatenate([blk, new]).astype(np.int32)
        if r >= 1 and r != 5:
            assert m == (300 // bs) * bs  # 288: the full blocks of the system prompt
        # append the suffix (positions m .. L-1) only
        kk, vv = kv_of(tokens, hkv, d, table_k, table_v)
        pos = np.arange(m, L)
        slots = torch.tensor(table[pos // bs].astype(np.int64) * bs + pos % bs, device="cuda")
        pkv.kv_append(k_cache, v_cache, kk[pos].cuda(), vv[pos].cuda(), slots)
        # extend the suffix rows over the matched prefix
        q = torch.randn((L - m, hq, d), generator=gen).to(torch.bfloat16).cuda()
        out = torch.full_like(q, float("nan"))
        bt = torch.tensor(table[None, :], dtype=torch.int32, device="cuda")
        pkv.paged_extend_attn(k_cache, v_cache, q, out,
                              torch.tensor([0, L - m], dtype=torch.int32, device="cuda"),
                              torch.tensor([m], dtype=torch.int32, device="cuda"), bt, sm_scale,
                              L - m, L)
        torch.cuda.synchronize()
        # oracle: full causal prefill of all L tokens on contiguous K/V, last L-m rows
        nbl = -(-L // bs)
        kc = torch.zeros((nbl, hkv, bs, d), dtype=torch.bfloat16)
        vc = torch.zeros_like(kc)
        for p in range(L):
            kc[p // bs, :, p % bs] = kk[p]
            vc[p // bs, :, p % bs] = vv[p]
        q_full = torch.zeros((L, hq, d), dtype=torch.bfloat16)
        q_full[m:] = q.cpu()
        ref, _, st = oracle.paged_extend(S(kc), S(vc), BF16, 1.0, 1.0, S(q_full), BF16,
                                         np.array([0, L], np.int32), np.array([0], np.int32),
                                         np.arange(nbl, dtype=np.int32)[None, :], hq, sm_scale)
        assert st == 0
        assert_attention_close(to_f64(out), ref[m:], BF16, what=f"request {r}")
        index.insert(np.array(tokens, np.int32), table)
        index.release(np.array(tokens, np.int32), m)
        if L % bs:
            index.free(table[-1:])
    assert pkv.get_device_error() == 0
