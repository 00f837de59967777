"""The roofline numerators of bench.py (algorithmic bytes and useful flops) against figures
worked by hand from the workloads' definitions."""
from types import SimpleNamespace

import torch

import bench
from paged_kv_cache_285_gb300 import workloads as W


def _case(lens, hq, hkv, d, bs, cache_dtype):
    b = len(lens)
    return SimpleNamespace(q=torch.zeros((b, hq, d)), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                           block_size=bs, cache_dtype=cache_dtype,
                           seq_lens=torch.tensor(lens, dtype=torch.int32))


def test_tiny_decode_step_bytes():
    # 4 requests {37, 60, 16, 1}, 4 q / 1 kv head, d64, fp16, bs16: K+V = 114 tokens x 256 B;
    # q and out 2 x 4 x 4 x 64 x 2 B; 3 + 4 + 1 + 1 = 9 block ids and 4 lengths (4 B each);
    # the append of one token per request: K and V rows read and written (2 B each) + an 8 B slot
    append, decode = bench.decode_step_bytes(_case([37, 60, 16, 1], 4, 1, 64, 16, W.F16))
    assert decode == 114 * 256 + 4096 + 9 * 4 + 4 * 4
    assert append == 4 * 1 * 64 * (2 + 2) * 2 + 4 * 8


def test_llama3_layer_bytes_per_token():
    # Llama-3-8B-shaped layer (8 kv heads, d128, bf16): 4,096 B of K+V per cached token, which
    # over 32 layers is the pages' 128 KiB per token
    lens = [1000, 3000]
    _, decode = bench.decode_step_bytes(_case(lens, 32, 8, 128, 16, W.BF16))
    fixed = 2 * 2 * 32 * 128 * 2 + 4 * (63 + 188) + 4 * 2
    assert decode - fixed == 4000 * 4096
    assert 4096 * 32 == 128 * 1024
    # an fp8 cache halves the K/V bytes
    _, d8 = bench.decode_step_bytes(_case(lens, 32, 8, 128, 16, W.E4M3))
    assert d8 - fixed == 4000 * 2048


def test_extend_useful_flops():
    # 1,900 cached + 100 computed tokens: rows see 1,901 .. 2,000 keys, 195,050 in all;
    # 4 x 128 x 32 x 195,050 = 3.196 GFLOP per request, 818.1 GFLOP for 256 requests
    assert sum(range(1901, 2001)) == 195_050
    assert bench.extend_useful_flops([1900], [100], 32, 128) == 4 * 128 * 32 * 195_050
    assert bench.extend_useful_flops([1900] * 256, [100] * 256, 32, 128) == 818_098_995_200
    # no prefix: a causal prefill of n rows sees n (n + 1) / 2 keys
    assert bench.extend_useful_flops([0, 5], [10, 0], 1, 1) == 4 * 55
