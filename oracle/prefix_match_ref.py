"""Longest cached prefix at block granularity, plain Python -- TEST INFRASTRUCTURE.

Only tests/ may import this module; the host prefix index (pkv_radix_*) shares
no code with it.

"PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", section 03: a new
request reuses the KV of the longest prefix it shares with requests served
before and prefills only the rest; with paged KV only whole blocks can be
shared.  This is that definition written out by brute force: compare the
request's tokens block by block with every stored sequence and keep the
longest run of equal whole blocks, with the physical blocks the first
sequence that holds that run was given.
"""
from __future__ import annotations


def common_blocks(a, b, block_size: int) -> int:
    """Number of leading whole blocks on which token lists a and b agree."""
    n = min(len(a), len(b)) // block_size
    k = 0
    while k < n and list(a[k * block_size:(k + 1) * block_size]) == \
            list(b[k * block_size:(k + 1) * block_size]):
        k += 1
    return k


def longest_block_prefix(stored, tokens, block_size: int):
    """stored: [(tokens, block_table)] in the order they were served.  Returns
    (matched whole blocks, their physical blocks) -- the blocks of the earliest
    stored sequence that reaches the longest match."""
    best, best_table = 0, None
    for seq, table in stored:
        k = common_blocks(seq, tokens, block_size)
        if k > best:
            best, best_table = k, table
    return best, ([] if best_table is None else list(best_table[:best]))
