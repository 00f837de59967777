"""Chain hashes of full KV blocks, plain Python -- TEST INFRASTRUCTURE.

Only tests/ may import this module; the CUDA library shares no code with it.

"PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", section 05: a block's
identifier combines its parent's, its own token ids and optional extra data
(a salt, section 06).  The pages fix no hash function; the one here is the
library's documented definition (pkv.h, pkv_chain_hash), written out step by
step with explicit 64-bit wraparound:

    G = 0x9E3779B97F4A7C15
    mix(z): the SplitMix64 finalizer
    content(block) = c after c = mix(c + G + (uint32)t) for every token t, c0 = 0
    h[0] = mix((salt ^ content(block 0)) + G);  h[i] = mix((h[i-1] ^ content(block i)) + G)
"""
from __future__ import annotations

M64 = (1 << 64) - 1
G = 0x9E3779B97F4A7C15


def mix(z: int) -> int:
    """SplitMix64's output function (Steele, Lea, Flood 2014; constants of Vigna's
    published version)."""
    z &= M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def splitmix64_stream(seed: int, n: int):
    """The SplitMix64 generator: state += G, output mix(state)."""
    s = seed & M64
    out = []
    for _ in range(n):
        s = (s + G) & M64
        out.append(mix(s))
    return out


def content(block_tokens) -> int:
    c = 0
    for t in block_tokens:
        c = mix(c + G + (int(t) & 0xFFFFFFFF))
    return c


def chain(tokens, block_size: int, salt: int = 0):
    """Hashes of the full blocks of one request's token ids, in order."""
    h = salt & M64
    out = []
    for i in range(len(tokens) // block_size):
        h = mix(((h ^ content(tokens[i * block_size:(i + 1) * block_size])) + G) & M64)
        out.append(h)
    return out
