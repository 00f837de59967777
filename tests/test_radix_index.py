"""Host prefix index (pkv_radix_*): the radix tree over token ids of
"PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", section 03, with
whole-block edges and leaf-first LRU eviction.

Pinned by the page's own examples (the "firm" insert next to dog, dot, pump,
fat, fire; a 1,900-token cached prefix of a 2,000-token request; 1,000
requests sharing one 1,000-token system prompt from "KV Cache 완전 정리",
RadixAttention section), by the eviction order the pages describe, and by a
brute-force model (longest whole-block common prefix against every stored
sequence) on random workloads."""
import numpy as np
import pytest

import paged_kv_cache_285_gb300 as pkv
from oracle.prefix_match_ref import common_blocks, longest_block_prefix

pytestmark = pytest.mark.filterwarnings("ignore")


def serve(x, tokens):
    """One request through the index: match, allocate the rest, insert, release.
    Returns (matched tokens, block table)."""
    bs = x.block_size
    m, blk = x.match(tokens)
    need = -(-len(tokens) // bs) - len(blk)
    new = x.alloc(need)
    table = np.concatenate([blk, new]).astype(np.int32)
    x.insert(tokens, table)
    x.release(tokens, m)
    if len(tokens) % bs:
        x.free(table[-1:])  # the partial tail block is not kept
    return m, table


def word(w):
    return [ord(c) for c in w]


def test_firm_insert_example():
    # the page's figure: dog, dot, pump, fat, fire in the tree; inserting "firm"
    # reuses f-i-r and adds a node for m
    x = pkv.RadixIndex(1, 64)
    for w in ["dog", "dot", "pump", "fat", "fire"]:
        serve(x, word(w))
    st = x.stats()
    # do|g|t, pump, f|at|ire: 14 token blocks on 7 edges, 5 leaves
    assert (st["tree_blocks"], st["nodes"], st["evictable_leaves"]) == (14, 7, 5)
    m, blk = x.match(word("firm"))
    assert m == 3  # f, i, r
    fire_m, fire_blk = x.match(word("fire"))
    assert fire_m == 4 and list(fire_blk[:3]) == list(blk)
    x.release(word("fire"), fire_m)
    x.release(word("firm"), m)
    serve(x, word("firm"))
    st = x.stats()
    # one new block (m); "ire" split into "ir" + "e", plus the new leaf "m"
    assert (st["tree_blocks"], st["nodes"], st["evictable_leaves"]) == (15, 9, 6)
    m, blk = x.match(word("firm"))
    assert m == 4 and list(blk[:3]) == list(fire_blk[:3])
    x.release(word("firm"), m)


def test_prefix_of_2000_token_request_block_rounded():
    # 1,900 of a 2,000-token request cached: with 16-token blocks the 118 full
    # blocks (1,888 tokens) are shared, the 12-token tail is recomputed
    rng = np.random.default_rng(0)
    prefix = rng.integers(0, 32000, 1900).astype(np.int32)
    x = pkv.RadixIndex(16, 1024)
    serve(x, prefix)
    req = np.concatenate([prefix, rng.integers(0, 32000, 100).astype(np.int32)])
    m, blk = x.match(req)
    assert m == 1888 and len(blk) == 118
    x.release(req, m)


def test_request_one_and_two_share_the_prefix():
    # Request I = prefix + suffix A, then Request II = prefix + suffix B reuses
    # KV(prefix) and prefills suffix B only
    rng = np.random.default_rng(1)
    pre = rng.integers(0, 100, 64).astype(np.int32)
    a = np.concatenate([pre, [1, 2, 3, 4, 5, 6, 7, 8]]).astype(np.int32)
    b = np.concatenate([pre, [9, 9, 9, 9, 9, 9, 9, 9]]).astype(np.int32)
    x = pkv.RadixIndex(8, 64)
    m1, t1 = serve(x, a)
    m2, t2 = serve(x, b)
    assert m1 == 0 and m2 == 64
    assert list(t1[:8]) == list(t2[:8]) and t1[8] != t2[8]


def test_chatbot_system_prompt_computed_once():
    # 1,000 requests, one shared 1,000-token system prompt + a different question
    # each: the prompt is prefilled once instead of 1,000 times (>= 99 % saved)
    rng = np.random.default_rng(2)
    system = rng.integers(0, 32000, 1000).astype(np.int32)
    x = pkv.RadixIndex(1, 1000 + 1000 * 20 + 16)
    prompt_prefill = 0
    for r in range(1000):
        q = rng.integers(0, 32000, 20).astype(np.int32)
        m, _ = serve(x, np.concatenate([system, q]))
        prompt_prefill += 1000 - min(m, 1000)
    assert prompt_prefill == 1000
    assert 1 - prompt_prefill / (1000 * 1000) >= 0.99


def test_leaf_first_lru_eviction_protects_shared_prefix_and_locks():
    x = pkv.RadixIndex(4, 12)
    shared = list(range(100, 108))           # 2 blocks, shared interior prefix
    a = shared + [1, 1, 1, 1]                # leaf A (1 block)
    b = shared + [2, 2, 2, 2]                # leaf B
    c = shared + [3, 3, 3, 3]                # leaf C
    for t in (a, b, c):
        serve(x, t)
    assert x.stats()["tree_blocks"] == 5
    # touch A and C: B is now the least recently used leaf
    for t in (a, c):
        m, _ = x.match(t)
        x.release(t, m)
    # hold C with a match (locked): it must survive any eviction
    mc, _ = x.match(c)
    got = x.alloc(7 + 1)  # 7 free blocks + 1 evicted
    assert len(got) == 8
    assert x.match(b)[0] == 8   # B's leaf went first; the shared prefix stayed
    x.release(b, 8)
    assert x.match(a)[0] == 12
    x.release(a, 12)
    # next: A (leaf), then nothing else is evictable while C holds the prefix
    got2 = x.alloc(1)
    assert x.match(a)[0] == 8
    x.release(a, 8)
    with pytest.raises(pkv.PkvError) as e:
        x.alloc(1)
    assert e.value.status == pkv.NO_SPACE
    assert x.match(c)[0] == 12  # still there
    x.release(c, 12)
    x.release(c, mc)
    # once unlocked, C goes, then the shared prefix (now a leaf)
    assert x.evict(3) == 3
    assert x.stats()["tree_blocks"] == 0
    x.free(np.concatenate([got, got2]))
    assert x.stats()["free_blocks"] == 12


def test_insert_releases_duplicate_blocks_and_rejects_bad_input():
    x = pkv.RadixIndex(4, 16)
    t = list(range(12))
    serve(x, t)
    # a second request computed the same 12 tokens in its own blocks without
    # matching: the tree keeps its blocks and frees the caller's
    own = x.alloc(3)
    rel = x.insert(t, own)
    assert sorted(rel) == sorted(own)
    assert x.stats()["caller_blocks"] == 0
    # free blocks, blocks listed twice, tree blocks freed by the caller: refused
    f = x.alloc(2)
    with pytest.raises(pkv.PkvError):
        x.insert(list(range(50, 58)), [f[0], f[0]])
    x.free(f)
    with pytest.raises(pkv.PkvError):
        x.insert(list(range(50, 58)), f)     # free blocks
    m, blk = x.match(t)
    with pytest.raises(pkv.PkvError):
        x.free(blk)                           # the tree's blocks
    with pytest.raises(pkv.PkvError):
        x.release(list(range(90, 94)), 4)     # a path nobody matched
    x.release(t, m)
    st = x.stats()
    assert st["free_blocks"] + st["tree_blocks"] + st["caller_blocks"] == 16


def test_brute_force_model_on_hand_cases():
    # the reference itself, on cases worked by hand
    assert common_blocks([1, 2, 3, 4, 5, 6], [1, 2, 3, 4, 9, 6], 2) == 2
    assert common_blocks([1, 2, 3], [1, 2, 3, 4], 2) == 1      # partial blocks never count
    assert common_blocks([7, 7], [8, 7], 1) == 0
    stored = [([1, 2, 3, 4], [10, 11]), ([1, 2, 3, 4, 5, 6], [20, 21, 22])]
    assert longest_block_prefix(stored, [1, 2, 3, 4, 5, 6, 7], 2) == (3, [20, 21, 22])
    assert longest_block_prefix(stored, [1, 2, 3, 4, 9, 9], 2) == (2, [10, 11])  # earliest wins
    assert longest_block_prefix(stored, [5, 5], 2) == (0, [])


def test_random_workload_against_brute_force_model():
    # without eviction (a pool large enough), every match equals the longest
    # whole-block common prefix with any sequence served before (the brute-force
    # reference in oracle/prefix_match_ref.py), and returns the blocks that
    # sequence was given; the pool is accounted exactly
    rng = np.random.default_rng(7)
    bs = 4
    x = pkv.RadixIndex(bs, 200000)
    stored = []   # (tokens, table) of every served sequence
    bases = [rng.integers(0, 5, rng.integers(0, 40)).astype(np.int32) for _ in range(12)]
    for it in range(600):
        base = bases[rng.integers(0, len(bases))]
        tail = rng.integers(0, 5, rng.integers(0, 30)).astype(np.int32)
        t = np.concatenate([base[: rng.integers(0, len(base) + 1)], tail]).astype(np.int32)
        best, best_blocks = longest_block_prefix(stored, t, bs)
        m, blk = x.match(t)
        assert m == best * bs, it
        assert list(blk) == best_blocks, it
        x.release(t, m)
        _, table = serve(x, t)
        stored.append((t, table))
        st = x.stats()
        assert st["free_blocks"] + st["tree_blocks"] + st["caller_blocks"] == 200000
        assert st["caller_blocks"] == 0


def test_random_workload_with_eviction_keeps_the_pool_consistent():
    rng = np.random.default_rng(9)
    bs = 4
    pool = 96
    x = pkv.RadixIndex(bs, pool)
    for it in range(2000):
        t = rng.integers(0, 4, rng.integers(1, 60)).astype(np.int32)
        try:
            m, table = serve(x, t)
        except pkv.PkvError as e:
            assert e.status == pkv.NO_SPACE
            # the matched path was locked before the allocation failed
            m, _ = x.match(t)
            x.release(t, m)
            x.release(t, m)
            continue
        st = x.stats()
        assert st["free_blocks"] + st["tree_blocks"] + st["caller_blocks"] == pool
        assert st["caller_blocks"] == 0 and st["tree_blocks"] <= pool
    # every tree block is unlocked and evictable at the end
    x.evict(pool)
    assert x.stats()["tree_blocks"] == 0 and x.stats()["free_blocks"] == pool


def test_native_trace_driver():
    # the C++ replay that bench.py reports (bench_native/radix_trace.cpp, built by the bench
    # against the library): runs the whole trace through the C ABI without an error, refuses
    # no request, and reuses the shared prompts
    import json
    import subprocess

    import bench
    from paged_kv_cache_285_gb300 import build as pkv_build
    pkv_build.build()
    exe = bench._build_radix_trace()
    assert exe is not None
    r = subprocess.run([exe, "3000"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    d = json.loads(r.stdout)
    assert d["requests"] == 3000 and d["refused"] == 0
    # 64 prompts of 1,000 tokens (62 whole blocks each) under 10..200 new tokens: once every
    # prompt is cached, about 992 of ~1,105 tokens of a request come from the index
    assert 0.8 < d["cached_token_frac"] < 0.9
