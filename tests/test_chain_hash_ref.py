"""Pins of the chain-hash oracle (oracle/chain_hash_ref.py): its mixing step
against the published SplitMix64 outputs, and the chaining properties the
pages state for block hashes ("PagedAttention과 RadixAttention으로 LLM KV 캐시
최적화", sections 05 and 06): equal token prefixes give equal chains, a change
in block j changes hash j and every later one but no earlier one, a salt
separates tenants, only full blocks are hashed."""
import random

from oracle import chain_hash_ref as ch


def test_mix_reproduces_published_splitmix64_outputs():
    # the first outputs of SplitMix64 seeded with 0, as published with the generator
    assert ch.splitmix64_stream(0, 3) == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_equal_prefixes_give_equal_chains():
    rnd = random.Random(1)
    pre = [rnd.randrange(0, 50000) for _ in range(64)]
    a = ch.chain(pre + [1, 2, 3, 4] * 4, 16)
    b = ch.chain(pre + [9, 9, 9, 9] * 4, 16)
    assert a[:4] == b[:4] and a[4] != b[4]


def test_change_in_one_block_changes_that_hash_and_all_later_ones():
    rnd = random.Random(2)
    t = [rnd.randrange(0, 50000) for _ in range(16 * 10)]
    h = ch.chain(t, 16)
    for j in (0, 3, 9):
        u = list(t)
        u[16 * j + 5] ^= 1
        g = ch.chain(u, 16)
        assert g[:j] == h[:j]
        assert all(x != y for x, y in zip(g[j:], h[j:]))


def test_salt_separates_tenants_and_partial_blocks_are_not_hashed():
    t = list(range(40))
    assert len(ch.chain(t, 16)) == 2 and ch.chain(t[:15], 16) == []
    a, b = ch.chain(t, 16, salt=1), ch.chain(t, 16, salt=2)
    assert all(x != y for x, y in zip(a, b))
    assert ch.chain(t, 16) == ch.chain(t, 16, salt=0)


def test_block_size_one_chain_is_a_fold_over_tokens():
    t = [5, 7, 11]
    h = 0
    for x in t:
        h = ch.mix(((h ^ ch.mix(0 + ch.G + x)) + ch.G) & ch.M64)
    assert ch.chain(t, 1)[-1] == h


def test_token_ids_enter_as_unsigned_32_bit_values():
    # an int32 token id is read as its unsigned 32-bit value, not sign-extended
    assert ch.chain([-1] * 4, 4) == ch.chain([0xFFFFFFFF] * 4, 4)
    assert ch.content([-1]) == ch.mix(ch.G + 0xFFFFFFFF)
    assert ch.content([-1]) != ch.mix((ch.G + ch.M64) & ch.M64)
