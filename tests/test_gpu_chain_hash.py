"""GPU parity of pkv_chain_hash against the oracle (oracle/chain_hash_ref.py):
bit-exact block hashes for several block sizes, salts, empty and partial
requests, a request with more blocks than one pass of the kernel covers, and
the max_blocks bound."""
import numpy as np
import pytest
import torch

import paged_kv_cache_285_gb300 as pkv
from oracle import chain_hash_ref as ch

pytestmark = pytest.mark.gpu


def run(seqs, bs, salts=None, max_blocks=None):
    lens = [len(s) for s in seqs]
    indptr = np.zeros(len(seqs) + 1, np.int32)
    indptr[1:] = np.cumsum(lens)
    toks = np.concatenate([np.asarray(s, np.int32) for s in seqs]) if sum(lens) else np.zeros(1, np.int32)
    mb = max_blocks if max_blocks is not None else max(1, max(l // bs for l in lens))
    sentinel = -7
    hashes = torch.full((len(seqs), mb), sentinel, dtype=torch.int64, device="cuda")
    salt_t = None
    if salts is not None:
        salt_t = torch.tensor(np.array(salts, dtype=np.uint64).view(np.int64), device="cuda")
    pkv.chain_hash(torch.tensor(toks, device="cuda"), torch.tensor(indptr, device="cuda"), bs, hashes,
                   salts=salt_t)
    torch.cuda.synchronize()
    return hashes.cpu().numpy().view(np.uint64), sentinel


@pytest.mark.parametrize("bs", [1, 16, 32])
def test_chain_hash_matches_oracle(bs):
    rng = np.random.default_rng(bs)
    seqs = [rng.integers(-2**31, 2**31 - 1, int(n), dtype=np.int64).astype(np.int32).tolist()
            for n in rng.integers(0, 700, 12)]
    seqs[0] = []
    seqs[1] = seqs[2][: len(seqs[2]) // 2]           # a prefix of another request
    salts = [int(x) for x in rng.integers(0, 2**63, 12)]
    salts[3] = 0
    got, sentinel = run(seqs, bs, salts)
    for b, s in enumerate(seqs):
        ref = ch.chain(s, bs, salts[b])
        assert [int(v) for v in got[b, :len(ref)]] == ref, b
        assert np.all(got[b, len(ref):].view(np.int64) == sentinel)


def test_long_request_spans_several_kernel_passes():
    rng = np.random.default_rng(5)
    s = rng.integers(0, 50000, 16 * 1000).astype(np.int32).tolist()  # 1,000 blocks
    got, _ = run([s, s[:16 * 300 + 7]], 16, [11, 11])
    ref = ch.chain(s, 16, 11)
    assert [int(v) for v in got[0]] == ref
    assert [int(v) for v in got[1, :300]] == ref[:300]


def test_max_blocks_bound_is_reported():
    s = list(range(64))
    got, _ = run([s], 16, max_blocks=2)
    assert [int(v) for v in got[0]] == ch.chain(s, 16)[:2]
    assert pkv.get_device_error() == 5


@pytest.mark.parametrize("bs", [129, 4096])
def test_odd_and_large_block_sizes(bs):
    # chunks hold at most 16,384 tokens, so large blocks take few per chunk
    rng = np.random.default_rng(bs)
    seqs = [rng.integers(0, 2**31 - 1, n).astype(np.int32).tolist() for n in (bs * 5 + 3, bs * 200, bs - 1)]
    got, sentinel = run(seqs, bs, [1, 2, 3])
    for b, s in enumerate(seqs):
        ref = ch.chain(s, bs, b + 1)
        assert [int(v) for v in got[b, :len(ref)]] == ref, b
        assert np.all(got[b, len(ref):].view(np.int64) == sentinel)
