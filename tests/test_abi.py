"""The C ABI without a GPU: libpkv.so builds, loads, exports every symbol that
include/pkv.h declares, and rejects bad arguments on the host before it
touches CUDA."""
import ctypes
import os
import re

import pytest
import torch

import paged_kv_cache_285_gb300 as pkv
from paged_kv_cache_285_gb300 import build as pkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return pkv.load()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn), encoding="utf-8").read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert {"pkv_kv_append", "pkv_paged_decode_attn", "pkv_paged_extend_attn"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"libpkv.so does not export {n}"


def test_status_strings_and_version(lib):
    assert pkv.status_string(0) == "PKV_OK"
    assert pkv.status_string(3) == "PKV_ERR_WORKSPACE"
    assert pkv.status_string(99) == "PKV_ERR_UNKNOWN"
    assert pkv.version() == 20100


def _desc(**kw):
    d = dict(num_blocks=8, block_size=16, num_kv_heads=2, head_dim=128, cache_dtype=1,
             k_scale=1.0, v_scale=1.0)
    d.update(kw)
    return pkv.CacheDesc(**d)


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: every call below fails validation first


def _decode(lib, desc, hq=4, act=1, batch=2, splits=0, scale=0.1, ws=None, ws_bytes=0):
    return lib.pkv_paged_decode_attn(ctypes.byref(desc), FAKE, FAKE, FAKE, FAKE, act, FAKE, 4,
                                     FAKE, batch, hq, scale, 64, splits, None, ws, ws_bytes, None)


def test_decode_argument_errors(lib):
    assert _decode(lib, _desc(), hq=3) == 1                 # Hq % Hkv != 0
    assert _decode(lib, _desc(head_dim=96)) == 2            # unsupported head_dim
    assert _decode(lib, _desc(block_size=8)) == 2           # unsupported block size
    assert _decode(lib, _desc(num_blocks=0)) == 1
    assert _decode(lib, _desc(), act=0) == 2                # bf16 cache with f16 queries
    assert _decode(lib, _desc(), act=2) == 1                # fp8 is not an act dtype
    assert _decode(lib, _desc(cache_dtype=2, k_scale=0.0)) == 1   # fp8 needs scales > 0
    assert _decode(lib, _desc(), scale=float("nan")) == 1
    assert _decode(lib, _desc(), batch=-1) == 1
    assert _decode(lib, _desc(), batch=0) == 0              # empty batch: nothing to do
    assert lib.pkv_paged_decode_attn(None, FAKE, FAKE, FAKE, FAKE, 1, FAKE, 4, FAKE, 2, 4, 0.1,
                                     64, 0, None, None, 0, None) == 1


def test_append_argument_errors(lib):
    d = _desc()
    call = lambda desc, act=1, n=4, slots=FAKE: lib.pkv_kv_append(
        ctypes.byref(desc), FAKE, FAKE, FAKE, FAKE, act, slots, n, None)
    assert call(d, n=-1) == 1
    assert call(d, n=0) == 0
    assert call(d, act=0) == 2
    assert call(d, slots=None) == 1
    assert call(_desc(head_dim=80)) == 2


def test_extend_argument_errors(lib):
    d = _desc()
    r = lib.pkv_paged_extend_attn(ctypes.byref(d), FAKE, FAKE, FAKE, FAKE, 1, FAKE, FAKE, FAKE, 4,
                                  1, 3, 0.1, 10, 10, 100, None, None, 0, None)
    assert r == 1                                            # Hq % Hkv != 0
    ext = lambda desc, hq=4, act=1: lib.pkv_paged_extend_attn(
        ctypes.byref(desc), FAKE, FAKE, FAKE, FAKE, act, FAKE, FAKE, FAKE, 4, 1, hq, 0.1, 10, 10,
        100, None, None, 0, None)
    assert ext(_desc(), hq=2 * 129) == 2                     # GQA group above 128 rows
    assert ext(_desc(head_dim=96)) == 2                      # unsupported head_dim
    assert ext(_desc(), act=0) == 2                          # bf16 cache with f16 queries
    assert ext(_desc(), act=2) == 1                          # fp8 is not an act dtype
    # no dtype needs scratch: fp8 caches are widened inside the kernel
    for dt in (0, 1, 2):
        for hd in (64, 128):
            assert lib.pkv_extend_workspace_bytes(ctypes.byref(_desc(cache_dtype=dt, head_dim=hd)),
                                                  4, 8, 400, 2000) == 0


def test_decode_workspace_plan(lib):
    # forced 4 splits over max_seq_len 1000: 63 tiles of 16 -> 16 tiles (256 tokens) per
    # split -> 4 splits; partials 2*8*4*128 floats (256-byte aligned) + 2*8*4 LSE floats
    d = _desc()
    assert pkv.decode_workspace_bytes(torch_free_cache(d), 2, 8, 1000, num_splits=4) == \
        2 * 8 * 4 * 128 * 4 + 2 * 8 * 4 * 4
    assert pkv.decode_workspace_bytes(torch_free_cache(d), 2, 8, 1000, num_splits=1) == 0


class torch_free_cache:
    """Stand-in with the shape/dtype the binding reads (no device memory)."""
    def __init__(self, d):
        import torch
        self.shape = (d.num_blocks, d.num_kv_heads, d.block_size, d.head_dim)
        self.dtype = torch.bfloat16

    def dim(self):
        return 4


def _shared(lib, desc, hq=8, act=1, batch=2, groups=1, scale=0.1, ws=None, ws_bytes=0):
    return lib.pkv_paged_decode_attn_shared_prefix(
        ctypes.byref(desc), FAKE, FAKE, None, None, FAKE, FAKE, act, FAKE, 4, FAKE, batch, hq,
        scale, FAKE, FAKE, groups, 2, 64, 100, 0, None, ws, ws_bytes, None)


def test_shared_prefix_decode_argument_errors(lib):
    assert _shared(lib, _desc(), hq=2 * 129) == 2             # group above one 128-row tile
    assert _shared(lib, _desc(), act=0) == 2                  # bf16 cache with f16 queries
    assert _shared(lib, _desc(), scale=-0.1) == 1             # the prefix pass needs scale > 0
    assert _shared(lib, _desc(), hq=3) == 1                   # Hq % Hkv != 0
    assert _shared(lib, _desc(), groups=0) == 1               # requests but no group
    assert _shared(lib, _desc(), batch=0) == 0                # empty batch: nothing to do
    # forced 2 splits over the members' own tokens (bound 100, + 15 for the prefix rounded
    # down to whole blocks): 8 tiles -> 4 per split; slots = 2 + the prefix's
    d = _desc()
    # (+ 256-byte alignment, then one int2 span per request)
    assert lib.pkv_shared_prefix_decode_workspace_bytes(ctypes.byref(d), 2, 8, 100, 100, 2) == \
        2 * 8 * 3 * 128 * 4 + 256 + 2 * 8
    # a 1,000-token prefix bound: 4 chunks of 256 keys -> 4 prefix slots + 2 own splits
    assert lib.pkv_shared_prefix_decode_workspace_bytes(ctypes.byref(d), 2, 8, 1000, 100, 2) == \
        2 * 8 * 6 * 128 * 4 + 512 + 2 * 8
    # at most 8 prefix chunks, however long the prefix
    assert lib.pkv_shared_prefix_decode_workspace_bytes(ctypes.byref(d), 2, 8, 100000, 100, 2) == \
        2 * 8 * 10 * 128 * 4 + 768 + 2 * 8
    assert lib.pkv_shared_prefix_decode_workspace_bytes(ctypes.byref(d), 2, 8, -1, 100, 2) == 0


def test_chain_hash_and_extend_append_argument_errors(lib):
    call = lambda tokens=FAKE, indptr=FAKE, b=2, bs=16, hashes=FAKE, mb=8: lib.pkv_chain_hash(
        tokens, indptr, b, bs, None, hashes, mb, None)
    assert call(bs=0) == 1
    assert call(bs=5000) == 1
    assert call(b=-1) == 1
    assert call(b=0) == 0 and call(mb=0) == 0
    assert call(tokens=None) == 1
    import torch
    with pytest.raises(ValueError):  # int64 token ids: refused by the binding
        pkv.chain_hash(torch.zeros(4, dtype=torch.int64), torch.zeros(2, dtype=torch.int32), 16,
                       torch.zeros((1, 1), dtype=torch.int64))
    ext = lambda desc, kn=FAKE: lib.pkv_paged_extend_attn_append(
        ctypes.byref(desc), FAKE, FAKE, kn, kn, FAKE, FAKE, 1, FAKE, FAKE, FAKE, 4, 1, 4, 0.1, 10,
        10, 100, None, None)
    assert ext(_desc(head_dim=96)) == 2                       # unsupported head_dim
    assert ext(_desc(cache_dtype=2, v_scale=float("inf"))) == 1   # fp8 scales finite and > 0
    assert ext(_desc(), kn=None) == 1                         # the suffix K/V are required


def test_shared_prefix_extend_argument_errors(lib):
    # every case is refused (or empty) before anything is enqueued
    call = lambda batch=2, groups=1, rows=10, gi=FAKE, gs=FAKE, hq=8, scale=0.1, desc=None, \
        ws=None, ws_bytes=0: lib.pkv_paged_extend_attn_shared_prefix(
            ctypes.byref(desc or _desc()), FAKE, FAKE, FAKE, FAKE, 1, FAKE, FAKE, FAKE, 4, batch,
            hq, scale, 20, gi, gs, groups, rows, 100, None, ws, ws_bytes, None)
    assert call(groups=0) == 1                                # requests but no group
    assert call(groups=3) == 1                                # more groups than requests
    assert call(groups=-1) == 1
    assert call(rows=-1) == 1                                 # negative row bound
    assert call(gi=None) == 1 and call(gs=None) == 1          # the groups are required
    assert call(hq=3) == 1                                    # Hq % Hkv != 0
    assert call(scale=float("nan")) == 1
    assert call(desc=_desc(head_dim=96)) == 2                 # unsupported head_dim
    assert call(batch=0, groups=0) == 0                       # empty batch: nothing to do
    assert call(rows=0) == 0                                  # no rows in any group
    # the optional workspace of a bf16 cache: an f16 copy of the V pool, 256-byte aligned
    need = lib.pkv_extend_shared_prefix_workspace_bytes(ctypes.byref(_desc()))
    assert need == 8 * 2 * 16 * 128 * 2
    assert call(ws=FAKE, ws_bytes=need - 1) == 3              # too small
    assert call(ws=ctypes.c_void_p(0x10010), ws_bytes=need) == 3  # misaligned
    # an fp8 cache: f16 copies of its K and V pools; an f16 cache takes none
    assert lib.pkv_extend_shared_prefix_workspace_bytes(ctypes.byref(_desc(cache_dtype=2))) == \
        2 * 8 * 2 * 16 * 128 * 2
    assert call(desc=_desc(cache_dtype=2), ws=FAKE, ws_bytes=need) == 3  # too small for K and V
    assert lib.pkv_extend_shared_prefix_workspace_bytes(ctypes.byref(_desc(cache_dtype=0))) == 0
    assert lib.pkv_extend_shared_prefix_workspace_bytes(ctypes.byref(_desc(head_dim=96))) == 0


def test_plain_extend_widen_workspace_size(lib):
    # the pools of the shared-prefix workspace, then int32 claims (a counter, a
    # flag and a list entry per block) rounded up to 256 bytes; 0 where nothing
    # is widened
    pool = 8 * 2 * 16 * 128 * 2
    assert lib.pkv_extend_widen_workspace_bytes(ctypes.byref(_desc())) == pool + 256
    assert lib.pkv_extend_widen_workspace_bytes(ctypes.byref(_desc(num_blocks=100))) == \
        100 * 2 * 16 * 128 * 2 + 1024
    assert lib.pkv_extend_widen_workspace_bytes(ctypes.byref(_desc(cache_dtype=2))) == \
        2 * pool + 256
    assert lib.pkv_extend_widen_workspace_bytes(ctypes.byref(_desc(cache_dtype=0))) == 0
    assert lib.pkv_extend_widen_workspace_bytes(ctypes.byref(_desc(head_dim=96))) == 0
    # pkv_extend_workspace_bytes still asks for nothing: the widening is optional
    assert lib.pkv_extend_workspace_bytes(ctypes.byref(_desc(cache_dtype=2)), 2, 4, 10, 100) == 0


def test_binding_refuses_wrong_index_dtypes():
    import torch
    c = torch.zeros((4, 2, 16, 128), dtype=torch.bfloat16)
    q = torch.zeros((2, 4, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError):  # int64 block tables
        pkv.paged_decode_attn(c, c, q, q, torch.zeros((2, 4), dtype=torch.int64),
                              torch.zeros(2, dtype=torch.int32), 0.1, 64)
    with pytest.raises(ValueError):  # int32 slots
        pkv.kv_append(c, c, q, q, torch.zeros(2, dtype=torch.int32))
    with pytest.raises(ValueError):  # int64 prefix lengths
        pkv.paged_extend_attn(c, c, q, q, torch.zeros(3, dtype=torch.int32),
                              torch.zeros(2, dtype=torch.int64),
                              torch.zeros((2, 4), dtype=torch.int32), 0.1, 1, 64)


def test_binding_refuses_inconsistent_shapes(lib):
    # the C ABI takes bare pointers, so the binding checks every tensor against the others
    # before anything is launched (CPU tensors: consistent ones stop at the device check)
    c = torch.zeros((4, 2, 16, 128), dtype=torch.bfloat16)
    q = torch.zeros((3, 8, 128), dtype=torch.bfloat16)
    kn = torch.zeros((3, 2, 128), dtype=torch.bfloat16)
    bt = torch.zeros((3, 4), dtype=torch.int32)
    sl = torch.zeros(3, dtype=torch.int32)
    ip = torch.zeros(4, dtype=torch.int32)
    gi = torch.zeros(2, dtype=torch.int32)
    gp = torch.zeros(1, dtype=torch.int32)
    bad = [
        ("v_cache", lambda: pkv.paged_decode_attn(c, c[:3], q, q, bt, sl, 0.1, 64)),
        ("out", lambda: pkv.paged_decode_attn(c, c, q, q[:2], bt, sl, 0.1, 64)),
        ("out", lambda: pkv.paged_decode_attn(c, c, q, q.float(), bt, sl, 0.1, 64)),
        ("q", lambda: pkv.paged_decode_attn(c, c, q[..., :64], q[..., :64], bt, sl, 0.1, 64)),
        ("block_tables", lambda: pkv.paged_decode_attn(c, c, q, q, bt[:2], sl, 0.1, 64)),
        ("seq_lens", lambda: pkv.paged_decode_attn(c, c, q, q, bt, sl[:2], 0.1, 64)),
        ("lse_out", lambda: pkv.paged_decode_attn(c, c, q, q, bt, sl, 0.1, 64,
                                                  lse_out=torch.zeros((3, 7)))),
        ("k_new", lambda: pkv.paged_decode_attn_append(c, c, kn[:2], kn[:2], q, q, bt, sl, 0.1, 64)),
        ("seq_lens", lambda: pkv.paged_decode_attn_noalloc(c, c, q, q, bt, sl[:2], 0.1, 64)),
        ("k_new", lambda: pkv.paged_decode_attn_shared_prefix(c, c, q, q, bt, sl, 0.1, gi, gp, 3, 32,
                                                              64, k_new=kn[:1], v_new=kn[:1])),
        ("k_new", lambda: pkv.kv_append(c, c, kn, kn, torch.zeros(2, dtype=torch.int64))),
        ("v_new", lambda: pkv.kv_append(c, c, kn, kn.half(), torch.zeros(3, dtype=torch.int64))),
        ("q_indptr", lambda: pkv.paged_extend_attn(c, c, q, q, ip[:3], sl, bt, 0.1, 8, 64)),
        ("block_tables", lambda: pkv.paged_extend_attn(c, c, q, q, ip, sl, bt[:1], 0.1, 8, 64)),
        ("k_new", lambda: pkv.paged_extend_attn_append(c, c, kn[:2], kn[:2], q, q, ip, sl, bt, 0.1,
                                                       8, 64)),
    ]
    for name, call in bad:
        with pytest.raises(ValueError, match=name):
            call()
    with pytest.raises(ValueError, match="device tensors"):
        pkv.paged_decode_attn(c, c, q, q, bt, sl, 0.1, 64)
    with pytest.raises(ValueError, match="device tensors"):
        pkv.paged_extend_attn_append(c, c, kn, kn, q, q, ip, sl, bt, 0.1, 8, 64)
