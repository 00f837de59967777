"""Seeded synthetic inputs for paged-KV attention.

This module draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA library's tests/benchmark and the fp64
oracle take their inputs from here, and nothing here calls either of them.

Shapes follow the examples on the pages:
  * tiny decode: 4 requests of 37/60/16/1 tokens, blocks drawn at random from a
    64-block pool ("PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화",
    section 02: a request only gets the blocks it needs; the block table maps
    logical blocks to scattered physical ones such as 7, 1, 3);
  * a Llama-3-8B-shaped layer (32 q heads, 8 kv heads, d128, same page,
    section 01);
  * a batch that shares one system-prompt prefix ("KV Cache 완전 정리 —
    PagedAttention vs RadixAttention, SGLang이 빠른 이유", section
    "RadixAttention — SGLang의 혁신": 1,000-token shared prompt, different
    questions) and a 1,900-token cached prefix + 100-token suffix (first page,
    section 03);
  * a 100,000-token, 32-layer long context (first page, section 01);
  * an fp8_e4m3 Llama-2-70B-shaped layer (64 q / 8 kv heads,
    "KV Cache에 대해 알아보자 (Feat. Attention)", §4).

Conventions: cache [num_blocks, Hkv, block_size, D]; q [tokens, Hq, D];
block_tables int32 [B, max_blocks]; seq_lens int32 [B]; slot of position p of
request b = block_tables[b][p // bs] * bs + p % bs (the slot-mapping input
format); -1 marks a slot to skip.  fp8 pools are stored as uint8 codes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

F16, BF16, E4M3 = 0, 1, 2
TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16, E4M3: torch.uint8}
DTYPE_NAME = {F16: "f16", BF16: "bf16", E4M3: "fp8_e4m3"}
ELEM_BYTES = {F16: 2, BF16: 2, E4M3: 1}


@dataclass
class PagedBatch:
    """A paged KV pool plus per-request block tables (one layer)."""
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    cache_dtype: int
    act_dtype: int
    k_scale: float
    v_scale: float
    block_tables: torch.Tensor
    num_q_heads: int
    sm_scale: float
    meta: dict = field(default_factory=dict)

    @property
    def num_blocks(self):
        return self.k_cache.shape[0]

    @property
    def num_kv_heads(self):
        return self.k_cache.shape[1]

    @property
    def block_size(self):
        return self.k_cache.shape[2]

    @property
    def head_dim(self):
        return self.k_cache.shape[3]


@dataclass
class DecodeCase(PagedBatch):
    seq_lens: torch.Tensor = None          # int32 [B], current token included
    q: torch.Tensor = None                 # [B, Hq, D] act dtype
    new_k: torch.Tensor = None             # [B, Hkv, D] act dtype: the current token's K
    new_v: torch.Tensor = None
    slot_last: torch.Tensor = None         # int64 [B]: slot of position seq_len-1
    slot_next: torch.Tensor = None         # int64 [B]: slot of position seq_len (or -1)


@dataclass
class ExtendCase(PagedBatch):
    q_indptr: torch.Tensor = None          # int32 [B+1]
    prefix_lens: torch.Tensor = None       # int32 [B]
    q: torch.Tensor = None                 # [sum S, Hq, D]
    suffix_k: torch.Tensor = None          # [sum S, Hkv, D] act dtype
    suffix_v: torch.Tensor = None
    suffix_slots: torch.Tensor = None      # int64 [sum S]


def _normal(shape, gen, device, scale=1.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x


def _fill_pool(nb, hkv, bs, d, dtype, gen, device, value_scale=1.0, chunk_blocks=4096):
    """Pool of N(0,1)*value_scale values.  fp8: codes of x / (amax/448), plus that scale."""
    if dtype != E4M3:
        out = torch.empty((nb, hkv, bs, d), dtype=TORCH_DTYPE[dtype], device=device)
        for s in range(0, nb, chunk_blocks):
            e = min(nb, s + chunk_blocks)
            out[s:e] = _normal((e - s, hkv, bs, d), gen, device, value_scale).to(out.dtype)
        return out, 1.0
    x = _normal((nb, hkv, bs, d), gen, device, value_scale)
    amax = float(x.abs().max())
    scale = amax / 448.0 if amax > 0 else 1.0
    codes = (x / scale).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes.contiguous(), scale


def _alloc_tables(caps, bs, pool_blocks, perm_gen, shared_blocks=0, max_blocks=None):
    """Host block allocator: every request gets ceil(cap/bs) blocks, the first
    `shared_blocks` of them common to all requests, the rest private; physical
    ids are drawn without replacement from a random permutation of the pool."""
    need = [max(0, math.ceil(c / bs)) for c in caps]
    private = sum(max(0, n - shared_blocks) for n in need)
    total = shared_blocks + private
    if pool_blocks is None:
        pool_blocks = total
    if total > pool_blocks:
        raise ValueError(f"pool of {pool_blocks} blocks cannot hold {total}")
    perm = torch.randperm(pool_blocks, generator=perm_gen).to(torch.int32)
    width = max_blocks if max_blocks is not None else max(1, max(need) if need else 1)
    tables = torch.full((len(caps), width), -1, dtype=torch.int32)
    shared = perm[:shared_blocks]
    nxt = shared_blocks
    for b, n in enumerate(need):
        k = min(n, shared_blocks)
        tables[b, :k] = shared[:k]
        m = n - k
        tables[b, k:n] = perm[nxt:nxt + m]
        nxt += m
    return tables, pool_blocks


def _slots(tables, positions, bs):
    pos = positions.to(torch.int64)
    width = tables.shape[1]
    lb = pos // bs
    inside = (pos >= 0) & (lb < width)
    blk = tables.to(torch.int64).gather(1, lb.clamp(0, width - 1)[:, None])[:, 0]
    slot = blk * bs + pos % bs
    return torch.where(inside & (blk >= 0), slot, torch.full_like(slot, -1))


def context_slots(case):
    """Slot of every cached position of a decode case, request by request
    (position t of request b -> block_tables[b][t // bs] * bs + t % bs): the
    slot mapping of a kv_append that fills each request's whole context."""
    lens = case.seq_lens.to(torch.int64)
    bs = case.k_cache.shape[2]
    starts = torch.cumsum(lens, 0) - lens
    rows_b = torch.repeat_interleave(torch.arange(lens.numel(), device=lens.device), lens)
    pos = torch.arange(rows_b.numel(), device=lens.device) - starts[rows_b]
    blk = case.block_tables.to(torch.int64)[rows_b, pos // bs]
    return blk * bs + pos % bs


def _replicate_prefix_tail(case_k, case_v, tables, prefix, bs):
    """Same K/V for the prefix's tail tokens in every request's private block."""
    tail = prefix % bs
    if tail == 0:
        return
    lb = prefix // bs
    src = int(tables[0, lb])
    for b in range(1, tables.shape[0]):
        dst = int(tables[b, lb])
        case_k[dst, :, :tail] = case_k[src, :, :tail]
        case_v[dst, :, :tail] = case_v[src, :, :tail]


def decode_case(seq_lens, num_q_heads, num_kv_heads, head_dim, block_size, cache_dtype,
                act_dtype, seed, device="cpu", pool_blocks=None, value_scale=1.0,
                shared_prefix=0, extra_capacity=1, sm_scale=None):
    """One decode layer.  seq_lens already count the current token."""
    perm_gen = torch.Generator().manual_seed(seed)
    gen = torch.Generator(device=device).manual_seed(seed + 1000)
    lens = [int(x) for x in seq_lens]
    caps = [n + extra_capacity for n in lens]
    shared_blocks = shared_prefix // block_size
    tables, nb = _alloc_tables(caps, block_size, pool_blocks, perm_gen, shared_blocks)
    k_cache, ks = _fill_pool(nb, num_kv_heads, block_size, head_dim, cache_dtype, gen, device,
                             value_scale)
    v_cache, vs = _fill_pool(nb, num_kv_heads, block_size, head_dim, cache_dtype, gen, device,
                             value_scale)
    if shared_prefix:
        _replicate_prefix_tail(k_cache, v_cache, tables, shared_prefix, block_size)
    adt = TORCH_DTYPE[act_dtype]
    b = len(lens)
    q = _normal((b, num_q_heads, head_dim), gen, device, value_scale).to(adt)
    nk = _normal((b, num_kv_heads, head_dim), gen, device, value_scale).to(adt)
    nv = _normal((b, num_kv_heads, head_dim), gen, device, value_scale).to(adt)
    sl = torch.tensor(lens, dtype=torch.int32)
    slot_last = _slots(tables, sl - 1, block_size)
    cap_pos = torch.tensor(lens, dtype=torch.int64)
    slot_next = _slots(tables, cap_pos, block_size)
    if extra_capacity < 1:
        slot_next = torch.full_like(slot_next, -1)
    dev = torch.device(device)
    return DecodeCase(
        k_cache=k_cache, v_cache=v_cache, cache_dtype=cache_dtype, act_dtype=act_dtype,
        k_scale=ks, v_scale=vs, block_tables=tables.to(dev), num_q_heads=num_q_heads,
        sm_scale=(1.0 / math.sqrt(head_dim)) if sm_scale is None else sm_scale,
        seq_lens=sl.to(dev), q=q, new_k=nk, new_v=nv, slot_last=slot_last.to(dev),
        slot_next=slot_next.to(dev),
        meta=dict(seed=seed, shared_prefix=shared_prefix, value_scale=value_scale))


def extend_case(prefix_lens, suffix_lens, num_q_heads, num_kv_heads, head_dim, block_size,
                cache_dtype, act_dtype, seed, device="cpu", shared_prefix=0, pool_blocks=None,
                value_scale=1.0, sm_scale=None):
    """Suffix prefill over cached prefixes.  The pool already holds every
    prefix AND suffix K/V (as if the suffix had been appended); suffix_k/v and
    suffix_slots are returned too so that an append can be run first."""
    perm_gen = torch.Generator().manual_seed(seed)
    gen = torch.Generator(device=device).manual_seed(seed + 1000)
    P = [int(x) for x in prefix_lens]
    S = [int(x) for x in suffix_lens]
    caps = [p + s for p, s in zip(P, S)]
    shared_blocks = shared_prefix // block_size
    tables, nb = _alloc_tables(caps, block_size, pool_blocks, perm_gen, shared_blocks)
    k_cache, ks = _fill_pool(nb, num_kv_heads, block_size, head_dim, cache_dtype, gen, device,
                             value_scale)
    v_cache, vs = _fill_pool(nb, num_kv_heads, block_size, head_dim, cache_dtype, gen, device,
                             value_scale)
    if shared_prefix:
        _replicate_prefix_tail(k_cache, v_cache, tables, shared_prefix, block_size)
    adt = TORCH_DTYPE[act_dtype]
    tot = sum(S)
    q = _normal((tot, num_q_heads, head_dim), gen, device, value_scale).to(adt)
    sk = _normal((tot, num_kv_heads, head_dim), gen, device, value_scale).to(adt)
    sv = _normal((tot, num_kv_heads, head_dim), gen, device, value_scale).to(adt)
    indptr = torch.zeros(len(S) + 1, dtype=torch.int32)
    indptr[1:] = torch.cumsum(torch.tensor(S, dtype=torch.int32), 0)
    rows_b = torch.repeat_interleave(torch.arange(len(S)), torch.tensor(S, dtype=torch.int64))
    pos = torch.tensor(P, dtype=torch.int64)[rows_b] + \
        (torch.arange(tot) - indptr[:-1].to(torch.int64)[rows_b])
    slots = _slots(tables[rows_b], pos, block_size)
    dev = torch.device(device)
    return ExtendCase(
        k_cache=k_cache, v_cache=v_cache, cache_dtype=cache_dtype, act_dtype=act_dtype,
        k_scale=ks, v_scale=vs, block_tables=tables.to(dev), num_q_heads=num_q_heads,
        sm_scale=(1.0 / math.sqrt(head_dim)) if sm_scale is None else sm_scale,
        q_indptr=indptr.to(dev), prefix_lens=torch.tensor(P, dtype=torch.int32).to(dev), q=q,
        suffix_k=sk, suffix_v=sv, suffix_slots=slots.to(dev),
        meta=dict(seed=seed, shared_prefix=shared_prefix, value_scale=value_scale))


# ---- the named workloads ---------------------------------------------------

def tiny_decode(device="cpu"):
    """4 requests {37,60,16,1}, 4 q / 1 kv head, d64, bs16, fp16, 64-block pool."""
    return decode_case([37, 60, 16, 1], 4, 1, 64, 16, F16, F16, seed=0, device=device,
                       pool_blocks=64, extra_capacity=1, sm_scale=1.0 / 8.0)


def uniform_lens(batch, lo, hi, seed):
    g = torch.Generator().manual_seed(seed + 7)
    return torch.randint(lo, hi + 1, (batch,), generator=g).tolist()


def llama3_8b_decode(device="cuda", batch=64, lo=512, hi=4096):
    """Llama-3-8B-shaped decode layer: 32q/8kv, d128, bf16, bs16, n ~ U[512,4096],
    values N(0,1)*0.5, blocks permuted across a pool sized to the total."""
    lens = uniform_lens(batch, lo, hi, seed=1)
    return decode_case(lens, 32, 8, 128, 16, BF16, BF16, seed=1, device=device,
                       value_scale=0.5, extra_capacity=0)


def shared_prefix_decode(device="cuda", batch=256, prefix=1000, lo=32, hi=256):
    """256 requests sharing one 1000-token prefix (62 shared blocks + an 8-token
    tail replicated per request) with unique suffixes U[32,256]."""
    suf = uniform_lens(batch, lo, hi, seed=2)
    lens = [prefix + s for s in suf]
    return decode_case(lens, 32, 8, 128, 16, BF16, BF16, seed=2, device=device,
                       shared_prefix=prefix, extra_capacity=0)


def shared_prefix_extend(device="cuda", batch=256, prefix=1900, suffix=100):
    """Suffix prefill: `batch` requests share one `prefix`-token cached prefix
    (full blocks shared, tail replicated), each with its own `suffix` tokens."""
    return extend_case([prefix] * batch, [suffix] * batch, 32, 8, 128, 16, BF16, BF16,
                       seed=3, device=device, shared_prefix=prefix)


def long_context_layers(device="cuda", batch=4, n=100_000, layers=32):
    """4 x 100k tokens, 32 layers of Llama-3-8B KV (8 kv heads, d128, fp16, bs32),
    32 q heads: one pool per layer, each with its own permutation."""
    cases = []
    for layer in range(layers):
        cases.append(decode_case([n] * batch, 32, 8, 128, 32, F16, F16, seed=100 + layer,
                                 device=device, extra_capacity=0))
    return cases


def fp8_70b_decode(device="cuda", batch=128, n=4096):
    """Llama-2-70B-shaped layer: 64q/8kv, d128, bs16, fp8_e4m3 K/V with per-tensor
    scale amax/448, bf16 q/out, seq_len 4096."""
    return decode_case([n] * batch, 64, 8, 128, 16, E4M3, BF16, seed=5, device=device,
                       extra_capacity=0)


def to_numpy_storage(t: torch.Tensor):
    """Host copy of a tensor's storage bits (uint16 for 16-bit floats, uint8 for codes)."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view("uint16")
    if t.dtype == torch.uint8:
        return t.numpy()
    return t.numpy()
