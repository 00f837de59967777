"""Second fp64 oracle, written in NumPy -- TEST INFRASTRUCTURE.

An independent restatement of the same definitions as ``pkv_oracle.c``
(gather the request's blocks through its block table, then textbook
softmax(QK^T * scale)V), used only to cross-check the C oracle on small cases.
It is vectorised per request and decodes elements with NumPy's own float16
and a bit-level bfloat16 / e4m3 decoder, so a slip in either version shows up
as a disagreement.

Definitions: "KV Cache에 대해 알아보자 (Feat. Attention)", §1 (attention) and §3
(decode attends over every cached token); "PagedAttention과 RadixAttention으로
LLM KV 캐시 최적화", section 02 (block table) and section 03 (suffix-only
prefill over a cached prefix).
"""
from __future__ import annotations

import numpy as np

F16, BF16, E4M3 = 0, 1, 2


def decode_storage(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Storage bits -> float64 values."""
    if dtype == F16:
        return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)
    if dtype == BF16:
        u32 = np.asarray(bits, np.uint16).astype(np.uint32) << 16
        return u32.view(np.float32).astype(np.float64)
    c = np.asarray(bits, np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    normal = (1.0 + man / 8.0) * np.exp2(exp - 7.0)
    sub = (man / 8.0) * np.exp2(-6.0)
    val = np.where(exp == 0, sub, normal)
    val = np.where((exp == 15) & (man == 7), np.nan, val)
    return sign * val


def gather(cache_vals: np.ndarray, table_row: np.ndarray, n: int, g: int) -> np.ndarray:
    """[num_blocks, Hkv, bs, D] values -> [n, D] for kv head g, in logical order."""
    bs = cache_vals.shape[2]
    t = np.arange(n)
    phys = np.asarray(table_row)[t // bs]
    return cache_vals[phys, g, t % bs, :]


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float):
    """q [R, D], k/v [n, D] -> (out [R, D], lse [R]); softmax along keys."""
    s = (q @ k.T) * scale
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    den = p.sum(axis=1, keepdims=True)
    return (p @ v) / den, (m + np.log(den))[:, 0]


def paged_decode(k_cache, v_cache, cache_dtype, k_scale, v_scale, q, q_dtype, block_tables,
                 seq_lens, num_q_heads, sm_scale):
    kv = decode_storage(k_cache, cache_dtype)
    vv = decode_storage(v_cache, cache_dtype)
    if cache_dtype == E4M3:
        kv = kv * float(k_scale)
        vv = vv * float(v_scale)
    qv = decode_storage(q, q_dtype)
    batch = len(seq_lens)
    hkv, d = kv.shape[1], kv.shape[3]
    grp = num_q_heads // hkv
    out = np.zeros((batch, num_q_heads, d))
    lse = np.full((batch, num_q_heads), -np.inf)
    for b in range(batch):
        n = int(seq_lens[b])
        if n == 0:
            continue
        for g in range(hkv):
            k = gather(kv, block_tables[b], n, g)
            v = gather(vv, block_tables[b], n, g)
            heads = slice(g * grp, (g + 1) * grp)
            o, l = attention(qv[b, heads, :], k, v, float(sm_scale))
            out[b, heads, :] = o
            lse[b, heads] = l
    return out, lse


def paged_extend(k_cache, v_cache, cache_dtype, k_scale, v_scale, q, q_dtype, q_indptr,
                 prefix_lens, block_tables, num_q_heads, sm_scale):
    kv = decode_storage(k_cache, cache_dtype)
    vv = decode_storage(v_cache, cache_dtype)
    if cache_dtype == E4M3:
        kv = kv * float(k_scale)
        vv = vv * float(v_scale)
    qv = decode_storage(q, q_dtype)
    hkv, d = kv.shape[1], kv.shape[3]
    grp = num_q_heads // hkv
    rows = int(q_indptr[-1])
    out = np.zeros((rows, num_q_heads, d))
    lse = np.zeros((rows, num_q_heads))
    for b in range(len(prefix_lens)):
        p = int(prefix_lens[b])
        r0, r1 = int(q_indptr[b]), int(q_indptr[b + 1])
        s_len = r1 - r0
        if s_len == 0:
            continue
        total = p + s_len
        for g in range(hkv):
            k = gather(kv, block_tables[b], total, g)
            v = gather(vv, block_tables[b], total, g)
            for h in range(g * grp, (g + 1) * grp):
                s = (qv[r0:r1, h, :] @ k.T) * float(sm_scale)      # [S, total]
                key = np.arange(total)[None, :]
                lim = p + np.arange(s_len)[:, None]
                s = np.where(key <= lim, s, -np.inf)
                m = s.max(axis=1, keepdims=True)
                e = np.exp(s - m)
                den = e.sum(axis=1, keepdims=True)
                out[r0:r1, h, :] = (e @ v) / den
                lse[r0:r1, h] = (m + np.log(den))[:, 0]
    return out, lse
