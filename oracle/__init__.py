"""Float64 CPU oracle for paged-KV attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never calls it and shares no
code with it.

Two independent implementations live here:

* ``pkv_oracle.c`` (plain C, fp64, OpenMP over query rows), loaded through
  ctypes -- the oracle used for parity and for the CPU baseline;
* ``ref_numpy.py`` (NumPy, fp64) -- a second, separately written version used
  only to cross-check the C code on small cases.

Beside the attention oracle, plain-Python references of the block-identity
parts: ``chain_hash_ref.py`` (salted chain hashes of full blocks) and
``prefix_match_ref.py`` (the longest cached prefix at block granularity, by
brute force).

Sources of the definitions (page title, section):
  * "KV Cache에 대해 알아보자 (Feat. Attention)", §1: softmax(QK^T/sqrt(d_k))V.
  * "PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", section 02:
    block table maps logical blocks to scattered physical blocks, read as one
    contiguous sequence.
  * same page, section 03: only the suffix after the longest cached prefix is
    computed (2,000-token request, 1,900 cached -> 100 prefilled).
  * "KV Cache에 대해 알아보자 (Feat. Attention)", §3: decode appends the new
    token's K/V to the cache and attends over every cached token.
  * "KV Cache 완전 정리 — PagedAttention vs RadixAttention, SGLang이 빠른 이유",
    section "FP8 KV 캐시": fp8_e4m3 cache dtype.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liborc.so")
_lock = threading.Lock()
_lib = None

F16, BF16, E4M3 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile ``pkv_oracle.c`` into ``oracle/liborc.so`` with gcc + OpenMP."""
    if not force and os.path.exists(_LIB_PATH) and \
            os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, D, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_float
        lib.orc_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_f16_to_double.restype = D
        lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_double.restype = D
        lib.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_to_double.restype = D
        lib.orc_e4m3_from_float.argtypes = [F]
        lib.orc_e4m3_from_float.restype = ctypes.c_uint8
        lib.orc_div_f32.argtypes = [F, F]
        lib.orc_div_f32.restype = F
        lib.orc_paged_decode.argtypes = [P, P, I, D, D, I, I, I, I, P, I, P, I, P, I, I, D,
                                         P, I, P, P, I]
        lib.orc_paged_decode.restype = I
        lib.orc_paged_extend.argtypes = [P, P, I, D, D, I, I, I, I, P, I, P, P, P, I, I, I,
                                         D, P, I, P, P, I]
        lib.orc_paged_extend.restype = I
        lib.orc_kv_append.argtypes = [P, P, I, F, F, I, I, I, I, P, P, I, P, I]
        lib.orc_kv_append.restype = I
        lib.orc_kv_bytes_per_token.argtypes = [I, I, I, I]
        lib.orc_kv_bytes_per_token.restype = ctypes.c_uint64
        lib.orc_max_threads.argtypes = []
        lib.orc_max_threads.restype = I
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(a: np.ndarray, dtype: int) -> np.ndarray:
    """View an element array as its raw storage (uint16 for f16/bf16, uint8 for e4m3)."""
    a = np.ascontiguousarray(a)
    want = np.uint8 if dtype == E4M3 else np.uint16
    if a.dtype == want:
        return a
    if a.dtype == np.float16 and dtype == F16:
        return a.view(np.uint16)
    raise TypeError(f"array of dtype {a.dtype} does not hold storage for dtype code {dtype}")


def max_threads() -> int:
    return int(_load().orc_max_threads())


def f16_to_double(bits: int) -> float:
    return float(_load().orc_f16_to_double(bits))


def bf16_to_double(bits: int) -> float:
    return float(_load().orc_bf16_to_double(bits))


def e4m3_to_double(code: int) -> float:
    return float(_load().orc_e4m3_to_double(code))


def e4m3_from_float(y: float) -> int:
    return int(_load().orc_e4m3_from_float(y))


def div_f32(x: float, s: float) -> float:
    return float(_load().orc_div_f32(x, s))


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """2 x layers x kv_heads x head_dim x bytes -- "KV Cache에 대해 알아보자", §4."""
    return int(_load().orc_kv_bytes_per_token(layers, kv_heads, head_dim, elem_bytes))


def paged_decode(k_cache, v_cache, cache_dtype, k_scale, v_scale, q, q_dtype,
                 block_tables, seq_lens, num_q_heads, sm_scale, pairs=None, threads=0):
    """Gather-then-textbook decode attention in fp64.

    k_cache/v_cache: storage arrays shaped [num_blocks, Hkv, bs, D] (uint16 for
    f16/bf16 bits, uint8 for e4m3).  q: storage array [B, Hq, D].
    Returns (out fp64 [B,Hq,D] or [len(pairs),D], lse fp64, status).
    """
    lib = _load()
    kc, vc = _bits(k_cache, cache_dtype), _bits(v_cache, cache_dtype)
    qb = _bits(q, q_dtype)
    nb, hkv, bs, d = kc.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    batch = sl.shape[0]
    if pairs is not None:
        pr = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
        out = np.zeros((pr.shape[0], d), np.float64)
        lse = np.zeros((pr.shape[0],), np.float64)
        npairs = pr.shape[0]
    else:
        pr = None
        out = np.zeros((batch, num_q_heads, d), np.float64)
        lse = np.zeros((batch, num_q_heads), np.float64)
        npairs = 0
    st = lib.orc_paged_decode(_ptr(kc), _ptr(vc), cache_dtype, float(k_scale), float(v_scale),
                              nb, hkv, bs, d, _ptr(qb), q_dtype, _ptr(bt), bt.shape[1],
                              _ptr(sl), batch, num_q_heads, float(sm_scale), _ptr(pr), npairs,
                              _ptr(out), _ptr(lse), int(threads))
    return out, lse, st


def paged_extend(k_cache, v_cache, cache_dtype, k_scale, v_scale, q, q_dtype, q_indptr,
                 prefix_lens, block_tables, num_q_heads, sm_scale, rows=None, threads=0):
    """Gather-then-textbook suffix prefill in fp64 (causal, aligned to the end)."""
    lib = _load()
    kc, vc = _bits(k_cache, cache_dtype), _bits(v_cache, cache_dtype)
    qb = _bits(q, q_dtype)
    nb, hkv, bs, d = kc.shape
    qi = np.ascontiguousarray(q_indptr, dtype=np.int32)
    pl = np.ascontiguousarray(prefix_lens, dtype=np.int32)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    batch = pl.shape[0]
    if rows is not None:
        rw = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 2)
        out = np.zeros((rw.shape[0], d), np.float64)
        lse = np.zeros((rw.shape[0],), np.float64)
        nrows = rw.shape[0]
    else:
        rw = None
        out = np.zeros((int(qi[-1]), num_q_heads, d), np.float64)
        lse = np.zeros((int(qi[-1]), num_q_heads), np.float64)
        nrows = 0
    st = lib.orc_paged_extend(_ptr(kc), _ptr(vc), cache_dtype, float(k_scale), float(v_scale),
                              nb, hkv, bs, d, _ptr(qb), q_dtype, _ptr(qi), _ptr(pl), _ptr(bt),
                              bt.shape[1], batch, num_q_heads, float(sm_scale), _ptr(rw), nrows,
                              _ptr(out), _ptr(lse), int(threads))
    return out, lse, st


def kv_append(k_cache, v_cache, cache_dtype, k_scale, v_scale, new_k, new_v, act_dtype,
              slot_mapping):
    """Apply an append to COPIES of the cache storage arrays; returns (k, v, status)."""
    lib = _load()
    kc = np.array(_bits(k_cache, cache_dtype), copy=True)
    vc = np.array(_bits(v_cache, cache_dtype), copy=True)
    nb, hkv, bs, d = kc.shape
    nk, nv = _bits(new_k, act_dtype), _bits(new_v, act_dtype)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    st = lib.orc_kv_append(_ptr(kc), _ptr(vc), cache_dtype, float(k_scale), float(v_scale),
                           nb, hkv, bs, d, _ptr(nk), _ptr(nv), act_dtype, _ptr(sm),
                           sm.shape[0])
    return kc, vc, st
