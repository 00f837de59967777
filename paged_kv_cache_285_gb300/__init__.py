"""Paged-KV attention for GB300 (sm_103a): a thin ctypes binding of libpkv.so.

Every call here only marshals arguments (PyTorch tensors -> device pointers,
the current CUDA stream) and forwards them to the C ABI declared in
``include/pkv.h``; all work runs in the library's CUDA kernels.  There is no
CPU fallback: if libpkv.so is missing or fails to load, every call raises.

The three calls (names as in pkv.h without the ``pkv_`` prefix):
  * kv_append          -- scatter new K/V rows into their cache slots;
  * paged_decode_attn  -- one query token per request over its paged K/V
                          (GQA, split-KV, online softmax, LSE merge);
  * paged_extend_attn  -- suffix prefill over cached prefix blocks + causal
                          suffix.
Also: paged_decode_attn_append and paged_extend_attn_append (the new tokens'
K/V written into the cache by the same call; in decode by the attention
kernel itself), paged_decode_attn_shared_prefix
(decode for groups of requests sharing a prefix, the prefix attended once per
group), RadixIndex (the host prefix index that hands out block tables and
prefix lengths; host int32 arrays in, host arrays out) and chain_hash (salted
chain hashes of full blocks, as block identifiers).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = ["F16", "BF16", "FP8_E4M3", "PkvError", "CacheDesc", "lib_path", "load",
           "kv_append", "paged_decode_attn", "paged_extend_attn", "decode_workspace_bytes",
           "extend_workspace_bytes", "get_device_error", "status_string", "version",
           "paged_decode_attn_append", "RadixIndex", "NO_SPACE", "chain_hash",
           "paged_decode_attn_shared_prefix", "shared_prefix_decode_workspace_bytes",
           "paged_extend_attn_append", "paged_extend_attn_shared_prefix",
           "extend_shared_prefix_workspace_bytes", "extend_widen_workspace_bytes"]

F16, BF16, FP8_E4M3 = 0, 1, 2
NO_SPACE = 5  # PKV_ERR_NO_SPACE
_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libpkv.so")
_lib = None
_lock = threading.Lock()


class RadixStats(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("free_blocks", ctypes.c_int32),
                ("tree_blocks", ctypes.c_int32), ("caller_blocks", ctypes.c_int32),
                ("nodes", ctypes.c_int32), ("evictable_leaves", ctypes.c_int32)]


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class CacheDesc(ctypes.Structure):
    """Mirror of pkv_cache_desc."""
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("cache_dtype", ctypes.c_int), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float)]


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load libpkv.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is not built; run paged_kv_cache_285_gb300.build.build()")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I32, SZ, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
        D = ctypes.POINTER(CacheDesc)
        lib.pkv_kv_append.argtypes = [D, P, P, P, P, ctypes.c_int, P, I32, P]
        lib.pkv_kv_append.restype = ctypes.c_int
        lib.pkv_decode_workspace_bytes.argtypes = [D, I32, I32, I32, I32]
        lib.pkv_decode_workspace_bytes.restype = SZ
        lib.pkv_paged_decode_attn.argtypes = [D, P, P, P, P, ctypes.c_int, P, I32, P, I32, I32, F,
                                              I32, I32, P, P, SZ, P]
        lib.pkv_paged_decode_attn.restype = ctypes.c_int
        lib.pkv_paged_decode_attn_append.argtypes = [D, P, P, P, P, P, P, ctypes.c_int, P, I32, P,
                                                      I32, I32, F, I32, I32, P, P, SZ, P]
        lib.pkv_paged_decode_attn_append.restype = ctypes.c_int
        lib.pkv_paged_decode_attn_noalloc.argtypes = [D, P, P, P, P, ctypes.c_int, P, I32, P, I32,
                                                       I32, F, I32, I32, P, P]
        lib.pkv_paged_decode_attn_noalloc.restype = ctypes.c_int
        lib.pkv_extend_workspace_bytes.argtypes = [D, I32, I32, I32, I32]
        lib.pkv_extend_workspace_bytes.restype = SZ
        lib.pkv_paged_extend_attn.argtypes = [D, P, P, P, P, ctypes.c_int, P, P, P, I32, I32, I32,
                                              F, I32, I32, I32, P, P, SZ, P]
        lib.pkv_paged_extend_attn.restype = ctypes.c_int
        lib.pkv_paged_extend_attn_append.argtypes = [D, P, P, P, P, P, P, ctypes.c_int, P, P, P, I32,
                                                     I32, I32, F, I32, I32, I32, P, P]
        lib.pkv_paged_extend_attn_append.restype = ctypes.c_int
        lib.pkv_paged_extend_attn_shared_prefix.argtypes = [D, P, P, P, P, ctypes.c_int, P, P, P,
                                                            I32, I32, I32, F, I32, P, P, I32, I32,
                                                            I32, P, P, SZ, P]
        lib.pkv_paged_extend_attn_shared_prefix.restype = ctypes.c_int
        lib.pkv_extend_shared_prefix_workspace_bytes.argtypes = [D]
        lib.pkv_extend_shared_prefix_workspace_bytes.restype = SZ
        lib.pkv_extend_widen_workspace_bytes.argtypes = [D]
        lib.pkv_extend_widen_workspace_bytes.restype = SZ
        lib.pkv_status_string.argtypes = [ctypes.c_int]
        lib.pkv_status_string.restype = ctypes.c_char_p
        lib.pkv_get_device_error.argtypes = [ctypes.POINTER(I32), I32, P]
        lib.pkv_get_device_error.restype = ctypes.c_int
        lib.pkv_version.argtypes = []
        lib.pkv_version.restype = I32
        lib.pkv_shared_prefix_decode_workspace_bytes.argtypes = [D, I32, I32, I32, I32, I32]
        lib.pkv_shared_prefix_decode_workspace_bytes.restype = SZ
        lib.pkv_paged_decode_attn_shared_prefix.argtypes = [D, P, P, P, P, P, P, ctypes.c_int, P,
                                                             I32, P, I32, I32, F, P, P, I32, I32,
                                                             I32, I32, I32, P, P, SZ, P]
        lib.pkv_paged_decode_attn_shared_prefix.restype = ctypes.c_int
        lib.pkv_chain_hash.argtypes = [P, P, I32, I32, P, P, I32, P]
        lib.pkv_chain_hash.restype = ctypes.c_int
        VP = ctypes.c_void_p
        lib.pkv_radix_create.argtypes = [I32, I32, ctypes.POINTER(VP)]
        lib.pkv_radix_create.restype = ctypes.c_int
        lib.pkv_radix_destroy.argtypes = [VP]
        lib.pkv_radix_destroy.restype = None
        lib.pkv_radix_match.argtypes = [VP, P, I32, P, I32, ctypes.POINTER(I32)]
        lib.pkv_radix_match.restype = ctypes.c_int
        lib.pkv_radix_release.argtypes = [VP, P, I32]
        lib.pkv_radix_release.restype = ctypes.c_int
        lib.pkv_radix_alloc.argtypes = [VP, I32, P]
        lib.pkv_radix_alloc.restype = ctypes.c_int
        lib.pkv_radix_free.argtypes = [VP, P, I32]
        lib.pkv_radix_free.restype = ctypes.c_int
        lib.pkv_radix_insert.argtypes = [VP, P, I32, P, P, ctypes.POINTER(I32)]
        lib.pkv_radix_insert.restype = ctypes.c_int
        lib.pkv_radix_evict.argtypes = [VP, I32, ctypes.POINTER(I32)]
        lib.pkv_radix_evict.restype = ctypes.c_int
        lib.pkv_radix_stats.argtypes = [VP, ctypes.POINTER(RadixStats)]
        lib.pkv_radix_stats.restype = ctypes.c_int
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().pkv_status_string(int(status)).decode()


def version() -> int:
    return int(load().pkv_version())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.uint8 or t.dtype == getattr(torch, "float8_e4m3fn", None):
        return FP8_E4M3
    raise TypeError(f"unsupported tensor dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libpkv takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libpkv takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _desc(k_cache: torch.Tensor, k_scale: float, v_scale: float) -> CacheDesc:
    if k_cache.dim() != 4:
        raise ValueError("cache must be [num_blocks, num_kv_heads, block_size, head_dim]")
    nb, hkv, bs, d = k_cache.shape
    return CacheDesc(nb, bs, hkv, d, _dtype_code(k_cache), float(k_scale), float(v_scale))


def _need(dtype, **tensors):
    """The index tensors of a call must have the dtype the C ABI reads."""
    for name, t in tensors.items():
        if t is not None and t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _shape(name, t, shape, dtype=None):
    """A tensor argument must have the shape (and dtype) the call derives from the others: the
    C ABI takes bare pointers and cannot see how large a buffer is."""
    if t is None:
        return
    want = tuple(int(x) for x in shape)
    if tuple(t.shape) != want:
        raise ValueError(f"{name} must have shape {want}, got {tuple(t.shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _cache_pair(k_cache, v_cache):
    """K and V pools [num_blocks, num_kv_heads, block_size, head_dim] of one dtype; returns
    (num_kv_heads, head_dim)."""
    if k_cache.dim() != 4:
        raise ValueError("cache must be [num_blocks, num_kv_heads, block_size, head_dim]")
    _shape("v_cache", v_cache, k_cache.shape, k_cache.dtype)
    return int(k_cache.shape[1]), int(k_cache.shape[3])


def _rows(name, t, head_dim):
    """[rows, heads, head_dim] activations; returns (rows, heads)."""
    if t.dim() != 3 or int(t.shape[2]) != head_dim:
        raise ValueError(f"{name} must be [rows, heads, {head_dim}], got {tuple(t.shape)}")
    return int(t.shape[0]), int(t.shape[1])


def _table(name, t, rows):
    if t.dim() != 2 or int(t.shape[0]) != rows:
        raise ValueError(f"{name} must be [{rows}, max_blocks_per_seq], got {tuple(t.shape)}")


def _decode_shapes(k_cache, v_cache, q, out, block_tables, seq_lens, lse_out, k_new=None,
                   v_new=None):
    """Shapes of a decode call; returns (batch, num_q_heads)."""
    hkv, d = _cache_pair(k_cache, v_cache)
    b, hq = _rows("q", q, d)
    _shape("out", out, q.shape, q.dtype)
    _table("block_tables", block_tables, b)
    _shape("seq_lens", seq_lens, (b,))
    _shape("lse_out", lse_out, (b, hq), torch.float32)
    _shape("k_new", k_new, (b, hkv, d), q.dtype)
    _shape("v_new", v_new, (b, hkv, d), q.dtype)
    return b, hq


def _extend_shapes(k_cache, v_cache, q, out, q_indptr, prefix_lens, block_tables, lse_out,
                   k_new=None, v_new=None):
    """Shapes of an extend call; returns (total_q_rows, num_q_heads, batch)."""
    hkv, d = _cache_pair(k_cache, v_cache)
    rows, hq = _rows("q", q, d)
    _shape("out", out, q.shape, q.dtype)
    if prefix_lens.dim() != 1:
        raise ValueError("prefix_lens must be [batch]")
    batch = int(prefix_lens.shape[0])
    _shape("q_indptr", q_indptr, (batch + 1,))
    _table("block_tables", block_tables, batch)
    _shape("lse_out", lse_out, (rows, hq), torch.float32)
    _shape("k_new", k_new, (rows, hkv, d), q.dtype)
    _shape("v_new", v_new, (rows, hkv, d), q.dtype)
    return rows, hq, batch


def _check(status: int, what: str):
    if status != 0:
        raise PkvError(status, what)


def kv_append(k_cache, v_cache, k_new, v_new, slot_mapping, k_scale=1.0, v_scale=1.0,
              stream=None):
    """pkv_kv_append: k_new/v_new [T, Hkv, D] act dtype, slot_mapping int64 [T]."""
    _need(torch.int64, slot_mapping=slot_mapping)
    hkv, d = _cache_pair(k_cache, v_cache)
    if slot_mapping.dim() != 1:
        raise ValueError("slot_mapping must be [num_tokens]")
    t = int(slot_mapping.shape[0])
    _shape("k_new", k_new, (t, hkv, d))
    _shape("v_new", v_new, (t, hkv, d), k_new.dtype)
    lib = load()
    desc = _desc(k_cache, k_scale, v_scale)
    st = lib.pkv_kv_append(ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache), _ptr(k_new),
                           _ptr(v_new), _dtype_code(k_new), _ptr(slot_mapping),
                           int(slot_mapping.shape[0]), _stream(stream))
    _check(st, "pkv_kv_append")


def decode_workspace_bytes(k_cache, batch, num_q_heads, max_seq_len, num_splits=0,
                           k_scale=1.0, v_scale=1.0) -> int:
    lib = load()
    desc = _desc(k_cache, k_scale, v_scale)
    return int(lib.pkv_decode_workspace_bytes(ctypes.byref(desc), batch, num_q_heads,
                                              max_seq_len, num_splits))


def paged_decode_attn(k_cache, v_cache, q, out, block_tables, seq_lens, sm_scale, max_seq_len,
                      k_scale=1.0, v_scale=1.0, num_splits=0, lse_out=None, workspace=None,
                      stream=None):
    """pkv_paged_decode_attn: q/out [B, Hq, D]; block_tables int32 [B, W]; seq_lens int32 [B].
    ``workspace`` is a uint8 device tensor of at least decode_workspace_bytes() bytes."""
    _need(torch.int32, block_tables=block_tables, seq_lens=seq_lens)
    b, hq = _decode_shapes(k_cache, v_cache, q, out, block_tables, seq_lens, lse_out)
    lib = load()
    desc = _desc(k_cache, k_scale, v_scale)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.pkv_paged_decode_attn(ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache), _ptr(q),
                                   _ptr(out), _dtype_code(q), _ptr(block_tables),
                                   int(block_tables.shape[1]), _ptr(seq_lens), b, hq,
                                   float(sm_scale), int(max_seq_len), int(num_splits),
                                   _ptr(lse_out), _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "pkv_paged_decode_attn")


def paged_decode_attn_append(k_cache, v_cache, k_new, v_new, q, out, block_tables, seq_lens,
                             sm_scale, max_seq_len, k_scale=1.0, v_scale=1.0, num_splits=0,
                             lse_out=None, workspace=None, stream=None):
    """pkv_paged_decode_attn_append: k_new/v_new [B, Hkv, D] are written to position
    seq_len-1 of each request and attended in the same launch."""
    _need(torch.int32, block_tables=block_tables, seq_lens=seq_lens)
    b, hq = _decode_shapes(k_cache, v_cache, q, out, block_tables, seq_lens, lse_out, k_new,
                           v_new)
    lib = load()
    desc = _desc(k_cache, k_scale, v_scale)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.pkv_paged_decode_attn_append(ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(out),
                                          _dtype_code(q), _ptr(block_tables),
                                          int(block_tables.shape[1]), _ptr(seq_lens), b, hq,
                                          float(sm_scale), int(max_seq_len), int(num_splits),
                                          _ptr(lse_out), _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "pkv_paged_decode_attn_append")


def paged_decode_attn_noalloc(k_cache, v_cache, q, out, block_tables, seq_lens, sm_scale,
                              max_seq_len, k_scale=1.0, v_scale=1.0, num_splits=0, lse_out=None,
                              stream=None):
    """pkv_paged_decode_attn_noalloc: paged_decode_attn with the split partials in the library's
    own scratch array (no workspace; calls on one device must not overlap)."""
    _need(torch.int32, block_tables=block_tables, seq_lens=seq_lens)
    b, hq = _decode_shapes(k_cache, v_cache, q, out, block_tables, seq_lens, lse_out)
    lib = load()
    desc = _desc(k_cache, k_scale, v_scale)
    st = lib.pkv_paged_decode_attn_noalloc(ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache),
                                           _ptr(q), _ptr(out), _dtype_code(q), _ptr(block_tables),
                                           int(block_tables.shape[1]), _ptr(seq_lens), b, hq,
                                           float(sm_scale), int(max_seq_len), int(num_splits),
                                           _ptr(lse_out), _stream(stream))
    _check(st, "pkv_paged_decode_attn_noalloc")


def shared_prefix_decode_workspace_bytes(k_cache, batch, num_q_heads, max_prefix_len,
                                         max_suffix_len, num_splits=0) -> int:
    lib = load()
    desc = _desc(k_cache, 1.0, 1.0)
    return int(lib.pkv_shared_prefix_decode_workspace_bytes(ctypes.byref(desc), batch, num_q_heads,
                                                            max_prefix_len, max_suffix_len,
                                                            num_splits))


def paged_decode_attn_shared_prefix(k_cache, v_cache, q, out, block_tables, seq_lens, sm_scale,
                                    group_indptr, group_prefix_lens, max_group_size,
                                    max_prefix_len, max_suffix_len, k_new=None, v_new=None,
                                    num_splits=0, lse_out=None, workspace=None, stream=None,
                                    k_scale=1.0, v_scale=1.0):
    """pkv_paged_decode_attn_shared_prefix: requests [group_indptr[g], group_indptr[g+1])
    share their first group_prefix_lens[g] tokens (read through the group's first member's
    block table), attended once per group; max_prefix_len / max_suffix_len bound the groups'
    prefixes and the members' own tokens; k_new/v_new as paged_decode_attn_append; k_scale /
    v_scale are an fp8 cache's scales."""
    _need(torch.int32, block_tables=block_tables, seq_lens=seq_lens)
    b, hq = _decode_shapes(k_cache, v_cache, q, out, block_tables, seq_lens, lse_out, k_new,
                           v_new)
    lib = load()
    desc = _desc(k_cache, k_scale, v_scale)
    if group_indptr.dim() != 1:
        raise ValueError("group_indptr must be int32 [num_groups + 1]")
    ng = int(group_indptr.shape[0]) - 1
    if group_indptr.dtype != torch.int32 or group_prefix_lens.dtype != torch.int32:
        raise ValueError("group_indptr and group_prefix_lens must be int32")
    if tuple(group_prefix_lens.shape) != (ng,):
        raise ValueError("group_prefix_lens must be int32 [num_groups]")
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.pkv_paged_decode_attn_shared_prefix(
        ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), _ptr(q),
        _ptr(out), _dtype_code(q), _ptr(block_tables), int(block_tables.shape[1]), _ptr(seq_lens),
        b, hq, float(sm_scale), _ptr(group_indptr), _ptr(group_prefix_lens), ng,
        int(max_group_size), int(max_prefix_len), int(max_suffix_len), int(num_splits),
        _ptr(lse_out),
        _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "pkv_paged_decode_attn_shared_prefix")


def extend_workspace_bytes(k_cache, batch, num_q_heads, total_q_rows, max_total_len,
                           k_scale=1.0, v_scale=1.0) -> int:
    lib = load()
    desc = _desc(k_cache, k_scale, v_scale)
    return int(lib.pkv_extend_workspace_bytes(ctypes.byref(desc), batch, num_q_heads,
                                              total_q_rows, max_total_len))


def paged_extend_attn(k_cache, v_cache, q, out, q_indptr, prefix_lens, block_tables, sm_scale,
                      max_suffix_len, max_total_len, k_scale=1.0, v_scale=1.0, lse_out=None,
                      workspace=None, stream=None):
    """pkv_paged_extend_attn: q/out [sum S, Hq, D]; q_indptr int32 [B+1]; prefix_lens int32 [B];
    workspace: None, or a uint8 device tensor of extend_widen_workspace_bytes() bytes or more
    (the pages read are then widened to 16 bits once per block; smaller ones are not used)."""
    _need(torch.int32, q_indptr=q_indptr, prefix_lens=prefix_lens, block_tables=block_tables)
    rows, hq, batch = _extend_shapes(k_cache, v_cache, q, out, q_indptr, prefix_lens,
                                     block_tables, lse_out)
    lib = load()
    desc = _desc(k_cache, k_scale, v_scale)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.pkv_paged_extend_attn(ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache), _ptr(q),
                                   _ptr(out), _dtype_code(q), _ptr(q_indptr), _ptr(prefix_lens),
                                   _ptr(block_tables), int(block_tables.shape[1]), batch, hq,
                                   float(sm_scale), rows, int(max_suffix_len),
                                   int(max_total_len), _ptr(lse_out), _ptr(workspace), ws_bytes,
                                   _stream(stream))
    _check(st, "pkv_paged_extend_attn")


def extend_widen_workspace_bytes(k_cache, k_scale=1.0, v_scale=1.0) -> int:
    """pkv_extend_widen_workspace_bytes: the optional widening workspace of paged_extend_attn
    (16-bit copies of a bf16 cache's V pool or of an fp8 cache's K and V pools, and the
    per-block claims; 0 for an f16 cache)."""
    lib = load()
    desc = _desc(k_cache, k_scale, v_scale)
    return int(lib.pkv_extend_widen_workspace_bytes(ctypes.byref(desc)))


def extend_shared_prefix_workspace_bytes(k_cache, k_scale=1.0, v_scale=1.0) -> int:
    """pkv_extend_shared_prefix_workspace_bytes: the optional workspace of
    paged_extend_attn_shared_prefix (f16 copies of a bf16 cache's V pool or of an fp8
    cache's K and V pools; 0 for an f16 cache)."""
    lib = load()
    desc = _desc(k_cache, k_scale, v_scale)
    return int(lib.pkv_extend_shared_prefix_workspace_bytes(ctypes.byref(desc)))


def paged_extend_attn_shared_prefix(k_cache, v_cache, q, out, q_indptr, prefix_lens, block_tables,
                                    group_indptr, group_shared_lens, sm_scale, max_group_rows,
                                    max_total_len, k_scale=1.0, v_scale=1.0, lse_out=None,
                                    workspace=None, stream=None):
    """pkv_paged_extend_attn_shared_prefix: as paged_extend_attn, for groups of requests
    (group_indptr int32 [G+1], consecutive requests) sharing the blocks of their first
    group_shared_lens[g] tokens (int32 [G]); the groups' rows are packed into shared tiles.
    workspace: None, or a uint8 device tensor of extend_shared_prefix_workspace_bytes() bytes
    (the pages of a bf16 or fp8 cache are then widened to f16 once per call instead of per
    tile)."""
    _need(torch.int32, q_indptr=q_indptr, prefix_lens=prefix_lens, block_tables=block_tables,
          group_indptr=group_indptr, group_shared_lens=group_shared_lens)
    rows, hq, batch = _extend_shapes(k_cache, v_cache, q, out, q_indptr, prefix_lens,
                                     block_tables, lse_out)
    ng = int(group_indptr.shape[0]) - 1
    if group_indptr.dim() != 1 or ng < 0 or tuple(group_shared_lens.shape) != (ng,):
        raise ValueError("group_indptr must be [G+1] and group_shared_lens [G]")
    for name, t in (("group_indptr", group_indptr), ("group_shared_lens", group_shared_lens)):
        if t.device != q.device:
            raise ValueError(f"{name} must be on {q.device}")
    lib = load()
    desc = _desc(k_cache, k_scale, v_scale)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib.pkv_paged_extend_attn_shared_prefix(
        ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache), _ptr(q), _ptr(out), _dtype_code(q),
        _ptr(q_indptr), _ptr(prefix_lens), _ptr(block_tables), int(block_tables.shape[1]), batch,
        hq, float(sm_scale), rows, _ptr(group_indptr), _ptr(group_shared_lens), ng,
        int(max_group_rows), int(max_total_len), _ptr(lse_out), _ptr(workspace), ws_bytes,
        _stream(stream))
    _check(st, "pkv_paged_extend_attn_shared_prefix")


def paged_extend_attn_append(k_cache, v_cache, k_new, v_new, q, out, q_indptr, prefix_lens,
                             block_tables, sm_scale, max_suffix_len, max_total_len, lse_out=None,
                             stream=None, k_scale=1.0, v_scale=1.0):
    """pkv_paged_extend_attn_append: k_new/v_new [sum S, Hkv, D] (q's dtype) are written to
    positions prefix_lens[b] + i (an fp8 cache stores them quantised with k_scale / v_scale) and
    attended in the same call."""
    _need(torch.int32, q_indptr=q_indptr, prefix_lens=prefix_lens, block_tables=block_tables)
    rows, hq, batch = _extend_shapes(k_cache, v_cache, q, out, q_indptr, prefix_lens,
                                     block_tables, lse_out, k_new, v_new)
    lib = load()
    desc = _desc(k_cache, k_scale, v_scale)
    st = lib.pkv_paged_extend_attn_append(ctypes.byref(desc), _ptr(k_cache), _ptr(v_cache),
                                          _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(out),
                                          _dtype_code(q), _ptr(q_indptr), _ptr(prefix_lens),
                                          _ptr(block_tables), int(block_tables.shape[1]), batch,
                                          hq, float(sm_scale), rows, int(max_suffix_len),
                                          int(max_total_len), _ptr(lse_out), _stream(stream))
    _check(st, "pkv_paged_extend_attn_append")


def chain_hash(tokens, token_indptr, block_size, hashes, salts=None, stream=None):
    """pkv_chain_hash: tokens int32 [T], token_indptr int32 [B+1], hashes int64 [B, max_blocks]
    (uint64 bits), salts int64 [B] (uint64 bits) or None; all device tensors."""
    lib = load()
    b = int(token_indptr.shape[0]) - 1
    if tokens.dtype != torch.int32 or token_indptr.dtype != torch.int32 or token_indptr.dim() != 1:
        raise ValueError("tokens and token_indptr must be int32 (token_indptr 1-D)")
    if hashes.dtype != torch.int64 or hashes.dim() != 2 or hashes.shape[0] != b:
        raise ValueError("hashes must be int64 [batch, max_blocks]")
    if salts is not None and (salts.dtype != torch.int64 or tuple(salts.shape) != (b,)):
        raise ValueError("salts must be int64 [batch]")
    _check(lib.pkv_chain_hash(_ptr(tokens), _ptr(token_indptr), b, int(block_size), _ptr(salts),
                              _ptr(hashes), int(hashes.shape[1]), _stream(stream)), "pkv_chain_hash")


def get_device_error(clear=True, stream=None) -> int:
    """Read (and by default clear) the library's device error word (synchronises)."""
    lib = load()
    w = ctypes.c_int32(0)
    _check(lib.pkv_get_device_error(ctypes.byref(w), int(bool(clear)), _stream(stream)),
           "pkv_get_device_error")
    return int(w.value)


def _host_i32(a):
    """Contiguous host int32 array and its address (numpy or a CPU tensor)."""
    import numpy as np
    if isinstance(a, torch.Tensor):
        a = a.detach().to("cpu").numpy()
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    return arr, (arr.ctypes.data if arr.size else None)


class RadixIndex:
    """pkv_radix_*: host prefix index over the block ids [0, num_blocks) of one pool.
    Token and block lists are host int32 arrays; results are numpy int32 arrays."""

    def __init__(self, block_size: int, num_blocks: int):
        self._lib = load()
        h = ctypes.c_void_p()
        _check(self._lib.pkv_radix_create(int(block_size), int(num_blocks), ctypes.byref(h)),
               "pkv_radix_create")
        self._h = h
        self.block_size = int(block_size)

    def close(self):
        if getattr(self, "_h", None):
            self._lib.pkv_radix_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def match(self, tokens):
        """(matched_tokens, blocks): the locked longest cached whole-block prefix."""
        import numpy as np
        t, tp = _host_i32(tokens)
        cap = t.size // self.block_size
        out = np.zeros(max(cap, 1), dtype=np.int32)
        m = ctypes.c_int32(0)
        _check(self._lib.pkv_radix_match(self._h, tp, int(t.size), out.ctypes.data, cap, ctypes.byref(m)),
               "pkv_radix_match")
        return int(m.value), out[: m.value // self.block_size].copy()

    def release(self, tokens, matched_tokens: int):
        t, tp = _host_i32(tokens)
        _check(self._lib.pkv_radix_release(self._h, tp, int(matched_tokens)), "pkv_radix_release")

    def alloc(self, count: int):
        import numpy as np
        out = np.zeros(max(int(count), 1), dtype=np.int32)
        _check(self._lib.pkv_radix_alloc(self._h, int(count), out.ctypes.data), "pkv_radix_alloc")
        return out[: int(count)].copy()

    def free(self, blocks):
        b, bp = _host_i32(blocks)
        _check(self._lib.pkv_radix_free(self._h, bp, int(b.size)), "pkv_radix_free")

    def insert(self, tokens, blocks):
        """Adopt the full blocks of a request; returns the caller blocks that were freed
        because the tree already held the same tokens."""
        import numpy as np
        t, tp = _host_i32(tokens)
        b, bp = _host_i32(blocks)
        rel = np.zeros(max(t.size // self.block_size, 1), dtype=np.int32)
        n = ctypes.c_int32(0)
        _check(self._lib.pkv_radix_insert(self._h, tp, int(t.size), bp, rel.ctypes.data, ctypes.byref(n)),
               "pkv_radix_insert")
        return rel[: n.value].copy()

    def evict(self, num_blocks: int) -> int:
        f = ctypes.c_int32(0)
        _check(self._lib.pkv_radix_evict(self._h, int(num_blocks), ctypes.byref(f)), "pkv_radix_evict")
        return int(f.value)

    def stats(self) -> dict:
        st = RadixStats()
        _check(self._lib.pkv_radix_stats(self._h, ctypes.byref(st)), "pkv_radix_stats")
        return {k: int(getattr(st, k)) for k, _ in RadixStats._fields_}
