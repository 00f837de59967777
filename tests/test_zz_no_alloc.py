"""pkv_paged_decode_attn_noalloc against pkv_paged_decode_attn.

The allocation-free entry point serves callers that cannot allocate device
memory (an engine plugin that only receives the call's tensors, a path where
cudaMalloc is not allowed); it keeps the split partials in a scratch array
built into the library.  Its results must match the regular entry point's,
call after call, even though every call reuses the same scratch.  This file is
named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_285_gb300 as pkv
from paged_kv_cache_285_gb300 import workloads as W
from tests.pkv_testlib import BF16, assert_attention_close, to_f64

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 * 1024 * 1024


def _lib():
    lib = pkv.load()
    fn = lib.pkv_paged_decode_attn_noalloc
    P, I32 = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [ctypes.POINTER(pkv.CacheDesc), P, P, P, P, ctypes.c_int, P, I32, P, I32, I32,
                   ctypes.c_float, I32, I32, P, P]
    fn.restype = ctypes.c_int
    return fn


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(fn, case, q, out, lse, max_len, splits):
    nb, hkv, bs, d = case.k_cache.shape
    desc = pkv.CacheDesc(nb, bs, hkv, d, case.cache_dtype, case.k_scale, case.v_scale)
    st = fn(ctypes.byref(desc), _ptr(case.k_cache), _ptr(case.v_cache), _ptr(q), _ptr(out),
            case.act_dtype, _ptr(case.block_tables), case.block_tables.shape[1],
            _ptr(case.seq_lens), q.shape[0], case.num_q_heads, case.sm_scale, max_len, splits,
            _ptr(lse), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


def _regular(case, q, max_len, splits):
    out = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device="cuda")
    ws_bytes = pkv.decode_workspace_bytes(case.k_cache, q.shape[0], case.num_q_heads, max_len,
                                          splits, case.k_scale, case.v_scale)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    pkv.paged_decode_attn(case.k_cache, case.v_cache, q, out, case.block_tables, case.seq_lens,
                          case.sm_scale, max_len, k_scale=case.k_scale, v_scale=case.v_scale,
                          num_splits=splits, lse_out=lse, workspace=ws)
    return out, lse


def test_noalloc_matches_regular_decode_twice():
    fn = _lib()
    lens = [700, 33, 1500, 257, 64, 1024]
    case = W.decode_case(lens, 32, 8, 128, 16, BF16, BF16, seed=90, device="cuda")
    max_len, splits = 1536, 6
    assert 0 < pkv.decode_workspace_bytes(case.k_cache, len(lens), 32, max_len, splits) <= SCRATCH_BYTES
    q2 = torch.randn_like(case.q, dtype=torch.float32).to(case.q.dtype)
    for q in (case.q, q2):                      # two calls in a row share the scratch
        out = torch.full_like(q, float("nan"))
        lse = torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(fn, case, q, out, lse, max_len, splits) == 0
        ref_out, ref_lse = _regular(case, q, max_len, splits)
        torch.cuda.synchronize()
        assert_attention_close(to_f64(out), to_f64(ref_out), BF16, what="noalloc vs regular")
        assert np.max(np.abs(lse.cpu().double().numpy() - ref_lse.cpu().double().numpy())) <= 1e-3


def test_noalloc_rejects_plans_beyond_the_scratch():
    fn = _lib()
    case = W.decode_case([40, 50], 8, 2, 128, 16, BF16, BF16, seed=91, device="cuda")
    out = torch.empty_like(case.q)
    # 2 requests x 8 heads x 8,000 splits x 129 floats x 4 bytes = 66 MB of partials > 16 MiB
    big = 128_000
    assert pkv.decode_workspace_bytes(case.k_cache, 2, 8, big, 8000) > SCRATCH_BYTES
    assert _noalloc(fn, case, case.q, out, None, big, 8000) == 3      # PKV_ERR_WORKSPACE
    assert _noalloc(fn, case, case.q, out, None, 64, 1) == 0          # one split needs no scratch
    torch.cuda.synchronize()
