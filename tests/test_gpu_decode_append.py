"""GPU tests of pkv_paged_decode_attn_append (the current token's K/V written
by the decode kernel itself): the same output bits and the same cache bytes
as pkv_kv_append at position seq_len-1 followed by pkv_paged_decode_attn, for
every cache dtype, several split counts, a request whose new token opens a
fresh block, a single-token request and an empty one; and parity with the
oracle applying its own append to the pre-append pool."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_285_gb300 as pkv
from paged_kv_cache_285_gb300 import workloads as W
from tests.pkv_testlib import BF16, E4M3, F16, assert_attention_close, to_f64

pytestmark = pytest.mark.gpu
S = W.to_numpy_storage


def _ws(case, n_max, splits):
    b = case.q.shape[0]
    nbytes = pkv.decode_workspace_bytes(case.k_cache, b, case.num_q_heads, n_max, splits,
                                        case.k_scale, case.v_scale)
    return torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")


def _run(case, fused, splits):
    lens = case.seq_lens
    n_max = int(lens.max())
    b = case.q.shape[0]
    out = torch.full_like(case.q, float("nan"))
    lse = torch.full((b, case.num_q_heads), float("nan"), dtype=torch.float32, device="cuda")
    kw = dict(k_scale=case.k_scale, v_scale=case.v_scale, num_splits=splits, lse_out=lse,
              workspace=_ws(case, n_max, splits))
    if fused:
        pkv.paged_decode_attn_append(case.k_cache, case.v_cache, case.new_k, case.new_v, case.q,
                                     out, case.block_tables, lens, case.sm_scale, n_max, **kw)
    else:
        pkv.kv_append(case.k_cache, case.v_cache, case.new_k, case.new_v, case.slot_last,
                      k_scale=case.k_scale, v_scale=case.v_scale)
        pkv.paged_decode_attn(case.k_cache, case.v_cache, case.q, out, case.block_tables, lens,
                              case.sm_scale, n_max, **kw)
    torch.cuda.synchronize()
    return out, lse


CASES = [
    # (seq_lens, hq, hkv, d, bs, cache dtype, act dtype)
    ([200, 3, 64, 17, 1, 0, 130], 8, 2, 128, 16, BF16, BF16),
    ([37, 60, 16, 1], 4, 1, 64, 16, F16, F16),
    ([33, 250, 4096, 65], 32, 8, 128, 32, BF16, BF16),
    ([200, 3, 64, 17], 64, 8, 128, 16, E4M3, BF16),
    ([45, 90, 16, 1], 8, 1, 64, 16, E4M3, F16),
    # groups above 8: every head chunk's CTA writes the current token's row (the same bytes)
    ([130, 17, 1, 600], 64, 4, 128, 16, BF16, BF16),
    ([300, 5, 33], 96, 8, 128, 16, E4M3, BF16),
]


@pytest.mark.parametrize("splits", [0, 1, 3])
@pytest.mark.parametrize("cfg", CASES, ids=lambda c: f"n{c[0]}-h{c[1]}x{c[2]}-d{c[3]}-bs{c[4]}-c{c[5]}-a{c[6]}")
def test_fused_append_equals_append_then_decode(cfg, splits):
    lens, hq, hkv, d, bs, ct, at = cfg
    seed = sum(lens) + hq + splits
    ref_case = W.decode_case(lens, hq, hkv, d, bs, ct, at, seed=seed, device="cuda")
    fused_case = W.decode_case(lens, hq, hkv, d, bs, ct, at, seed=seed, device="cuda")
    k0, v0 = S(ref_case.k_cache), S(ref_case.v_cache)
    out_r, lse_r = _run(ref_case, False, splits)
    out_f, lse_f = _run(fused_case, True, splits)
    # identical cache bytes and identical results (the same kernel reads the same bytes)
    assert np.array_equal(S(ref_case.k_cache), S(fused_case.k_cache))
    assert np.array_equal(S(ref_case.v_cache), S(fused_case.v_cache))
    assert torch.equal(out_r.view(torch.int16), out_f.view(torch.int16))
    assert torch.equal(lse_r.view(torch.int32), lse_f.view(torch.int32))
    # and the oracle, appending on its own copy of the pre-append pool
    kr, vr, st = oracle.kv_append(k0, v0, ct, ref_case.k_scale, ref_case.v_scale, S(ref_case.new_k),
                                  S(ref_case.new_v), at, ref_case.slot_last.cpu().numpy())
    assert st == 0
    assert np.array_equal(kr, S(fused_case.k_cache)) and np.array_equal(vr, S(fused_case.v_cache))
    ref, ref_lse, st = oracle.paged_decode(kr, vr, ct, ref_case.k_scale, ref_case.v_scale,
                                           S(ref_case.q), at, ref_case.block_tables.cpu().numpy(),
                                           ref_case.seq_lens.cpu().numpy(), hq, ref_case.sm_scale)
    assert st == 0
    got = to_f64(out_f)
    assert_attention_close(got, ref, at, fp8=(ct == E4M3), what=str(cfg))
    assert pkv.get_device_error() == 0


def test_fused_append_llama3_8b_layer():
    # the benchmark's layer: fused step == append + decode, bit for bit
    a = W.llama3_8b_decode(device="cuda")
    bcase = W.llama3_8b_decode(device="cuda")
    out_r, _ = _run(a, False, 0)
    out_f, _ = _run(bcase, True, 0)
    assert torch.equal(out_r.view(torch.int16), out_f.view(torch.int16))
    assert torch.equal(a.k_cache.view(torch.int16), bcase.k_cache.view(torch.int16))
    assert torch.equal(a.v_cache.view(torch.int16), bcase.v_cache.view(torch.int16))
    assert pkv.get_device_error() == 0


def test_fused_append_rejects_half_inputs():
    case = W.decode_case([20], 4, 1, 64, 16, F16, F16, seed=3, device="cuda")
    with pytest.raises((pkv.PkvError, ValueError)):
        pkv.paged_decode_attn_append(case.k_cache, case.v_cache, case.new_k, None, case.q,
                                     torch.empty_like(case.q), case.block_tables, case.seq_lens,
                                     case.sm_scale, 20)


class _Mapped:
    """Device-addressable view of a pinned host tensor (the GPU reads and writes
    it directly over the host link)."""

    def __init__(self, t):
        self.__cuda_array_interface__ = {"shape": tuple(t.shape), "typestr": _typestr(t.dtype),
                                         "data": (t.data_ptr(), False), "version": 3}


def _typestr(dt):
    return {torch.int32: "<i4", torch.float32: "<f4", torch.float16: "<f2",
            torch.int16: "<i2"}[dt]


def _on_host(t):
    """A pinned host copy of t and a CUDA tensor addressing the same host bytes
    (16-bit floats travel as int16: only their bits matter)."""
    bits = t.view(torch.int16) if t.element_size() == 2 and t.is_floating_point() else t
    h = bits.cpu().pin_memory()
    d = torch.as_tensor(_Mapped(h), device="cuda")
    assert d.data_ptr() == h.data_ptr()
    return h, (d.view(t.dtype) if d.dtype != t.dtype else d)


@pytest.mark.parametrize("cfg", [CASES[0], CASES[3]], ids=["bf16", "fp8"])
def test_zero_copy_host_buffers_give_the_same_bits(cfg):
    # q, the new K/V, block tables, seq_lens, out and lse_out in pinned host
    # memory, read and written by the kernels over the host link: the same bits
    # as the same call on device buffers (caches and workspace stay on device)
    lens, hq, hkv, d, bs, dt, act = cfg
    dev = W.decode_case(lens, hq, hkv, d, bs, dt, act, seed=77, device="cuda")
    host = W.decode_case(lens, hq, hkv, d, bs, dt, act, seed=77, device="cuda")
    ref_out, ref_lse = _run(dev, True, 0)
    n_max = int(host.seq_lens.max())
    b = host.q.shape[0]
    args = {}
    keep = []
    for name in ("q", "new_k", "new_v", "block_tables", "seq_lens"):
        h, view = _on_host(getattr(host, name))
        keep.append(h)
        args[name] = view
    out_h, out_v = _on_host(torch.full_like(host.q, float("nan")))
    lse_h, lse_v = _on_host(torch.full((b, hq), float("nan"), dtype=torch.float32, device="cuda"))
    pkv.paged_decode_attn_append(host.k_cache, host.v_cache, args["new_k"], args["new_v"],
                                 args["q"], out_v, args["block_tables"], args["seq_lens"],
                                 host.sm_scale, n_max, k_scale=host.k_scale, v_scale=host.v_scale,
                                 lse_out=lse_v, workspace=_ws(host, n_max, 0))
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.int16), ref_out.view(torch.int16).cpu())
    assert torch.equal(lse_h, ref_lse.cpu())
    assert np.array_equal(S(host.k_cache), S(dev.k_cache))
    assert np.array_equal(S(host.v_cache), S(dev.v_cache))
    assert pkv.get_device_error() == 0
