"""GPU parity of the extend kernels' softmax when a row's maximum grows along
its keys.  The kernels keep a running maximum as the exponent's base and move
it only when a key tile's maximum exceeds it by more than 2^8, rescaling O in
TMEM then.  Random data never does that after the first tile, so these cases
scale each key tile's K by a factor that grows with its position (the pool's
values, read the same way by the oracle), and check on the host that some
fully visible tile after the first does raise a row's maximum past that
margin.  Plain, widened, shared-prefix and fp8 paths, head_dim 64 and 128,
against the fp64 oracle."""
import math

import numpy as np
import pytest
import torch

import paged_kv_cache_285_gb300 as pkv
from paged_kv_cache_285_gb300 import workloads as W
from tests.pkv_testlib import BF16, E4M3, F16
from tests.test_gpu_extend import check
from tests.test_gpu_extend_shared_prefix import check as check_shared
from tests.test_gpu_extend_shared_prefix import grouped_extend_case, run_shared

pytestmark = pytest.mark.gpu
BN = 128  # keys per tile of the extend kernels


def grow_keys(case, g, q_mul):
    """K of key tile t (keys 128 t .. 128 t + 127 of a request) times
    g^(t - t_max): every physical block once (shared blocks hold the same
    positions in every table that names them); the queries times q_mul."""
    bs = case.k_cache.shape[2]
    tables = case.block_tables.cpu().numpy()
    tot = (case.prefix_lens.cpu() + (case.q_indptr[1:] - case.q_indptr[:-1]).cpu()).numpy()
    t_max = (int(tot.max()) - 1) // BN
    seen = {}
    for b in range(tables.shape[0]):
        for i in range(math.ceil(int(tot[b]) / bs)):
            seen.setdefault(int(tables[b, i]), (i * bs) // BN)
    for blk, t in seen.items():
        f = g ** (t - t_max)
        if case.k_cache.dtype == torch.uint8:
            v = case.k_cache[blk].view(torch.float8_e4m3fn).float() * f
            case.k_cache[blk] = v.to(torch.float8_e4m3fn).view(torch.uint8)
        else:
            case.k_cache[blk] = (case.k_cache[blk].float() * f).to(case.k_cache.dtype)
    case.q.copy_((case.q.float() * q_mul).to(case.q.dtype))


def assert_max_grows(case, margin=8.0):
    """Some row's running maximum (base 2, over whole key tiles before its
    diagonal) grows by more than `margin` at a tile after the first."""
    if case.k_cache.dtype == torch.uint8:
        k = case.k_cache.cpu().view(torch.float8_e4m3fn).double().numpy() * case.k_scale
    else:
        k = case.k_cache.cpu().double().numpy()
    q = case.q.float().cpu().numpy().astype(np.float64)
    tables = case.block_tables.cpu().numpy()
    qi = case.q_indptr.cpu().numpy()
    P = case.prefix_lens.cpu().numpy()
    bs, hkv = k.shape[2], k.shape[1]
    G = q.shape[1] // hkv
    scale = case.sm_scale * math.log2(math.e)
    for b in range(len(P)):
        if qi[b + 1] == qi[b] or P[b] < 2 * BN:
            continue
        full = int(P[b]) // BN  # tiles every suffix row sees whole
        keys = np.concatenate([k[tables[b, i]] for i in range(math.ceil(full * BN / bs))], axis=1)
        for h in range(q.shape[1]):
            s = keys[h // G, :full * BN] @ q[qi[b], h] * scale
            m = np.maximum.accumulate(s.reshape(full, BN).max(axis=1))
            if np.any(m[1:] - m[:-1] > margin):
                return
    raise AssertionError("no row's maximum grows past the margin: the case misses its path")


def run_plain(case, workspace=False):
    out = torch.full_like(case.q, float("nan"))
    rows, hq, _ = case.q.shape
    lse = torch.full((rows, hq), float("nan"), dtype=torch.float32, device="cuda")
    suf = (case.q_indptr[1:] - case.q_indptr[:-1]).cpu()
    tot = case.prefix_lens.cpu() + suf
    ws = None
    if workspace:
        n = pkv.extend_widen_workspace_bytes(case.k_cache, case.k_scale, case.v_scale)
        ws = torch.full((max(n, 256),), 0xFF, dtype=torch.uint8, device="cuda")
    pkv.paged_extend_attn(case.k_cache, case.v_cache, case.q, out, case.q_indptr,
                          case.prefix_lens, case.block_tables, case.sm_scale, int(suf.max()),
                          int(tot.max()), k_scale=case.k_scale, v_scale=case.v_scale,
                          lse_out=lse, workspace=ws)
    torch.cuda.synchronize()
    return out, lse


CASES = [
    # (prefix_lens, suffix_lens, hq, hkv, bs, cache dtype, act dtype, head_dim,
    #  growth per key tile, query factor): 4 to 46 (row, tile) steps past the margin
    ([700, 260], [130, 70], 8, 2, 16, BF16, BF16, 128, 1.6, 16.0),
    ([900, 400, 33], [40, 129, 7], 16, 2, 32, F16, F16, 128, 2.5, 16.0),
    ([700, 260], [130, 70], 8, 2, 16, BF16, BF16, 64, 1.6, 16.0),
    ([1100], [60], 32, 8, 16, BF16, BF16, 128, 1.6, 24.0),
    ([1100], [60], 32, 8, 16, BF16, BF16, 128, 2.0, 24.0),
    ([700, 300], [100, 50], 8, 2, 16, E4M3, BF16, 128, 1.6, 16.0),
    ([700, 300], [100, 50], 8, 2, 16, E4M3, F16, 64, 1.6, 16.0),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: (
    f"P{c[0]}-S{c[1]}-h{c[2]}x{c[3]}-bs{c[4]}-c{c[5]}-a{c[6]}-hd{c[7]}-g{c[8]}-q{c[9]}"))
def test_extend_with_growing_maximum(cfg):
    P, Sx, hq, hkv, bs, cdt, adt, hd, g, q_mul = cfg
    case = W.extend_case(P, Sx, hq, hkv, hd, bs, cdt, adt, seed=400 + hd + len(P), device="cuda")
    grow_keys(case, g, q_mul)
    assert_max_grows(case)
    fp8 = cdt == E4M3
    out, lse = run_plain(case)
    check(case, out, lse, "growing max " + str(cfg), fp8=fp8)
    if cdt != F16:
        wo, wl = run_plain(case, workspace=True)
        check(case, wo, wl, "growing max, widened " + str(cfg), fp8=fp8)
        if not (fp8 and adt == BF16):
            assert torch.equal(out.view(torch.int16), wo.view(torch.int16))
            assert torch.equal(lse.view(torch.int32), wl.view(torch.int32))
    assert pkv.get_device_error() == 0


@pytest.mark.parametrize("cdt,hd", [(BF16, 128), (BF16, 64), (E4M3, 128)])
def test_shared_prefix_extend_with_growing_maximum(cdt, hd):
    # three requests over a 640-token shared prefix (5 key tiles), one alone
    P, Sx, groups, shared = [640, 700, 660, 300], [60, 45, 130, 20], [0, 3, 4], [640, 0]
    case = grouped_extend_case(P, Sx, groups, shared, 8, 2, hd, 16, cdt, BF16, seed=410 + hd)
    grow_keys(case, 2.5, 16.0)
    assert_max_grows(case)
    for ws in (False, True):
        out, lse = run_shared(case, groups, shared, workspace=ws)
        check_shared(case, out, lse, f"shared prefix, growing max, workspace {ws}",
                     fp8=cdt == E4M3)
    assert pkv.get_device_error() == 0
