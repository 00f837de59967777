"""GPU checks of pkv_paged_extend_attn's optional widening workspace: each
cache block the call reads is widened once into 16-bit pools (V to f16 for a
bf16 cache; K to the queries' type and V to f16 for an fp8 cache), a block
that several requests share claimed by the first of them.  The same
conversions as the per-tile path, so the output and LSE bits match it, except
for an fp8 cache under bf16 queries (the queries stay bf16 for S = Q K^T),
checked against the fp64 oracle instead.  The workspace arrives filled with
garbage: the call may rely neither on its pools nor on its claim flags."""
import numpy as np
import pytest
import torch

import paged_kv_cache_285_gb300 as pkv
from paged_kv_cache_285_gb300 import workloads as W
from tests.pkv_testlib import BF16, E4M3, F16
from tests.test_gpu_extend import check

pytestmark = pytest.mark.gpu


def run(case, workspace=None):
    out = torch.full_like(case.q, float("nan"))
    rows, hq, _ = case.q.shape
    lse = torch.full((rows, hq), float("nan"), dtype=torch.float32, device="cuda")
    suf = (case.q_indptr[1:] - case.q_indptr[:-1]).cpu()
    tot = case.prefix_lens.cpu() + suf
    pkv.paged_extend_attn(case.k_cache, case.v_cache, case.q, out, case.q_indptr,
                          case.prefix_lens, case.block_tables, case.sm_scale, int(suf.max()),
                          int(tot.max()), k_scale=case.k_scale, v_scale=case.v_scale,
                          lse_out=lse, workspace=workspace)
    torch.cuda.synchronize()
    return out, lse


def garbage_workspace(case, extra=0, fill=0xFF):
    n = pkv.extend_widen_workspace_bytes(case.k_cache, case.k_scale, case.v_scale)
    assert n > 0
    # 0xFF everywhere: NaN in both 16-bit pools, and every claim flag already set
    return torch.full((n + extra,), fill, dtype=torch.uint8, device="cuda")


def same_bits(a, b):
    (oa, la), (ob, lb) = a, b
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(la.view(torch.int32), lb.view(torch.int32))


CASES = [
    # (prefix_lens, suffix_lens, hq, hkv, bs, cache dtype, act dtype, head_dim)
    ([0, 13, 30, 200], [37, 19, 130, 1], 8, 2, 16, BF16, BF16, 128),
    ([1900], [100], 32, 8, 16, BF16, BF16, 128),
    ([129, 64, 1], [200, 17, 256], 64, 8, 16, BF16, BF16, 64),
    ([100, 0], [300, 129], 8, 8, 32, BF16, BF16, 128),
    ([40, 7, 0, 300, 0], [0, 50, 0, 3, 0], 8, 2, 16, BF16, BF16, 128),
    ([33, 0, 90], [70, 45, 130], 12, 4, 16, E4M3, F16, 128),
    ([0, 13, 30, 200], [37, 19, 130, 1], 8, 2, 16, E4M3, F16, 64),
    ([500, 7], [40, 250], 24, 4, 32, E4M3, F16, 128),
    ([0, 13, 30, 200], [37, 19, 130, 1], 8, 2, 16, E4M3, BF16, 128),
    ([1900], [100], 32, 8, 16, E4M3, BF16, 128),
    ([129, 64, 1], [200, 17, 256], 64, 8, 16, E4M3, BF16, 64),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: (
    f"P{c[0]}-S{c[1]}-h{c[2]}x{c[3]}-bs{c[4]}-c{c[5]}-a{c[6]}-hd{c[7]}"))
def test_widened_extend(cfg):
    P, Sx, hq, hkv, bs, cdt, adt, hd = cfg
    case = W.extend_case(P, Sx, hq, hkv, hd, bs, cdt, adt, seed=300 + sum(Sx) + hd,
                         device="cuda")
    plain = run(case)
    wide = run(case, garbage_workspace(case))
    fp8 = cdt == E4M3
    check(case, *wide, "widened " + str(cfg), fp8=fp8)
    if not (fp8 and adt == BF16):
        same_bits(plain, wide)
    assert pkv.get_device_error() == 0


@pytest.mark.parametrize("cdt,adt", [(BF16, BF16), (E4M3, F16), (E4M3, BF16)])
def test_shared_blocks_are_widened_once_and_read_by_all(cdt, adt):
    # 64 requests whose tables share a 1,900-token prefix (118 whole blocks):
    # one of them claims each shared block; sampled rows of every request
    case = W.extend_case([1900] * 64, [100] * 64, 32, 8, 128, 16, cdt, adt, seed=310,
                         device="cuda", shared_prefix=1900)
    plain = run(case)
    wide = run(case, garbage_workspace(case))
    rng = np.random.default_rng(7)
    rows = [(int(r), int(h)) for r, h in zip(rng.integers(0, case.q.shape[0], 256),
                                             rng.integers(0, 32, 256))]
    check(case, *wide, "shared blocks widened", rows=rows, fp8=cdt == E4M3)
    if cdt == BF16 or adt == F16:
        same_bits(plain, wide)
    assert pkv.get_device_error() == 0


def test_workspace_reused_after_the_cache_changed():
    # the claim flags are cleared by every call: a second call over new page
    # contents widens them again instead of reading the first call's copies
    case = W.extend_case([64, 200], [30, 77], 8, 2, 128, 16, BF16, BF16, seed=320, device="cuda")
    ws = garbage_workspace(case)
    run(case, ws)
    torch.manual_seed(321)
    case.v_cache.copy_(torch.randn_like(case.v_cache, dtype=torch.float32).to(torch.bfloat16))
    case.k_cache.copy_(torch.randn_like(case.k_cache, dtype=torch.float32).to(torch.bfloat16))
    plain = run(case)
    wide = run(case, ws)
    same_bits(plain, wide)
    check(case, *wide, "reused workspace")


def test_small_workspace_takes_the_per_tile_path():
    # a workspace below the widening size (the 0 bytes pkv_extend_workspace_bytes
    # asks for, or one byte short) is not used: the same bits as none
    case = W.extend_case([30, 200], [50, 77], 8, 2, 128, 16, E4M3, BF16, seed=330, device="cuda")
    need = pkv.extend_widen_workspace_bytes(case.k_cache, case.k_scale, case.v_scale)
    plain = run(case)
    short = torch.full((need - 1,), 0xFF, dtype=torch.uint8, device="cuda")
    same_bits(plain, run(case, short))
    # a larger one is used (fp8 under bf16 queries: bf16 scores, other bits)
    wide = run(case, garbage_workspace(case, extra=4096))
    check(case, *wide, "larger workspace", fp8=True)
    assert pkv.get_device_error() == 0


def test_f16_cache_needs_no_widening():
    case = W.extend_case([30], [50], 8, 2, 128, 16, F16, F16, seed=340, device="cuda")
    assert pkv.extend_widen_workspace_bytes(case.k_cache) == 0
    ws = torch.full((1 << 16,), 0xFF, dtype=torch.uint8, device="cuda")
    same_bits(run(case), run(case, ws))


@pytest.mark.parametrize("hd", [128, 64])
def test_widened_garbage_past_end_is_ignored(hd):
    # NaN codes past the last key of a block are widened too; the kernel still
    # zeroes the keys past the end before P V
    case = W.extend_case([30], [20], 8, 2, hd, 16, E4M3, BF16, seed=350, device="cuda")
    total = 50
    blk = int(case.block_tables[0, (total - 1) // 16])
    case.k_cache[blk, :, total % 16:] = 0x7F
    case.v_cache[blk, :, total % 16:] = 0xFF
    check(case, *run(case, garbage_workspace(case)), "widened garbage tail", fp8=True)


def test_widened_extend_on_the_benchmark_workload():
    # the 256-request suffix prefill of the shared-prefix workload through the
    # plain call, with and without the workspace: every bit the same (bf16)
    case = W.shared_prefix_extend(device="cuda")
    same_bits(run(case), run(case, garbage_workspace(case)))
    assert pkv.get_device_error() == 0


def test_request_longer_than_the_length_hint_is_widened_whole():
    # the kernels read every key through the table whatever max_total_len says;
    # the widening passes, whose grids that hint sizes, cover every block too
    # (a 5,000-token request is 313 blocks; the hint's grid claims 256 at once)
    case = W.extend_case([4950, 20], [50, 30], 8, 2, 128, 16, E4M3, BF16, seed=360, device="cuda")
    suf = (case.q_indptr[1:] - case.q_indptr[:-1]).cpu()
    outs = []
    for ws in (None, garbage_workspace(case)):
        out = torch.full_like(case.q, float("nan"))
        lse = torch.full(case.q.shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        pkv.paged_extend_attn(case.k_cache, case.v_cache, case.q, out, case.q_indptr,
                              case.prefix_lens, case.block_tables, case.sm_scale, int(suf.max()),
                              100, k_scale=case.k_scale, v_scale=case.v_scale, lse_out=lse,
                              workspace=ws)
        torch.cuda.synchronize()
        outs.append((out, lse))
    for out, lse in outs:
        check(case, out, lse, "length hint below the request", fp8=True)
    assert pkv.get_device_error() == 0
