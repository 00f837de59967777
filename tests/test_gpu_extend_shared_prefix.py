"""GPU parity of pkv_paged_extend_attn_shared_prefix (suffix prefill with the
rows of each group's requests packed into shared tiles) against the fp64
oracle's plain extend: one group over a long shared prefix, several groups with
different shared lengths (block-aligned and not), groups of one request, a
shared length of 0, empty requests, one-token suffixes (many requests per tile
pair), GQA groups 1 to 16, head_dim 64 and 128, both block sizes, 16-bit and
fp8 caches; the benchmark's 256-request workload (sampled rows); and the
device-side checks of the grouping contract."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_285_gb300 as pkv
from paged_kv_cache_285_gb300 import workloads as W
from tests.pkv_testlib import BF16, E4M3, F16, assert_attention_close, to_f64

pytestmark = pytest.mark.gpu
S = W.to_numpy_storage


def grouped_extend_case(P, Sx, groups, shared, hq, hkv, hd, bs, cdt, adt, seed):
    """extend_case whose group members point the first shared[g] // bs entries of
    their tables at the group's first member's blocks (the blocks they share)."""
    case = W.extend_case(P, Sx, hq, hkv, hd, bs, cdt, adt, seed=seed, device="cuda")
    tables = case.block_tables.cpu()
    for g in range(len(groups) - 1):
        a, b = groups[g], groups[g + 1]
        nb = shared[g] // bs
        for r in range(a + 1, b):
            tables[r, :nb] = tables[a, :nb]
    case.block_tables.copy_(tables.to(case.block_tables.device))
    return case


def run_shared(case, groups, shared, max_group_rows=None, lse=True, workspace=False):
    """workspace: give the call its optional workspace (bf16 caches widen their V
    pages into it first), filled with 0xFF bytes (NaN halves) beforehand."""
    rows, hq, _ = case.q.shape
    ws = None
    if workspace:
        nbytes = pkv.extend_shared_prefix_workspace_bytes(case.k_cache, case.k_scale, case.v_scale)
        ws = torch.full((max(nbytes, 256),), 0xFF, dtype=torch.uint8, device="cuda")
    out = torch.full_like(case.q, float("nan"))
    lse_t = torch.full((rows, hq), float("nan"), dtype=torch.float32, device="cuda") if lse else None
    qi = case.q_indptr.cpu()
    gi = torch.tensor(groups, dtype=torch.int32)
    if max_group_rows is None:
        max_group_rows = int((qi[gi[1:].long()] - qi[gi[:-1].long()]).max())
    tot = case.prefix_lens.cpu() + (qi[1:] - qi[:-1])
    pkv.paged_extend_attn_shared_prefix(
        case.k_cache, case.v_cache, case.q, out, case.q_indptr, case.prefix_lens,
        case.block_tables, gi.to("cuda"), torch.tensor(shared, dtype=torch.int32, device="cuda"),
        case.sm_scale, max_group_rows, int(tot.max()), k_scale=case.k_scale, v_scale=case.v_scale,
        lse_out=lse_t, workspace=ws)
    torch.cuda.synchronize()
    return out, lse_t


def check(case, out, lse, what, rows=None, fp8=False):
    args = (S(case.k_cache), S(case.v_cache), case.cache_dtype, case.k_scale, case.v_scale,
            S(case.q), case.act_dtype, case.q_indptr.cpu().numpy(), case.prefix_lens.cpu().numpy(),
            case.block_tables.cpu().numpy(), case.num_q_heads, case.sm_scale)
    ref, ref_lse, st = oracle.paged_extend(*args, rows=rows)
    assert st == 0
    got, gl = to_f64(out), lse.cpu().double().numpy()
    if rows is not None:
        got = np.stack([got[r, h] for r, h in rows])
        gl = np.array([gl[r, h] for r, h in rows])
    assert_attention_close(got, ref, case.act_dtype, fp8=fp8, what=what)
    assert np.max(np.abs(gl - ref_lse)) <= (3e-2 if fp8 else 1e-3), what


CASES = [
    # (prefix_lens, suffix_lens, groups (request offsets), shared lens, hq, hkv, bs, cache, act, hd)
    # one group, shared prefix ending mid-block (rounded down to whole blocks)
    ([300, 310, 305], [40, 70, 25], [0, 3], [300], 8, 2, 16, BF16, BF16, 128),
    # two groups, one of a single request; shared lengths 0 and block-aligned
    ([64, 90, 0, 33], [100, 50, 7, 130], [0, 2, 4], [64, 0], 16, 4, 16, BF16, BF16, 128),
    # many one-token suffixes: dozens of requests in one tile pair
    ([200] * 40, [1] * 40, [0, 40], [200], 32, 8, 16, F16, F16, 128),
    # empty requests inside a group, GQA 3 (42-token tiles), block size 32
    ([96, 96, 128, 100, 97], [0, 60, 0, 45, 90], [0, 5], [96], 12, 4, 32, BF16, BF16, 128),
    # MHA and GQA 16; three groups
    ([500, 520, 40, 41, 1000], [20, 200, 64, 3, 129], [0, 2, 4, 5], [500, 40, 999], 16, 16, 16,
     F16, F16, 128),
    ([150, 160, 170], [30, 40, 50], [0, 3], [150], 32, 2, 16, BF16, BF16, 128),
    # head_dim 64
    ([300, 310, 305], [40, 70, 25], [0, 3], [300], 8, 2, 16, BF16, BF16, 64),
    ([64, 90, 0, 33], [100, 50, 7, 130], [0, 2, 4], [64, 0], 16, 4, 32, F16, F16, 64),
    # fp8 e4m3 caches with either act dtype
    ([300, 310, 305], [40, 70, 25], [0, 3], [300], 8, 2, 16, E4M3, BF16, 128),
    ([64, 90, 0, 33], [100, 50, 7, 130], [0, 2, 4], [64, 0], 16, 4, 16, E4M3, F16, 64),
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: f"P{c[0][:3]}-S{c[1][:3]}-g{c[2]}-W{c[3]}-"
                                                     f"h{c[4]}x{c[5]}-bs{c[6]}-{c[7]}{c[8]}-hd{c[9]}")
def test_shared_prefix_extend_matches_oracle(cfg):
    P, Sx, groups, shared, hq, hkv, bs, cdt, adt, hd = cfg
    case = grouped_extend_case(P, Sx, groups, shared, hq, hkv, hd, bs, cdt, adt,
                               seed=sum(P) + sum(Sx) + hq + hd)
    out, lse = run_shared(case, groups, shared)
    check(case, out, lse, str(cfg), fp8=(cdt == E4M3))
    assert pkv.get_device_error() == 0


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: f"P{c[0][:3]}-g{c[2]}-W{c[3]}-h{c[4]}x{c[5]}-"
                                                     f"bs{c[6]}-{c[7]}{c[8]}-hd{c[9]}")
def test_workspace_gives_the_same_bits(cfg):
    # a bf16 cache's V pages (an fp8 cache's K and V pages) widened once per call
    # into the workspace and read from there, against the per-tile conversion in
    # shared memory: the same conversions, so the same output and LSE bits -- except
    # for an fp8 cache under bf16 queries, whose K is widened to bf16 so that the
    # queries need no rounding to f16 (as the per-tile path does): checked against
    # the oracle and within rounding of the per-tile path; an f16 cache takes no
    # workspace
    P, Sx, groups, shared, hq, hkv, bs, cdt, adt, hd = cfg
    case = grouped_extend_case(P, Sx, groups, shared, hq, hkv, hd, bs, cdt, adt,
                               seed=sum(P) + sum(Sx) + hq + hd + 1)
    nbytes = pkv.extend_shared_prefix_workspace_bytes(case.k_cache, case.k_scale, case.v_scale)
    pool16 = (case.v_cache.numel() * 2 + 255) // 256 * 256  # elements x 2 bytes
    assert nbytes == {BF16: pool16, E4M3: 2 * pool16}.get(cdt, 0)
    out_a, lse_a = run_shared(case, groups, shared)
    out_b, lse_b = run_shared(case, groups, shared, workspace=True)
    if cdt == E4M3 and adt == BF16:
        check(case, out_b, lse_b, str(cfg) + " with workspace", fp8=True)
        assert np.max(np.abs(to_f64(out_a) - to_f64(out_b))) <= 1.6e-2  # two bf16 ulps at 1
        assert torch.allclose(lse_a, lse_b, atol=1e-3, rtol=0)
    else:
        assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
        assert torch.equal(lse_a.view(torch.int32), lse_b.view(torch.int32))
    assert pkv.get_device_error() == 0


def test_workspace_on_the_benchmark_workload():
    # 256 requests over one shared 1,900-token prefix: every output bit the same
    # with the V pages widened once per call
    case = W.shared_prefix_extend(device="cuda")
    out_a, lse_a = run_shared(case, [0, 256], [1900])
    out_b, lse_b = run_shared(case, [0, 256], [1900], workspace=True)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(lse_a.view(torch.int32), lse_b.view(torch.int32))
    assert pkv.get_device_error() == 0


def test_shared_prefix_extend_equals_plain_extend():
    # same rows through the plain call: the two layouts agree to rounding
    P, Sx, groups, shared = [64, 90, 0, 33], [100, 50, 7, 130], [0, 2, 4], [64, 0]
    case = grouped_extend_case(P, Sx, groups, shared, 16, 4, 128, 16, BF16, BF16, seed=5)
    out_s, lse_s = run_shared(case, groups, shared)
    out_p = torch.empty_like(case.q)
    lse_p = torch.empty_like(lse_s)
    pkv.paged_extend_attn(case.k_cache, case.v_cache, case.q, out_p, case.q_indptr,
                          case.prefix_lens, case.block_tables, case.sm_scale, 130, 163,
                          lse_out=lse_p)
    torch.cuda.synchronize()
    a, b = to_f64(out_s), to_f64(out_p)
    assert np.max(np.abs(a - b)) <= 4e-3
    assert torch.allclose(lse_s, lse_p, atol=1e-4, rtol=0)


def test_shared_prefix_extend_workload_sampled():
    # the benchmark's launch: 256 requests x 100 suffix rows over one shared 1,900-token
    # prefix (1,888 tokens in shared blocks); rows from packed tiles that straddle
    # requests, every head, against the oracle
    case = W.shared_prefix_extend(device="cuda")
    out, lse = run_shared(case, [0, 256], [1900])
    reqs = [0, 1, 63, 64, 127, 200, 254, 255]
    toks = [0, 27, 28, 31, 32, 60, 96, 99]
    rows = [(r * 100 + i, h) for r in reqs for i in toks for h in range(32)]
    check(case, out, lse, "shared-prefix extend (packed)", rows=rows)
    assert pkv.get_device_error() == 0


def test_shared_prefix_extend_rejects_a_short_prefix_on_the_device():
    # a member whose prefix is shorter than the group's shared length breaks the
    # contract: its tile pair is not computed and the length error is reported
    case = grouped_extend_case([96, 40], [20, 20], [0, 2], [32], 8, 2, 128, 16, BF16, BF16, seed=3)
    assert pkv.get_device_error() == 0
    out, _ = run_shared(case, [0, 2], [64], lse=False)
    assert pkv.get_device_error() == 3
    assert torch.isnan(out.float()).all()  # nothing written


def test_shared_prefix_extend_reports_rows_beyond_the_hint():
    case = grouped_extend_case([40, 41], [100, 100], [0, 2], [32], 8, 2, 128, 16, BF16, BF16,
                               seed=4)
    assert pkv.get_device_error() == 0
    run_shared(case, [0, 2], [32], max_group_rows=64, lse=False)
    assert pkv.get_device_error() == 3


def test_shared_prefix_extend_host_refusals():
    case = grouped_extend_case([40], [10], [0, 1], [32], 8, 2, 128, 16, BF16, BF16, seed=6)
    out = torch.empty_like(case.q)
    gi = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    gs = torch.tensor([32], dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):  # group lengths of the wrong shape
        pkv.paged_extend_attn_shared_prefix(case.k_cache, case.v_cache, case.q, out,
                                            case.q_indptr, case.prefix_lens, case.block_tables,
                                            gi, gs[:0], case.sm_scale, 10, 50)
    with pytest.raises(RuntimeError):  # negative row hint
        pkv.paged_extend_attn_shared_prefix(case.k_cache, case.v_cache, case.q, out,
                                            case.q_indptr, case.prefix_lens, case.block_tables,
                                            gi, gs, case.sm_scale, -1, 50)
    assert pkv.get_device_error() == 0
