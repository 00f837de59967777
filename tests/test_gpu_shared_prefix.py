"""GPU parity of pkv_paged_decode_attn_shared_prefix (decode for groups of
requests that share a cached prefix, the prefix attended once per group on
the tensor cores and merged by LSE with each request's own tokens) against
the fp64 oracle's plain decode over every request's whole sequence.

"KV Cache 완전 정리 — PagedAttention vs RadixAttention, SGLang이 빠른 이유",
section "RadixAttention — SGLang의 혁신" (many requests, one shared prompt);
"PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", section 03.
Groups share their whole prefix blocks (the members' tables point at the
first member's blocks) and hold copies of the prefix's partial last block, as
a paged cache stores a shared prefix."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_285_gb300 as pkv
from paged_kv_cache_285_gb300 import workloads as W
from tests.pkv_testlib import BF16, E4M3, F16, assert_attention_close, to_f64

pytestmark = pytest.mark.gpu
S = W.to_numpy_storage


def grouped_case(groups, suffixes, hq, hkv, bs, dt, seed, hd=128, act=None):
    """groups: [(members, P)]; suffixes: one own-token count per request (>= 0); dt is the
    cache dtype, act the query / output dtype (dt unless the cache is fp8)."""
    lens = []
    it = iter(suffixes)
    for size, prefix in groups:
        lens += [prefix + next(it) for _ in range(size)]
    case = W.decode_case(lens, hq, hkv, hd, bs, dt, dt if act is None else act, seed=seed,
                         device="cuda")
    tables = case.block_tables.cpu()
    indptr, plens, start = [0], [], 0
    for size, prefix in groups:
        full, tail = prefix // bs, prefix % bs
        for m in range(start + 1, start + size):
            tables[m, :full] = tables[start, :full]
            if tail:
                src, dst = int(tables[start, full]), int(tables[m, full])
                case.k_cache[dst, :, :tail] = case.k_cache[src, :, :tail]
                case.v_cache[dst, :, :tail] = case.v_cache[src, :, :tail]
        start += size
        indptr.append(start)
        plens.append(prefix)
    case.block_tables = tables.to("cuda")
    gi = torch.tensor(indptr, dtype=torch.int32, device="cuda")
    gp = torch.tensor(plens, dtype=torch.int32, device="cuda")
    max_group = max(size for size, _ in groups)
    max_suffix = max(n - plens[g] for g, (a, e) in enumerate(zip(indptr[:-1], indptr[1:]))
                     for n in lens[a:e])
    return case, gi, gp, max_group, max_suffix


def run_cascade(case, gi, gp, max_group, max_suffix, splits=0, append=False):
    b = case.q.shape[0]
    out = torch.full_like(case.q, float("nan"))
    lse = torch.full((b, case.num_q_heads), float("nan"), dtype=torch.float32, device="cuda")
    max_prefix = int(gp.max()) if gp.numel() else 0
    nbytes = pkv.shared_prefix_decode_workspace_bytes(case.k_cache, b, case.num_q_heads,
                                                      max_prefix, max_suffix, splits)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    kw = dict(k_new=case.new_k, v_new=case.new_v) if append else {}
    pkv.paged_decode_attn_shared_prefix(case.k_cache, case.v_cache, case.q, out, case.block_tables,
                                        case.seq_lens, case.sm_scale, gi, gp, max_group,
                                        max_prefix, max_suffix, num_splits=splits, lse_out=lse,
                                        workspace=ws,
                                        k_scale=case.k_scale, v_scale=case.v_scale, **kw)
    torch.cuda.synchronize()
    return out, lse


def oracle_ref(case, pools=None, pairs=None):
    k, v = (S(case.k_cache), S(case.v_cache)) if pools is None else pools
    ref, ref_lse, st = oracle.paged_decode(k, v, case.cache_dtype, case.k_scale, case.v_scale,
                                           S(case.q),
                                           case.act_dtype, case.block_tables.cpu().numpy(),
                                           case.seq_lens.cpu().numpy(), case.num_q_heads,
                                           case.sm_scale, pairs=pairs)
    assert st == 0
    return ref, ref_lse


def check(case, out, lse, what, pools=None):
    ref, ref_lse = oracle_ref(case, pools)
    fp8 = case.cache_dtype == E4M3
    assert_attention_close(to_f64(out), ref, case.act_dtype, fp8=fp8, what=what)
    gl = lse.cpu().double().numpy()
    fin = np.isfinite(ref_lse)
    assert np.all(np.isfinite(gl) == fin), what
    assert np.max(np.abs(gl[fin] - ref_lse[fin]), initial=0) <= (3e-2 if fp8 else 1e-3), what


def rand_suffixes(n, lo, hi, seed):
    return np.random.default_rng(seed).integers(lo, hi + 1, n).tolist()


CASES = [
    # (groups [(members, P)], suffix range, hq, hkv, bs, dtype)
    ([(64, 500)], (1, 300), 32, 8, 16, BF16),
    ([(1, 0), (5, 100), (70, 1000), (3, 37), (1, 16), (2, 0)], (1, 200), 8, 2, 16, F16),
    ([(40, 256)], (1, 90), 64, 8, 32, BF16),
    ([(9, 48), (7, 480)], (1, 70), 8, 8, 16, F16),
    ([(33, 160), (2, 64)], (1, 50), 16, 8, 32, BF16),
    # long own-token runs: with one split a CTA covers > 512 tokens (the deeper
    # pipeline variant of the decode)
    ([(12, 200)], (600, 1000), 16, 8, 16, BF16),
    ([(4, 96), (6, 32)], (520, 700), 8, 2, 32, F16),
    # GQA groups above 8 (the decode takes them in chunks of 8 heads) and not a power of two
    ([(10, 300), (3, 32)], (1, 200), 64, 4, 16, BF16),
    ([(7, 128)], (1, 90), 12, 4, 32, F16),
]


@pytest.mark.parametrize("splits", [0, 1, 3])
@pytest.mark.parametrize("cfg", CASES, ids=lambda c: f"g{len(c[0])}-h{c[2]}x{c[3]}-bs{c[4]}-d{c[5]}")
def test_groups_match_oracle(cfg, splits):
    groups, (lo, hi), hq, hkv, bs, dt = cfg
    nreq = sum(s for s, _ in groups)
    case, gi, gp, mg, ms = grouped_case(groups, rand_suffixes(nreq, lo, hi, nreq + splits), hq,
                                        hkv, bs, dt, seed=nreq + hq + splits)
    out, lse = run_cascade(case, gi, gp, mg, ms, splits)
    check(case, out, lse, f"{cfg} splits={splits}")
    assert pkv.get_device_error() == 0


MORE_CASES = [
    # (groups, suffix range, hq, hkv, bs, cache dtype, act dtype, head_dim)
    ([(64, 500)], (1, 300), 32, 8, 16, BF16, BF16, 64),
    ([(1, 0), (5, 100), (30, 1000), (3, 37)], (1, 200), 4, 1, 16, F16, F16, 64),
    ([(12, 200)], (600, 1000), 16, 8, 32, BF16, BF16, 64),
    ([(64, 500)], (1, 300), 32, 8, 16, E4M3, BF16, 128),
    ([(1, 0), (5, 100), (30, 1000), (3, 37)], (1, 200), 8, 2, 16, E4M3, F16, 128),
    ([(40, 256)], (1, 90), 64, 8, 32, E4M3, BF16, 64),
    ([(12, 200)], (600, 1000), 16, 8, 16, E4M3, F16, 64),
]


@pytest.mark.parametrize("splits", [0, 3])
@pytest.mark.parametrize("cfg", MORE_CASES,
                         ids=lambda c: f"g{len(c[0])}-h{c[2]}x{c[3]}-bs{c[4]}-c{c[5]}a{c[6]}-hd{c[7]}")
def test_groups_match_oracle_d64_and_fp8(cfg, splits):
    groups, (lo, hi), hq, hkv, bs, dt, act, hd = cfg
    nreq = sum(s for s, _ in groups)
    case, gi, gp, mg, ms = grouped_case(groups, rand_suffixes(nreq, lo, hi, nreq + splits + hd), hq,
                                        hkv, bs, dt, seed=nreq + hq + splits + hd, hd=hd, act=act)
    out, lse = run_cascade(case, gi, gp, mg, ms, splits)
    check(case, out, lse, f"{cfg} splits={splits}")
    assert pkv.get_device_error() == 0


@pytest.mark.parametrize("dt,act,hd", [(E4M3, BF16, 128), (E4M3, F16, 64), (BF16, BF16, 64)])
def test_fused_append_d64_and_fp8(dt, act, hd):
    groups = [(20, 320), (6, 40)]
    suf = rand_suffixes(26, 1, 120, 6)
    case, gi, gp, mg, ms = grouped_case(groups, suf, 32, 8, 16, dt, seed=22, hd=hd, act=act)
    k0, v0 = S(case.k_cache), S(case.v_cache)
    out, lse = run_cascade(case, gi, gp, mg, ms, append=True)
    kr, vr, st = oracle.kv_append(k0, v0, case.cache_dtype, case.k_scale, case.v_scale,
                                  S(case.new_k), S(case.new_v), case.act_dtype,
                                  case.slot_last.cpu().numpy())
    assert st == 0
    assert np.array_equal(kr, S(case.k_cache)) and np.array_equal(vr, S(case.v_cache))
    check(case, out, lse, "fused append", pools=(kr, vr))
    assert pkv.get_device_error() == 0


def test_members_with_no_own_tokens():
    # seq_len == the shared prefix (whole blocks): only the prefix pass contributes
    case, gi, gp, mg, ms = grouped_case([(4, 64), (3, 96)], [0, 5, 0, 31, 0, 0, 1], 8, 2, 16,
                                        BF16, seed=11)
    out, lse = run_cascade(case, gi, gp, mg, ms)
    check(case, out, lse, "no own tokens")
    assert pkv.get_device_error() == 0


def test_fused_append_matches_append_then_oracle():
    groups = [(20, 320), (6, 40)]
    suf = rand_suffixes(26, 1, 120, 5)
    case, gi, gp, mg, ms = grouped_case(groups, suf, 32, 8, 16, BF16, seed=21)
    k0, v0 = S(case.k_cache), S(case.v_cache)
    out, lse = run_cascade(case, gi, gp, mg, ms, append=True)
    kr, vr, st = oracle.kv_append(k0, v0, case.cache_dtype, 1.0, 1.0, S(case.new_k),
                                  S(case.new_v), case.act_dtype, case.slot_last.cpu().numpy())
    assert st == 0
    assert np.array_equal(kr, S(case.k_cache)) and np.array_equal(vr, S(case.v_cache))
    check(case, out, lse, "fused append", pools=(kr, vr))
    assert pkv.get_device_error() == 0


def test_no_shared_prefix_equals_plain_decode():
    # every group's prefix 0: the cascade is plain split decode + merge
    case, gi, gp, mg, ms = grouped_case([(3, 0), (5, 0)], [100, 7, 64, 1, 300, 33, 16, 90], 32, 8,
                                        16, F16, seed=31)
    out, lse = run_cascade(case, gi, gp, mg, ms, splits=2)
    check(case, out, lse, "prefix 0")
    assert pkv.get_device_error() == 0


def test_shared_prefix_decode_workload_sampled():
    # the benchmark layer: 256 requests, one 1,000-token prompt (62 shared blocks +
    # an 8-token tail in each request's own block), own tokens U[32, 256]
    case = W.shared_prefix_decode(device="cuda")
    b = case.q.shape[0]
    gi = torch.tensor([0, b], dtype=torch.int32, device="cuda")
    gp = torch.tensor([1000], dtype=torch.int32, device="cuda")
    ms = int(case.seq_lens.max()) - 1000
    out, lse = run_cascade(case, gi, gp, b, ms)
    pairs = [(r, h) for r in (0, 1, 77, 128, 255) for h in (0, 5, 31)]
    ref, ref_lse = oracle_ref(case, pairs=pairs)
    got = np.stack([to_f64(out)[r, h] for r, h in pairs])
    assert_attention_close(got, ref, case.act_dtype, what="shared prefix workload")
    gl = np.array([float(lse[r, h]) for r, h in pairs])
    assert np.max(np.abs(gl - ref_lse)) <= 1e-3
    # and the plain decode on the same inputs agrees within the same bound
    plain = torch.empty_like(case.q)
    ws = torch.empty(max(pkv.decode_workspace_bytes(case.k_cache, b, case.num_q_heads,
                                                    int(case.seq_lens.max()), 0), 1),
                     dtype=torch.uint8, device="cuda")
    pkv.paged_decode_attn(case.k_cache, case.v_cache, case.q, plain, case.block_tables,
                          case.seq_lens, case.sm_scale, int(case.seq_lens.max()), workspace=ws)
    torch.cuda.synchronize()
    d = (to_f64(plain) - to_f64(out))
    assert np.max(np.abs(d)) <= 8e-3
    assert pkv.get_device_error() == 0


def test_prefix_longer_than_a_member_is_reported():
    # P_g above one member's seq_len: flagged in the device error word, no fault
    case, gi, gp, mg, ms = grouped_case([(3, 64)], [40, 40, 40], 8, 2, 16, F16, seed=41)
    case.seq_lens[2] = 50  # < 64
    run_cascade(case, gi, gp, mg, ms)
    assert pkv.get_device_error() == 3


def test_prefix_beyond_the_hint_is_reported():
    # max_prefix_len 256 (one 256-key chunk) under a 600-token prefix: the keys past the
    # chunk are not attended and the device error word says so
    case, gi, gp, mg, ms = grouped_case([(4, 600)], [30, 30, 30, 30], 8, 2, 16, BF16, seed=42)
    b = case.q.shape[0]
    ws = torch.empty(pkv.shared_prefix_decode_workspace_bytes(case.k_cache, b, 8, 256, ms, 0),
                     dtype=torch.uint8, device="cuda")
    pkv.get_device_error()  # clear
    pkv.paged_decode_attn_shared_prefix(case.k_cache, case.v_cache, case.q, torch.empty_like(case.q),
                                        case.block_tables, case.seq_lens, case.sm_scale, gi, gp, mg,
                                        256, ms, workspace=ws)
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 3


def test_long_shared_prefix_in_chunks():
    # one group of 3 members over a 5,000-token prefix: few work items, so the prefix pass
    # cuts the keys into chunks (one more partial each in the merge)
    case, gi, gp, mg, ms = grouped_case([(3, 5000)], [40, 7, 130], 8, 2, 16, BF16, seed=43)
    out, lse = run_cascade(case, gi, gp, mg, ms)
    check(case, out, lse, "5,000-token prefix in chunks")
    assert pkv.get_device_error() == 0


def test_unsupported_and_bad_arguments_are_refused_on_the_host():
    gi = torch.tensor([0, 2], dtype=torch.int32, device="cuda")
    gp = torch.tensor([32], dtype=torch.int32, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    cbig = W.decode_case([40, 50], 2 * 129, 2, 64, 16, F16, F16, seed=1, device="cuda")
    with pytest.raises(pkv.PkvError) as e:  # a group of 129 heads does not fit one row tile
        pkv.paged_decode_attn_shared_prefix(cbig.k_cache, cbig.v_cache, cbig.q,
                                            torch.empty_like(cbig.q), cbig.block_tables,
                                            cbig.seq_lens, cbig.sm_scale, gi, gp, 2, 32, 20,
                                            workspace=ws)
    assert e.value.status == 2
    c = W.decode_case([40, 50], 8, 2, 128, 16, BF16, BF16, seed=2, device="cuda")
    small = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attn_shared_prefix(c.k_cache, c.v_cache, c.q, torch.empty_like(c.q),
                                            c.block_tables, c.seq_lens, c.sm_scale, gi, gp, 2, 32,
                                            20, workspace=small)
    assert e.value.status == 3
    with pytest.raises(pkv.PkvError) as e:  # a negative softmax scale
        pkv.paged_decode_attn_shared_prefix(c.k_cache, c.v_cache, c.q, torch.empty_like(c.q),
                                            c.block_tables, c.seq_lens, -0.1, gi, gp, 2, 32, 20,
                                            workspace=ws)
    assert e.value.status == 1


def test_request_outside_every_group_is_reported():
    # groups cover requests 0..2 of 5: requests 3 and 4 attend their whole sequence through
    # their own tables (correct values) and the device error word reports the gap
    case, gi, gp, mg, ms = grouped_case([(3, 64), (1, 0), (1, 0)], [20, 30, 40, 50, 60], 8, 2, 16,
                                        BF16, seed=51)
    gi = gi[:2].contiguous()   # [0, 3]: one group only
    gp = gp[:1].contiguous()
    out, lse = run_cascade(case, gi, gp, mg, max(ms, 124))
    check(case, out, lse, "uncovered requests")
    assert pkv.get_device_error() == 3


def test_merge_is_bit_identical_across_calls():
    # the prefix pass runs beside the own-token decode, in whatever order the
    # GPU schedules them; the merge takes the parts in a fixed slot order, so the
    # output and LSE bits do not depend on it
    case, gi, gp, mg, ms = grouped_case([(64, 500), (9, 1000)], rand_suffixes(73, 0, 300, 7),
                                        32, 8, 16, BF16, seed=51)
    runs = [run_cascade(case, gi, gp, mg, ms, splits=sp) for sp in (0, 0, 0, 2, 2)]
    for out, lse in runs[1:3]:
        assert torch.equal(out, runs[0][0]) and torch.equal(lse, runs[0][1])
    assert torch.equal(runs[4][0], runs[3][0]) and torch.equal(runs[4][1], runs[3][1])
    check(case, runs[0][0], runs[0][1], "repeated calls")
    check(case, runs[3][0], runs[3][1], "repeated calls, 2 splits")
    assert pkv.get_device_error() == 0


def test_workspace_with_stale_contents():
    # the workspace needs no initial contents: one holding any bytes (here all
    # ones, then the previous call's state) gives the same result as a fresh one
    case, gi, gp, mg, ms = grouped_case([(20, 320), (6, 40)], rand_suffixes(26, 1, 120, 8),
                                        32, 8, 16, F16, seed=52)
    b = case.q.shape[0]
    nbytes = pkv.shared_prefix_decode_workspace_bytes(case.k_cache, b, case.num_q_heads, 320, ms, 0)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        out = torch.full_like(case.q, float("nan"))
        pkv.paged_decode_attn_shared_prefix(case.k_cache, case.v_cache, case.q, out,
                                            case.block_tables, case.seq_lens, case.sm_scale, gi, gp,
                                            mg, 320, ms, workspace=ws)
        torch.cuda.synchronize()
        outs.append(out)
    fresh, _ = run_cascade(case, gi, gp, mg, ms)
    assert torch.equal(outs[0], fresh) and torch.equal(outs[1], fresh)
    assert pkv.get_device_error() == 0


def test_empty_requests_get_zero_output():
    # a request with no token at all (no prefix, seq_len 0) has no partial to
    # merge: out = 0, lse = -inf
    case, gi, gp, mg, ms = grouped_case([(3, 0), (2, 64)], [0, 17, 0, 5, 9], 8, 2, 16, BF16,
                                        seed=53)
    out, lse = run_cascade(case, gi, gp, mg, ms)
    for r in (0, 2):
        assert torch.count_nonzero(out[r]) == 0
        assert torch.all(torch.isneginf(lse[r]))
    check(case, out, lse, "empty requests")
    assert pkv.get_device_error() == 0
