"""GPU checks of how the calls sit on CUDA streams: each call is ordered on the
stream it is given like any kernel, can be captured into a CUDA graph, and
gives the same bits whatever stream or host thread issues it.  The
shared-prefix decode runs its prefix pass on a side stream the library keeps
per device (forked from the caller's stream by an event and joined back before
the merge), so it is the call these checks are most about: a graph captured
from it must take the side stream's work along, and callers on several host
threads must not mix up their forks and joins."""
import threading

import pytest
import torch

import paged_kv_cache_285_gb300 as pkv
from paged_kv_cache_285_gb300 import workloads as W
from tests.pkv_testlib import BF16
from tests.test_gpu_shared_prefix import check, grouped_case, rand_suffixes

pytestmark = pytest.mark.gpu

GROUPS = [(40, 500), (3, 64), (1, 0), (20, 1000)]


def spd_case(seed):
    suf = rand_suffixes(sum(n for n, _ in GROUPS), 1, 200, seed)
    return grouped_case(GROUPS, suf, 32, 8, 16, BF16, seed=seed)


class SpdCall:
    """One caller's buffers for pkv_paged_decode_attn_shared_prefix."""

    def __init__(self, case, gi, gp, max_group, max_suffix):
        self.case, self.gi, self.gp = case, gi, gp
        self.max_group, self.max_suffix = max_group, max_suffix
        self.max_prefix = int(gp.max())
        b = case.q.shape[0]
        self.q = case.q.clone()
        self.out = torch.full_like(case.q, float("nan"))
        self.lse = torch.full((b, case.num_q_heads), float("nan"), dtype=torch.float32,
                              device="cuda")
        n = pkv.shared_prefix_decode_workspace_bytes(case.k_cache, b, case.num_q_heads,
                                                     self.max_prefix, max_suffix, 0)
        self.ws = torch.empty(n, dtype=torch.uint8, device="cuda")

    def __call__(self, stream=None):
        c = self.case
        pkv.paged_decode_attn_shared_prefix(
            c.k_cache, c.v_cache, self.q, self.out, c.block_tables, c.seq_lens, c.sm_scale,
            self.gi, self.gp, self.max_group, self.max_prefix, self.max_suffix,
            lse_out=self.lse, workspace=self.ws, stream=stream)


def bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def test_shared_prefix_decode_in_a_cuda_graph():
    case, gi, gp, mg, ms = spd_case(seed=71)
    eager = SpdCall(case, gi, gp, mg, ms)
    eager()
    torch.cuda.synchronize()
    check(case, eager.out, eager.lse, "eager shared-prefix decode")
    call = SpdCall(case, gi, gp, mg, ms)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            call()
    for _ in range(3):
        call.out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(bits(call.out), bits(eager.out))
        assert torch.equal(bits(call.lse), bits(eager.lse))
    # new queries written into the captured input: the replay reads them
    newq = torch.randn_like(case.q, dtype=torch.float32).to(case.q.dtype)
    call.q.copy_(newq)
    eager.q.copy_(newq)
    eager()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(bits(call.out), bits(eager.out))
    assert pkv.get_device_error() == 0


def test_decode_and_extend_in_one_cuda_graph():
    dec = W.decode_case([700, 33, 2000, 1], 32, 8, 128, 16, BF16, BF16, seed=72, device="cuda")
    ext = W.extend_case([300, 0], [90, 40], 8, 2, 128, 16, BF16, BF16, seed=73, device="cuda")
    b = dec.q.shape[0]
    wsb = pkv.decode_workspace_bytes(dec.k_cache, b, dec.num_q_heads, 2000)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    d_out, e_out = torch.empty_like(dec.q), torch.empty_like(ext.q)

    def step():
        pkv.paged_decode_attn(dec.k_cache, dec.v_cache, dec.q, d_out, dec.block_tables,
                              dec.seq_lens, dec.sm_scale, 2000, workspace=ws)
        pkv.paged_extend_attn(ext.k_cache, ext.v_cache, ext.q, e_out, ext.q_indptr,
                              ext.prefix_lens, ext.block_tables, ext.sm_scale, 90, 390)

    step()
    torch.cuda.synchronize()
    d_ref, e_ref = d_out.clone(), e_out.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            step()
    d_out.fill_(float("nan"))
    e_out.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(bits(d_out), bits(d_ref))
    assert torch.equal(bits(e_out), bits(e_ref))


def test_calls_from_several_host_threads():
    # four host threads, each with its own stream and buffers, issue shared-prefix
    # decodes (one fork and join each on the library's side stream) and plain
    # decodes at the same time; every result has the bits of a single-threaded call
    case, gi, gp, mg, ms = spd_case(seed=74)
    dec = W.decode_case([900, 40, 1500], 32, 8, 128, 16, BF16, BF16, seed=75, device="cuda")
    dwsb = pkv.decode_workspace_bytes(dec.k_cache, 3, dec.num_q_heads, 1500)
    ref_calls = []
    qs = [torch.randn_like(case.q, dtype=torch.float32).to(case.q.dtype) for _ in range(4)]
    for q in qs:
        c = SpdCall(case, gi, gp, mg, ms)
        c.q.copy_(q)
        c()
        ref_calls.append(c)
    d_ref = torch.empty_like(dec.q)
    dws = torch.empty(max(dwsb, 256), dtype=torch.uint8, device="cuda")
    pkv.paged_decode_attn(dec.k_cache, dec.v_cache, dec.q, d_ref, dec.block_tables, dec.seq_lens,
                          dec.sm_scale, 1500, workspace=dws)
    torch.cuda.synchronize()

    errors = []
    results = [None] * 4

    def worker(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                c = SpdCall(case, gi, gp, mg, ms)
                c.q.copy_(qs[i])
                d_out = torch.empty_like(dec.q)
                ws = torch.empty(max(dwsb, 256), dtype=torch.uint8, device="cuda")
                for _ in range(20):
                    c(stream=s)
                    pkv.paged_decode_attn(dec.k_cache, dec.v_cache, dec.q, d_out,
                                          dec.block_tables, dec.seq_lens, dec.sm_scale, 1500,
                                          workspace=ws, stream=s)
                s.synchronize()
                results[i] = (c.out.clone(), c.lse.clone(), d_out.clone())
        except Exception as e:  # reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads), "a worker did not finish"
    assert not errors, errors
    for i, (out, lse, d_out) in enumerate(results):
        assert torch.equal(bits(out), bits(ref_calls[i].out)), i
        assert torch.equal(bits(lse), bits(ref_calls[i].lse)), i
        assert torch.equal(bits(d_out), bits(d_ref)), i
    assert pkv.get_device_error() == 0
