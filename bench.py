"""Benchmark of the paged-KV attention hot path on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl pkv|reference]

One step of the default workload (a Llama-3-8B-shaped decode layer: 64
requests, seq_lens uniform in [512, 4096], 32 q / 8 kv heads, d128, bf16,
16-token blocks randomly permuted over the pool) is the whole decode hot path:
kv_append of every request's current token into its slot, then
paged_decode_attn (split-KV + LSE merge) over every cached token.  The same
line reports the suffix-prefill hot path (paged_extend_attn over a shared
1,900-token cached prefix, 256 requests x 100 suffix tokens) in its own
object.

Printed (rank 0, one JSON line): value = algorithmic HBM bytes of the step /
device time (GB/s), decode tokens/s, the roofline of the dominant call
(paged_decode_attn) against the measured copy bandwidth, the fp64 CPU oracle
as a baseline, an end-to-end number through host buffers and the SM clocks
sampled while timing.  `--impl reference` times the fp64 CPU oracle itself
on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "paged decode attn HBM GB/s (% of GB300 peak) & tokens/s; extend TFLOP/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# GB300 datasheet figures (context beside the measured peaks): HBM3e bandwidth and dense bf16
NOMINAL_HBM_GBS = 7900.0
NOMINAL_BF16_TFLOPS = 2250.0


# ---------------------------------------------------------------------------------
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def src_hash(*rel):
    """Hash of the sources a kernel is built from; "path#A,B" takes only the
    definitions of structs A and B from that file (the parameter layouts the
    kernel reads)."""
    h = hashlib.sha256()
    for r in rel:
        path, _, structs = r.partition("#")
        with open(os.path.join(ROOT, path), "rb") as f:
            data = f.read()
        if structs:
            text = data.decode("utf-8")
            parts = []
            for name in structs.split(","):
                i = text.index("struct " + name + " {")
                parts.append(text[i:text.index("\n};", i) + 3])
            data = "\n".join(parts).encode("utf-8")
        h.update(data)
    return h.hexdigest()[:16]


def profiled_traffic(name, sources, key="dram_bytes_per_launch"):
    """DRAM bytes per launch (the summary's `key` line) from a committed ncu summary, if the
    kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", name)
    try:
        kv = {}
        with open(path, encoding="utf-8") as f:
            for line in f:
                if line.startswith("- ") and ":" in line:
                    k, v = line[2:].split(":", 1)
                    kv[k.strip()] = v.strip().strip("`")
        if kv.get("source_sha256_16") != src_hash(*sources):
            return None
        return float(kv[key])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed loop runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.samples = []
        if self.proc is None:
            return False
        time.sleep(0.2)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append(parts)
        return False

    def summary(self):
        if not getattr(self, "samples", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = sorted(float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit())
        mx = max((float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for s in self.samples:
            for n, v in zip(names, s[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(self.samples)}


class L2Flush:
    """Writes then reads a 256 MiB buffer (2x the 129 MB L2): afterwards L2 holds
    only clean lines of this buffer, so the next timed kernel neither hits its own
    data nor pays for writing back dirty flush lines."""

    def __init__(self, dev):
        self.buf = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.buf.fill_(1)
        self.sink = self.buf.sum()


# ---------------------------------------------------------------------------------
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value over all ranks (the slowest rank sets the job's time)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------------
def extend_useful_flops(prefix_lens, suffix_lens, num_q_heads, head_dim):
    """Useful flops of a suffix prefill: suffix row i of a request with prefix P sees P + i + 1
    keys, and each (row, head, key) costs 2 * head_dim for the score and 2 * head_dim for its
    share of P V (padding rows and masked keys a kernel computes are not counted)."""
    keys = sum(p * s + s * (s + 1) // 2 for p, s in zip(prefix_lens, suffix_lens))
    return 4.0 * head_dim * num_q_heads * keys


def decode_step_bytes(case):
    """Algorithmic HBM bytes of one step: append of B tokens + decode over sum(seq_lens)."""
    from paged_kv_cache_285_gb300 import workloads as W
    b = case.q.shape[0]
    hq, hkv, d = case.num_q_heads, case.num_kv_heads, case.head_dim
    ce = W.ELEM_BYTES[case.cache_dtype]
    ae = 2
    ntok = int(case.seq_lens.sum())
    nblk = int(sum(math.ceil(int(n) / case.block_size) for n in case.seq_lens.tolist()))
    append = b * hkv * d * (ae + ce) * 2 + 8 * b
    decode = ntok * hkv * d * ce * 2 + 2 * b * hq * d * ae + 4 * nblk + 4 * b
    return append, decode


def run_decode_bench(args, world, rank, local):
    import paged_kv_cache_285_gb300 as pkv
    from paged_kv_cache_285_gb300 import workloads as W

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pkv.load()
    makers = {"llama3_8b_layer": (W.llama3_8b_decode, 4096),
              "fp8_70b_layer": (W.fp8_70b_decode, 4096),
              "shared_prefix_decode": (W.shared_prefix_decode, 1256),
              "tiny": (lambda device: W.tiny_decode(device=device), 60)}
    mk, max_len = makers[args.workload]
    case = mk(device="cuda")
    b = case.q.shape[0]
    out = torch.empty_like(case.q)
    ws_bytes = pkv.decode_workspace_bytes(case.k_cache, b, case.num_q_heads, max_len, 0,
                                          case.k_scale, case.v_scale)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)

    def append():
        pkv.kv_append(case.k_cache, case.v_cache, case.new_k, case.new_v, case.slot_last,
                      k_scale=case.k_scale, v_scale=case.v_scale)

    def decode():
        pkv.paged_decode_attn(case.k_cache, case.v_cache, case.q, out, case.block_tables,
                              case.seq_lens, case.sm_scale, max_len, k_scale=case.k_scale,
                              v_scale=case.v_scale, workspace=ws)

    def fused():  # the current token appended by the decode kernel itself
        pkv.paged_decode_attn_append(case.k_cache, case.v_cache, case.new_k, case.new_v, case.q,
                                     out, case.block_tables, case.seq_lens, case.sm_scale,
                                     max_len, k_scale=case.k_scale, v_scale=case.v_scale,
                                     workspace=ws)

    for _ in range(args.warmup):
        append()
        decode()
        fused()
    torch.cuda.synchronize()
    # The step's launches are captured once into CUDA graphs and replayed, so the
    # device time is not stretched by host-side enqueue cost (Python + ctypes).
    g_step, g_dec, g_fused = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(g_step, stream=cap):
            append()
            decode()
        with torch.cuda.graph(g_dec, stream=cap):
            decode()
        with torch.cuda.graph(g_fused, stream=cap):
            fused()
    stream.wait_stream(cap)
    for _ in range(args.warmup):
        g_step.replay()
        g_dec.replay()
        g_fused.replay()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for i in range(K):
            flush()                             # evict the pool from L2 between steps
            ev[i][0].record(stream)
            g_step.replay()
            ev[i][1].record(stream)
            flush()
            ev[i][2].record(stream)
            g_dec.replay()                      # the decode call alone, for its roofline
            ev[i][3].record(stream)
            flush()
            ev[i][4].record(stream)
            g_fused.replay()                    # the step with the append fused into decode
            ev[i][5].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    dec_ms = [e[2].elapsed_time(e[3]) for e in ev]
    fused_ms = [e[4].elapsed_time(e[5]) for e in ev]
    ms_sep = max_over_ranks(sum(step_ms) / K, world)
    ms_dec = sum(dec_ms) / K
    ms_step_max = max_over_ranks(sum(fused_ms) / K, world)
    ms_step_med = max_over_ranks(_median(fused_ms), world)
    ms_dec_med = _median(dec_ms)

    app_b, dec_b = decode_step_bytes(case)
    step_bytes = app_b + dec_b
    hbm, bf16, bf16_sus, peak_src = peaks()
    value = world * step_bytes / (ms_step_max * 1e-3) / 1e9
    dec_gbs = dec_b / (ms_dec * 1e-3) / 1e9
    splits_plan = ws_bytes > 0
    dec_launches = 1 + (1 if splits_plan else 0)    # decode_kernel (+ merge_kernel)

    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step_max, 5),
        "ms_per_step_median": round(ms_step_med, 5),
        "value_median": round(world * step_bytes / (ms_step_med * 1e-3) / 1e9, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": W.DTYPE_NAME[case.cache_dtype],
        "data": "synthetic (seeded N(0,1) K/V/q, random block permutation)",
        "config": {"workload": args.workload, "batch": b, "num_q_heads": case.num_q_heads,
                   "num_kv_heads": case.num_kv_heads, "head_dim": case.head_dim,
                   "block_size": case.block_size, "cache_dtype": W.DTYPE_NAME[case.cache_dtype],
                   "act_dtype": W.DTYPE_NAME[case.act_dtype],
                   "cached_tokens": int(case.seq_lens.sum()),
                   "step": "paged_decode_attn_append: the current token's K/V (1 per request) "
                           "appended by the decode kernel, then attention; one CUDA graph",
                   "l2": "256 MiB buffer written then read between timed steps (outside the events)",
                   "parallelism": f"replicas x{world}"},
        "pct_of_peak": round(100.0 * value / world / hbm, 1),
        "tokens_per_s": round(world * b / (ms_step_max * 1e-3), 1),
        # timed region per iteration: append + decode, decode alone, fused step
        "gpu_launches": (1 + 3 * dec_launches) * K,
        "separate_step": {"step": "kv_append + paged_decode_attn, one CUDA graph",
                          "ms_per_step": round(ms_sep, 5),
                          "value": round(world * step_bytes / (ms_sep * 1e-3) / 1e9, 1),
                          "unit": "GB/s"},
    }
    traffic = profiled_traffic("decode_kernel_llama3_8b_layer.md",
                               ["paged_kv_cache_285_gb300/csrc/decode.cu",
                                "paged_kv_cache_285_gb300/csrc/ptx.cuh",
                                "paged_kv_cache_285_gb300/csrc/internal.h"
                                "#DecodeParams,DecodeExtraParams"]) \
        if args.workload == "llama3_8b_layer" else None
    res["roofline"] = {"kernel": "paged_decode_attn (decode_kernel + merge_kernel)",
                       "bound": "hbm", "achieved": round(dec_gbs, 1), "peak": hbm,
                       "unit": "GB/s", "frac": round(dec_gbs / hbm, 4),
                       "peak_source": f"{peak_src} (hbm_gbs)",
                       "achieved_median": round(dec_b / (ms_dec_med * 1e-3) / 1e9, 1),
                       "frac_of_nominal": round(dec_gbs / NOMINAL_HBM_GBS, 4),
                       "nominal_peak": NOMINAL_HBM_GBS,
                       "algorithmic_bytes_per_launch": dec_b,
                       "traffic": traffic}
    res["clocks"] = clk.summary()
    res["wall_s_timed"] = round(t_wall, 3)

    # end to end through the C ABI with host buffers: per step the inputs of the
    # step (q, the new token's K/V, seq_lens, block tables) go host->device
    # from pinned memory and the output comes back device->host
    res["e2e"] = e2e_decode(case, pkv, max_len, ws, out, stream, K, world)
    if args.no_side:
        return res
    if args.extend and rank == 0 and world == 1:
        res["extend"] = run_extend_bench(args, dev, bf16, bf16_sus, peak_src)
    if rank == 0 and world == 1:
        res["prefix_index"] = run_prefix_index_bench()
        res["chain_hash"] = run_chain_hash_bench(dev, hbm, peak_src)
        res["shared_prefix_decode"] = run_shared_prefix_bench(dev, hbm, peak_src)
        res["more_decode_configs"] = run_more_decode_configs_bench(dev, hbm, peak_src)
        res["append_fill"] = run_append_fill_bench(dev, hbm, peak_src)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline_decode(case, budget_s=args.cpu_seconds)
    return res


class _HostView:
    """Device-side view of pinned host memory (unified addressing: the GPU reads
    and writes it over the host link), for copy kernels instead of copy-engine
    transfers."""

    def __init__(self, t):
        self.__cuda_array_interface__ = {"shape": (t.numel() * t.element_size(),),
                                         "typestr": "|u1", "data": (t.data_ptr(), False),
                                         "version": 3}


def e2e_decode(case, pkv, max_len, ws, out, stream, K, world):
    """The fused decode step through the public API from host buffers: each step's
    inputs (q, the current token's K/V, seq_lens, block tables) sit in one pinned
    staging buffer (256-byte-aligned views) and cross to the device in one copy
    kernel that reads the pinned buffer over the host link; the output crosses
    back the same way.  Copy kernels rather than the copy engine: the step then
    never switches between engines (same bytes, same link)."""
    names = ["q", "new_k", "new_v", "seq_lens", "block_tables"]
    offs, total = {}, 0
    for n in names:
        t = getattr(case, n)
        offs[n] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device=out.device)

    def views(buf):
        v = {}
        for n in names:
            t = getattr(case, n)
            nb = t.numel() * t.element_size()
            v[n] = buf[offs[n]:offs[n] + nb].view(t.dtype).view(t.shape)
        return v

    host, dev_t = views(host_buf), views(dev_buf)
    for n in names:
        host[n].copy_(getattr(case, n).cpu())
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = total
    d2h = out_h.numel() * out_h.element_size()
    host_on_dev = torch.as_tensor(_HostView(host_buf), device=out.device)
    out_h_on_dev = torch.as_tensor(_HostView(out_h), device=out.device)
    assert host_on_dev.data_ptr() == host_buf.data_ptr()
    out_bytes = out.view(torch.uint8).view(-1)

    def step():
        dev_buf.copy_(host_on_dev)
        pkv.paged_decode_attn_append(case.k_cache, case.v_cache, dev_t["new_k"], dev_t["new_v"],
                                     dev_t["q"], out, dev_t["block_tables"], dev_t["seq_lens"],
                                     case.sm_scale, max_len, k_scale=case.k_scale,
                                     v_scale=case.v_scale, workspace=ws)
        out_h_on_dev.copy_(out_bytes)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    # the output that crossed the link is the device's, byte for byte
    assert torch.equal(out_h.view(torch.uint8), out.view(torch.uint8).cpu())
    # the whole step (input copy, the API call, output copy) replayed as one graph
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            step()
    stream.wait_stream(cap)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.uint8), out.view(torch.uint8).cpu())
    flush = L2Flush(out.device)
    tot = 0.0
    for _ in range(K):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        e1.synchronize()
        tot += e0.elapsed_time(e1)
    ms_staged = max_over_ranks(tot / K, world)

    # Zero-copy: the same API call given device-addressable views of the pinned
    # buffers themselves, so the decode kernel reads q, the new K/V, lengths and
    # block tables over the host link and the output is written there; no copy
    # launch.  Same bytes cross the link every step.
    host_zc = views(host_on_dev)
    out_zc = out_h_on_dev.view(out.dtype).view(out.shape)

    def step_zc():
        pkv.paged_decode_attn_append(case.k_cache, case.v_cache, host_zc["new_k"], host_zc["new_v"],
                                     host_zc["q"], out_zc, host_zc["block_tables"],
                                     host_zc["seq_lens"], case.sm_scale, max_len,
                                     k_scale=case.k_scale, v_scale=case.v_scale, workspace=ws)

    # every step appends the same token at the same slot, so the cache and the
    # output are the same whichever form ran before
    step_zc()
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.uint8), out.view(torch.uint8).cpu())
    graph_zc = torch.cuda.CUDAGraph()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph_zc, stream=cap):
            step_zc()
    stream.wait_stream(cap)
    for _ in range(3):
        graph_zc.replay()
    torch.cuda.synchronize()
    assert torch.equal(out_h.view(torch.uint8), out.view(torch.uint8).cpu())
    tot = 0.0
    for _ in range(K):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph_zc.replay()
        e1.record(stream)
        e1.synchronize()
        tot += e0.elapsed_time(e1)
    ms_zc = max_over_ranks(tot / K, world)

    app_b, dec_b = decode_step_bytes(case)
    gbs = lambda ms: round(world * (app_b + dec_b) / (ms * 1e-3) / 1e9, 1)
    return {"value": gbs(ms_zc), "unit": "GB/s",
            "ms_per_step": round(ms_zc, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "transfer": "zero-copy: the API call reads its inputs from and writes its output to "
                        "pinned host buffers over the host link (GB300 addresses host memory "
                        "directly); no copy launch",
            "launch": "the step (the API call) captured once as a CUDA graph and replayed",
            "staged": {"value": gbs(ms_staged), "ms_per_step": round(ms_staged, 5),
                       "transfer": "one copy kernel each way over the host link, pinned host "
                                   "buffers, then the API call on device buffers"}}


def _median(xs):
    ys = sorted(xs)
    n = len(ys)
    return ys[n // 2] if n % 2 else 0.5 * (ys[n // 2 - 1] + ys[n // 2])


def _time_extend_case(case, P, Sfx, n, flush, with_append, ws=None):
    """Mean and median device time of paged_extend_attn on `case` (L2 flushed before each
    call; `ws` its optional widening workspace); with_append: also the step with the
    suffix's kv_append before it and the one-call paged_extend_attn_append.  Returns a dict
    of lists of ms."""
    import paged_kv_cache_285_gb300 as pkv
    out = torch.empty_like(case.q)
    sc = dict(k_scale=case.k_scale, v_scale=case.v_scale)

    def append():
        pkv.kv_append(case.k_cache, case.v_cache, case.suffix_k, case.suffix_v, case.suffix_slots,
                      **sc)

    def extend():
        pkv.paged_extend_attn(case.k_cache, case.v_cache, case.q, out, case.q_indptr,
                              case.prefix_lens, case.block_tables, case.sm_scale, Sfx, P + Sfx,
                              workspace=ws, **sc)

    def fused():
        pkv.paged_extend_attn_append(case.k_cache, case.v_cache, case.suffix_k, case.suffix_v,
                                     case.q, out, case.q_indptr, case.prefix_lens,
                                     case.block_tables, case.sm_scale, Sfx, P + Sfx, **sc)

    for _ in range(3):
        if with_append:
            append()
            fused()
        extend()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    t = {"extend": [], "step": [], "fused": []}
    for _ in range(n):
        flush()
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(stream)
        if with_append:
            append()
        e1.record(stream)
        extend()
        e2.record(stream)
        e2.synchronize()
        t["extend"].append(e1.elapsed_time(e2))
        t["step"].append(e0.elapsed_time(e2))
        if with_append:
            flush()
            e3, e4 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
            e3.record(stream)
            fused()
            e4.record(stream)
            e4.synchronize()
            t["fused"].append(e3.elapsed_time(e4))
    return t


def _time_extend_shared(case, groups, shared, max_group_rows, max_total, n, flush, ws=None):
    """Device times (ms) of paged_extend_attn_shared_prefix on `case` with the given groups
    (and the optional workspace `ws`), L2 flushed before each call."""
    import paged_kv_cache_285_gb300 as pkv
    out = torch.empty_like(case.q)
    gi = torch.tensor(groups, dtype=torch.int32, device=case.q.device)
    gs = torch.tensor(shared, dtype=torch.int32, device=case.q.device)

    def call():
        pkv.paged_extend_attn_shared_prefix(case.k_cache, case.v_cache, case.q, out, case.q_indptr,
                                            case.prefix_lens, case.block_tables, gi, gs,
                                            case.sm_scale, max_group_rows, max_total,
                                            k_scale=case.k_scale, v_scale=case.v_scale,
                                            workspace=ws)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    ts = []
    for _ in range(n):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    return ts


def _extend_with_workspace(case, P, Sfx, n, flush, flops, bf16):
    """paged_extend_attn with its optional widening workspace (each block read widened to
    16 bits once per call; the widening pass inside the timed call), or None where the
    cache dtype needs none."""
    import paged_kv_cache_285_gb300 as pkv
    wsb = pkv.extend_widen_workspace_bytes(case.k_cache, case.k_scale, case.v_scale)
    if not wsb:
        return None
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    tw = _time_extend_case(case, P, Sfx, n, flush, False, ws=ws)["extend"]
    del ws
    tw_mean = sum(tw) / n
    tfw = flops / (tw_mean * 1e-3) / 1e12
    return {"ms_per_call": round(tw_mean, 5), "ms_per_call_median": round(_median(tw), 5),
            "tflops": round(tfw, 1), "frac": round(tfw / bf16, 4),
            "frac_of_nominal": round(tfw / NOMINAL_BF16_TFLOPS, 4), "workspace_bytes": wsb}


def run_extend_bench(args, dev, bf16, bf16_sus, peak_src):
    """paged_extend_attn on 256 requests x 100 suffix tokens over a shared 1,900-token
    prefix (useful causal flops only); the step with the suffix's kv_append as a
    separate launch and as paged_extend_attn_append.  The same workload is also timed with
    an fp8 e4m3 cache (bf16 queries), at head_dim 64, and through
    paged_extend_attn_shared_prefix (the 256 requests as one group)."""
    import paged_kv_cache_285_gb300 as pkv
    from paged_kv_cache_285_gb300 import workloads as W
    try:
        case = W.shared_prefix_extend(device="cuda")
    except Exception as e:  # pragma: no cover
        return {"error": str(e)}
    rows = case.q.shape[0]
    P, Sfx = 1900, 100
    B = case.prefix_lens.shape[0]
    n = max(5, min(50, args.steps))
    flush = L2Flush(dev)
    try:
        t = _time_extend_case(case, P, Sfx, n, flush, True)
    except pkv.PkvError as e:
        return {"status": "not built", "error": str(e)}
    t_ext = sum(t["extend"]) / n
    t_step = sum(t["step"]) / n
    t_fused = sum(t["fused"]) / n
    med_ext = _median(t["extend"])
    hq, d = case.num_q_heads, case.head_dim
    # the suffix's kv_append: K and V rows read from the inputs and written to the cache
    t_app = t_step - t_ext
    app_bytes = rows * case.num_kv_heads * d * 2 * 2 * 2 + 8 * rows
    hbm = peaks()[0]
    flops = extend_useful_flops([P] * B, [Sfx] * B, hq, d)
    tf = flops / (t_ext * 1e-3) / 1e12
    res = {"workload": "shared_prefix_extend", "batch": B, "prefix": P, "suffix": Sfx,
           "num_q_heads": hq, "num_kv_heads": case.num_kv_heads, "head_dim": d,
           "ms_per_call": round(t_ext, 5), "ms_per_call_median": round(med_ext, 5),
           "ms_per_step_with_append": round(t_step, 5),
           "ms_per_step_fused_append": round(t_fused, 5),
           "kv_append": {"tokens": rows, "ms": round(t_app, 5), "bytes": app_bytes,
                         "gbs": round(app_bytes / (t_app * 1e-3) / 1e9, 1),
                         "frac_of_hbm": round(app_bytes / (t_app * 1e-3) / 1e9 / hbm, 4)},
           "tflops": round(tf, 1), "tflops_median": round(flops / (med_ext * 1e-3) / 1e12, 1),
           "useful_flops_per_call": flops,
           "roofline": {"kernel": "paged_extend_attn", "bound": "tensor", "achieved": round(tf, 1),
                        "peak": bf16, "unit": "TFLOP/s", "frac": round(tf / bf16, 4),
                        "peak_source": f"{peak_src} (bf16_tflops burst)",
                        "frac_of_nominal": round(tf / NOMINAL_BF16_TFLOPS, 4),
                        "nominal_peak": NOMINAL_BF16_TFLOPS,
                        "traffic": profiled_traffic(
                            "extend_kernel_shared_prefix_extend.md",
                            ["paged_kv_cache_285_gb300/csrc/extend.cu",
                             "paged_kv_cache_285_gb300/csrc/ptx.cuh",
                             "paged_kv_cache_285_gb300/csrc/tcgen05.cuh",
                             "paged_kv_cache_285_gb300/csrc/internal.h"
                             "#ExtendParams,ExtendPartialParams,FastDiv"])}}
    ww = _extend_with_workspace(case, P, Sfx, n, flush, flops, bf16)
    if ww:
        # the widened kernel's DRAM bytes per launch (the widening pass not included)
        ww["traffic"] = profiled_traffic(
            "extend_kernel_shared_prefix_extend.md",
            ["paged_kv_cache_285_gb300/csrc/extend.cu", "paged_kv_cache_285_gb300/csrc/ptx.cuh",
             "paged_kv_cache_285_gb300/csrc/tcgen05.cuh",
             "paged_kv_cache_285_gb300/csrc/internal.h#ExtendParams,ExtendPartialParams,FastDiv"],
            key="dram_bytes_per_launch_workspace")
        res["with_workspace"] = ww
    del case
    # the same workload over an fp8 cache (codes widened inside the kernel) and at d64
    for key, cdt, hd in (("extend_fp8", W.E4M3, 128), ("extend_d64", W.BF16, 64)):
        try:
            c = W.extend_case([P] * B, [Sfx] * B, hq, 8, hd, 16, cdt, W.BF16, seed=3,
                              device="cuda", shared_prefix=P)
            tt = _time_extend_case(c, P, Sfx, n, flush, False)
        except pkv.PkvError as e:
            res[key] = {"status": "failed", "error": str(e)}
            continue
        te, tm = sum(tt["extend"]) / n, _median(tt["extend"])
        fl = extend_useful_flops([P] * B, [Sfx] * B, hq, hd)
        tfx = fl / (te * 1e-3) / 1e12
        res[key] = {"cache_dtype": W.DTYPE_NAME[cdt], "act_dtype": "bf16", "head_dim": hd,
                    "ms_per_call": round(te, 5), "ms_per_call_median": round(tm, 5),
                    "useful_flops_per_call": fl, "tflops": round(tfx, 1),
                    "frac": round(tfx / bf16, 4), "frac_of_nominal": round(tfx / NOMINAL_BF16_TFLOPS, 4),
                    "peak_source": f"{peak_src} (bf16_tflops burst)",
                    "workspace_bytes": pkv.extend_workspace_bytes(c.k_cache, B, hq, rows, P + Sfx,
                                                                  k_scale=c.k_scale,
                                                                  v_scale=c.v_scale),
                    "cache_bytes": 2 * c.k_cache.numel() * c.k_cache.element_size()}
        ww = _extend_with_workspace(c, P, Sfx, n, flush, fl, bf16)
        if ww:
            res[key]["with_workspace"] = ww
        del c
    # the same rows through the shared-prefix call: one group, the 1,900-token prompt shared
    # (118 whole blocks), the 256 x 100 rows packed into tiles without per-request padding
    shared = {}
    for key, cdt, hd in (("bf16", W.BF16, 128), ("fp8", W.E4M3, 128), ("d64", W.BF16, 64)):
        try:
            c = W.extend_case([P] * B, [Sfx] * B, hq, 8, hd, 16, cdt, W.BF16, seed=3,
                              device="cuda", shared_prefix=P)
            ts = _time_extend_shared(c, [0, B], [P], B * Sfx, P + Sfx, n, flush)
        except pkv.PkvError as e:
            shared[key] = {"status": "failed", "error": str(e)}
            continue
        te, tm = sum(ts) / n, _median(ts)
        fl = extend_useful_flops([P] * B, [Sfx] * B, hq, hd)
        tfx = fl / (te * 1e-3) / 1e12
        shared[key] = {"cache_dtype": W.DTYPE_NAME[cdt], "act_dtype": "bf16", "head_dim": hd,
                       "ms_per_call": round(te, 5), "ms_per_call_median": round(tm, 5),
                       "useful_flops_per_call": fl, "tflops": round(tfx, 1),
                       "frac": round(tfx / bf16, 4),
                       "frac_of_nominal": round(tfx / NOMINAL_BF16_TFLOPS, 4)}
        # with the optional workspace: a bf16 cache's V pages widened to f16 once per
        # call (the widening pass is inside the timed call), then read by the kernel
        wsb = pkv.extend_shared_prefix_workspace_bytes(c.k_cache, c.k_scale, c.v_scale)
        if wsb:
            ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
            tw = _time_extend_shared(c, [0, B], [P], B * Sfx, P + Sfx, n, flush, ws=ws)
            tw_mean = sum(tw) / n
            tfw = fl / (tw_mean * 1e-3) / 1e12
            shared[key]["with_workspace"] = {
                "ms_per_call": round(tw_mean, 5), "ms_per_call_median": round(_median(tw), 5),
                "tflops": round(tfw, 1), "frac": round(tfw / bf16, 4),
                "frac_of_nominal": round(tfw / NOMINAL_BF16_TFLOPS, 4), "workspace_bytes": wsb}
            del ws
        del c
    res["extend_shared_prefix"] = {
        "call": "paged_extend_attn_shared_prefix, groups [0, 256], shared 1,900 tokens",
        "peak_source": f"{peak_src} (bf16_tflops burst)", **shared}
    # the same workload and useful flops through the call made for it (rows packed
    # across the requests that share the prefix), with its workspace
    ww = shared.get("bf16", {}).get("with_workspace")
    if ww:
        res["roofline_shared_prefix_call"] = {
            "kernel": "paged_extend_attn_shared_prefix (one group; workspace: V pages widened to "
                      "f16 once per call, the widening pass inside the timed call)",
            "bound": "tensor", "achieved": ww["tflops"], "peak": bf16, "unit": "TFLOP/s",
            "frac": ww["frac"], "peak_source": f"{peak_src} (bf16_tflops burst)",
            "frac_of_nominal": ww["frac_of_nominal"], "nominal_peak": NOMINAL_BF16_TFLOPS,
            "traffic": profiled_traffic(
                "extend_kernel_shared_prefix_extend.md",
                ["paged_kv_cache_285_gb300/csrc/extend.cu", "paged_kv_cache_285_gb300/csrc/ptx.cuh",
                 "paged_kv_cache_285_gb300/csrc/tcgen05.cuh",
                 "paged_kv_cache_285_gb300/csrc/internal.h#ExtendParams,ExtendPartialParams,FastDiv"],
                key="dram_bytes_per_launch_shared_prefix_workspace")}
    return res


def run_prefix_index_bench(n_requests=20000, seed=0):
    """The host prefix index (RadixIndex) on a chat-like trace: 64 system prompts
    of 1,000 tokens, a question of 10..200 tokens per request, 16-token blocks, a
    pool of 8,192 blocks so that eviction runs; every request does match, alloc,
    insert, release and frees its partial tail, through the public binding."""
    import numpy as np
    import paged_kv_cache_285_gb300 as pkv
    rng = np.random.default_rng(seed)
    bs, pool = 16, 8192
    prompts = [rng.integers(0, 32000, 1000).astype(np.int32) for _ in range(64)]
    reqs = [np.concatenate([prompts[rng.integers(0, 64)],
                            rng.integers(0, 32000, rng.integers(10, 201)).astype(np.int32)])
            for _ in range(n_requests)]
    x = pkv.RadixIndex(bs, pool)
    hit = total = refused = 0
    t0 = time.perf_counter()
    for t in reqs:
        m, blk = x.match(t)
        try:
            new = x.alloc(-(-len(t) // bs) - len(blk))
        except pkv.PkvError:
            x.release(t, m)
            refused += 1
            continue
        table = np.concatenate([blk, new])
        x.insert(t, table)
        x.release(t, m)
        if len(t) % bs:
            x.free(table[-1:])
        hit += m
        total += len(t)
    dt = time.perf_counter() - t0
    return {"workload": "64 x 1,000-token system prompts + 10..200-token questions, bs 16, "
                        "8,192-block pool", "requests": n_requests,
            "requests_per_s": round(n_requests / dt, 1),
            "cached_token_frac": round(hit / max(total, 1), 4), "refused": refused,
            "note": "host C++ index driven through the Python binding (5 calls per request)",
            "native_c_abi": _radix_trace_native(n_requests)}


def _build_radix_trace():
    """Compile bench_native/radix_trace.cpp (a benchmark driver, not part of the library)
    against libpkv.so; returns the executable's path or None."""
    import shutil
    here = os.path.dirname(os.path.abspath(__file__))
    src = os.path.join(here, "bench_native", "radix_trace.cpp")
    libdir = os.path.join(here, "paged_kv_cache_285_gb300")
    exe = os.path.join(here, "bench_native", "radix_trace")
    if os.path.exists(exe) and os.path.getmtime(exe) >= max(
            os.path.getmtime(src), os.path.getmtime(os.path.join(libdir, "libpkv.so"))):
        return exe
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        return None
    tmp = exe + f".tmp{os.getpid()}"
    r = subprocess.run([cxx, "-O3", "-std=c++17", f"-I{os.path.join(here, 'include')}",
                        "-I/usr/local/cuda/include", src, "-o", tmp, f"-L{libdir}", "-lpkv",
                        f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    if r.returncode != 0:
        return None
    os.replace(tmp, exe)
    return exe


def _radix_trace_native(n_requests):
    """The same trace recipe replayed by a C++ driver (bench_native/radix_trace.cpp) through
    the C ABI: the index's throughput without the binding's per-call overhead."""
    exe = _build_radix_trace()
    if exe is None:
        return {"status": "not built"}
    try:
        r = subprocess.run([exe, str(n_requests)], capture_output=True, text=True, timeout=120)
        if r.returncode != 0:
            return {"status": f"exit {r.returncode}"}
        d = json.loads(r.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError) as e:
        return {"status": f"failed: {e}"}
    d["note"] = "C++ driver through the C ABI, std::mt19937_64 trace of the same recipe"
    return d


def run_shared_prefix_bench(dev, hbm, peak_src, n=20):
    """Decode of 256 requests sharing one 1,000-token prompt (62 shared 16-token
    blocks + an 8-token tail in each request's own block), own tokens U[32, 256],
    32 q / 8 kv heads, d128, bf16: plain paged_decode_attn (every request reads
    the prefix) against paged_decode_attn_shared_prefix (the prefix once per
    group on the tensor cores, LSE merge), both in CUDA graphs, L2 flushed."""
    import paged_kv_cache_285_gb300 as pkv
    from paged_kv_cache_285_gb300 import workloads as W
    case = W.shared_prefix_decode(device="cuda")
    b, hq, hkv, d, bs = case.q.shape[0], case.num_q_heads, case.num_kv_heads, case.head_dim, 16
    lens = case.seq_lens.tolist()
    max_len = max(lens)
    prefix = 1000
    shared = (prefix // bs) * bs
    gi = torch.tensor([0, b], dtype=torch.int32, device=dev)
    gp = torch.tensor([prefix], dtype=torch.int32, device=dev)
    out_p, out_c = torch.empty_like(case.q), torch.empty_like(case.q)
    ws_p = torch.empty(max(pkv.decode_workspace_bytes(case.k_cache, b, hq, max_len, 0), 256),
                       dtype=torch.uint8, device=dev)
    ws_c = torch.empty(pkv.shared_prefix_decode_workspace_bytes(case.k_cache, b, hq, prefix,
                                                                max_len - prefix, 0),
                       dtype=torch.uint8, device=dev)

    def plain():
        pkv.paged_decode_attn(case.k_cache, case.v_cache, case.q, out_p, case.block_tables,
                              case.seq_lens, case.sm_scale, max_len, workspace=ws_p)

    def cascade():
        pkv.paged_decode_attn_shared_prefix(case.k_cache, case.v_cache, case.q, out_c,
                                            case.block_tables, case.seq_lens, case.sm_scale, gi,
                                            gp, b, prefix, max_len - prefix, workspace=ws_c)

    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        plain()
        cascade()
    torch.cuda.synchronize()
    graphs = []
    cap = torch.cuda.Stream()
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        for fn in (plain, cascade):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                fn()
            graphs.append(g)
    stream.wait_stream(cap)
    flush = L2Flush(dev)
    tot = [0.0, 0.0]
    for _ in range(n):
        for k, g in enumerate(graphs):
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            tot[k] += e0.elapsed_time(e1)
    ms_p, ms_c = tot[0] / n, tot[1] / n
    # warm: 10 calls back to back in one graph (no host launch between them),
    # so each call finds what the previous one left in L2 (the shared blocks,
    # partly the rest)
    reps = 10
    warm = []
    with torch.cuda.stream(cap):
        wgraphs = []
        for fn in (plain, cascade):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                for _ in range(reps):
                    fn()
            wgraphs.append(g)
    stream.wait_stream(cap)
    for g in wgraphs:
        g.replay()
        tw = []
        for _ in range(5):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            tw.append(e0.elapsed_time(e1) / reps)
        warm.append(_median(tw))
    kv_tok = hkv * d * 2 * 2  # K + V bytes per token (bf16)
    qo = 2 * b * hq * d * 2
    logical = sum(lens) * kv_tok + qo
    unique = (shared + sum(x - shared for x in lens)) * kv_tok + qo
    diff = (out_p.float() - out_c.float()).abs().max().item()
    return {"workload": "256 requests sharing one 1,000-token prompt (62 shared blocks), own "
                        "tokens U[32,256], 32q/8kv, d128, bf16, bs16",
            "plain_ms": round(ms_p, 5), "shared_prefix_ms": round(ms_c, 5),
            "speedup": round(ms_p / ms_c, 3),
            "plain_ms_warm": round(warm[0], 5), "shared_prefix_ms_warm": round(warm[1], 5),
            "logical_bytes": logical, "unique_bytes": unique,
            "plain_gbs_logical": round(logical / (ms_p * 1e-3) / 1e9, 1),
            "shared_prefix_gbs_logical": round(logical / (ms_c * 1e-3) / 1e9, 1),
            "shared_prefix_gbs_unique": round(unique / (ms_c * 1e-3) / 1e9, 1),
            "shared_prefix_frac_of_hbm_unique": round(unique / (ms_c * 1e-3) / 1e9 / hbm, 4),
            "peak_source": f"{peak_src} (hbm_gbs)",
            "max_abs_diff_plain_vs_shared_prefix": diff,
            "l2": "256 MiB buffer written then read between calls; *_warm: 10 calls back to "
                  "back in one graph, no flush (median of 5 replays)"}


def run_more_decode_configs_bench(dev, hbm, peak_src, n=10):
    """Two more of the pages' workload shapes, timed like the headline step (each
    request's current token appended by the decode kernel, then attention; one
    CUDA graph; L2 flushed between steps): the Llama-2-70B-shaped fp8 layer, and
    the long-context step over all 32 layers of 4 x 100,000 tokens."""
    import paged_kv_cache_285_gb300 as pkv
    from paged_kv_cache_285_gb300 import workloads as W
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(dev)

    def prepare(case, max_len):
        b = case.q.shape[0]
        out = torch.empty_like(case.q)
        wsb = pkv.decode_workspace_bytes(case.k_cache, b, case.num_q_heads, max_len, 0,
                                         case.k_scale, case.v_scale)
        ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device=dev)
        return lambda: pkv.paged_decode_attn_append(
            case.k_cache, case.v_cache, case.new_k, case.new_v, case.q, out, case.block_tables,
            case.seq_lens, case.sm_scale, max_len, k_scale=case.k_scale, v_scale=case.v_scale,
            workspace=ws)

    def time_step(fns):
        for _ in range(3):
            for f in fns:
                f()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for f in fns:
                    f()
        stream.wait_stream(cap)
        g.replay()
        tot = 0.0
        for _ in range(n):
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            tot += e0.elapsed_time(e1)
        return tot / n

    res = {}
    case = W.fp8_70b_decode(device="cuda")
    ms = time_step([prepare(case, 4096)])
    nbytes = sum(decode_step_bytes(case))
    res["fp8_70b_layer"] = {
        "workload": "128 requests x 4,096 tokens, 64q/8kv, d128, fp8_e4m3 K/V, bf16 q/out, bs16",
        "ms_per_step": round(ms, 5), "step_bytes": nbytes,
        "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
        "frac_of_hbm": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4)}
    del case
    torch.cuda.empty_cache()
    cases = W.long_context_layers(device="cuda")
    ms = time_step([prepare(c, 100_000) for c in cases])
    nbytes = sum(sum(decode_step_bytes(c)) for c in cases)
    res["long_context_32_layers"] = {
        "workload": "4 requests x 100,000 tokens, 32 layers (one pool each), 32q/8kv, d128, fp16, bs32",
        "ms_per_step": round(ms, 5), "step_bytes": nbytes,
        "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
        "frac_of_hbm": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4),
        "tokens_per_s": round(4 / (ms * 1e-3), 1)}
    del cases
    torch.cuda.empty_cache()
    res["peak_source"] = f"{peak_src} (hbm_gbs)"
    return res


def run_chain_hash_bench(dev, hbm, peak_src, n=20, seed=0):
    """pkv_chain_hash over a prefill batch: 1,024 requests of 4,096 token ids,
    16-token blocks, a salt per request; algorithmic bytes = the token ids read
    (4 B each) + the hashes written (8 B per block) + offsets and salts."""
    import paged_kv_cache_285_gb300 as pkv
    g = torch.Generator(device="cpu").manual_seed(seed)
    B, L, bs = 1024, 4096, 16
    toks = torch.randint(0, 128256, (B * L,), generator=g, dtype=torch.int32).to(dev)
    indptr = (torch.arange(B + 1, dtype=torch.int32) * L).to(dev)
    salts = torch.randint(-2**62, 2**62, (B,), generator=g, dtype=torch.int64).to(dev)
    hashes = torch.empty((B, L // bs), dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        pkv.chain_hash(toks, indptr, bs, hashes, salts=salts)
    flush = L2Flush(dev)
    tot = 0.0
    for _ in range(n):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pkv.chain_hash(toks, indptr, bs, hashes, salts=salts)
        e1.record(stream)
        e1.synchronize()
        tot += e0.elapsed_time(e1)
    ms = tot / n
    nbytes = 4 * B * L + 8 * B * (L // bs) + 4 * (B + 1) + 8 * B
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": "1,024 requests x 4,096 token ids, 16-token blocks, salted",
            "ms_per_call": round(ms, 5), "tokens_per_s": round(B * L / (ms * 1e-3), 1),
            "achieved_gbs": round(gbs, 1), "hbm_peak_gbs": hbm, "frac_of_hbm": round(gbs / hbm, 4),
            "peak_source": f"{peak_src} (hbm_gbs)", "algorithmic_bytes": nbytes,
            "bound": "latency: each request's chain is %d dependent hash steps" % (L // bs),
            "l2": "256 MiB buffer written then read between calls; *_warm: 10 calls back to "
                  "back in one graph, no flush (median of 5 replays)"}


def run_append_fill_bench(dev, hbm, peak_src, n=10):
    """pkv_kv_append as a bulk fill: every position of a layer's context written in
    one call (the Llama-3-8B-shaped layer kept in bf16, the Llama-2-70B-shaped
    layer stored as fp8 e4m3); algorithmic bytes = the K and V rows read (bf16) +
    the slot ids (8 B per token) + the K and V rows written (cache dtype)."""
    import paged_kv_cache_285_gb300 as pkv
    from paged_kv_cache_285_gb300 import workloads as W
    stream = torch.cuda.current_stream(dev)
    flush = L2Flush(dev)
    res = {}
    layers = (
        ("llama3_8b_layer_bf16", W.llama3_8b_decode,
         "64 requests, n ~ U[512,4096], 8 kv heads, d128, bf16 -> bf16 cache, bs16"),
        ("llama2_70b_layer_fp8", W.fp8_70b_decode,
         "128 requests x 4,096 tokens, 8 kv heads, d128, bf16 -> fp8_e4m3 cache, bs16"))
    for name, make, what in layers:
        case = make(device=dev)
        slots = W.context_slots(case)
        t, hkv, d = slots.numel(), case.k_cache.shape[1], case.k_cache.shape[3]
        g = torch.Generator(device=dev).manual_seed(7)
        nk = torch.randn((t, hkv, d), generator=g, device=dev).to(torch.bfloat16)
        nv = torch.randn((t, hkv, d), generator=g, device=dev).to(torch.bfloat16)

        def call():
            pkv.kv_append(case.k_cache, case.v_cache, nk, nv, slots, k_scale=case.k_scale,
                          v_scale=case.v_scale)

        for _ in range(3):
            call()
        torch.cuda.synchronize()
        tot = 0.0
        for _ in range(n):
            flush()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            call()
            e1.record(stream)
            e1.synchronize()
            tot += e0.elapsed_time(e1)
        ms = tot / n
        nbytes = t * hkv * d * (2 + case.k_cache.element_size()) * 2 + 8 * t
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = {"workload": what, "tokens": t, "ms_per_call": round(ms, 5),
                     "bytes": nbytes, "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / hbm, 4)}
        del case, slots, nk, nv
        torch.cuda.empty_cache()
    res["peak_source"] = f"{peak_src} (hbm_gbs)"
    res["l2"] = "256 MiB buffer written then read between calls"
    return res


def cpu_baseline_decode(case, budget_s=10.0):
    """The fp64 C oracle (OpenMP over (request, head)) on this host, on whole passes
    over the same decode layer until `budget_s` seconds have been spent."""
    import oracle
    from paged_kv_cache_285_gb300 import workloads as W
    S = W.to_numpy_storage
    k, v, q = S(case.k_cache), S(case.v_cache), S(case.q)
    bt, sl = case.block_tables.cpu().numpy(), case.seq_lens.cpu().numpy()
    app_b, dec_b = decode_step_bytes(case)
    # sample: the first requests of the batch, enlarged until one pass takes >= 1/4 budget
    nreq = 4
    while True:
        pairs = [(bb, h) for bb in range(nreq) for h in range(case.num_q_heads)]
        t0 = time.perf_counter()
        oracle.paged_decode(k, v, case.cache_dtype, case.k_scale, case.v_scale, q, case.act_dtype,
                            bt, sl, case.num_q_heads, case.sm_scale, pairs=pairs)
        dt = time.perf_counter() - t0
        if dt >= budget_s / 4 or nreq >= len(sl):
            break
        nreq = min(len(sl), nreq * 2)
    passes, tot = 1, dt
    while tot < budget_s:
        t0 = time.perf_counter()
        oracle.paged_decode(k, v, case.cache_dtype, case.k_scale, case.v_scale, q, case.act_dtype,
                            bt, sl, case.num_q_heads, case.sm_scale, pairs=pairs)
        tot += time.perf_counter() - t0
        passes += 1
    frac = float(sl[:nreq].sum()) / float(sl.sum())
    sample_bytes = dec_b * frac
    return {"value": round(sample_bytes * passes / tot / 1e9, 4), "unit": "GB/s",
            "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"fp64 C oracle decode of requests 0..{nreq - 1} of {len(sl)} "
                      f"(all {case.num_q_heads} heads), {passes} passes in {tot:.1f} s"}


def run_reference(args, world, rank):
    """The fp64 CPU oracle timed as the reference arm (rank 0 only)."""
    if rank != 0:
        return None
    from paged_kv_cache_285_gb300 import workloads as W
    case = W.llama3_8b_decode(device="cpu") if args.workload == "llama3_8b_layer" else None
    if case is None:
        return {"impl": "reference", "unavailable": f"no oracle arm for workload {args.workload}"}
    base = cpu_baseline_decode(case, budget_s=max(2.0, min(20.0, args.cpu_seconds)))
    val = base["value"]
    return {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "step": "decode attention, fp64 CPU oracle"},
            "cpu_baseline": base,
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_only(args, local):
    import paged_kv_cache_285_gb300 as pkv
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pkv.load()
    hbm, bf16, bf16_sus, peak_src = peaks()
    fns = {"extend": lambda: run_extend_bench(args, dev, bf16, bf16_sus, peak_src),
           "shared_prefix_decode": lambda: run_shared_prefix_bench(dev, hbm, peak_src),
           "append_fill": lambda: run_append_fill_bench(dev, hbm, peak_src),
           "more_decode_configs": lambda: run_more_decode_configs_bench(dev, hbm, peak_src),
           "chain_hash": lambda: run_chain_hash_bench(dev, hbm, peak_src),
           "prefix_index": run_prefix_index_bench}
    return {"only": args.only, args.only: fns[args.only]()}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--workload", default="llama3_8b_layer",
                    choices=["llama3_8b_layer", "fp8_70b_layer", "shared_prefix_decode", "tiny"])
    ap.add_argument("--no-extend", dest="extend", action="store_false")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side", action="store_true",
                    help="the decode step only: no extend, no side benchmarks (profiling)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--only", default=None,
                    choices=["extend", "shared_prefix_decode", "append_fill", "more_decode_configs",
                             "chain_hash", "prefix_index"],
                    help="run one side benchmark alone (for profiling on a small device footprint); "
                         "prints that object only, not the benchmark line")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)
    world, rank, local = dist_setup(args.gpus)
    if args.only is not None:
        res = run_only(args, local)
    elif args.impl == "reference":
        res = run_reference(args, world, rank)
    else:
        res = run_decode_bench(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
