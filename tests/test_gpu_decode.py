"""GPU parity of pkv_paged_decode_attn against the fp64 oracle.

Small cases span several 16-token tiles, partial last blocks, every supported
head_dim / block_size / dtype, GQA groups from 1 to 16 (powers of two and
others), forced split counts and the edge cases; the workload-sized cases run in the launch configuration the benchmark
times, compared in full where the oracle is fast enough and on sampled
(request, head) pairs otherwise."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_285_gb300 as pkv
from paged_kv_cache_285_gb300 import workloads as W
from tests.pkv_testlib import BF16, E4M3, F16, assert_attention_close, to_f64

pytestmark = pytest.mark.gpu
S = W.to_numpy_storage


def gpu_decode(case, num_splits=0, max_seq_len=None, lens=None):
    lens = case.seq_lens if lens is None else lens
    b = case.q.shape[0]
    n_max = int(lens.max()) if max_seq_len is None else max_seq_len
    out = torch.full_like(case.q, float("nan"))
    lse = torch.full((b, case.num_q_heads), float("nan"), dtype=torch.float32, device="cuda")
    ws_bytes = pkv.decode_workspace_bytes(case.k_cache, b, case.num_q_heads, n_max, num_splits,
                                          case.k_scale, case.v_scale)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    pkv.paged_decode_attn(case.k_cache, case.v_cache, case.q, out, case.block_tables, lens,
                          case.sm_scale, n_max, k_scale=case.k_scale, v_scale=case.v_scale,
                          num_splits=num_splits, lse_out=lse, workspace=ws)
    torch.cuda.synchronize()
    return out, lse


def append_both(case):
    """GPU append of the current token at position seq_len-1; the oracle applies its
    own append to a host copy of the pre-append pool (no oracle input comes from the GPU)."""
    k0, v0 = S(case.k_cache), S(case.v_cache)
    pkv.kv_append(case.k_cache, case.v_cache, case.new_k, case.new_v, case.slot_last,
                  k_scale=case.k_scale, v_scale=case.v_scale)
    kr, vr, st = oracle.kv_append(k0, v0, case.cache_dtype, case.k_scale, case.v_scale,
                                  S(case.new_k), S(case.new_v), case.act_dtype,
                                  case.slot_last.cpu().numpy())
    assert st == 0
    return kr, vr


def oracle_decode(case, pairs=None, lens=None, pools=None):
    lens = case.seq_lens if lens is None else lens
    kh, vh = (S(case.k_cache), S(case.v_cache)) if pools is None else pools
    out, lse, st = oracle.paged_decode(kh, vh, case.cache_dtype,
                                       case.k_scale, case.v_scale, S(case.q), case.act_dtype,
                                       case.block_tables.cpu().numpy(), lens.cpu().numpy(),
                                       case.num_q_heads, case.sm_scale, pairs=pairs)
    assert st == 0
    return out, lse


def check(case, out, lse, what, pairs=None, pools=None):
    ref, ref_lse = oracle_decode(case, pairs=pairs, pools=pools)
    got = to_f64(out)
    gl = lse.cpu().double().numpy()
    if pairs is not None:
        got = np.stack([got[b, h] for b, h in pairs])
        gl = np.array([gl[b, h] for b, h in pairs])
    assert_attention_close(got, ref, case.act_dtype, fp8=False, what=what)
    fin = np.isfinite(ref_lse)
    assert np.all(np.isfinite(gl) == fin), what
    assert np.max(np.abs(gl[fin] - ref_lse[fin]), initial=0) <= 1e-3, what


CONFIGS = [
    # (lens, hq, hkv, d, bs, cache, act)
    ([37, 60, 16, 1], 4, 1, 64, 16, F16, F16),
    ([1, 15, 16, 17, 31, 32, 33, 100], 8, 2, 128, 16, BF16, BF16),
    ([5, 64, 65, 200, 33], 8, 8, 128, 32, F16, F16),
    ([300, 17, 48], 16, 2, 64, 32, BF16, BF16),
    ([129, 1, 77, 256], 32, 8, 128, 16, BF16, BF16),
    ([200, 3, 64], 64, 8, 128, 16, E4M3, BF16),
    ([45, 90, 16], 8, 1, 64, 16, E4M3, F16),
    ([33, 250], 4, 2, 128, 32, E4M3, F16),
    ([40, 7, 500], 4, 4, 64, 16, F16, F16),
    # GQA groups above 8 (one CTA per 8 heads of a kv head) and not powers of two
    ([130, 17, 600], 64, 4, 128, 16, BF16, BF16),
    ([33, 90], 12, 1, 64, 32, F16, F16),
    ([300, 5], 96, 8, 128, 16, E4M3, BF16),
    ([77, 200, 1], 6, 2, 128, 16, BF16, BF16),
]


@pytest.mark.parametrize("cfg", CONFIGS, ids=lambda c: f"h{c[1]}x{c[2]}-d{c[3]}-bs{c[4]}-c{c[5]}a{c[6]}")
@pytest.mark.parametrize("splits", [0, 1, 2, 7])
def test_decode_small(cfg, splits):
    lens, hq, hkv, d, bs, cdt, adt = cfg
    case = W.decode_case(lens, hq, hkv, d, bs, cdt, adt, seed=sum(lens) + hq + d, device="cuda")
    out, lse = gpu_decode(case, num_splits=splits)
    check(case, out, lse, f"{cfg} splits={splits}")
    assert pkv.get_device_error() == 0


def test_tiny_config_with_append():
    # tiny workload: append the current token at position seq_len-1, then decode
    case = W.tiny_decode(device="cuda")
    pools = append_both(case)
    for splits in (0, 1, 2, 3, 4):
        out, lse = gpu_decode(case, num_splits=splits)
        check(case, out, lse, f"tiny splits={splits}", pools=pools)


def test_single_token_is_exact():
    for cdt, adt in ((F16, F16), (BF16, BF16)):
        case = W.decode_case([1, 1, 1], 8, 2, 128, 16, cdt, adt, seed=60, device="cuda")
        out, _ = gpu_decode(case)
        for b in range(3):
            blk = int(case.block_tables[b, 0])
            for h in range(8):
                torch.testing.assert_close(out[b, h], case.v_cache[blk, h // 4, 0], rtol=0, atol=0)


def test_empty_sequences_and_batch():
    case = W.decode_case([0, 20, 0], 8, 2, 128, 16, BF16, BF16, seed=61, device="cuda",
                         extra_capacity=1)
    out, lse = gpu_decode(case, max_seq_len=64)
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    assert torch.all(torch.isneginf(lse[0])) and torch.all(torch.isneginf(lse[2]))
    check(case, out, lse, "empty rows")
    # batch of zero requests is a no-op
    pkv.paged_decode_attn(case.k_cache, case.v_cache, case.q[:0], out[:0], case.block_tables[:0],
                          case.seq_lens[:0], case.sm_scale, 64)


def test_garbage_beyond_sequence_end_is_ignored():
    # slots past seq_len in the last block hold inf/nan: they must not leak in
    case = W.decode_case([20, 37, 5], 8, 2, 128, 16, BF16, BF16, seed=62, device="cuda",
                         extra_capacity=12)
    for b, n in enumerate([20, 37, 5]):
        blk = int(case.block_tables[b, (n - 1) // 16])
        off = n % 16
        if off:
            case.k_cache[blk, :, off:] = float("inf")
            case.v_cache[blk, :, off:] = float("nan")
    out, lse = gpu_decode(case, num_splits=2)
    check(case, out, lse, "garbage tail")


def test_block_permutation_is_bit_identical():
    case = W.decode_case([300, 17, 129, 64], 32, 8, 128, 16, BF16, BF16, seed=63, device="cuda")
    out0, lse0 = gpu_decode(case)
    nb = case.k_cache.shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(1)).cuda()
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(nb, device="cuda")
    case.k_cache = case.k_cache[perm].contiguous()
    case.v_cache = case.v_cache[perm].contiguous()
    t = case.block_tables.long()
    case.block_tables = torch.where(t >= 0, inv[t.clamp(min=0)], t).to(torch.int32).contiguous()
    out1, lse1 = gpu_decode(case)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_shared_prefix_equals_private_copies_bit_identical():
    case = W.decode_case([1000 + s for s in (40, 200, 33, 129)], 32, 8, 128, 16, BF16, BF16,
                         seed=64, device="cuda", shared_prefix=1000)
    out0, lse0 = gpu_decode(case)
    t = case.block_tables.clone()
    shared = 1000 // 16
    extra_k, extra_v = [], []
    nb = case.k_cache.shape[0]
    for b in range(1, t.shape[0]):
        for j in range(shared):
            extra_k.append(case.k_cache[t[b, j]])
            extra_v.append(case.v_cache[t[b, j]])
            t[b, j] = nb + len(extra_k) - 1
    case.k_cache = torch.cat([case.k_cache, torch.stack(extra_k)]).contiguous()
    case.v_cache = torch.cat([case.v_cache, torch.stack(extra_v)]).contiguous()
    case.block_tables = t.contiguous()
    out1, lse1 = gpu_decode(case)
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_bad_block_id_reads_zeros_and_is_reported():
    case = W.decode_case([40], 8, 2, 128, 16, BF16, BF16, seed=65, device="cuda")
    case.block_tables[0, 1] = 10_000_000
    out, lse = gpu_decode(case)
    assert torch.isfinite(out).all()
    assert pkv.get_device_error() == 1


# ---- workload-sized cases (the benchmark's launch configuration) -------------------

def _sample_pairs(b, hq, k, seed):
    rng = np.random.default_rng(seed)
    idx = rng.choice(b * hq, size=min(k, b * hq), replace=False)
    return [(int(i // hq), int(i % hq)) for i in sorted(idx)]


def test_llama3_8b_layer_full():
    case = W.llama3_8b_decode(device="cuda")
    pools = append_both(case)
    out, lse = gpu_decode(case, max_seq_len=4096)
    check(case, out, lse, "llama3-8b layer", pools=pools)


def test_shared_prefix_decode_sampled():
    case = W.shared_prefix_decode(device="cuda")
    out, lse = gpu_decode(case, max_seq_len=1256)
    check(case, out, lse, "shared prefix", pairs=_sample_pairs(256, 32, 256, 1))


def test_fp8_70b_layer_sampled():
    # every one of the 64 heads of 12 requests spread over the batch (768 of 8,192 rows)
    case = W.fp8_70b_decode(device="cuda")
    pools = append_both(case)
    out, lse = gpu_decode(case, max_seq_len=4096)
    reqs = [0, 1, 17, 31, 32, 63, 64, 77, 95, 100, 126, 127]
    pairs = [(b, h) for b in reqs for h in range(64)]
    check(case, out, lse, "fp8 70b layer", pairs=pairs, pools=pools)


def test_long_context_layers_full():
    # three of the 32 layers at full size (4 x 100,000 tokens, bs 32, fp16), every
    # (request, head) row against the oracle: the split-KV plan of the benchmark at 100k
    for layer in (0, 15, 31):
        case = W.decode_case([100_000] * 4, 32, 8, 128, 32, F16, F16, seed=100 + layer,
                             device="cuda", extra_capacity=0)
        out, lse = gpu_decode(case, max_seq_len=100_000)
        check(case, out, lse, f"long context layer {layer}")
        del case, out, lse
        torch.cuda.empty_cache()
