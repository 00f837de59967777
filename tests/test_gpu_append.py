"""GPU parity of pkv_kv_append against the oracle: bit-exact over the whole
cache pool (so a stray write anywhere shows up), for 16-bit copies and the fp8
store, plus skipped / out-of-pool slots."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_285_gb300 as pkv
from paged_kv_cache_285_gb300 import workloads as W
from tests.pkv_testlib import BF16, E4M3, F16

pytestmark = pytest.mark.gpu
S = W.to_numpy_storage


def _check_append(k_cache, v_cache, cdt, ks, vs, new_k, new_v, adt, slots):
    k0, v0 = S(k_cache), S(v_cache)
    pkv.kv_append(k_cache, v_cache, new_k, new_v, slots, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    kr, vr, st = oracle.kv_append(k0, v0, cdt, ks, vs, S(new_k), S(new_v), adt, slots.cpu().numpy())
    np.testing.assert_array_equal(S(k_cache), kr)
    np.testing.assert_array_equal(S(v_cache), vr)
    return st


def test_tiny_append_next_position():
    # one token per request at position seq_len; the 16-token request needs its new block
    case = W.tiny_decode(device="cuda")
    assert _check_append(case.k_cache, case.v_cache, F16, 1, 1, case.new_k, case.new_v, F16,
                         case.slot_next) == 0
    assert pkv.get_device_error() == 0


@pytest.mark.parametrize("cdt,adt", [(BF16, BF16), (F16, F16), (E4M3, BF16), (E4M3, F16)])
def test_bulk_suffix_append(cdt, adt):
    # 32 requests x 100 suffix tokens after a shared 1,900-token prefix
    case = W.extend_case([1900] * 32, [100] * 32, 32, 8, 128, 16, cdt, adt, seed=50,
                         device="cuda", shared_prefix=1900)
    assert _check_append(case.k_cache, case.v_cache, cdt, case.k_scale, case.v_scale, case.suffix_k,
                         case.suffix_v, adt, case.suffix_slots) == 0


@pytest.mark.parametrize("adt", [BF16, F16])
def test_fp8_store_edge_values(adt):
    # saturation, ties between codes, subnormals and signed zero through the real kernel
    d, hkv = 64, 1
    k = torch.zeros((4, hkv, 16, d), dtype=torch.uint8, device="cuda")
    v = torch.zeros_like(k)
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    finite = codes.view(torch.float8_e4m3fn).float()
    finite = finite[torch.isfinite(finite)].unique()
    mids = (finite[1:] + finite[:-1]) / 2
    extra = torch.tensor([0.0, -0.0, 500.0, -1e4, 1e30, float("inf"), float("-inf"), 448.0,
                          464.0, -464.0, 2.0 ** -10, 3 * 2.0 ** -10])
    vals = torch.cat([finite, mids, extra])
    tdt = torch.bfloat16 if adt == BF16 else torch.float16
    vals = vals[: (vals.numel() // d) * d]
    rows = vals.numel() // d
    x = vals.reshape(rows, hkv, d).to(tdt)
    slots = torch.arange(rows, dtype=torch.int64) * 3 % 64
    _check_append(k, v, E4M3, 0.5, 1.0, x.cuda(), (-x).cuda(), adt, slots.cuda())


def test_skip_negative_and_out_of_pool():
    case = W.decode_case([20, 30, 5], 8, 2, 128, 16, BF16, BF16, seed=51, device="cuda")
    nb = case.k_cache.shape[0]
    slots = torch.tensor([-1, nb * 16 + 3, 17], dtype=torch.int64, device="cuda")
    assert pkv.get_device_error() == 0
    st = _check_append(case.k_cache, case.v_cache, BF16, 1, 1, case.new_k, case.new_v, BF16, slots)
    assert st == 1
    assert pkv.get_device_error() == 2  # PKV_DEVERR_BAD_SLOT, then cleared
    assert pkv.get_device_error() == 0


def test_zero_tokens_is_noop():
    case = W.decode_case([20], 8, 2, 128, 16, BF16, BF16, seed=52, device="cuda")
    before = S(case.k_cache)
    pkv.kv_append(case.k_cache, case.v_cache, case.new_k[:0], case.new_v[:0],
                  case.slot_last[:0])
    torch.cuda.synchronize()
    np.testing.assert_array_equal(S(case.k_cache), before)


def _fill_inputs(case, seed):
    slots = W.context_slots(case)
    t, hkv, d = slots.numel(), case.k_cache.shape[1], case.k_cache.shape[3]
    g = torch.Generator(device="cuda").manual_seed(seed)
    new_k = torch.randn((t, hkv, d), generator=g, device="cuda").to(torch.bfloat16)
    new_v = torch.randn((t, hkv, d), generator=g, device="cuda").to(torch.bfloat16)
    return slots, new_k, new_v


def test_full_context_fill_llama3_8b_layer():
    # every position of the Llama-3-8B-shaped layer (64 requests, ~147k tokens) in one call:
    # each slot's row holds its input row bit for bit, every other byte of the pool is unchanged
    case = W.llama3_8b_decode(device="cuda")
    slots, new_k, new_v = _fill_inputs(case, 60)
    nb, hkv, bs, d = case.k_cache.shape
    k0, v0 = case.k_cache.clone(), case.v_cache.clone()
    pkv.kv_append(case.k_cache, case.v_cache, new_k, new_v, slots)
    torch.cuda.synchronize()
    written = torch.zeros(nb * bs, dtype=torch.bool, device="cuda")
    written[slots] = True
    assert int(written.sum()) == slots.numel()  # the slot mapping has no repeats
    for pool, before, new in ((case.k_cache, k0, new_k), (case.v_cache, v0, new_v)):
        assert torch.equal(pool[slots // bs, :, slots % bs, :].view(torch.int16), new.view(torch.int16))
        rows = pool.permute(0, 2, 1, 3).reshape(nb * bs, hkv, d)
        rows0 = before.permute(0, 2, 1, 3).reshape(nb * bs, hkv, d)
        assert torch.equal(rows[~written].view(torch.int16), rows0[~written].view(torch.int16))
    assert pkv.get_device_error() == 0


def test_full_context_fill_fp8_70b_layer_sampled():
    # the Llama-2-70B-shaped layer (128 x 4,096 tokens) stored as fp8 e4m3 in one call;
    # 514 sampled rows (the first and last among them) against the oracle's encoder
    case = W.fp8_70b_decode(device="cuda")
    slots, new_k, new_v = _fill_inputs(case, 61)
    nb, hkv, bs, d = case.k_cache.shape
    pkv.kv_append(case.k_cache, case.v_cache, new_k, new_v, slots, k_scale=case.k_scale,
                  v_scale=case.v_scale)
    torch.cuda.synchronize()
    t = slots.numel()
    rng = np.random.default_rng(61)
    idx = np.unique(np.concatenate([[0, t - 1], rng.choice(t, 512, replace=False)]))
    n = idx.size
    nblk = -(-n // bs)
    small = np.zeros((nblk, hkv, bs, d), dtype=np.uint8)
    sel = torch.as_tensor(idx, device="cuda")
    kr, vr, st = oracle.kv_append(small, small.copy(), E4M3, case.k_scale, case.v_scale,
                                  S(new_k[sel]), S(new_v[sel]), BF16, np.arange(n, dtype=np.int64))
    assert st == 0
    ss = slots[sel]
    for pool, ref in ((case.k_cache, kr), (case.v_cache, vr)):
        got = S(pool[ss // bs, :, ss % bs, :])
        want = ref.transpose(0, 2, 1, 3).reshape(nblk * bs, hkv, d)[:n]
        np.testing.assert_array_equal(got, want)
    assert pkv.get_device_error() == 0


# K and V scales of the exhaustive fp8 store tests: ordinary amax / 448 values (random and
# round ones), scale 1, the ends of the range where the store skips its division, and
# scales outside it
_FP8_SCALES = [(1.0, 3.0), (1 / 448, 5 / 448), (4 / 448, 4.7316 / 448), (0.83 / 448, 13.1 / 448),
               (2.0 ** -64, 2.0 ** 64), (2.0 ** -70, 1e30), (3e-30, 0.3), (7.0, 2.0 ** -60)]


def _all_patterns(adt, nan):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    exp_mask, man_mask = (0x7F80, 0x007F) if adt == BF16 else (0x7C00, 0x03FF)
    is_nan = ((bits & exp_mask) == exp_mask) & ((bits & man_mask) != 0)
    sel = bits[is_nan] if nan else bits[~is_nan]
    d = 128
    sel = np.resize(sel, -(-sel.size // d) * d)  # whole rows (repeats a few patterns)
    tdt = torch.bfloat16 if adt == BF16 else torch.float16
    return torch.from_numpy(sel.view(np.int16).copy()).view(tdt).reshape(-1, 1, d)


@pytest.mark.parametrize("adt", [BF16, F16])
def test_fp8_store_every_finite_and_infinite_input(adt):
    # every non-NaN 16-bit pattern, K and V with different scales, against the oracle's
    # e4m3(fp32(x) / scale): the store's division-free path and its fallback agree with it
    x = _all_patterns(adt, nan=False)
    rows, bs = x.shape[0], 16
    slots = torch.arange(rows, dtype=torch.int64, device="cuda")
    for ks, vs in _FP8_SCALES:
        k = torch.zeros((-(-rows // bs), 1, bs, 128), dtype=torch.uint8, device="cuda")
        v = torch.zeros_like(k)
        assert _check_append(k, v, E4M3, ks, vs, x.cuda(), x.flip(0).cuda(), adt, slots) == 0


@pytest.mark.parametrize("adt", [BF16, F16])
def test_fp8_store_nan_inputs(adt):
    x = _all_patterns(adt, nan=True)
    rows, bs = x.shape[0], 16
    slots = torch.arange(rows, dtype=torch.int64, device="cuda")
    k = torch.zeros((-(-rows // bs), 1, bs, 128), dtype=torch.uint8, device="cuda")
    v = torch.zeros_like(k)
    assert _check_append(k, v, E4M3, 1 / 448, 1.0, x.cuda(), x.cuda(), adt, slots) == 0
