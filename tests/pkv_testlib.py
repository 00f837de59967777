"""Shared helpers for the tests: building small paged pools from values, and
the output comparison rule.

Comparison rule (the tolerance the attention results are held to):
  * 16-bit outputs: every element lies within 2e-3 plus half an output ulp
    of the fp64 oracle (rounding a bf16 value in [1, 2) alone can move it by
    3.9e-3, so the 2e-3 bound applies to the error beyond the output's own
    rounding), and the relative L2 error against the fp64 oracle rounded once
    (round-to-nearest-even) to the output dtype is <= 1e-3 (against the
    unrounded oracle, bf16 rounding alone gives ~1.6e-3).
  * fp8 caches: max-abs <= 3e-2 against the oracle run on the same codes.
"""
from __future__ import annotations

import numpy as np
import torch

F16, BF16, E4M3 = 0, 1, 2


def bits_of(values, dtype):
    """float array -> storage bits (uint16 for f16/bf16)."""
    v = np.asarray(values, dtype=np.float64)
    if dtype == F16:
        return v.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        t = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16)
    raise ValueError(dtype)


def empty_pool(num_blocks, hkv, bs, d, dtype, fill=0.0):
    if dtype == E4M3:
        return np.zeros((num_blocks, hkv, bs, d), np.uint8)
    return np.broadcast_to(bits_of([fill], dtype), (num_blocks, hkv, bs, d)).copy()


def put_sequence(pool, table_row, g, seq_bits):
    """Write seq_bits[t, :] as logical token t of kv head g through table_row."""
    bs = pool.shape[2]
    for t in range(seq_bits.shape[0]):
        pool[table_row[t // bs], g, t % bs, :] = seq_bits[t]


def round_to(x, dtype):
    """fp64 -> nearest value of the act dtype (round to nearest even), as fp64."""
    t = torch.from_numpy(np.asarray(x, np.float64))
    tdt = torch.float16 if dtype == F16 else torch.bfloat16
    return t.to(tdt).to(torch.float64).numpy()


def half_ulp(x, dtype):
    a = np.abs(np.asarray(x, np.float64))
    mant = 10 if dtype == F16 else 7
    e = np.floor(np.log2(np.maximum(a, 1e-30)))
    e = np.maximum(e, -14 if dtype == F16 else -126)
    return np.ldexp(1.0, (e - mant - 1).astype(int))


def assert_attention_close(gpu, ref, act_dtype, fp8=False, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    if gpu.size == 0:
        return
    if fp8:
        err = np.max(np.abs(gpu - ref))
        assert err <= 3e-2, f"{what}: fp8 max-abs {err:.3e} > 3e-2"
        return
    # max-abs: the error beyond the output's own rounding (half an ulp of the act
    # dtype at the exact value) stays within 2e-3
    excess = np.abs(gpu - ref) - half_ulp(ref, act_dtype)
    worst = float(np.max(excess))
    assert worst <= 2e-3, f"{what}: max-abs beyond output rounding {worst:.3e} > 2e-3"
    # relative L2 against the oracle rounded once to the output dtype
    ref_r = round_to(ref, act_dtype)
    den = np.linalg.norm(ref_r)
    rel = np.linalg.norm(gpu - ref_r) / den if den > 0 else np.linalg.norm(gpu - ref_r)
    assert rel <= 1e-3, f"{what}: rel-L2 {rel:.3e} > 1e-3 (vs rounded oracle)"


def to_f64(t: torch.Tensor):
    return t.detach().to("cpu").to(torch.float64).numpy()
