"""Helpers of the GPU parity tests: moving device tensors to numpy views the
oracle reads, sentinel-filled buffers, and the merge tolerances.

Tolerances (written here once, used by every merge comparison):
  * fp32 payload: max |gpu - oracle| <= 1e-5 on `out` (the bound stated for
    fp32 inputs); out_lse: |d| <= 1e-5 + 1e-6 |oracle|.
  * bf16 / fp16 payload: the stated bound, max |gpu - oracle| / max |oracle|
    <= 2e-2 over each compared tensor, AND a per-element bound derived from
    the arithmetic: one round-to-nearest into the output type (relative error
    <= 2^-9 for bf16, 2^-12 for fp16, doubled for margin) plus fp32
    accumulation error (<= 1e-5 absolute at these magnitudes):
        bf16: |d| <= 4e-3 |oracle| + 1e-5      fp16: |d| <= 5e-4 |oracle| + 1e-5
  * fp8 e4m3 payload: one round-to-nearest into e4m3 of the fp32 sum, so
    every element lies within half an e4m3 ulp of the oracle value (ulp =
    2^(floor(log2|x|) - 3) for |x| >= 2^-6, 2^-9 below), plus the fp32
    accumulation slack 1e-5 (1 + |oracle|).  The 2e-2 norm-wise bound stated
    for 16-bit payloads is not applied: one e4m3 rounding alone can reach
    2^-4 relative.
  * Non-finite oracle values (NaN, +-inf) must be matched exactly by class.
"""
from __future__ import annotations

import numpy as np
import torch

NP_PAYLOAD = {torch.float32: np.float32, torch.float16: np.float16, torch.bfloat16: np.uint16,
              torch.float8_e4m3fn: np.uint8}
ORACLE_DT = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16",
             torch.float8_e4m3fn: "fp8"}
ELEM_REL = {torch.float32: 0.0, torch.float16: 5e-4, torch.bfloat16: 4e-3}


def to_np(t: torch.Tensor) -> np.ndarray:
    """Contiguous host copy with the oracle's payload representation (bf16 as
    uint16, fp8 as uint8)."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def sentinel_like(shape, dtype, device, byte=0x5A) -> torch.Tensor:
    t = torch.empty(shape, dtype=dtype, device=device)
    t.view(torch.uint8).fill_(byte)
    return t


def np_sentinel(shape, np_dtype, byte=0x5A) -> np.ndarray:
    a = np.empty(shape, dtype=np_dtype)
    a.view(np.uint8)[...] = byte
    return a


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def _class_mask(want: np.ndarray, got: np.ndarray, what: str) -> np.ndarray:
    nan_w, nan_g = np.isnan(want), np.isnan(got)
    assert np.array_equal(nan_w, nan_g), f"{what}: NaN positions differ ({nan_w.sum()} vs {nan_g.sum()})"
    inf_w = np.isinf(want)
    assert np.array_equal(inf_w, np.isinf(got)), f"{what}: inf positions differ"
    assert np.array_equal(want[inf_w], got[inf_w]), f"{what}: inf signs differ"
    return ~(nan_w | inf_w)


def e4m3_ulp(a: np.ndarray) -> np.ndarray:
    """Spacing of e4m3 values around |a|: 2^(e - 3) in the binade [2^e, 2^(e+1)),
    2^-9 among the subnormals (|a| < 2^-6)."""
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    return np.exp2(e - 3)


def assert_merge_close(got: torch.Tensor, want: np.ndarray, what: str = "out") -> dict:
    """Compare a merged payload tensor with the oracle's fp64 result."""
    dt = got.dtype
    g = to_f64(got).reshape(want.shape)
    fin = _class_mask(want, g, what)
    d = np.abs(g[fin] - want[fin])
    w = np.abs(want[fin])
    stats = {"max_abs": float(d.max(initial=0.0)), "n": int(fin.sum())}
    if dt == torch.float32:
        assert stats["max_abs"] <= 1e-5, f"{what}: max abs error {stats['max_abs']:.3e} > 1e-5"
    elif dt == torch.float8_e4m3fn:
        bound = 0.5 * e4m3_ulp(w) + 1e-5 * (1.0 + w)
        bad = d > bound
        assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond half an e4m3 ulp, "
                               f"worst excess {float((d - bound).max()):.3e}")
    else:
        scale = max(float(w.max(initial=0.0)), 1e-30)
        stats["rel"] = stats["max_abs"] / scale
        assert stats["rel"] <= 2e-2, f"{what}: relative error {stats['rel']:.3e} > 2e-2"
        bound = ELEM_REL[dt] * w + 1e-5
        bad = d > bound
        assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond the rounding bound, "
                               f"worst excess {float((d - bound).max()):.3e}")
    return stats


def assert_lse_close(got: torch.Tensor, want: np.ndarray, what: str = "out_lse") -> float:
    g = to_f64(got).reshape(want.shape)
    fin = _class_mask(want, g, what)
    d = np.abs(g[fin] - want[fin])
    bad = d > 1e-5 + 1e-6 * np.abs(want[fin])
    assert not bad.any(), f"{what}: {int(bad.sum())} values beyond 1e-5 + 1e-6|G|, max {d.max():.3e}"
    return float(d.max(initial=0.0))


def assert_bytes_equal(got: torch.Tensor, want: np.ndarray, what: str) -> None:
    gb = got.detach().contiguous().cpu().view(torch.uint8).numpy().reshape(-1)
    wb = np.ascontiguousarray(want).view(np.uint8).reshape(-1)
    assert gb.size == wb.size, f"{what}: size {gb.size} vs {wb.size}"
    if not np.array_equal(gb, wb):
        bad = np.flatnonzero(gb != wb)
        raise AssertionError(f"{what}: {bad.size} bytes differ, first at byte {bad[0]}")
