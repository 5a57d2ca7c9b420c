"""Comparators between a device result and the oracle (test infrastructure only).

Tolerances are the workload's acceptance rules:
  - routing indices, the compacted index and the top-k selection: bit-exact;
  - a router swap between experts e, e' (across the top-k boundary or within the rank
    order) is allowed iff their oracle scores differ by less than 1e-5; the output is then
    compared with the oracle re-run on the device's choice;
  - routing weights: |dw| <= 1e-5 * max(1, |w|) (fp32 against fp64);
  - bf16 outputs: per element |dy| <= 2 bf16 ulp of y_ref, or |dy| <= 1e-2 |y_ref|;
    an element with |y_ref| < 1e-3 * rms(row) (cancellation near zero) that fails both is
    judged against 1e-2 * 1e-3 * rms(row) instead, and counted.
  - the intermediate bf16 activations h (the first of the two rounding points): every
    element equal to the oracle's or one bf16 ulp away (fp32 accumulation can land on the
    other side of a rounding midpoint than fp64), at most H_FLIP_BUDGET of them; y is then
    compared with the oracle's down projection and combine applied to the device's h, so
    that a legitimate flip of h is not counted against y.
"""
from __future__ import annotations

import numpy as np
import torch

TIE_GAP = 1e-5
H_FLIP_BUDGET = 0.01


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits).view(np.int16)
    return torch.from_numpy(b.copy()).view(torch.bfloat16).double().numpy()


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significant bits; subnormal spacing 2^-133)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    return np.ldexp(1.0, (e - 7).astype(int))


def y_report(y_dev_bits: np.ndarray, y_ref_bits: np.ndarray) -> dict:
    y = bf16_bits_to_f64(y_dev_bits)
    r = bf16_bits_to_f64(y_ref_bits)
    d = np.abs(y - r)
    ok = (d <= 2 * bf16_ulp(r)) | (d <= 1e-2 * np.abs(r))
    rms = np.sqrt(np.mean(r * r, axis=-1, keepdims=True))
    small = np.abs(r) < 1e-3 * rms
    rescued = ~ok & small & (d <= 1e-2 * 1e-3 * rms)
    fail = ~ok & ~rescued
    return {
        "n": int(y.size), "exact": int(np.sum(y_dev_bits == y_ref_bits)),
        "near_zero_rescued": int(np.sum(rescued)), "fail": int(np.sum(fail)),
        "max_abs": float(d.max()) if d.size else 0.0,
    }


def routing_report(idx_dev: np.ndarray, idx_ref: np.ndarray, s_ref: np.ndarray) -> dict:
    """Rows where the device's expert list differs from the oracle's; each difference must
    be a permitted near-tie (all swapped experts within TIE_GAP of the scores they replace)."""
    bad, swapped = [], []
    for r in range(idx_ref.shape[0]):
        a, b = idx_dev[r].tolist(), idx_ref[r].tolist()
        if a == b:
            continue
        swapped.append(r)
        ok = len(set(a)) == len(a)
        for j, (ea, eb) in enumerate(zip(a, b)):
            if ea != eb and abs(s_ref[r, ea] - s_ref[r, eb]) >= TIE_GAP:
                ok = False
        if not ok:
            bad.append(r)
    return {"rows_swapped": swapped, "rows_bad": bad}


def weights_ok(w_dev: np.ndarray, w_ref: np.ndarray) -> bool:
    return bool(np.all(np.abs(w_dev.astype(np.float64) - w_ref) <= 1e-5 * np.maximum(1.0, np.abs(w_ref))))


def h_report(h_dev_bits: np.ndarray, h_ref_bits: np.ndarray) -> dict:
    """Device h against the oracle's: exact, one bf16 ulp apart, or worse."""
    a = np.ascontiguousarray(h_dev_bits).view(np.uint16).astype(np.int64)
    b = np.ascontiguousarray(h_ref_bits).view(np.uint16).astype(np.int64)

    def ordered(v):  # bf16 bits -> integers in numeric order (adjacent values differ by 1)
        return np.where(v & 0x8000, -(v & 0x7FFF), v & 0x7FFF)

    d = np.abs(ordered(a) - ordered(b))
    n = int(d.size)
    return {"n": n, "exact": int(np.sum(d == 0)), "one_ulp": int(np.sum(d == 1)),
            "worse": int(np.sum(d > 1)), "ok": bool(np.all(d <= 1) and np.sum(d == 1) <= H_FLIP_BUDGET * n)}
