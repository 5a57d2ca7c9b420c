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
  - the intermediate bf16 activations h (the first of the two rounding points) and y
    near cancellation: the device accumulates in fp32 where the oracle uses fp64, so a
    result may round to a different bf16 neighbour. An element passes if it is the bf16
    rounding of some value within the fp32 accumulation band of the oracle's exact value:
    |g_dev - g| <= ACC_REL * sum|g terms| (same for u and y), propagated through
    silu(g) * u with silu's Lipschitz constant 1.1, plus the fp32 evaluation of silu and
    the product (FP32_EVAL relative). y is compared with the oracle's down projection and
    combine applied to the device's own h, so a legitimate difference in h is not counted
    against y.
"""
from __future__ import annotations

import numpy as np
import torch

TIE_GAP = 1e-5
H_FLIP_BUDGET = 0.01
ACC_REL = 2.0 ** -14       # fp32 accumulation over <= 16384 terms in ~150 sequential steps
FP32_EVAL = 2.0 ** -20     # expf, division and products of the fp32 epilogue


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


def _in_band(dev_bits: np.ndarray, lo: np.ndarray, hi: np.ndarray) -> np.ndarray:
    """True where the device's bf16 value lies between bf16_rne(lo) and bf16_rne(hi)."""
    import oracle
    v = bf16_bits_to_f64(dev_bits)
    vlo = bf16_bits_to_f64(oracle.bf16_rne_array(lo))
    vhi = bf16_bits_to_f64(oracle.bf16_rne_array(hi))
    return (v >= vlo) & (v <= vhi)


def h_band_report(h_dev_bits: np.ndarray, aux: np.ndarray) -> dict:
    """h from the device against the fp32 band around the oracle's exact silu(g) * u.
    aux [..., 4] = (g, u, sum|g terms|, sum|u terms|) from oracle.moe_forward."""
    g, u, ag, au = aux[..., 0], aux[..., 1], aux[..., 2], aux[..., 3]
    sig = 1.0 / (1.0 + np.exp(-g))
    silu = g * sig
    h = silu * u
    dg, du = ACC_REL * ag, ACC_REL * au
    B = 1.1 * dg * (np.abs(u) + du) + np.abs(silu) * du + FP32_EVAL * np.abs(h)
    ok = _in_band(h_dev_bits, h - B, h + B)
    return {"n": int(ok.size), "outside": int(np.sum(~ok)), "ok": bool(np.all(ok))}


def y_band_report(y_dev_bits: np.ndarray, y_ref_bits: np.ndarray, yaux: np.ndarray) -> dict:
    """y from the device against the oracle applied to the device's h: the stated tolerance
    (2 bf16 ulp or 1e-2 relative), or inside the fp32 accumulation band.
    yaux [..., 2] = (y before rounding, sum of the absolute values of its terms)."""
    rep = y_report(y_dev_bits, y_ref_bits)
    y = bf16_bits_to_f64(y_dev_bits)
    r = bf16_bits_to_f64(y_ref_bits)
    d = np.abs(y - r)
    tol_ok = (d <= 2 * bf16_ulp(r)) | (d <= 1e-2 * np.abs(r))
    yraw, ay = yaux[..., 0], yaux[..., 1]
    band_ok = _in_band(y_dev_bits, yraw - ACC_REL * ay, yraw + ACC_REL * ay)
    ok = tol_ok | band_ok
    rep.update({"band_only": int(np.sum(band_ok & ~tol_ok)), "outside": int(np.sum(~ok)),
                "ok": bool(np.all(ok))})
    return rep
