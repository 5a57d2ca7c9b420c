"""Comparators between a device result and the oracle (test infrastructure only).

Tolerances are the workload's acceptance rules:
  - routing indices, the compacted index and the top-k selection: bit-exact;
  - a router swap between experts e, e' (across the top-k boundary or within the rank
    order) is allowed iff their oracle scores differ by less than 1e-5; the output is then
    compared with the oracle re-run on the device's choice;
  - routing weights: |dw| <= 1e-5 * max(1, |w|) (fp32 against fp64);
  - bf16 outputs y: per element |dy| <= 2 bf16 ulp of y_ref, or |dy| <= 1e-2 |y_ref|;
    an element with |y_ref| < 1e-3 * rms(row) (cancellation near zero) that fails both is
    judged against 1e-2 * 1e-3 * rms(row) instead, and counted.

The layer has two bf16 rounding points (h = silu(g) * u, and y). The device forms g, u
and y in fp32, the oracle in fp64, so near a rounding boundary the two may round to
neighbouring bf16 values. Where floating point takes such a decision, the comparison
takes the device's decision and checks that it is a legitimate one:
  - h: each device value must be the bf16 rounding of some value inside the fp32
    accumulation band around the oracle's exact silu(g) * u (`h_band_report`);
  - y: the device's y must lie inside the band of the oracle applied, in fp64, to the
    device's own h and routing weights (`y_band_report`);
  - y against the full oracle (`y_full_report`): an element outside the stated tolerance
    is accepted only when its deviation is no larger than the deviation that the device's
    own (band-checked) h and w produce in exact arithmetic, plus the band and the two
    final roundings. Such elements are counted; the tests hold them to a budget.

The band (`accumulation_band`) is derived from how the kernels accumulate, not fitted:
products of a bf16 activation and a 4-bit weight are exact in fp32; each Q4 block (32
values) is two m16n8k16 tensor-core MMAs chained through the accumulator, whose internal
addition of 16 products plus the accumulator is taken as up to 17 truncating steps of
relative error 2^-23 each (no rounding mode is documented for it); the block's fp16 scale
is applied by one fp32 fma into a per-lane chain of `chain` blocks; `partials` such chain
results are then added one by one in a fixed order. First-order error analysis of that
evaluation gives |fp32 result - exact| <= u * sum|terms| with
    u = 2^-24 * (2 * 2 * 17 + chain + partials),
since no partial sum exceeds sum|terms|. For the verify layer (hidden 4096, intermediate
1024, top-8) this is about 2^-17.5 for g and u and 2^-17.2 for y (down projection and
combine), against the 2 bf16 ulp (2^-7 relative) of the output tolerance.
"""
from __future__ import annotations

import numpy as np
import torch

TIE_GAP = 1e-5
H_FLIP_BUDGET = 1e-3        # h elements that differ from the oracle's rounding (all in band)
Y_EXPLAINED_BUDGET = 1e-3   # y elements outside the tolerance, explained by h / w decisions
FP32_EVAL = 2.0 ** -20      # expf, division and products of the fp32 SwiGLU epilogue


def accumulation_band(chain: int, partials: int) -> float:
    """Relative bound (to sum|terms|) of an fp32 Q4 dot product evaluated as described in
    the module docstring: two chained MMAs per block, `chain` block-scale fmas in one
    lane's chain, `partials` chain results added in order."""
    return 2.0 ** -24 * (2 * 2 * 17 + chain + partials)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits).view(np.int16)
    return torch.from_numpy(b.copy()).view(torch.bfloat16).double().numpy()


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (8 significant bits; subnormal spacing 2^-133)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    return np.ldexp(1.0, (e - 7).astype(int))


def _tolerance_ok(y: np.ndarray, r: np.ndarray):
    """Per element: within 2 bf16 ulp or 1e-2 relative of r, or (|r| < 1e-3 rms of its
    row) within 1e-5 rms. Returns (ok, rescued-by-the-near-zero-clause)."""
    d = np.abs(y - r)
    ok = (d <= 2 * bf16_ulp(r)) | (d <= 1e-2 * np.abs(r))
    rms = np.sqrt(np.mean(r * r, axis=-1, keepdims=True))
    small = np.abs(r) < 1e-3 * rms
    rescued = ~ok & small & (d <= 1e-2 * 1e-3 * rms)
    return ok | rescued, rescued


def y_report(y_dev_bits: np.ndarray, y_ref_bits: np.ndarray) -> dict:
    y = bf16_bits_to_f64(y_dev_bits)
    r = bf16_bits_to_f64(y_ref_bits)
    ok, rescued = _tolerance_ok(y, r)
    d = np.abs(y - r)
    return {
        "n": int(y.size), "exact": int(np.sum(y_dev_bits == y_ref_bits)),
        "near_zero_rescued": int(np.sum(rescued)), "fail": int(np.sum(~ok)),
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
    """Device h against the oracle's: exact, one bf16 ulp apart, or further."""
    a = np.ascontiguousarray(h_dev_bits).view(np.uint16).astype(np.int64)
    b = np.ascontiguousarray(h_ref_bits).view(np.uint16).astype(np.int64)

    def ordered(v):  # bf16 bits -> integers in numeric order (adjacent values differ by 1)
        return np.where(v & 0x8000, -(v & 0x7FFF), v & 0x7FFF)

    d = np.abs(ordered(a) - ordered(b))
    n = int(d.size)
    return {"n": n, "exact": int(np.sum(d == 0)), "one_ulp": int(np.sum(d == 1)),
            "further": int(np.sum(d > 1)), "differ": int(np.sum(d > 0))}


def _in_band(dev_bits: np.ndarray, lo: np.ndarray, hi: np.ndarray) -> np.ndarray:
    """True where the device's bf16 value lies between bf16_rne(lo) and bf16_rne(hi)."""
    import oracle
    v = bf16_bits_to_f64(dev_bits)
    vlo = bf16_bits_to_f64(oracle.bf16_rne_array(lo))
    vhi = bf16_bits_to_f64(oracle.bf16_rne_array(hi))
    return (v >= vlo) & (v <= vhi)


def h_band_report(h_dev_bits: np.ndarray, aux: np.ndarray, rel: float) -> dict:
    """h from the device against the fp32 band around the oracle's exact silu(g) * u.
    aux [..., 4] = (g, u, sum|g terms|, sum|u terms|) from oracle.moe_forward; `rel` the
    accumulation band of g and u. The band of h propagates dg and du through silu(g) * u
    (|silu'| <= 1.1) and adds the fp32 evaluation of the epilogue."""
    g, u, ag, au = aux[..., 0], aux[..., 1], aux[..., 2], aux[..., 3]
    sig = 1.0 / (1.0 + np.exp(-g))
    silu = g * sig
    h = silu * u
    dg, du = rel * ag, rel * au
    B = 1.1 * dg * (np.abs(u) + du) + np.abs(silu) * du + FP32_EVAL * np.abs(h)
    ok = _in_band(h_dev_bits, h - B, h + B)
    return {"n": int(ok.size), "outside": int(np.sum(~ok)), "ok": bool(np.all(ok)),
            "band_rel": rel}


def y_band_report(y_dev_bits: np.ndarray, y_ref_bits: np.ndarray, yaux: np.ndarray,
                  rel: float) -> dict:
    """y from the device against the oracle applied, in fp64, to the device's own h and
    routing weights (y_ref_bits, yaux): the stated tolerance, or inside the fp32
    accumulation band `rel`. yaux [..., 2] = (y before rounding, sum of |its terms|).
    `band_only` counts elements that only the band accepts."""
    rep = y_report(y_dev_bits, y_ref_bits)
    y = bf16_bits_to_f64(y_dev_bits)
    r = bf16_bits_to_f64(y_ref_bits)
    tol_ok, _ = _tolerance_ok(y, r)
    yraw, ay = yaux[..., 0], yaux[..., 1]
    band_ok = _in_band(y_dev_bits, yraw - rel * ay, yraw + rel * ay)
    ok = tol_ok | band_ok
    rep.update({"band_only": int(np.sum(band_ok & ~tol_ok)), "outside": int(np.sum(~ok)),
                "ok": bool(np.all(ok)), "band_rel": rel})
    return rep


def y_full_report(y_dev_bits: np.ndarray, y_ref_bits: np.ndarray, yraw_dev: np.ndarray,
                  yraw_ref: np.ndarray, ay: np.ndarray, rel: float) -> dict:
    """y from the device against the full oracle y_ref. yraw_ref: the oracle's y before
    rounding; yraw_dev: the oracle's y before rounding from the device's h and w (both
    fp64); ay: sum of |terms| of y; rel: the accumulation band.
    An element outside the stated tolerance is `explained` when
        |y_dev - y_ref| <= |yraw_dev - yraw_ref| + rel * ay + ulp(y_dev)/2 + ulp(y_ref)/2,
    i.e. no larger than what the device's own rounding decisions in h and w, its fp32
    band and the two final roundings can produce; otherwise it fails."""
    y = bf16_bits_to_f64(y_dev_bits)
    r = bf16_bits_to_f64(y_ref_bits)
    tol_ok, rescued = _tolerance_ok(y, r)
    d = np.abs(y - r)
    allowed = np.abs(yraw_dev - yraw_ref) + rel * ay + 0.5 * bf16_ulp(y) + 0.5 * bf16_ulp(r)
    explained = ~tol_ok & (d <= allowed)
    fail = ~tol_ok & ~explained
    return {"n": int(y.size), "exact": int(np.sum(y_dev_bits == y_ref_bits)),
            "near_zero_rescued": int(np.sum(rescued)), "explained": int(np.sum(explained)),
            "fail": int(np.sum(fail)), "max_abs": float(d.max()) if d.size else 0.0}


def kernel_bands(H: int, I: int, k: int) -> tuple[float, float]:
    """Accumulation bands of the library's Q4 kernels for a layer of hidden H,
    intermediate I and top-k (relative to sum|terms|): (g and u, y).
    Gate/up: K = H is cut into chunks of 32 tiles (2 per consumer warp) or, when the larger
    stages do not fit, of 16 tiles (1 per warp), tiles of two blocks; a lane's chain holds
    its blocks of every chunk, and the 16 consumer warps' chains are added in warp order.
    Down: one warp owns a 16-row tile row for all of K = I in two chains (even and odd
    tiles, two blocks each), added once; the combine adds the k weighted expert outputs to
    the shared one by k fmas in rank order."""
    T_h, T_i = H // 64, I // 64
    chain_gu = min(2 * T_h, max(4 * -(-T_h // 32), 2 * -(-T_h // 16)))
    chain_dn = 2 * -(-T_i // 2)
    return accumulation_band(chain_gu, 16), accumulation_band(chain_dn, 2) + 2.0 ** -24 * k


def moe_check(host: dict, x_bits: np.ndarray, k: int, y_dev: np.ndarray, idx_dev: np.ndarray,
              w_dev: np.ndarray, h_dev: np.ndarray) -> dict:
    """Every check of one device MoE call against the oracle. host: the layer as numpy
    arrays of raw bits; x_bits bf16 bits [R,H]; device results y (bf16 bits), topk_idx,
    topk_w, and h (bf16 bits [R,1+k,I], read from the workspace). Returns a report; the
    caller asserts report["ok"] (the report says which check failed otherwise)."""
    import oracle
    H, I = x_bits.shape[1], host["gate_qs"].shape[1]
    rel_gu, rel_y = kernel_bands(H, I, k)
    ref = oracle.moe_forward(host, x_bits, k, want_h=True)
    rep = {"routing": routing_report(idx_dev, ref["idx"], ref["s"])}
    if rep["routing"]["rows_swapped"]:
        ref = oracle.moe_forward(host, x_bits, k, idx_in=idx_dev, want_h=True)
    rep["weights_ok"] = weights_ok(w_dev, ref["w"])
    rep["h_band"] = h_band_report(h_dev, ref["aux"], rel_gu)
    rep["h"] = h_report(h_dev, ref["h"])
    # the second half of the layer in fp64 from the device's own h and w, and from the
    # oracle's (whose rounding must give the oracle's y)
    wd = w_dev.astype(np.float64)
    y_dh, yaux_dev = oracle.moe_down_combine(host, k, ref["idx"], wd, h_dev, want_aux=True)
    y_rh, yaux_ref = oracle.moe_down_combine(host, k, ref["idx"], ref["w"], ref["h"], want_aux=True)
    rep["oracle_consistent"] = bool(np.array_equal(y_rh, ref["y"]))
    rep["y_vs_device_h"] = y_band_report(y_dev, y_dh, yaux_dev, rel_y)
    rep["y_vs_oracle"] = y_full_report(y_dev, ref["y"], yaux_dev[..., 0], yaux_ref[..., 0],
                                       yaux_dev[..., 1], rel_y)
    n_h, n_y = rep["h"]["n"], rep["y_vs_oracle"]["n"]
    rep["ok"] = bool(
        not rep["routing"]["rows_bad"] and rep["weights_ok"] and rep["oracle_consistent"]
        and rep["h_band"]["ok"] and rep["h"]["differ"] <= H_FLIP_BUDGET * n_h
        and rep["y_vs_device_h"]["ok"] and rep["y_vs_device_h"]["band_only"] <= Y_EXPLAINED_BUDGET * n_y
        and rep["y_vs_oracle"]["fail"] == 0
        and rep["y_vs_oracle"]["explained"] <= Y_EXPLAINED_BUDGET * n_y)
    return rep
