"""Python view of the plain C oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the benchmark's
CPU-baseline / reference leg, never by the library. It shares no code with the CUDA path
and imports nothing from it. Inputs are numpy arrays of raw bits (bf16/fp16 as uint16).

Parity pins: every function here is checked against something other than itself in
tests/test_oracle_pins.py (golden fixtures written by hand from the definitions, closed
forms, brute force on tiny inputs, library routines on special cases).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SRC = HERE / "oracle.c"
LIB = HERE / "liboracle.so"
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra"]


def build(force: bool = False) -> Path:
    if force or not LIB.exists() or LIB.stat().st_mtime < SRC.stat().st_mtime:
        cc = os.environ.get("CC", "gcc")
        subprocess.run([cc, *CFLAGS, str(SRC), "-o", str(LIB), "-lm"], check=True)
    return LIB


_lib = None


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(str(LIB))
        P = C.c_void_p
        L.orc_bf16_to_f64.argtypes = [C.c_uint16]; L.orc_bf16_to_f64.restype = C.c_double
        L.orc_f16_to_f64.argtypes = [C.c_uint16]; L.orc_f16_to_f64.restype = C.c_double
        L.orc_bf16_rne.argtypes = [C.c_double]; L.orc_bf16_rne.restype = C.c_uint16
        L.orc_q4_value.argtypes = [P, P, C.c_int64, C.c_int64, C.c_int64]
        L.orc_q4_value.restype = C.c_double
        L.orc_router.argtypes = [P, C.c_int32, C.c_int32, P, C.c_int32, C.c_int32, P, P, P]
        L.orc_router.restype = None
        L.orc_moe_forward.argtypes = [P, P, C.c_int32, P, P, P, P, P, P, P]
        L.orc_moe_forward.restype = None
        L.orc_moe_down_combine.argtypes = [P, C.c_int32, P, P, P, P, P]
        L.orc_bf16_rne_array.argtypes = [P, P, C.c_int64]
        L.orc_bf16_rne_array.restype = None
        L.orc_moe_down_combine.restype = None
        L.orc_block_score.argtypes = [P, P, P, C.c_int32, C.c_int32]
        L.orc_block_score.restype = C.c_float
        L.orc_select.argtypes = [C.c_int32] * 6 + [P, C.c_int64, P, P, P, P, C.c_int32,
                                                   C.c_int32, P, P, P, P, P]
        L.orc_select.restype = None
        L.orc_q8_value.argtypes = [P, P, C.c_int64, C.c_int64, C.c_int64]
        L.orc_q8_value.restype = C.c_double
        L.orc_q8_project.argtypes = [P, P, C.c_int64, C.c_int64, P, C.c_int32, P, P]
        L.orc_q8_project.restype = None
        L.orc_verify_greedy.argtypes = [P, C.c_int32, C.c_int32, P, P]
        L.orc_verify_greedy.restype = C.c_int32
        L.orc_verify_sample.argtypes = [P, C.c_int32, C.c_int32, C.c_double, P, P, P, P, P]
        L.orc_verify_sample.restype = C.c_int32
        L.orc_committed_tokens.argtypes = [P, C.c_int32]
        L.orc_committed_tokens.restype = C.c_int32
        L.orc_sparse_attention.argtypes = [P, P, P, C.c_int64, C.c_int32, C.c_int32, C.c_int32,
                                           P, C.c_int32, C.c_int32, P, P]
        L.orc_sparse_attention.restype = C.c_int32
        _lib = L
    return _lib


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


class _OrcMoeLayer(C.Structure):
    _fields_ = [("H", C.c_int32), ("E", C.c_int32), ("I", C.c_int32), ("k", C.c_int32)] + [
        (n, C.c_void_p) for n in (
            "router_w", "gate_qs", "gate_sc", "up_qs", "up_sc", "down_qs", "down_sc",
            "sg_qs", "sg_sc", "su_qs", "su_sc", "sd_qs", "sd_sc")]


# ------------------------------------------------------------------ scalar helpers --
def bf16_to_f64(b: int) -> float:
    return lib().orc_bf16_to_f64(int(b))


def f16_to_f64(h: int) -> float:
    return lib().orc_f16_to_f64(int(h))


def bf16_rne(v: float) -> int:
    return int(lib().orc_bf16_rne(float(v)))


def q4_value(qs: np.ndarray, sc: np.ndarray, K: int, row: int, k: int) -> float:
    qs = np.ascontiguousarray(qs, dtype=np.uint8)
    sc = _u16(sc)
    return lib().orc_q4_value(_p(qs), _p(sc), K, row, k)


# -------------------------------------------------------------------------- router --
def router(x: np.ndarray, wr: np.ndarray, k: int):
    """x bf16 bits [R,H], wr bf16 bits [E,H] -> idx int32 [R,k], w f64 [R,k], s f64 [R,E]."""
    x, wr = _u16(x), _u16(wr)
    R, H = x.shape
    E = wr.shape[0]
    idx = np.empty((R, k), np.int32)
    w = np.empty((R, k), np.float64)
    s = np.empty((R, E), np.float64)
    lib().orc_router(_p(x), R, H, _p(wr), E, k, _p(idx), _p(w), _p(s))
    return idx, w, s


# ----------------------------------------------------------------------- MoE layer --
def _layer_struct(layer: dict, k: int):
    keep = {}

    def arr(name, dtype):
        a = np.ascontiguousarray(layer[name])
        assert a.dtype == dtype, (name, a.dtype)
        keep[name] = a
        return a.ctypes.data

    E, H = layer["router_w"].shape
    I = layer["gate_qs"].shape[1]
    st = _OrcMoeLayer(H, E, I, k, arr("router_w", np.uint16),
                      arr("gate_qs", np.uint8), arr("gate_sc", np.uint16),
                      arr("up_qs", np.uint8), arr("up_sc", np.uint16),
                      arr("down_qs", np.uint8), arr("down_sc", np.uint16),
                      arr("sh_gate_qs", np.uint8), arr("sh_gate_sc", np.uint16),
                      arr("sh_up_qs", np.uint8), arr("sh_up_sc", np.uint16),
                      arr("sh_down_qs", np.uint8), arr("sh_down_sc", np.uint16))
    return st, keep, (H, E, I)


def moe_down_combine(layer: dict, k: int, idx: np.ndarray, w: np.ndarray, h: np.ndarray,
                     want_aux: bool = False):
    """y bf16 bits [R,H] from given activations h bf16 bits [R,1+k,I], experts idx [R,k]
    and weights w [R,k] (the layer's second half, fp64). With want_aux, also returns
    yaux [R,H,2] = (y before rounding, sum of the absolute values of its terms)."""
    st, keep, (H, E, I) = _layer_struct(layer, k)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float64)
    h = _u16(h)
    R = idx.shape[0]
    assert h.shape == (R, 1 + k, I)
    y = np.empty((R, H), np.uint16)
    yaux = np.empty((R, H, 2), np.float64) if want_aux else None
    lib().orc_moe_down_combine(C.byref(st), R, _p(idx), _p(w), _p(h), _p(y), _p(yaux))
    return (y, yaux) if want_aux else y


def bf16_rne_array(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().orc_bf16_rne_array(_p(v), _p(out), v.size)
    return out


def moe_forward(layer: dict, x: np.ndarray, k: int, idx_in: np.ndarray | None = None,
                want_h: bool = False):
    """layer: dict of numpy arrays (router_w, gate/up/down, sh_gate/sh_up/sh_down qs and sc,
    bf16/fp16 as uint16). x bf16 bits [R,H].
    Returns dict(y uint16 [R,H], idx, w, s, h uint16 [R,1+k,I] or None, aux f64
    [R,1+k,I,4] = (g, u, sum|g terms|, sum|u terms|) or None)."""
    keep = {}

    def arr(name, dtype):
        a = np.ascontiguousarray(layer[name])
        assert a.dtype == dtype, (name, a.dtype)
        keep[name] = a
        return a.ctypes.data

    E, H = layer["router_w"].shape
    I = layer["gate_qs"].shape[1]
    st = _OrcMoeLayer(H, E, I, k, arr("router_w", np.uint16),
                      arr("gate_qs", np.uint8), arr("gate_sc", np.uint16),
                      arr("up_qs", np.uint8), arr("up_sc", np.uint16),
                      arr("down_qs", np.uint8), arr("down_sc", np.uint16),
                      arr("sh_gate_qs", np.uint8), arr("sh_gate_sc", np.uint16),
                      arr("sh_up_qs", np.uint8), arr("sh_up_sc", np.uint16),
                      arr("sh_down_qs", np.uint8), arr("sh_down_sc", np.uint16))
    x = _u16(x)
    R = x.shape[0]
    y = np.empty((R, H), np.uint16)
    idx = np.empty((R, k), np.int32)
    w = np.empty((R, k), np.float64)
    s = np.empty((R, E), np.float64)
    h = np.empty((R, 1 + k, I), np.uint16) if want_h else None
    aux = np.empty((R, 1 + k, I, 4), np.float64) if want_h else None
    idx_in_a = None if idx_in is None else np.ascontiguousarray(idx_in, dtype=np.int32)
    lib().orc_moe_forward(C.byref(st), _p(x), R, _p(idx_in_a), _p(y), _p(idx), _p(w), _p(s), _p(h),
                          _p(aux))
    return {"y": y, "idx": idx, "w": w, "s": s, "h": h, "aux": aux}


# -------------------------------------------------------------------- block select --
def block_score(q: np.ndarray, key: np.ndarray, w: np.ndarray) -> float:
    """q bf16 bits [Hh,D], key bf16 bits [D], w f32 [Hh] -> canonical fp32 score."""
    q, key = _u16(q), _u16(key)
    w = np.ascontiguousarray(w, dtype=np.float32)
    Hh, D = q.shape
    return float(np.float32(lib().orc_block_score(_p(q), _p(key), _p(w), Hh, D)))


def select(keys: np.ndarray, q: np.ndarray, hw: np.ndarray, mask: np.ndarray, limit: np.ndarray,
           topk: int, layers=None):
    """keys bf16 bits [L,N,D]; q bf16 bits [L,R,Hh,D]; hw f32 [L,R,Hh]; mask uint32 [L,R,W];
    limit int32 [L,R]. layers: optional (l0, l1) range. Returns dict(sel, nsel, cidx,
    ccount, cscore) as full [L,R,...] arrays (rows outside the range undefined)."""
    keys, q = _u16(keys), _u16(q)
    hw = np.ascontiguousarray(hw, dtype=np.float32)
    mask = np.ascontiguousarray(mask).view(np.uint32)
    limit = np.ascontiguousarray(limit, dtype=np.int32)
    L, N, D = keys.shape
    R, Hh = q.shape[1], q.shape[2]
    l0, l1 = (0, L) if layers is None else layers
    sel = np.full((L, R, topk), -2, np.int32)
    nsel = np.full((L, R), -2, np.int32)
    cidx = np.full((L, R, N), -2, np.int32)
    ccount = np.full((L, R), -2, np.int32)
    cscore = np.zeros((L, R, N), np.float32)
    lib().orc_select(L, R, Hh, D, N, topk, _p(keys), N * D, _p(q), _p(hw), _p(mask), _p(limit),
                     l0, l1, _p(sel), _p(nsel), _p(cidx), _p(ccount), _p(cscore))
    return {"sel": sel, "nsel": nsel, "cidx": cidx, "ccount": ccount, "cscore": cscore}


def committed_tokens(accepted: np.ndarray, R: int) -> int:
    a = np.ascontiguousarray(accepted, dtype=np.uint8)
    return int(lib().orc_committed_tokens(_p(a), R))


def verify_greedy(logits: np.ndarray, draft: np.ndarray) -> np.ndarray:
    """Tokens emitted by one greedy verify step: logits fp32 [R][V], draft int32 [R-1]."""
    z = np.ascontiguousarray(logits, dtype=np.float32)
    R, V = z.shape
    d = np.ascontiguousarray(draft, dtype=np.int32).reshape(-1)
    assert d.size == R - 1
    out = np.zeros(R, dtype=np.int32)
    n = lib().orc_verify_greedy(_p(z), R, V, _p(d) if d.size else None, _p(out))
    return out[:n]


def verify_sample(logits: np.ndarray, T: float, qd: np.ndarray, draft: np.ndarray,
                  u_acc: np.ndarray, u_res: np.ndarray) -> np.ndarray:
    """Tokens emitted by one verify step with exact speculative sampling at temperature T:
    logits fp32 [R][V], qd fp64 [R-1][V] (the drafter's distributions), draft int32 [R-1],
    u_acc fp64 [R-1], u_res fp64 [R] (uniforms in [0, 1))."""
    if not (np.isfinite(T) and T > 0):
        raise ValueError(f"temperature must be finite and > 0 (got {T})")
    z = np.ascontiguousarray(logits, dtype=np.float32)
    R, V = z.shape
    q = np.ascontiguousarray(qd, dtype=np.float64).reshape(max(R - 1, 0), V)
    d = np.ascontiguousarray(draft, dtype=np.int32).reshape(-1)
    ua = np.ascontiguousarray(u_acc, dtype=np.float64).reshape(-1)
    ur = np.ascontiguousarray(u_res, dtype=np.float64).reshape(-1)
    assert d.size == R - 1 and ua.size == R - 1 and ur.size == R
    out = np.zeros(R, dtype=np.int32)
    n = lib().orc_verify_sample(_p(z), R, V, float(T), _p(q) if q.size else None,
                                _p(d) if d.size else None, _p(ua) if ua.size else None,
                                _p(ur), _p(out))
    if n < 0:
        raise ValueError(f"orc_verify_sample refused temperature {T}")
    return out[:n]


def q8_value(qs: np.ndarray, sc: np.ndarray, K: int, row: int, k: int) -> float:
    q = np.ascontiguousarray(qs, dtype=np.int8)
    s = _u16(sc)
    return float(lib().orc_q8_value(_p(q), _p(s), K, row, k))


def q8_project(qs: np.ndarray, sc: np.ndarray, x: np.ndarray):
    """R rows through one Q8 matrix: qs int8 [rows][K], sc fp16 bits [rows][K/32], x bf16
    bits [R][K] -> (y fp64 [R][rows], y rounded to bf16 bits [R][rows])."""
    q = np.ascontiguousarray(qs, dtype=np.int8)
    s = _u16(sc)
    xb = _u16(x)
    rows, K = q.shape
    R = xb.shape[0]
    y = np.zeros((R, rows), np.float64)
    yb = np.zeros((R, rows), np.uint16)
    lib().orc_q8_project(_p(q), _p(s), rows, K, _p(xb), R, _p(y), _p(yb))
    return y, yb


def sparse_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, sel: np.ndarray,
                     block: int = 4):
    """One layer: q bf16 bits [R][Hq][D], k and v bf16 bits [T][D], sel int32 [R][K]
    (selected block ids, -1 padded) -> (o fp64 [R][Hq][D], o bf16 bits [R][Hq][D])."""
    qb = _u16(q)
    kb = _u16(k)
    vb = _u16(v)
    s = np.ascontiguousarray(sel, dtype=np.int32)
    R, Hq, D = qb.shape
    T = kb.shape[0]
    assert kb.shape == (T, D) and vb.shape == (T, D) and s.shape[0] == R
    o = np.zeros((R, Hq, D), np.float64)
    ob = np.zeros((R, Hq, D), np.uint16)
    st = lib().orc_sparse_attention(_p(qb), _p(kb), _p(vb), T, D, R, Hq, _p(s), s.shape[1],
                                    block, _p(o), _p(ob))
    if st < 0:
        raise ValueError("a selected block lies outside the key range")
    return o, ob
