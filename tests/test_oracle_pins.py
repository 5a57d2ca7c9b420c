"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each pin would fail under a plausible mistake in the oracle: a wrong nibble order or sign
offset (Q4 golden blocks, one-hot columns), a double rounding or wrong tie rule (bf16
golden cases, torch's converter), a transposed operand or dropped term (dequantise-then-
numpy-matmul layer check), a wrong selection order or tie-break (full sorts, all-equal
scores), a wrong summation order in the block score (hand-worked fp32 cases), a wrong
byte order or sign in Q8 values (hand-worked blocks, one-hot columns), a wrong
acceptance rule or residual in the verify step (the acceptance probability min(1, p/q) and
the first emitted token's distribution equal to the target's, both in closed form over a
stratified grid of the uniforms; the inverse CDF against scipy's softmax; the greedy limit).
"""
import json
import math

import numpy as np
import pytest
import torch

import oracle
import synth

# ------------------------------------------------------------------- helpers (tests) --


def np_dequant(qs: np.ndarray, sc: np.ndarray) -> np.ndarray:
    """Independent numpy dequantisation of a Q4 matrix: [..., rows, K/2] bytes and fp16-bit
    scales [..., rows, K/32] -> fp64 [..., rows, K]."""
    lo = (qs & 15).astype(np.int64) - 8
    hi = (qs >> 4).astype(np.int64) - 8
    q = np.stack([lo, hi], axis=-1).reshape(qs.shape[:-1] + (qs.shape[-1] * 2,))
    s = sc.view(np.float16).astype(np.float64)
    return q.astype(np.float64) * np.repeat(s, 32, axis=-1)


def bf16_to_np(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()


def layer_numpy(d: dict) -> dict:
    out = {}
    for k, v in d.items():
        v = v.contiguous()
        if v.dtype in (torch.bfloat16, torch.float16):
            out[k] = v.view(torch.int16).numpy().view(np.uint16)
        else:
            out[k] = v.numpy()
    return out


# ------------------------------------------------------------------- number formats --


def test_f16_decode_matches_numpy_all_patterns():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = h.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in h])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_bf16_decode_matches_torch():
    b = np.arange(0, 65536, 97, dtype=np.uint32).astype(np.uint16)
    ref = bf16_to_np(b)
    got = np.array([oracle.bf16_to_f64(int(x)) for x in b])
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_bf16_rne_golden(golden_dir):
    d = json.loads((golden_dir / "bf16_rne.json").read_text())
    for c in d["cases"]:
        assert oracle.bf16_rne(c["value"]) == int(c["bits"], 16), c


def test_bf16_rne_matches_torch_on_fp32_values():
    # torch rounds fp32 -> bf16 to nearest even; on fp32 inputs there is no double rounding.
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(4000), rng.standard_normal(2000) * 1e-38,
                        rng.standard_normal(2000) * 1e30]).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_rne(float(x)) for x in v], dtype=np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------------- Q4 format ----


def test_q4_golden_blocks(golden_dir):
    d = json.loads((golden_dir / "q4_block.json").read_text())
    for blk in d["blocks"]:
        qs = np.frombuffer(bytes.fromhex(blk["bytes_hex"]), dtype=np.uint8).reshape(1, 16)
        sc = np.array([[int(blk["scale_f16_hex"], 16)]], dtype=np.uint16)
        for k in range(32):
            assert oracle.q4_value(qs, sc, 32, 0, k) == blk["scale"] * blk["q"][k]
        # the numpy helper used by the other pins agrees with the hand-worked values too
        assert np.array_equal(np_dequant(qs, sc)[0], blk["scale"] * np.array(blk["q"]))


# ---------------------------------------------------------------------- Q8 weights ----


def np_dequant_q8(qs: np.ndarray, sc: np.ndarray) -> np.ndarray:
    """Independent numpy dequantisation of a Q8 matrix: int8 [rows, K] and fp16-bit scales
    [rows, K/32] -> fp64 [rows, K]."""
    s = sc.view(np.float16).astype(np.float64)
    return qs.astype(np.float64) * np.repeat(s, 32, axis=-1)


def test_q8_golden_blocks(golden_dir):
    d = json.loads((golden_dir / "q8_block.json").read_text())
    for blk in d["blocks"]:
        qs = np.frombuffer(bytes.fromhex(blk["bytes_hex"]), dtype=np.int8).reshape(1, 32)
        sc = np.array([[int(blk["scale_f16_hex"], 16)]], dtype=np.uint16)
        for k in range(32):
            assert oracle.q8_value(qs, sc, 32, 0, k) == blk["scale"] * blk["q"][k]
        assert np.array_equal(np_dequant_q8(qs, sc)[0], blk["scale"] * np.array(blk["q"]))


def _q8_case(rows, K, R, seed):
    rng = np.random.default_rng(seed)
    qs = rng.integers(-128, 128, size=(rows, K), dtype=np.int64).astype(np.int8)
    sc = (rng.uniform(0.5, 2.0, size=(rows, K // 32)) * 2.0 ** -7).astype(np.float16).view(np.uint16)
    x = torch.randn(R, K).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return qs, sc, x


def test_q8_project_onehot_gives_the_column():
    qs, sc, _ = _q8_case(40, 96, 1, seed=5)
    W = np_dequant_q8(qs, sc)
    for k in (0, 31, 32, 95):
        x = np.zeros((1, 96), np.uint16)
        x[0, k] = 0x3F80   # bf16 1.0
        y, _ = oracle.q8_project(qs, sc, x)
        assert np.array_equal(y[0], W[:, k])


def test_q8_project_against_numpy_and_row_pairing():
    qs, sc, x = _q8_case(72, 256, 6, seed=6)
    y, yb = oracle.q8_project(qs, sc, x)
    ref = bf16_to_np(x) @ np_dequant_q8(qs, sc).T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    # one bf16 rounding of the fp64 value (torch's converter rounds to nearest even)
    want = torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(yb, want)
    # the rows share the weights but not their results: each row alone gives the same
    for r in range(6):
        y1, yb1 = oracle.q8_project(qs, sc, x[r:r + 1])
        assert np.array_equal(y1[0], y[r]) and np.array_equal(yb1[0], yb[r])


# ------------------------------------------------------------------------- router ----


def test_router_onehot_closed_form():
    # x = e_i gives z_e = Wr[e, i] exactly; top-2 of column i.
    E, H, k = 4, 32, 2
    wr = np.zeros((E, H), np.float32)
    wr[:, 5] = [0.5, -1.0, 2.0, 0.25]
    x = np.zeros((1, H), np.float32)
    x[0, 5] = 1.0
    to_bits = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    idx, w, s = oracle.router(to_bits(x), to_bits(wr), k)
    assert idx.tolist() == [[2, 0]]
    sig = lambda z: 1.0 / (1.0 + math.exp(-z))
    assert s[0].tolist() == pytest.approx([sig(0.5), sig(-1.0), sig(2.0), sig(0.25)], abs=1e-15)
    tot = sig(2.0) + sig(0.5)
    assert w[0].tolist() == pytest.approx([sig(2.0) / tot, sig(0.5) / tot], abs=1e-15)


def test_router_all_equal_scores_take_lowest_indices():
    E, H, k = 16, 64, 5
    x = synth.to_numpy_bits(synth.activations(3, H, seed=4))
    wr = np.zeros((E, H), np.uint16)
    idx, w, _ = oracle.router(x, wr, k)
    assert idx.tolist() == [list(range(k))] * 3
    assert np.all(w == 1.0 / k)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_router_full_sort_and_library_matmul(seed):
    shape = synth.TINY_MOE
    d = layer_numpy(synth.moe_layer(shape, seed=seed))
    x = synth.to_numpy_bits(synth.activations(4, shape.H, seed=seed))
    idx, w, s = oracle.router(x, d["router_w"], shape.k)
    z = bf16_to_np(x) @ bf16_to_np(d["router_w"]).T          # library matmul, fp64
    ref_s = 1.0 / (1.0 + np.exp(-z))
    assert np.allclose(s, ref_s, rtol=0, atol=1e-14)
    for r in range(x.shape[0]):
        order = np.lexsort((np.arange(shape.E), -s[r]))    # full sort: score desc, index asc
        assert idx[r].tolist() == order[: shape.k].tolist()
        assert len(set(idx[r].tolist())) == shape.k
        assert w[r].sum() == pytest.approx(1.0, abs=1e-12)
        assert np.allclose(w[r], s[r, idx[r]] / s[r, idx[r]].sum(), rtol=1e-15)
        # monotone: the same experts rank first by logit
        assert set(np.argsort(-z[r], kind="stable")[: shape.k].tolist()) == set(idx[r].tolist())


def test_router_brute_force_subsets():
    # Among all k-subsets, the oracle's choice has the largest score sum.
    import itertools
    E, H, k = 7, 32, 3
    d = layer_numpy(synth.moe_layer(synth.MoeShape(H=H, E=E, I=32, k=k), seed=11))
    x = synth.to_numpy_bits(synth.activations(2, H, seed=11))
    idx, _, s = oracle.router(x, d["router_w"], k)
    for r in range(2):
        best = max(itertools.combinations(range(E), k), key=lambda c: sum(s[r, list(c)]))
        assert sorted(best) == sorted(idx[r].tolist())


# ------------------------------------------------------------------ expert / layer ----


def _onehot_layer(H=64, E=4, I=32, k=2, seed=3):
    d = layer_numpy(synth.moe_layer(synth.MoeShape(H=H, E=E, I=I, k=k), seed=seed))
    return d, H, E, I, k


def test_expert_onehot_input_gives_dequantised_column():
    d, H, E, I, k = _onehot_layer()
    col = 37
    x = np.zeros((1, H), np.uint16)
    x[0, col] = 0x3F80  # 1.0
    out = oracle.moe_forward(d, x, k, want_h=True)
    g = np_dequant(d["sh_gate_qs"], d["sh_gate_sc"])[:, col]
    u = np_dequant(d["sh_up_qs"], d["sh_up_sc"])[:, col]
    want = [oracle.bf16_rne(gi / (1.0 + math.exp(-gi)) * ui) for gi, ui in zip(g, u)]
    assert out["h"][0, 0].tolist() == want
    for j in range(k):
        e = out["idx"][0, j]
        g = np_dequant(d["gate_qs"][e], d["gate_sc"][e])[:, col]
        u = np_dequant(d["up_qs"][e], d["up_sc"][e])[:, col]
        want = [oracle.bf16_rne(gi / (1.0 + math.exp(-gi)) * ui) for gi, ui in zip(g, u)]
        assert out["h"][0, 1 + j].tolist() == want


def test_expert_all_ones_weights_sum_inputs():
    # q = 1 everywhere (nibble 9, bytes 0x99), scale 1: g = u = sum(x) for every output row.
    d, H, E, I, k = _onehot_layer()
    for nm in ("sh_gate", "sh_up"):
        d[nm + "_qs"] = np.full_like(d[nm + "_qs"], 0x99)
        d[nm + "_sc"] = np.full_like(d[nm + "_sc"], 0x3C00)  # fp16 1.0
    x = synth.to_numpy_bits(synth.activations(1, H, seed=8))
    out = oracle.moe_forward(d, x, k, want_h=True)
    sx = math.fsum(bf16_to_np(x)[0])
    want = oracle.bf16_rne(sx / (1.0 + math.exp(-sx)) * sx)
    assert np.all(out["h"][0, 0] == want)


@pytest.mark.parametrize("seed,R", [(0, 1), (1, 3)])
def test_layer_matches_dequantise_then_numpy_matmul(seed, R):
    shape = synth.TINY_MOE
    d = layer_numpy(synth.moe_layer(shape, seed=seed))
    x = synth.to_numpy_bits(synth.activations(R, shape.H, seed=seed))
    out = oracle.moe_forward(d, x, shape.k, want_h=True)
    xf = bf16_to_np(x)
    z = xf @ bf16_to_np(d["router_w"]).T
    s = 1.0 / (1.0 + np.exp(-z))

    def expert(gq, gs, uq, us, dq, dsc, xr):
        g = np_dequant(gq, gs) @ xr
        u = np_dequant(uq, us) @ xr
        hv = g / (1.0 + np.exp(-g)) * u
        hb = torch.from_numpy(hv.astype(np.float32)).to(torch.bfloat16).double().numpy()
        return hb, np_dequant(dq, dsc) @ hb

    for r in range(R):
        order = np.lexsort((np.arange(shape.E), -s[r]))[: shape.k]
        wts = s[r, order] / s[r, order].sum()
        hsh, acc = expert(d["sh_gate_qs"], d["sh_gate_sc"], d["sh_up_qs"], d["sh_up_sc"],
                          d["sh_down_qs"], d["sh_down_sc"], xf[r])
        hs = [hsh]
        for j, e in enumerate(order):
            he, o = expert(d["gate_qs"][e], d["gate_sc"][e], d["up_qs"][e], d["up_sc"][e],
                           d["down_qs"][e], d["down_sc"][e], xf[r])
            hs.append(he)
            acc = acc + wts[j] * o
        assert out["idx"][r].tolist() == order.tolist()
        # h: the reference rounds through fp32, so allow one bf16 ulp on rare ties
        got_h = bf16_to_np(out["h"][r])
        want_h = np.stack(hs)
        ulp = np.abs(want_h) * 2.0 ** -7 + 1e-30
        assert np.all(np.abs(got_h - want_h) <= ulp)
        assert np.mean(got_h == want_h) > 0.999
        got_y = bf16_to_np(out["y"][r])
        ulp_y = np.maximum(np.abs(acc) * 2.0 ** -7, 1e-6)
        assert np.all(np.abs(got_y - acc) <= 2 * ulp_y)


def test_down_combine_from_own_h_reproduces_y():
    shape = synth.TINY_MOE
    d = layer_numpy(synth.moe_layer(shape, seed=7))
    x = synth.to_numpy_bits(synth.activations(3, shape.H, seed=7))
    out = oracle.moe_forward(d, x, shape.k, want_h=True)
    y = oracle.moe_down_combine(d, shape.k, out["idx"], out["w"], out["h"])
    assert np.array_equal(y, out["y"])
    # and it is linear in h: zero activations give zero output
    assert np.all(oracle.moe_down_combine(d, shape.k, out["idx"], out["w"],
                                          np.zeros_like(out["h"])) == 0)


def test_band_checks_accept_exact_and_reject_perturbed():
    from oracle import compare
    shape = synth.TINY_MOE
    d = layer_numpy(synth.moe_layer(shape, seed=8))
    x = synth.to_numpy_bits(synth.activations(2, shape.H, seed=8))
    out = oracle.moe_forward(d, x, shape.k, want_h=True)
    rel_gu, rel_y = compare.kernel_bands(shape.H, shape.I, shape.k)
    assert compare.h_band_report(out["h"], out["aux"], rel_gu)["ok"]
    bad = out["h"].copy()
    bad.reshape(-1)[::97] ^= 0x0040          # flip a mantissa bit in ~1% of elements
    assert not compare.h_band_report(bad, out["aux"], rel_gu)["ok"]
    y, yaux = oracle.moe_down_combine(d, shape.k, out["idx"], out["w"], out["h"], want_aux=True)
    assert compare.y_band_report(y, y, yaux, rel_y)["ok"]
    ybad = y.copy()
    ybad.reshape(-1)[::50] ^= 0x0100          # perturb ~2% of the outputs by 2^-5 or more
    assert not compare.y_band_report(ybad, y, yaux, rel_y)["ok"]


def _moe_numpy_case(seed=9, R=3):
    shape = synth.TINY_MOE
    d = layer_numpy(synth.moe_layer(shape, seed=seed))
    x = synth.to_numpy_bits(synth.activations(R, shape.H, seed=seed))
    out = oracle.moe_forward(d, x, shape.k, want_h=True)
    return shape, d, x, out


def test_moe_check_accepts_the_oracle_itself():
    from oracle import compare
    shape, d, x, out = _moe_numpy_case()
    rep = compare.moe_check(d, x, shape.k, out["y"], out["idx"], out["w"].astype(np.float32),
                            out["h"])
    assert rep["ok"], rep
    assert rep["y_vs_oracle"]["exact"] == rep["y_vs_oracle"]["n"]


def test_moe_check_rejects_planted_mistakes():
    # Mistakes planted in copies of the oracle's own results (on the CPU): each must be
    # caught by the check that covers it.
    from oracle import compare
    shape, d, x, out = _moe_numpy_case()
    w32 = out["w"].astype(np.float32)
    # an h value moved far outside its band
    h_bad = out["h"].copy()
    h_bad[1, 0, 5] ^= 0x0200
    rep = compare.moe_check(d, x, shape.k, out["y"], out["idx"], w32, h_bad)
    assert not rep["h_band"]["ok"] and not rep["ok"]
    # a y value off by a quarter of its magnitude: outside the tolerance, not explained
    y_bad = out["y"].copy()
    y_bad[2, 7] ^= 0x0020
    rep = compare.moe_check(d, x, shape.k, y_bad, out["idx"], w32, out["h"])
    assert rep["y_vs_oracle"]["fail"] >= 1 and not rep["ok"]
    # swapped expert order in one row (not a near-tie)
    idx_bad = out["idx"].copy()
    idx_bad[0, [0, 1]] = idx_bad[0, [1, 0]]
    rep = compare.moe_check(d, x, shape.k, out["y"], idx_bad, w32, out["h"])
    assert rep["routing"]["rows_bad"] == [0] and not rep["ok"]
    # routing weights off by 1e-4
    rep = compare.moe_check(d, x, shape.k, out["y"], out["idx"], w32 + np.float32(1e-4), out["h"])
    assert not rep["weights_ok"] and not rep["ok"]


def test_accumulation_band_matches_its_derivation():
    from oracle import compare
    # 2 MMAs x 17 truncating steps of 2^-23, plus one rounding per chained block and per
    # added partial, each 2^-24
    assert compare.accumulation_band(0, 0) == 34 * 2.0 ** -23
    assert compare.accumulation_band(8, 16) == (68 + 24) * 2.0 ** -24
    rel_gu, rel_y = compare.kernel_bands(4096, 1024, 8)
    assert 2.0 ** -18 < rel_gu < 2.0 ** -17 and 2.0 ** -18 < rel_y < 2.0 ** -17


def test_layer_rows_independent():
    shape = synth.TINY_MOE
    d = layer_numpy(synth.moe_layer(shape, seed=5))
    x = synth.to_numpy_bits(synth.activations(3, shape.H, seed=5))
    full = oracle.moe_forward(d, x, shape.k)
    for r in range(3):
        one = oracle.moe_forward(d, x[r:r + 1], shape.k)
        assert np.array_equal(one["y"][0], full["y"][r])
        assert np.array_equal(one["idx"][0], full["idx"][r])


def test_layer_idx_override_reweights_from_scores():
    shape = synth.TINY_MOE
    d = layer_numpy(synth.moe_layer(shape, seed=6))
    x = synth.to_numpy_bits(synth.activations(1, shape.H, seed=6))
    base = oracle.moe_forward(d, x, shape.k)
    swapped = base["idx"][:, ::-1].copy()
    alt = oracle.moe_forward(d, x, shape.k, idx_in=swapped)
    assert alt["idx"].tolist() == swapped.tolist()
    assert np.allclose(alt["w"], base["w"][:, ::-1], rtol=1e-15)


# ---------------------------------------------------------------------- block select --


def _bf16_bits(vals) -> np.ndarray:
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_block_score_golden_order(golden_dir):
    d = json.loads((golden_dir / "canonical_score.json").read_text())
    for c in d["cases"]:
        Hh = len(c["heads"])
        q = np.zeros((Hh, 128), np.float32)
        for h, vals in enumerate(c["heads"]):
            q[h, : len(vals)] = vals
        key = np.zeros(128, np.float32)
        key[: len(c["key"])] = c["key"]
        got = oracle.block_score(_bf16_bits(q), _bf16_bits(key), np.array(c["w"], np.float32))
        assert got == c["score"], c["name"]


def test_block_score_integer_inputs_exact():
    # small integers: every product and partial sum is exact in fp32, so the canonical
    # score equals the exact integer value.
    rng = np.random.default_rng(7)
    for _ in range(50):
        Hh = int(rng.integers(1, 9))
        q = rng.integers(-4, 5, (Hh, 128))
        k = rng.integers(-4, 5, 128)
        w = rng.integers(-3, 4, Hh)
        exact = int(sum(int(w[h]) * max(0, int(q[h] @ k)) for h in range(Hh)))
        got = oracle.block_score(_bf16_bits(q.astype(np.float32)), _bf16_bits(k.astype(np.float32)),
                                 w.astype(np.float32))
        assert got == exact


def _unpack(mask: np.ndarray, N: int) -> np.ndarray:
    by = mask.astype("<u4").view(np.uint8)
    return np.unpackbits(by.reshape(mask.shape[:-1] + (-1,)), axis=-1, bitorder="little")[..., :N].astype(bool)


@pytest.mark.parametrize("shared", [True, False])
def test_select_compaction_and_full_sort(shared):
    shape = synth.SelectShape(L=2, R=3, Hh=4, N=333, topk=40)
    inp = synth.select_inputs(shape, seed=2, shared_mask=shared)
    keys, q = synth.to_numpy_bits(inp["keys"]), synth.to_numpy_bits(inp["q"])
    hw, mask, limit = inp["head_w"].numpy(), inp["mask"].numpy().view(np.uint32), inp["limit"].numpy()
    out = oracle.select(keys, q, hw, mask, limit, shape.topk)
    bits = _unpack(mask, shape.N)
    for l in range(shape.L):
        for r in range(shape.R):
            adm = np.flatnonzero(bits[l, r] & (np.arange(shape.N) < limit[l, r]))
            n = out["ccount"][l, r]
            assert n == len(adm)
            assert out["cidx"][l, r, :n].tolist() == adm.tolist()
            sc = out["cscore"][l, r, :n]
            for j in (0, n // 2, n - 1):
                assert sc[j] == oracle.block_score(q[l, r], keys[l, adm[j]], hw[l, r])
            order = np.lexsort((adm, -sc.astype(np.float64)))[: shape.topk]
            want = np.sort(adm[order])
            m = min(shape.topk, n)
            assert out["nsel"][l, r] == m
            assert out["sel"][l, r, :m].tolist() == want.tolist()
            assert np.all(out["sel"][l, r, m:] == -1)


def test_select_fp64_sanity():
    # every selected block scores (in fp64) at least as high as every unselected one,
    # up to the fp32 rounding of the canonical order.
    shape = synth.SelectShape(L=1, R=2, Hh=8, N=2048, topk=512)
    inp = synth.select_inputs(shape, seed=9)
    keys, q = synth.to_numpy_bits(inp["keys"]), synth.to_numpy_bits(inp["q"])
    hw, mask, limit = inp["head_w"].numpy(), inp["mask"].numpy().view(np.uint32), inp["limit"].numpy()
    out = oracle.select(keys, q, hw, mask, limit, shape.topk)
    kf, qf = bf16_to_np(keys), bf16_to_np(q)
    for r in range(shape.R):
        n = out["ccount"][0, r]
        adm = out["cidx"][0, r, :n]
        d = np.einsum("hd,nd->nh", qf[0, r], kf[0, adm])
        s64 = np.maximum(d, 0.0) @ hw[0, r].astype(np.float64)
        scale = np.abs(hw[0, r]).sum() * np.abs(d).max()
        chosen = np.isin(adm, out["sel"][0, r])
        assert s64[chosen].min() >= s64[~chosen].max() - 1e-5 * scale


def test_select_ties_take_lowest_indices():
    # identical keys: every admitted block has the same score -> the lowest admitted ones.
    shape = synth.SelectShape(L=1, R=2, Hh=2, N=200, topk=16)
    inp = synth.select_inputs(shape, seed=1)
    keys = np.tile(synth.to_numpy_bits(inp["keys"])[:, :1, :], (1, shape.N, 1))
    q = synth.to_numpy_bits(inp["q"])
    hw, mask, limit = inp["head_w"].numpy(), inp["mask"].numpy().view(np.uint32), inp["limit"].numpy()
    out = oracle.select(keys, q, hw, mask, limit, shape.topk)
    for r in range(shape.R):
        assert out["sel"][0, r].tolist() == out["cidx"][0, r, : shape.topk].tolist()


def test_select_fewer_admitted_than_k_pads():
    shape = synth.SelectShape(L=1, R=1, Hh=1, N=64, topk=8)
    inp = synth.select_inputs(shape, seed=0)
    keys, q = synth.to_numpy_bits(inp["keys"]), synth.to_numpy_bits(inp["q"])
    hw, limit = inp["head_w"].numpy(), inp["limit"].numpy()
    mask = np.zeros((1, 1, 2), np.uint32)
    mask[0, 0, 0] = (1 << 3) | (1 << 17) | (1 << 30)
    out = oracle.select(keys, q, hw, mask, limit, shape.topk)
    assert out["sel"][0, 0].tolist() == [3, 17, 30, -1, -1, -1, -1, -1]
    assert out["nsel"][0, 0] == 3


def test_select_single_head_is_partial_sort_of_relu_dot():
    # tiny workload: one head, w = 1: score = relu(q . k) (about half exactly 0) and the
    # selection is a textbook partial sort with the lower index first among equals.
    shape = synth.TINY_SELECT
    inp = synth.select_inputs(shape, seed=0)
    keys, q = synth.to_numpy_bits(inp["keys"]), synth.to_numpy_bits(inp["q"])
    hw = np.ones((1, 1, 1), np.float32)
    mask, limit = inp["mask"].numpy().view(np.uint32), inp["limit"].numpy()
    out = oracle.select(keys, q, hw, mask, limit, shape.topk)
    bits = _unpack(mask, shape.N)[0, 0] & (np.arange(shape.N) < limit[0, 0])
    adm = np.flatnonzero(bits)
    dots = (bf16_to_np(keys)[0, adm] @ bf16_to_np(q)[0, 0, 0]).astype(np.float64)
    sc = out["cscore"][0, 0, : len(adm)]
    assert np.allclose(sc, np.maximum(dots, 0), rtol=1e-5, atol=1e-4)
    assert np.sum(sc == 0) > 0
    pairs = sorted(zip((-sc).tolist(), adm.tolist()))[: shape.topk]
    assert out["sel"][0, 0].tolist() == sorted(b for _, b in pairs)


# ------------------------------------------------------------- speculative bookkeeping --


def test_committed_tokens_small_cases():
    assert oracle.committed_tokens(np.array([1, 1, 0, 1, 1], np.uint8), 6) == 3
    assert oracle.committed_tokens(np.array([0, 1, 1, 1, 1], np.uint8), 6) == 1
    assert oracle.committed_tokens(np.ones(5, np.uint8), 6) == 6
    assert oracle.committed_tokens(np.zeros(0, np.uint8), 1) == 1


@pytest.mark.parametrize("a,R", [(0.5, 6), (0.7, 6), (0.9, 6), (0.7, 2)])
def test_committed_tokens_bernoulli_mean_closed_form(a, R):
    acc = synth.draft_acceptance(20000, R, a, seed=0)
    mean = np.mean([oracle.committed_tokens(acc[t], R) for t in range(acc.shape[0])])
    assert mean == pytest.approx((1 - a ** R) / (1 - a), rel=0.01)


# --------------------------------------------------------------- verify acceptance --


def test_verify_greedy_hand_cases():
    z = np.array([[0.0, 3.0, 1.0], [5.0, 0.0, 0.0], [0.0, 0.0, 9.0]], np.float32)
    # every draft equals its row's argmax: both accepted, then the bonus token of row 2
    assert oracle.verify_greedy(z, np.array([1, 0])).tolist() == [1, 0, 2]
    # the first draft is wrong: nothing accepted, the correction is row 0's argmax
    assert oracle.verify_greedy(z, np.array([2, 0])).tolist() == [1]
    # the second draft is wrong: one accepted, then row 1's argmax
    assert oracle.verify_greedy(z, np.array([1, 2])).tolist() == [1, 0]
    # a single row (no drafts): its argmax
    assert oracle.verify_greedy(z[:1], np.zeros(0, np.int32)).tolist() == [1]


def test_verify_greedy_tie_goes_to_lower_id():
    z = np.array([[1.0, 7.0, 7.0, 2.0], [0.0, 0.0, 0.0, 4.0]], np.float32)
    assert oracle.verify_greedy(z, np.array([1])).tolist() == [1, 3]
    assert oracle.verify_greedy(z, np.array([2])).tolist() == [1]


def _grid(G):
    return (np.arange(G) + 0.5) / G   # stratified midpoints of [0, 1)


def _softmax64(z, T):
    from scipy.special import softmax
    return softmax(np.asarray(z, np.float64) / T)


def test_verify_sample_acceptance_probability_closed_form():
    # one draft d: the fraction of u_acc values that accept it is min(1, p[d] / q[d])
    z = np.array([[0.3, -1.0, 2.0, 0.5, 0.0], [0.0, 0.0, 0.0, 0.0, 0.0]], np.float32)
    T = 0.8
    p = _softmax64(z[0], T)
    q = np.array([0.05, 0.4, 0.2, 0.3, 0.05])
    G = 2000
    for d in range(5):
        acc = sum(int(oracle.verify_sample(z, T, q[None], np.array([d]), np.array([u]),
                                           np.array([0.5, 0.5])).size == 2)
                  for u in _grid(G))
        assert acc / G == pytest.approx(min(1.0, p[d] / q[d]), abs=1.0 / G)


def test_verify_sample_first_token_follows_target_exactly():
    # exact speculative sampling: with the draft drawn from q, the first emitted token is
    # distributed as p whatever q is (accepted draft, or the residual's correction)
    z = np.array([[0.3, -1.0, 2.0, 0.5, 0.0], [1.0, 0.0, 0.0, 0.0, 0.0]], np.float32)
    T = 0.8
    p = _softmax64(z[0], T)
    q = np.array([0.05, 0.4, 0.2, 0.3, 0.05])
    G = 300
    dist = np.zeros(5)
    for d in range(5):
        for ua in _grid(G):
            for ur in _grid(G):
                tok = oracle.verify_sample(z, T, q[None], np.array([d]), np.array([ua]),
                                           np.array([ur, 0.5]))[0]
                dist[tok] += q[d] / (G * G)
    assert np.allclose(dist, p, atol=4.0 / G)


@pytest.mark.parametrize("u", [0.0, 0.1, 0.37, 0.5, 0.81, 0.999])
def test_verify_sample_bonus_token_is_the_softmax_inverse_cdf(u):
    # a single row: the token drawn with u is the first whose cumulative softmax exceeds u
    z = np.array([[0.2, 1.5, -0.3, 0.9, 0.0, 2.2]], np.float32)
    T = 1.3
    cdf = np.cumsum(_softmax64(z[0], T))
    want = int(np.searchsorted(cdf, u, side="right"))
    got = oracle.verify_sample(z, T, np.zeros((0, 6)), np.zeros(0, np.int32), np.zeros(0),
                               np.array([u]))
    assert got.tolist() == [want]


def test_verify_sample_low_temperature_is_greedy():
    # as T -> 0 the target rows become one-hot at their argmax; with one-hot drafter
    # distributions on the drafted tokens the sampled step equals the greedy one
    rng = np.random.default_rng(3)
    R, V = 6, 50
    z = rng.normal(size=(R, V)).astype(np.float32) * 4
    best = np.argmax(z, axis=1)
    for draft in (best[:-1].copy(), np.array([best[0], best[1], (best[2] + 1) % V, 0, 0])):
        q = np.zeros((R - 1, V))
        q[np.arange(R - 1), draft] = 1.0
        got = oracle.verify_sample(z, 1e-3, q, draft, np.full(R - 1, 0.5), np.full(R, 0.5))
        assert got.tolist() == oracle.verify_greedy(z, draft).tolist()


@pytest.mark.parametrize("T", [0.0, -1.0, float("inf"), float("nan")])
def test_verify_sample_rejects_a_temperature_without_a_softmax(T):
    z = np.zeros((1, 4), np.float32)
    with pytest.raises(ValueError):
        oracle.verify_sample(z, T, np.zeros((0, 4)), np.zeros(0, np.int32), np.zeros(0),
                             np.array([0.5]))
    # and the C function itself refuses it before writing anything
    import ctypes as C
    out = np.full(1, -7, np.int32)
    zz = np.ascontiguousarray(z)
    ur = np.array([0.5])
    n = oracle.lib().orc_verify_sample(zz.ctypes.data, 1, 4, T, None, None, None,
                                       ur.ctypes.data, out.ctypes.data)
    assert n == -1 and out[0] == -7


# ------------------------------------------------------------- sparse attention --

def _bf16_bits(a: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def _bits_to_f64(b: np.ndarray) -> np.ndarray:
    return torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).double().numpy()


def _attn_case(R, Hq, D, N, K, seed, bs=4):
    rng = np.random.default_rng(seed)
    q = _bf16_bits(rng.standard_normal((R, Hq, D)))
    k = _bf16_bits(rng.standard_normal((N * bs, D)))
    v = _bf16_bits(rng.standard_normal((N * bs, D)))
    sel = np.full((R, K), -1, np.int32)
    for r in range(R):
        n = int(rng.integers(1, K + 1))
        sel[r, :n] = np.sort(rng.choice(N, size=n, replace=False))
    return q, k, v, sel


def test_sparse_attention_matches_a_dense_masked_softmax():
    # an independent restatement: gather the selected tokens, scipy's softmax over
    # q.k / sqrt(D), weighted sum of the values
    from scipy.special import softmax
    R, Hq, D, N, K = 3, 4, 32, 40, 9
    q, k, v, sel = _attn_case(R, Hq, D, N, K, seed=1)
    o, ob = oracle.sparse_attention(q, k, v, sel)
    qf, kf, vf = _bits_to_f64(q), _bits_to_f64(k), _bits_to_f64(v)
    for r in range(R):
        toks = np.concatenate([np.arange(4 * b, 4 * b + 4) for b in sel[r] if b >= 0])
        s = qf[r] @ kf[toks].T / np.sqrt(D)
        want = softmax(s, axis=1) @ vf[toks]
        assert np.allclose(o[r], want, rtol=1e-12, atol=1e-14)
    # one bf16 rounding of the fp64 result (torch rounds fp64 -> bf16 once)
    want_b = torch.from_numpy(o).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ob, want_b)


def test_sparse_attention_equal_keys_give_the_mean_value():
    # every selected token has the same key: the weights are uniform and the output is the
    # plain mean of the selected tokens' values
    R, Hq, D, N, K = 2, 3, 16, 12, 4
    q, k, v, sel = _attn_case(R, Hq, D, N, K, seed=2)
    k[:] = k[0]
    o, _ = oracle.sparse_attention(q, k, v, sel)
    vf = _bits_to_f64(v)
    for r in range(R):
        toks = np.concatenate([np.arange(4 * b, 4 * b + 4) for b in sel[r] if b >= 0])
        for h in range(Hq):
            assert np.allclose(o[r, h], vf[toks].mean(axis=0), rtol=1e-13, atol=1e-15)


def test_sparse_attention_one_dominant_token():
    # a key equal to 16 x the query: its score exceeds every other by far more than 40, so
    # the output is that token's value to within e^-40
    R, Hq, D, N, K = 1, 1, 32, 8, 3
    q, k, v, sel = _attn_case(R, Hq, D, N, K, seed=3)
    sel[0] = [1, 4, 6]
    kf = _bits_to_f64(k)
    k[4 * 4 + 2] = _bf16_bits(16.0 * _bits_to_f64(q[0, 0]))
    o, _ = oracle.sparse_attention(q, k, v, sel)
    assert np.allclose(o[0, 0], _bits_to_f64(v)[4 * 4 + 2], rtol=1e-12, atol=1e-12)
    del kf


def test_sparse_attention_padding_empty_rows_and_range():
    R, Hq, D, N, K = 2, 2, 8, 6, 3
    q, k, v, sel = _attn_case(R, Hq, D, N, K, seed=4)
    sel[1] = -1
    o, ob = oracle.sparse_attention(q, k, v, sel)
    assert (o[1] == 0).all() and (ob[1] == 0).all()
    # the same selection with extra -1 entries gives the same output
    wide = np.concatenate([sel, np.full((R, 5), -1, np.int32)], axis=1)
    o2, _ = oracle.sparse_attention(q, k, v, wide)
    assert np.array_equal(o, o2)
    bad = sel.copy()
    bad[0, 0] = N
    with pytest.raises(ValueError):
        oracle.sparse_attention(q, k, v, bad)
