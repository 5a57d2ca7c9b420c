"""The tensor-core scoring interval of ds_select_blocks (called through the C ABI).

The selection is exact because every admitted block's canonical score lies within
kn * G of its tensor-core score s (kn: the key-norm bound, G: the row's bound of
2^-13 * sum_h |w_h| ||q_h||, both read back from the workspace). These tests check that
bound entry by entry against the oracle's canonical score on inputs built to strain it:
key and query entries spread over 2^-12 .. 2^12, keys made nearly orthogonal to a head's
query (heavy cancellation, dot products at the ReLU boundary), head weights of both
signs; and, in the same calls, the selection bit for bit against the oracle. The largest
observed |s - s_canonical| / (kn G) is printed.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsm():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from q4_moe_speculative_gb300.build import build_library
    build_library()
    import q4_moe_speculative_gb300 as m
    m._native.load()
    return m


def bf16(a: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bits (round to nearest even, through torch)."""
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def wide_range(rng, shape):
    """Values +-2^e * (1 + m/128), e uniform in [-12, 12]: exact in bf16."""
    e = rng.integers(-12, 13, size=shape)
    m = rng.integers(0, 128, size=shape)
    sgn = rng.choice([-1.0, 1.0], size=shape)
    return sgn * np.ldexp(1.0 + m / 128.0, e)


def adversarial(shape: synth.SelectShape, seed: int, kind: str) -> dict:
    rng = np.random.default_rng(seed)
    L, R, Hh, N, D = shape.L, shape.R, shape.Hh, shape.N, shape.D
    q = wide_range(rng, (L, R, Hh, D))
    if kind == "range":
        keys = wide_range(rng, (L, N, D))
    else:
        # cancellation: each key is a wide-range vector with its component along one head's
        # query (of row 0 or 1, head b % Hh) removed, so that q . k is small next to the sum
        # of |q_i k_i|; half of them are then nudged across zero
        keys = wide_range(rng, (L, N, D))
        for l in range(L):
            for b in range(N):
                qq = q[l, b % min(R, 2), b % Hh]
                keys[l, b] -= (keys[l, b] @ qq) / (qq @ qq) * qq
                if b & 1:
                    keys[l, b] += 1e-3 * rng.standard_normal() * np.abs(keys[l, b]).max() * qq / np.linalg.norm(qq)
    w = rng.standard_normal((L, R, Hh)).astype(np.float32)
    mask, limit = synth.admission_mask(shape, seed, shared=False)
    return {"keys": torch.from_numpy(bf16(keys).view(np.int16)).view(torch.bfloat16),
            "q": torch.from_numpy(bf16(q).view(np.int16)).view(torch.bfloat16),
            "head_w": torch.from_numpy(w),
            "mask": torch.from_numpy(mask.view(np.int32).copy()),
            "limit": torch.from_numpy(limit)}


def check_bound_and_selection(dsm, inp, topk, layers, sample=None, seed=0):
    dv = {k: v.to("cuda") for k, v in inp.items()}
    args = (dv["keys"], dv["q"], dv["head_w"], dv["mask"], dv["limit"], topk)
    ws = torch.empty(dsm.select_workspace_size(*args), dtype=torch.uint8, device="cuda")
    sel, nsel, _, _ = dsm.select_blocks(*args, workspace=ws, keep_workspace=True)
    torch.cuda.synchronize()
    assert dsm.workspace_status(ws) == 0
    views = {k: v.cpu().numpy() for k, v in dsm.select_workspace_views(*args, ws).items()}
    keys = synth.to_numpy_bits(inp["keys"])
    q = synth.to_numpy_bits(inp["q"])
    hw = inp["head_w"].numpy()
    mask = inp["mask"].numpy().view(np.uint32)
    limit = inp["limit"].numpy()
    L, R = q.shape[0], q.shape[1]
    # every (layer, row, union entry) the row admits, or a seeded sample of them
    cand = []
    for l in range(L):
        n = views["union_count"][l]
        blocks = views["union"][l, :n]
        for r in range(R):
            adm = ((mask[l, r, blocks >> 5] >> (blocks & 31)) & 1).astype(bool) & (blocks < limit[l, r])
            cand.extend((l, r, e) for e in np.flatnonzero(adm))
    if sample is not None and len(cand) > sample:
        pick = np.random.default_rng(seed).choice(len(cand), sample, replace=False)
        cand = [cand[i] for i in pick]
    worst = 0.0
    for l, r, e in cand:
        b = views["union"][l, e]
        s = float(views["scores"][l, r, e])
        eps = float(views["key_norms"][l, e]) * float(views["row_scales"][l, r])   # fp64 product
        c = oracle.block_score(q[l, r], keys[l, b], hw[l, r])
        assert np.isfinite(s) and eps > 0
        assert abs(s - c) <= eps, (l, r, int(b), s, c, eps)
        if eps > 0:
            worst = max(worst, abs(s - c) / eps)
    ref = oracle.select(keys, q, hw, mask, limit, topk, layers=layers)
    sel, nsel = sel.cpu().numpy(), nsel.cpu().numpy()
    for l in range(*layers):
        assert np.array_equal(nsel[l], ref["nsel"][l]), l
        assert np.array_equal(sel[l], ref["sel"][l]), l
    print(f"checked {len(cand)} entries; largest |s - s_canonical| / (kn G) = {worst:.3e}")
    return worst


@pytest.mark.parametrize("kind", ["range", "cancel"])
def test_interval_holds_on_adversarial_inputs(dsm, kind):
    shape = synth.SelectShape(L=2, R=6, Hh=8, N=3000, topk=512)
    inp = adversarial(shape, seed=41 if kind == "range" else 42, kind=kind)
    worst = check_bound_and_selection(dsm, inp, shape.topk, layers=(0, shape.L))
    assert worst < 1.0


def test_interval_holds_at_300k_context(dsm):
    # the full 300k / 43-layer case, N(0, 1) inputs: a seeded sample of 20,000 admitted
    # entries against the bound, and the selection of two layers bit for bit
    shape = synth.SELECT_300K
    inp = synth.select_inputs(shape, seed=3, device="cpu", shared_mask=True)
    check_bound_and_selection(dsm, inp, shape.topk, layers=(0, 2), sample=20000, seed=3)
