"""Verify acceptance on the GPU (ds_verify_greedy, ds_verify_sample) against the oracle.

Page "DeepSeek V4.1F Q4 on M3 Ultra with native DSpark MTP (40tps / 800tps)", paragraph
"DSpark": greedy verify gives the same output as decoding without the drafter; at
temperature > 0 the verify step does exact speculative sampling.

Greedy acceptance is integer work on fp32 comparisons: tokens and counts must equal the
oracle's exactly. Sampling decisions are taken in fp64 on both sides; the GPU adds the
vocabulary in a fixed parallel order where the oracle adds it in token order, so the two
can differ only for a decision whose margin (|u q[d] - p[d]| / p[d], or the distance of
u x total to the nearest cumulative boundary / total) is within rounding. Such steps are
counted (a margin below 1e-11 marks one) and must be rare; every other step must match
exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import q4_moe_speculative_gb300 as dsm

pytestmark = pytest.mark.gpu

AMBIGUOUS = 1e-11


def run_greedy(z, draft):
    dev = torch.device("cuda")
    zt = torch.from_numpy(z).to(dev)
    dt = torch.from_numpy(draft).to(dev) if z.shape[1] > 1 else None
    ws = torch.empty(dsm._native.load().ds_verify_workspace_size(*z.shape), dtype=torch.uint8,
                     device=dev)
    out, n = dsm.verify_greedy(zt, dt, workspace=ws)
    torch.cuda.synchronize()
    assert dsm.workspace_status(ws) == 0
    return out.cpu().numpy(), n.cpu().numpy()


def run_sample(d, T):
    dev = torch.device("cuda")
    t = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in d.items()
         if k in ("logits", "qd", "draft", "u_acc", "u_res")}
    R = d["logits"].shape[1]
    ws = torch.empty(dsm._native.load().ds_verify_workspace_size(*d["logits"].shape),
                     dtype=torch.uint8, device=dev)
    out, n = dsm.verify_sample(t["logits"], T, t["qd"] if R > 1 else None,
                               t["draft"] if R > 1 else None, t["u_acc"] if R > 1 else None,
                               t["u_res"], workspace=ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), n.cpu().numpy(), dsm.workspace_status(ws)


def decision_margin(z, T, qd, draft, ua, ur):
    """Smallest relative margin of the decisions the step takes (fp64, token order)."""
    R, V = z.shape
    margin = np.inf
    for r in range(R):
        x = z[r].astype(np.float64) / T
        e = np.exp(x - x.max())
        p = e / e.sum()
        if r == R - 1:
            w = p
            u = ur[r]
            break
        d = draft[r]
        lhs, rhs = ua[r] * qd[r][d], p[d]
        margin = min(margin, abs(lhs - rhs) / max(rhs, 1e-300))
        if lhs < rhs:
            continue
        res = np.maximum(p - qd[r], 0.0)
        w = res if res.sum() > 0 else p
        u = ur[r]
        break
    total = w.sum()
    cs = np.cumsum(w)
    t = u * total
    x = int(np.searchsorted(cs, t, side="right"))
    lo = cs[x - 1] if x > 0 else 0.0
    hi = cs[x] if x < V else total
    return min(margin, (t - lo) / total, (hi - t) / total)


def expect_rows(out, n, want_list):
    for b, want in enumerate(want_list):
        assert n[b] == len(want), (b, n[b], want)
        assert out[b, :n[b]].tolist() == list(want), (b, out[b].tolist(), want)
        assert (out[b, n[b]:] == -1).all()


@pytest.mark.parametrize("B,R,V", [(12, 6, synth.VOCAB), (8, 6, 4097), (5, 3, 5), (3, 1, 1000),
                                   (2, 6, 1), (4, 16, 12289)])
def test_greedy_matches_oracle(B, R, V):
    d = synth.greedy_inputs(B, R, V, seed=B * 100 + R)
    out, n = run_greedy(d["logits"], d["draft"])
    want = [oracle.verify_greedy(d["logits"][b], d["draft"][b]) for b in range(B)]
    expect_rows(out, n, want)
    # every prefix length occurs across the steps of the largest case
    if (B, R) == (12, 6):
        assert sorted(set(n.tolist())) == list(range(1, 7))


def check_sample_case(d, T, max_ambiguous=0):
    out, n, st = run_sample(d, T)
    assert st == 0
    B = d["logits"].shape[0]
    R = d["logits"].shape[1]
    amb = 0
    for b in range(B):
        qd = d["qd"][b] if R > 1 else np.zeros((0, d["logits"].shape[2]))
        dr = d["draft"][b] if R > 1 else np.zeros(0, np.int32)
        ua = d["u_acc"][b] if R > 1 else np.zeros(0)
        want = oracle.verify_sample(d["logits"][b], T, qd, dr, ua, d["u_res"][b])
        if decision_margin(d["logits"][b], T, qd, dr, ua, d["u_res"][b]) < AMBIGUOUS:
            amb += 1
            continue
        assert n[b] == len(want), (b, n[b], want.tolist())
        assert out[b, :n[b]].tolist() == want.tolist(), (b, out[b].tolist(), want.tolist())
        assert (out[b, n[b]:] == -1).all()
    assert amb <= max_ambiguous, amb
    return n


@pytest.mark.parametrize("T,alpha,seed", [(1.0, 0.7, 0), (0.6, 0.9, 1), (1.7, 0.3, 2),
                                          (1.0, 0.02, 3)])
def test_sample_matches_oracle_full_vocabulary(T, alpha, seed):
    d = synth.verify_inputs(16, 6, synth.VOCAB, seed=seed, alpha=alpha)
    n = check_sample_case(d, T)
    assert n.min() >= 1 and n.max() <= 6


@pytest.mark.parametrize("B,R,V", [(9, 6, 10007), (6, 2, 4096), (4, 1, 300), (5, 4, 7),
                                   (3, 16, 4099)])
def test_sample_matches_oracle_ragged_sizes(B, R, V):
    d = synth.verify_inputs(B, R, V, seed=V + R)
    check_sample_case(d, 0.9)


def test_sample_accepts_everything_with_an_exact_drafter():
    # qd = one-hot at the planted token and a target that puts all its mass there at low
    # temperature: every draft is kept and the bonus token is the planted one
    d = synth.verify_inputs(6, 6, 5000, seed=7, peak=400.0, alpha=1.0)
    d["draft"] = d["strong"][:, :5].copy()
    n = check_sample_case(d, 0.5)
    assert (n == 6).all()


def test_sample_draft_outside_the_vocabulary_is_flagged_and_rejected():
    d = synth.verify_inputs(2, 6, 1000, seed=11)
    d["draft"][0, 2] = -1
    d["draft"][1, 0] = 1000
    out, n, st = run_sample(d, 1.0)
    assert st == 6   # DS_ERR_DEVICE_CHECK
    assert n[1] == 1 and n[0] <= 3


def test_sample_statistics_follow_the_target():
    # exact speculative sampling: the first emitted token is distributed as p_0 whatever
    # the drafter; over many steps with a poor drafter the empirical frequency of the
    # planted token equals p_0 of that token (one row of logits repeated)
    B, R, V = 4096, 2, 64
    base = synth.verify_inputs(1, R, V, seed=5, peak=2.0, alpha=0.5)
    d = {k: np.repeat(v, B, axis=0) for k, v in base.items()}
    rng = np.random.default_rng(9)
    d["draft"] = rng.integers(0, V, size=(B, R - 1)).astype(np.int32)
    d["qd"] = np.full((B, R - 1, V), 1.0 / V)
    d["u_acc"] = rng.random((B, R - 1))
    d["u_res"] = rng.random((B, R))
    out, n, st = run_sample(d, 1.0)
    assert st == 0
    x = d["logits"][0, 0].astype(np.float64)
    p = np.exp(x - x.max())
    p /= p.sum()
    freq = np.bincount(out[:, 0], minlength=V) / B
    assert np.abs(freq - p).max() < 4.5 * np.sqrt(p.max() / B)
