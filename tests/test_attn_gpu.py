"""Sparse attention over the selected blocks on the GPU (ds_sparse_attention) against the
oracle.

Page "DeepSeek V4.1F Q4 on M3 Ultra with native DSpark MTP (40tps / 800tps)", paragraph
"Decode at depth": each layer attends to the blocks its selection picks; the attention
arithmetic is the plain softmax reading stated in the header.

Tolerance (derived from the arithmetic): q.k sums of 128 exact bf16 products in fp32, the
exponentials in fp32, p carried as two bf16 parts (about 2^-16 relative), the weighted sum
of at most 2048 tokens in fp32: every output element must lie within 2 bf16 ulp or 1e-2
relative of the oracle's bf16 result, with the near-zero clause of the MoE outputs (an
element below 1e-3 of its head's rms is judged against 1e-5 of that rms); and within
2^-12 of the head's value rms plus one bf16 ulp of the fp64 result.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import compare
import q4_moe_speculative_gb300 as dsm

pytestmark = pytest.mark.gpu


def random_sel(L, R, N, K, seed, fill=None):
    """Ascending block ids, -1 padded; `fill` entries per row (random count if None)."""
    rng = np.random.default_rng(seed)
    sel = np.full((L, R, K), -1, np.int32)
    for l in range(L):
        for r in range(R):
            n = int(rng.integers(0, min(K, N) + 1)) if fill is None else min(fill, K, N)
            sel[l, r, :n] = np.sort(rng.choice(N, size=n, replace=False))
    return sel


def check(inp, sel, bs=4):
    dev = torch.device("cuda")
    q, k, v = inp["q"].to(dev), inp["k"].to(dev), inp["v"].to(dev)
    st = torch.from_numpy(sel).to(dev)
    out = dsm.sparse_attention(q, k, v, st, bs)
    torch.cuda.synchronize()
    o = synth.to_numpy_bits(out)
    qb, kb, vb = (synth.to_numpy_bits(inp[x]) for x in ("q", "k", "v"))
    L = qb.shape[0]
    worst = 0.0
    for l in range(L):
        o64, obf = oracle.sparse_attention(qb[l], kb[l], vb[l], sel[l], bs)
        rep = compare.y_report(o[l].reshape(-1, 128), obf.reshape(-1, 128))
        assert rep["fail"] == 0, (l, rep)
        od = compare.bf16_bits_to_f64(o[l])
        vrms = np.sqrt(np.mean(compare.bf16_bits_to_f64(vb[l]) ** 2))
        excess = np.abs(od - o64) - (2.0 ** -12 * vrms + compare.bf16_ulp(o64))
        worst = max(worst, float(excess.max()))
    assert worst <= 0, worst
    return o


@pytest.mark.parametrize("L,R,Hq,N,K,bs,sigma", [
    (2, 6, 16, 2048, 512, 4, 1.0),     # the 8k context shape
    (2, 6, 16, 2048, 512, 4, 4.0),     # peaked attention
    (3, 3, 8, 300, 100, 4, 1.0),       # ragged: K not a multiple of the 4-entry groups
    (1, 2, 1, 64, 37, 4, 2.0),
    (2, 4, 16, 500, 64, 1, 1.0),       # one token per block
    (1, 2, 5, 40, 9, 16, 1.0),         # 16 tokens per block
    (1, 8, 16, 4096, 2048, 4, 1.0),    # the widest selection
])
def test_attention_matches_oracle(L, R, Hq, N, K, bs, sigma):
    inp = synth.attention_inputs(L, R, Hq, N * bs, seed=N + K + R, sigma=sigma)
    sel = random_sel(L, R, N, K, seed=K + bs)
    check(inp, sel, bs)


def test_attention_on_the_selection_of_the_select_call():
    # the selection written by ds_select_blocks at 8k context drives the attention
    sh = synth.SELECT_8K
    s_in = synth.select_inputs(sh, seed=3, device="cuda")
    sel_t, nsel, _, _ = dsm.select_blocks(s_in["keys"], s_in["q"], s_in["head_w"],
                                          s_in["mask"], s_in["limit"], sh.topk)
    inp = synth.attention_inputs(sh.L, sh.R, 16, sh.N * 4, seed=5)
    sel = sel_t.cpu().numpy()
    assert (nsel.cpu().numpy() == 512).all()
    check(inp, sel, 4)


def test_empty_rows_and_invalid_ids_give_zero_or_are_skipped():
    L, R, Hq, N, K = 1, 4, 16, 100, 32
    inp = synth.attention_inputs(L, R, Hq, N * 4, seed=9)
    sel = random_sel(L, R, N, K, seed=10, fill=20)
    sel[0, 1] = -1                      # no block: zero output
    o = check(inp, sel, 4)
    assert (o[0, 1] == 0).all()
    # ids at or beyond N are skipped like -1 (the oracle is given the same row without them)
    bad = sel.copy()
    bad[0, 2, 20:24] = [N, N + 5, 1 << 20, -7]
    dev = torch.device("cuda")
    out = dsm.sparse_attention(inp["q"].to(dev), inp["k"].to(dev), inp["v"].to(dev),
                               torch.from_numpy(bad).to(dev), 4)
    ref = dsm.sparse_attention(inp["q"].to(dev), inp["k"].to(dev), inp["v"].to(dev),
                               torch.from_numpy(sel).to(dev), 4)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_deterministic():
    inp = synth.attention_inputs(2, 6, 16, 8192, seed=12)
    sel = random_sel(2, 6, 2048, 512, seed=13, fill=512)
    dev = torch.device("cuda")
    args = (inp["q"].to(dev), inp["k"].to(dev), inp["v"].to(dev), torch.from_numpy(sel).to(dev))
    a = dsm.sparse_attention(*args)
    b = dsm.sparse_attention(*args)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
