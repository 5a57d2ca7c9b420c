"""GPU parity of ds_select_blocks against the oracle (through the C ABI): the compacted
index, the admitted counts and the top-k selection must match bit for bit."""
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


def to_dev(inp: dict) -> dict:
    return {k: v.to("cuda") for k, v in inp.items()}


def run_dev(dsm, inp, topk, canonical=False):
    sel, nsel, cidx, ccount = dsm.select_blocks(inp["keys"], inp["q"], inp["head_w"], inp["mask"],
                                                inp["limit"], topk, want_compacted=True,
                                                canonical=canonical)
    torch.cuda.synchronize()
    return sel.cpu().numpy(), nsel.cpu().numpy(), cidx.cpu().numpy(), ccount.cpu().numpy()


def run_ref(inp, topk, layers=None):
    keys = synth.to_numpy_bits(inp["keys"])
    q = synth.to_numpy_bits(inp["q"])
    hw = inp["head_w"].cpu().numpy()
    mask = inp["mask"].cpu().numpy().view(np.uint32)
    limit = inp["limit"].cpu().numpy()
    return oracle.select(keys, q, hw, mask, limit, topk, layers=layers)


def assert_equal_rows(dev, ref, layers):
    sel, nsel, cidx, ccount = dev
    for l in layers:
        assert np.array_equal(ccount[l], ref["ccount"][l]), l
        assert np.array_equal(nsel[l], ref["nsel"][l]), l
        assert np.array_equal(sel[l], ref["sel"][l]), l
        for r in range(ccount.shape[1]):
            n = ccount[l, r]
            assert np.array_equal(cidx[l, r, :n], ref["cidx"][l, r, :n]), (l, r)


def check(dsm, inp, topk, layers=None, canonical=False):
    dev = run_dev(dsm, to_dev(inp), topk, canonical=canonical)
    L = inp["keys"].shape[0]
    rng = (0, L) if layers is None else layers
    ref = run_ref(inp, topk, layers=rng)
    assert_equal_rows(dev, ref, range(*rng))
    return dev, ref


def test_tiny_single_head(dsm):
    shape = synth.TINY_SELECT
    inp = synth.select_inputs(shape, seed=0)
    inp["head_w"] = torch.ones_like(inp["head_w"])
    dev, ref = check(dsm, inp, shape.topk)
    assert dev[1][0, 0] == shape.topk


@pytest.mark.parametrize("canonical", [False, True])
@pytest.mark.parametrize("shared", [True, False])
def test_8k_context(dsm, shared, canonical):
    shape = synth.SELECT_8K
    inp = synth.select_inputs(shape, seed=3, shared_mask=shared)
    check(dsm, inp, shape.topk, canonical=canonical)


def test_ragged_sizes(dsm):
    shape = synth.SelectShape(L=3, R=5, Hh=3, N=1000, topk=100)
    inp = synth.select_inputs(shape, seed=4, shared_mask=False)
    check(dsm, inp, shape.topk)


@pytest.mark.parametrize("count", [0, 1, 511, 512, 513, 2047])
def test_exact_admitted_counts(dsm, count):
    shape = synth.SelectShape(L=1, R=2, Hh=8, N=2048, topk=512)
    inp = synth.select_inputs(shape, seed=5)
    rng = np.random.default_rng(count)
    bits = np.zeros((1, 2, shape.N), bool)
    for r in range(2):
        bits[0, r, rng.choice(shape.N, size=count, replace=False)] = True
    inp["mask"] = torch.from_numpy(synth.pack_bits(bits).view(np.int32).copy())
    inp["limit"] = torch.full((1, 2), shape.N, dtype=torch.int32)
    dev, _ = check(dsm, inp, shape.topk)
    assert np.all(dev[1] == min(count, 512))


@pytest.mark.parametrize("canonical", [False, True])
def test_all_equal_scores_take_lowest_indices(dsm, canonical):
    # every key identical: all admitted scores tie; a bucket far above the shared-memory
    # residual bound (thousands of equal keys) exercises the global-memory passes.
    shape = synth.SelectShape(L=1, R=3, Hh=8, N=20000, topk=512)
    inp = synth.select_inputs(shape, seed=6)
    inp["keys"] = inp["keys"][:, :1, :].expand(-1, shape.N, -1).contiguous()
    dev, ref = check(dsm, inp, shape.topk, canonical=canonical)
    for r in range(3):
        assert np.array_equal(dev[0][0, r], dev[2][0, r, :512])


@pytest.mark.parametrize("canonical", [False, True])
def test_zero_score_ties_single_head(dsm, canonical):
    # one head, w = 1: score = relu(q.k), about half exactly +0; top-k reaches into the zeros
    shape = synth.SelectShape(L=2, R=2, Hh=1, N=4000, topk=1500)
    inp = synth.select_inputs(shape, seed=7)
    inp["head_w"] = torch.ones_like(inp["head_w"])
    check(dsm, inp, shape.topk, canonical=canonical)


def test_many_heads_and_rows(dsm):
    # R * Hh = 128 (the widest tensor-core tile) and a layer stride with padding
    shape = synth.SelectShape(L=2, R=8, Hh=16, N=3000, topk=256)
    inp = synth.select_inputs(shape, seed=12)
    check(dsm, inp, shape.topk)


def test_eight_rows_eight_heads_long_rows(dsm):
    # R = 8 at 8 heads (the static epilogue with every row slot used: the key-norm bound of
    # each 32 entries takes its own reduction), rows long enough for the chunk-maxima
    # threshold and the chunk-level first test
    shape = synth.SelectShape(L=2, R=8, Hh=8, N=30000, topk=512)
    inp = synth.select_inputs(shape, seed=14, shared_mask=False)
    check(dsm, inp, shape.topk)


def test_candidate_band_overflow_falls_back(dsm):
    # keys in 3 distinct values: thousands of near-equal tensor-core scores around the
    # threshold overflow the candidate bound; the row is re-scored canonically.
    shape = synth.SelectShape(L=1, R=2, Hh=8, N=30000, topk=512)
    inp = synth.select_inputs(shape, seed=13)
    base = inp["keys"][:, :3, :]
    pick = torch.from_numpy(np.random.default_rng(0).integers(0, 3, shape.N))
    inp["keys"] = base[:, pick, :].contiguous()
    check(dsm, inp, shape.topk)


def test_negative_weights(dsm):
    shape = synth.SelectShape(L=1, R=4, Hh=8, N=3000, topk=512)
    inp = synth.select_inputs(shape, seed=8)
    inp["head_w"] = -inp["head_w"].abs()
    check(dsm, inp, shape.topk)


def test_layers_batched_equal_single_layer_calls(dsm):
    shape = synth.SelectShape(L=4, R=6, Hh=8, N=5000, topk=512)
    inp = to_dev(synth.select_inputs(shape, seed=9))
    full = run_dev(dsm, inp, shape.topk)
    for l in range(shape.L):
        one = run_dev(dsm, {k: v[l:l + 1].contiguous() for k, v in inp.items()}, shape.topk)
        assert np.array_equal(one[0][0], full[0][l])
        assert np.array_equal(one[1][0], full[1][l])
    again = run_dev(dsm, inp, shape.topk)
    for a, b in zip(full[:2], again[:2]):           # sel, nsel
        assert np.array_equal(a, b)
    assert np.array_equal(full[3], again[3])        # ccount
    for l in range(shape.L):                        # cidx up to the admitted count
        for r in range(shape.R):
            n = full[3][l, r]
            assert np.array_equal(full[2][l, r, :n], again[2][l, r, :n])


def test_300k_context_sampled_layers(dsm):
    # full workload (43 layers x 6 rows x 75,000 blocks) in the configuration the benchmark
    # times; the oracle checks three layers completely, every layer is checked for its
    # structural properties.
    shape = synth.SELECT_300K
    inp_host = synth.select_inputs(shape, seed=0, device="cpu")
    dev = run_dev(dsm, to_dev(inp_host), shape.topk)
    sel, nsel, cidx, ccount = dev
    for l in (0, 21, 42):
        ref = run_ref(inp_host, shape.topk, layers=(l, l + 1))
        assert_equal_rows(dev, ref, [l])
    assert np.all(nsel == 512)
    assert np.all(np.diff(sel, axis=-1) > 0)
    mask = inp_host["mask"].numpy().view(np.uint32)
    word = mask[np.arange(43)[:, None, None], np.arange(6)[None, :, None], sel // 32]
    assert np.all((word >> (sel % 32)) & 1)
    assert np.all(sel < inp_host["limit"].numpy()[..., None])


def test_status_word_clean(dsm):
    shape = synth.SELECT_8K
    inp = to_dev(synth.select_inputs(shape, seed=1))
    ws = torch.empty(dsm.select_workspace_size(inp["keys"], inp["q"], inp["head_w"], inp["mask"],
                                               inp["limit"], 512), dtype=torch.uint8, device="cuda")
    dsm.select_blocks(inp["keys"], inp["q"], inp["head_w"], inp["mask"], inp["limit"], 512,
                      workspace=ws)
    assert dsm.workspace_status(ws) == 0


@pytest.mark.parametrize("canonical", [False, True])
def test_mixed_density_and_empty_layers(dsm, canonical):
    # layer 0: every block below 4000 admitted, 10% above; layer 1: limit 0 (nothing);
    # layer 2: 20% everywhere; layer 3: every block, limits ending inside a 128-block tile
    shape = synth.SelectShape(L=4, R=3, Hh=8, N=9000, topk=512)
    inp = synth.select_inputs(shape, seed=8, shared_mask=False)
    rng = np.random.default_rng(8)
    N = shape.N
    bits = np.zeros((4, 3, N), bool)
    bits[0, :, :4000] = True
    bits[0, :, 4000:] = rng.random((3, N - 4000)) < 0.1
    bits[1] = rng.random((3, N)) < 0.7
    bits[2] = rng.random((3, N)) < 0.2
    bits[3] = True
    limit = np.full((4, 3), N, dtype=np.int32)
    limit[1] = 0
    limit[3] = [N - 37, N - 100, 5000]
    inp["mask"] = torch.from_numpy(synth.pack_bits(bits).view(np.int32).copy())
    inp["limit"] = torch.from_numpy(limit)
    dev, _ = check(dsm, inp, shape.topk, canonical=canonical)
    assert np.all(dev[1][1] == 0)


def test_chunk_threshold_paths(dsm):
    # Rows long enough (at least K chunks of 32 union entries) that the top-k takes its
    # collection threshold from the per-chunk score maxima. Layer 0: row 0 admits one
    # window of 3000 blocks (fewer than K chunks hold an admitted entry: the sampled
    # threshold), row 1 70%, row 2 every block; layer 1: 5% per row (most chunks hold one
    # or two admitted entries); layer 2: a shared 70% mask with a causal limit inside a
    # chunk on row 2.
    shape = synth.SelectShape(L=3, R=3, Hh=8, N=40000, topk=512)
    inp = synth.select_inputs(shape, seed=31, shared_mask=False)
    rng = np.random.default_rng(31)
    N = shape.N
    bits = np.zeros((3, 3, N), bool)
    bits[0, 0, 20000:23000] = True
    bits[0, 1] = rng.random(N) < 0.7
    bits[0, 2] = True
    bits[1] = rng.random((3, N)) < 0.05
    bits[2] = (rng.random(N) < 0.7)[None, :]
    limit = np.full((3, 3), N, dtype=np.int32)
    limit[2, 2] = 30017
    inp["mask"] = torch.from_numpy(synth.pack_bits(bits).view(np.int32).copy())
    inp["limit"] = torch.from_numpy(limit)
    dev, _ = check(dsm, inp, shape.topk)
    assert np.all(dev[1] == shape.topk)


@pytest.mark.parametrize("canonical", [False, True])
def test_twelve_heads_odd_block_count(dsm, canonical):
    # Hh = 12 (the generic scoring and re-score paths), 3 rows, an odd block count (score
    # rows padded to a multiple of 4, the last collection group ragged) and K = 300
    shape = synth.SelectShape(L=2, R=3, Hh=12, N=12345, topk=300)
    inp = synth.select_inputs(shape, seed=21)
    check(dsm, inp, shape.topk, canonical=canonical)


def test_dropped_workspace_is_rewritten_by_the_next_call(dsm):
    # By default the top-k drops the scores, key norms and union lists from L2 once read
    # (their workspace bytes become undefined); the next call on the same workspace must
    # rebuild everything it reads. Three calls on one workspace (dropping, keeping,
    # dropping) and a call on a fresh workspace give the same selection, bit for bit.
    shape = synth.SelectShape(L=6, R=6, Hh=8, N=20000, topk=512)
    inp = to_dev(synth.select_inputs(shape, seed=21))
    args = (inp["keys"], inp["q"], inp["head_w"], inp["mask"], inp["limit"], 512)
    ws = torch.empty(dsm.select_workspace_size(*args), dtype=torch.uint8, device="cuda")
    outs = []
    for keep in (False, True, False):
        sel, nsel, _, _ = dsm.select_blocks(*args, workspace=ws, keep_workspace=keep)
        torch.cuda.synchronize()
        assert dsm.workspace_status(ws) == 0
        outs.append((sel.cpu().clone(), nsel.cpu().clone()))
    fresh = dsm.select_blocks(*args)
    torch.cuda.synchronize()
    for sel, nsel in outs:
        assert torch.equal(sel, fresh[0].cpu()) and torch.equal(nsel, fresh[1].cpu())
    ref = run_ref(inp, 512, layers=(0, 2))
    assert np.array_equal(outs[2][0].numpy()[:2], ref["sel"][:2])
