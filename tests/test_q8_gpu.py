"""Paired Q8 projections on the GPU (ds_q8_tile, ds_q8_project) against the oracle.

Page "DeepSeek V4.1F Q4 on M3 Ultra with native DSpark MTP (40tps / 800tps)", paragraph
"DSpark": the verify rows share one weight stream through paired Q8 projections.

Contract checked here:
  * the tile-major form is the header's byte permutation, every byte;
  * every bf16 output is within 2 bf16 ulp or 1e-2 relative of the oracle (fp64 products,
    one rounding), with the near-zero clause of the MoE outputs;
  * tighter: each output is a rounding of a value within the fp32 accumulation band of
    the exact sum (int8 x bf16 products are exact; K / 512 block-scale fmas per warp chain
    and 16 warp partials added in order), i.e. |y - y_exact| <= band * sum|terms| + 1 ulp;
  * an R-row call writes the same bytes as R one-row calls, and runs are deterministic.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import compare
import q4_moe_speculative_gb300 as dsm

pytestmark = pytest.mark.gpu


def expected_tiles(qs: np.ndarray, sc: np.ndarray) -> np.ndarray:
    """The header's tile-major Q8 layout restated with numpy indexing."""
    rows, K = qs.shape
    U, Tk = rows // 16, K // 64
    out = np.zeros((U, Tk, 1088), np.uint8)
    qb = qs.view(np.uint8)
    scb = sc.view(np.uint16)
    for u in range(U):
        for kt in range(Tk):
            t = out[u, kt]
            for j in range(2):
                kb = 64 * kt + 32 * j
                for L in range(32):
                    g, q = L >> 2, L & 3
                    parts = [qb[16 * u + g, kb + 4 * q: kb + 4 * q + 4],
                             qb[16 * u + g + 8, kb + 4 * q: kb + 4 * q + 4],
                             qb[16 * u + g, kb + 16 + 4 * q: kb + 16 + 4 * q + 4],
                             qb[16 * u + g + 8, kb + 16 + 4 * q: kb + 16 + 4 * q + 4]]
                    t[512 * j + 16 * L: 512 * j + 16 * L + 16] = np.concatenate(parts)
            for g in range(8):
                s4 = np.array([scb[16 * u + g, 2 * kt], scb[16 * u + g + 8, 2 * kt],
                               scb[16 * u + g, 2 * kt + 1], scb[16 * u + g + 8, 2 * kt + 1]],
                              np.uint16)
                t[1024 + 8 * g: 1024 + 8 * g + 8] = s4.view(np.uint8)
    return out


@pytest.mark.parametrize("rows,K", [(16, 64), (48, 192), (32, 512)])
def test_tile_layout_every_byte(rows, K):
    qs, sc = synth.q8_matrix(rows, K, seed=rows + K, device="cuda")
    t = dsm.q8_tile(qs, sc)
    torch.cuda.synchronize()
    want = expected_tiles(qs.cpu().numpy(), sc.cpu().view(torch.int16).numpy())
    assert np.array_equal(t.cpu().numpy(), want)


def project_case(rows, K, R, seed):
    dev = torch.device("cuda")
    qs, sc = synth.q8_matrix(rows, K, seed=seed, device=dev)
    x = synth.activations(R, K, seed=seed + 1, device=dev)
    tiles = dsm.q8_tile(qs, sc)
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    y = dsm.q8_project(tiles, x, workspace=ws)
    torch.cuda.synchronize()
    assert dsm.workspace_status(ws) == 0
    q_np = qs.cpu().numpy()
    s_np = sc.cpu().view(torch.int16).numpy().view(np.uint16)
    x_np = synth.to_numpy_bits(x)
    y64, ybf = oracle.q8_project(q_np, s_np, x_np)
    return tiles, x, y, y64, ybf, q_np, s_np, x_np


def check_outputs(y, y64, ybf, q_np, s_np, x_np, K):
    yd = synth.to_numpy_bits(y)
    rep = compare.y_report(yd, ybf)
    assert rep["fail"] == 0, rep
    # the accumulation band: |y_dev - y_exact| <= band * sum|terms| + one bf16 ulp
    W = np.abs(q_np.astype(np.float64)) * np.repeat(
        s_np.view(np.float16).astype(np.float64), 32, axis=1)
    xa = np.abs(compare.bf16_bits_to_f64(x_np))
    A = xa @ W.T                                            # [R][rows]
    band = compare.accumulation_band(K // 512, 16)
    yv = compare.bf16_bits_to_f64(yd)
    excess = np.abs(yv - y64) - (band * A + compare.bf16_ulp(y64))
    assert excess.max() <= 0, float(excess.max())
    return rep


@pytest.mark.parametrize("rows,K,R", [(4096, 4096, 6), (64, 1024, 1), (112, 3072, 3),
                                      (16, 1024, 8), (2048, 8192, 6), (4800, 2048, 2),
                                      (160, 5120, 5)])
def test_project_matches_oracle(rows, K, R):
    tiles, x, y, y64, ybf, q_np, s_np, x_np = project_case(rows, K, R, seed=rows + K + R)
    rep = check_outputs(y, y64, ybf, q_np, s_np, x_np, K)
    assert rep["exact"] >= 0.9 * rep["n"], rep


def test_rows_share_the_stream_byte_identically():
    rows, K, R = 1024, 4096, 6
    tiles, x, y, *_ = project_case(rows, K, R, seed=17)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    singles = [dsm.q8_project(tiles, x[r:r + 1].contiguous(), workspace=ws) for r in range(R)]
    pair = dsm.q8_project(tiles, x[[4, 1]].contiguous(), workspace=ws)
    again = dsm.q8_project(tiles, x, workspace=ws)
    torch.cuda.synchronize()
    yb = y.view(torch.int16).cpu()
    for r in range(R):
        assert torch.equal(singles[r].view(torch.int16).cpu()[0], yb[r])
    assert torch.equal(pair.view(torch.int16).cpu()[0], yb[4])
    assert torch.equal(pair.view(torch.int16).cpu()[1], yb[1])
    assert torch.equal(again.view(torch.int16).cpu(), yb)


def test_unsupported_sizes_are_reported():
    dev = torch.device("cuda")
    qs, sc = synth.q8_matrix(32, 576, seed=1, device=dev)
    tiles = dsm.q8_tile(qs, sc)
    x = synth.activations(2, 576, seed=2, device=dev)
    with pytest.raises(dsm.DsmoeError) as e:
        dsm.q8_project(tiles, x)
    assert e.value.status == 2   # K not a multiple of 1024
    qs, sc = synth.q8_matrix(32, 1536, seed=1, device=dev)
    x = synth.activations(2, 1536, seed=2, device=dev)
    with pytest.raises(dsm.DsmoeError) as e:
        dsm.q8_project(dsm.q8_tile(qs, sc), x)
    assert e.value.status == 2
