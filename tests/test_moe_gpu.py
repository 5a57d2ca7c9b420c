"""GPU parity of ds_moe_verify_forward against the oracle (called through the C ABI).

Routing indices bit-exact (near-ties under 1e-5 may swap, then the output is compared with
the oracle re-run on the device's choice), routing weights within 1e-5, bf16 outputs
within 2 bf16 ulp or 1e-2 relative; an R-row call must write the same bytes as R one-row
calls.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import compare

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


def host_layer(d: dict) -> dict:
    return {k: synth.to_numpy_bits(v) for k, v in d.items()}


def check_case(dsm, d_dev, host, x_dev, k):
    """Router (exact up to permitted near-ties), weights, h (the first bf16 rounding point:
    exact or a budget of one-ulp flips), and y against the oracle's down projection and
    combine applied to the device's h."""
    layer = dsm.MoeLayer.from_dict(d_dev, k)
    R = x_dev.shape[0]
    ws = torch.empty(dsm.moe_workspace_size(layer, R), dtype=torch.uint8, device="cuda")
    y, idx, w = dsm.moe_verify_forward(layer, x_dev, workspace=ws)
    torch.cuda.synchronize()
    h_dev = synth.to_numpy_bits(dsm.moe_workspace_h(layer, R, ws))
    x = synth.to_numpy_bits(x_dev)
    y_b, idx_n, w_n = synth.to_numpy_bits(y), idx.cpu().numpy(), w.cpu().numpy()
    ref = oracle.moe_forward(host, x, k, want_h=True)
    rep = compare.routing_report(idx_n, ref["idx"], ref["s"])
    assert not rep["rows_bad"], rep
    if rep["rows_swapped"]:
        ref = oracle.moe_forward(host, x, k, idx_in=idx_n, want_h=True)
    assert compare.weights_ok(w_n, ref["w"])
    hb = compare.h_band_report(h_dev, ref["aux"])
    assert hb["ok"], hb
    y_from_h, yaux = oracle.moe_down_combine(host, k, ref["idx"], ref["w"], h_dev, want_aux=True)
    yr = compare.y_band_report(y_b, y_from_h, yaux)
    assert yr["ok"], yr
    yr["vs_full_oracle"] = compare.y_report(y_b, ref["y"])
    yr["h"] = compare.h_report(h_dev, ref["h"])
    return yr


def make(shape, R, seed, dev="cuda"):
    d = synth.moe_layer(shape, seed=seed, device=dev)
    x = synth.activations(R, shape.H, seed=seed, device=dev)
    return d, x


def test_tiny_config(dsm):
    shape = synth.TINY_MOE
    d, x = make(shape, 1, 0)
    yr = check_case(dsm, d, host_layer(d), x, shape.k)
    assert yr["vs_full_oracle"]["exact"] >= 0.95 * yr["n"]


@pytest.mark.parametrize("R", [1, 4, 6])
def test_ragged_multi_tile(dsm, R):
    # H = 34 blocks and I = 10 blocks: both end in a partial 4-block tile.
    shape = synth.MoeShape(H=1088, E=40, I=320, k=6)
    d, x = make(shape, R, 10 + R)
    check_case(dsm, d, host_layer(d), x, shape.k)


def test_all_experts_selected_and_top1(dsm):
    for shape in (synth.MoeShape(H=256, E=4, I=64, k=4), synth.MoeShape(H=256, E=9, I=128, k=1)):
        d, x = make(shape, 3, 21)
        check_case(dsm, d, host_layer(d), x, shape.k)


def test_large_hidden_chunks(dsm):
    # H > 4096 exercises the K loop over several 128-block chunks; I > 1024 the down chunks.
    shape = synth.MoeShape(H=8192, E=12, I=2048, k=2)
    d, x = make(shape, 2, 5)
    check_case(dsm, d, host_layer(d), x, shape.k)


@pytest.fixture(scope="module")
def verify_case(dsm):
    shape = synth.VERIFY_MOE
    d, x = make(shape, 6, 0)
    return shape, d, x


def test_verify_config_r6_matches_oracle(dsm, verify_case):
    shape, d, x = verify_case
    yr = check_case(dsm, d, host_layer(d), x, shape.k)
    assert yr["vs_full_oracle"]["exact"] >= 0.9 * yr["n"]
    assert yr["h"]["exact"] >= 0.99 * yr["h"]["n"]
    assert yr["h"]["worse"] <= 1e-3 * yr["h"]["n"]


def test_r_rows_equal_single_row_calls(dsm, verify_case):
    shape, d, x = verify_case
    layer = dsm.MoeLayer.from_dict(d, shape.k)
    y6, i6, w6 = dsm.moe_verify_forward(layer, x)
    for r in range(6):
        y1, i1, w1 = dsm.moe_verify_forward(layer, x[r:r + 1].contiguous())
        assert torch.equal(y1[0].view(torch.int16), y6[r].view(torch.int16)), r
        assert torch.equal(i1[0], i6[r])
        assert torch.equal(w1[0].view(torch.int32), w6[r].view(torch.int32))
    # a different mix of rows does not change a row's bytes either
    sub = x[[4, 1]].contiguous()
    y2, _, _ = dsm.moe_verify_forward(layer, sub)
    assert torch.equal(y2[0].view(torch.int16), y6[4].view(torch.int16))
    assert torch.equal(y2[1].view(torch.int16), y6[1].view(torch.int16))


def test_run_to_run_and_dirty_workspace(dsm, verify_case):
    shape, d, x = verify_case
    layer = dsm.MoeLayer.from_dict(d, shape.k)
    ws = torch.empty(dsm.moe_workspace_size(layer, 6), dtype=torch.uint8, device="cuda")
    ya, ia, _ = dsm.moe_verify_forward(layer, x, workspace=ws)
    ya = ya.clone()
    ws.fill_(0xA5)
    yb, ib, _ = dsm.moe_verify_forward(layer, x, workspace=ws)
    assert torch.equal(ya.view(torch.int16), yb.view(torch.int16))
    assert torch.equal(ia, ib)
    assert dsm.workspace_status(ws) == 0


def test_staging_limit_is_reported(dsm):
    # R * (2H + 64) bytes of verify rows must fit in shared memory beside the weight ring
    shape = synth.MoeShape(H=16384, E=2, I=64, k=1)
    d, x = make(shape, 6, 3)
    layer = dsm.MoeLayer.from_dict(d, shape.k)
    with pytest.raises(dsm.DsmoeError) as ei:
        dsm.moe_verify_forward(layer, x)
    assert ei.value.status == 2    # DS_ERR_UNSUPPORTED
    y, _, _ = dsm.moe_verify_forward(layer, x[:2].contiguous())   # R = 2 fits
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()


def test_gpu_validation_errors(dsm):
    shape = synth.TINY_MOE
    d, x = make(shape, 7, 1)
    layer = dsm.MoeLayer.from_dict(d, shape.k)
    with pytest.raises(dsm.DsmoeError):
        dsm.moe_verify_forward(layer, x)            # R = 7
    with pytest.raises(ValueError):
        dsm.moe_verify_forward(layer, x[:2].float())
