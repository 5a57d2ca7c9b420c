"""GPU parity of ds_moe_verify_forward against the oracle (called through the C ABI).

Every case runs compare.moe_check: routing indices bit-exact (near-ties under 1e-5 may
swap, then the output is compared with the oracle re-run on the device's choice),
routing weights within 1e-5; h (the first bf16 rounding point) the rounding of a value
inside the derived fp32 accumulation band around the exact value, with at most 0.1% of
h elements rounded differently from the oracle; y inside the band of the oracle applied
to the device's own h and w; and y against the full oracle within 2 bf16 ulp or 1e-2
relative (near-zero clause for |y| < 1e-3 rms) for every element, except elements whose
deviation the device's own band-checked h and w decisions explain, at most 0.1% of them.
An R-row call must write the same bytes as R one-row calls.
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
    layer = dsm.MoeLayer.from_dict(d_dev, k)
    R = x_dev.shape[0]
    ws = torch.empty(dsm.moe_workspace_size(layer, R), dtype=torch.uint8, device="cuda")
    y, idx, w = dsm.moe_verify_forward(layer, x_dev, workspace=ws)
    torch.cuda.synchronize()
    assert dsm.workspace_status(ws) == 0
    h_dev = synth.to_numpy_bits(dsm.moe_workspace_h(layer, R, ws))
    rep = compare.moe_check(host, synth.to_numpy_bits(x_dev), k, synth.to_numpy_bits(y),
                            idx.cpu().numpy(), w.cpu().numpy(), h_dev)
    print({key: rep[key] for key in ("h", "y_vs_device_h", "y_vs_oracle")})
    assert rep["ok"], rep
    return rep


def make(shape, R, seed, dev="cuda"):
    d = synth.moe_layer(shape, seed=seed, device=dev)
    x = synth.activations(R, shape.H, seed=seed, device=dev)
    return d, x


def test_tiny_config(dsm):
    shape = synth.TINY_MOE
    d, x = make(shape, 1, 0)
    rep = check_case(dsm, d, host_layer(d), x, shape.k)
    assert rep["y_vs_oracle"]["explained"] == 0


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
    check_case(dsm, d, host_layer(d), x, shape.k)


@pytest.mark.parametrize("R,seed", [(1, 3), (2, 6), (4, 4), (6, 1), (6, 2)])
def test_verify_config_other_rows_and_seeds(dsm, R, seed):
    shape = synth.VERIFY_MOE
    d, x = make(shape, R, seed)
    check_case(dsm, d, host_layer(d), x, shape.k)


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


def test_largest_hidden_size(dsm):
    # hidden 16384 at R = 6: the verify rows' tensor-core fragments live in tensor memory
    # (16 K chunks' worth fill its 512 columns), so shared memory holds only the ring
    shape = synth.MoeShape(H=16384, E=4, I=64, k=2)
    d, x = make(shape, 6, 3)
    check_case(dsm, d, host_layer(d), x, shape.k)


def test_gpu_validation_errors(dsm):
    shape = synth.TINY_MOE
    d, x = make(shape, 7, 1)
    layer = dsm.MoeLayer.from_dict(d, shape.k)
    with pytest.raises(dsm.DsmoeError):
        dsm.moe_verify_forward(layer, x)            # R = 7
    with pytest.raises(ValueError):
        dsm.moe_verify_forward(layer, x[:2].float())
