"""ds_moe_verify_forward_noalloc (the verify step on the library's own scratch array)
against ds_moe_verify_forward with a caller workspace, both called through the C ABI.

Two no-alloc calls in a row with different inputs and row counts (the second runs on the
scratch the first left dirty), each compared with the workspace entry point on the same
inputs. Both entry points run the same deterministic kernels, so every output must be
byte-identical. The device status of the scratch must read DS_OK after each call, and the
second call must not change the device's free memory. This file is named to be collected
last, and passes alone in a fresh process as well.
"""
import numpy as np
import pytest
import torch

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


def outputs(R, H, k):
    return (torch.empty((R, H), dtype=torch.bfloat16, device="cuda"),
            torch.full((R, k), -7, dtype=torch.int32, device="cuda"),
            torch.full((R, k), float("nan"), dtype=torch.float32, device="cuda"))


def assert_same_bytes(got, want):
    y, idx, w = (t.cpu() for t in got)
    y_ref, idx_ref, w_ref = (t.cpu() for t in want)
    assert torch.equal(idx, idx_ref)
    assert torch.equal(w.view(torch.int32), w_ref.view(torch.int32))
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))


@pytest.mark.parametrize("shape", [synth.VERIFY_MOE, synth.TINY_MOE], ids=["verify", "tiny"])
def test_two_calls_in_a_row_match_the_workspace_entry_point(dsm, shape):
    d = synth.moe_layer(shape, seed=31, device="cuda")
    layer = dsm.MoeLayer.from_dict(d, shape.k)
    rows = (6, 3)
    xs = [synth.activations(R, shape.H, seed=40 + R, device="cuda") for R in rows]
    outs = [outputs(R, shape.H, shape.k) for R in rows]

    dsm.moe_verify_forward_noalloc(layer, xs[0], *outs[0])
    assert dsm.noalloc_status() == 0
    free_before = torch.cuda.mem_get_info()[0]
    dsm.moe_verify_forward_noalloc(layer, xs[1], *outs[1])
    assert dsm.noalloc_status() == 0
    assert torch.cuda.mem_get_info()[0] == free_before

    for x, got in zip(xs, outs):
        want = dsm.moe_verify_forward(layer, x)
        torch.cuda.synchronize()
        assert_same_bytes(got, want)


def test_oversized_layer_is_refused_with_the_limit(dsm):
    shape = synth.MoeShape(H=16384, E=16, I=64, k=16)
    d = synth.moe_layer(shape, seed=5, device="cuda")
    layer = dsm.MoeLayer.from_dict(d, shape.k)
    assert dsm.moe_workspace_size(layer, 6) > dsm._native.DS_NOALLOC_SCRATCH_BYTES
    x = synth.activations(6, shape.H, seed=5, device="cuda")
    y, idx, w = outputs(6, shape.H, shape.k)
    with pytest.raises(RuntimeError, match="scratch"):
        dsm.moe_verify_forward_noalloc(layer, x, y, idx, w)
    assert torch.all(idx.cpu() == -7)  # nothing ran
    assert np.isnan(w.cpu().numpy()).all()
