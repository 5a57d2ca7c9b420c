"""ds_q4_tile (planar Q4 -> the tile-major form the MoE kernels stream) against the layout
definition in include/dsmoe.h, restated here with numpy index arithmetic: every output
byte must match. Called through the C ABI."""
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


def expected_tiles(qs: np.ndarray, sc: np.ndarray, G: int = 1) -> np.ndarray:
    """qs uint8 [rows, K/2], sc uint16 [rows, K/32] of ONE matrix -> uint8 [rows/16 * K/64,
    576], tiles at the positions the grouped order gives them."""
    rows, K = qs.shape[0], qs.shape[1] * 2
    T, TR = K // 64, rows // 16
    words = np.ascontiguousarray(qs).view("<u4").reshape(rows, K // 32, 4)  # [row][block][w]
    t, u, L = np.meshgrid(np.arange(TR), np.arange(T), np.arange(32), indexing="ij")
    g, w = L // 4, L % 4
    r0, r1 = 16 * t + g, 16 * t + g + 8
    nib = np.stack([words[r0, 2 * u, w], words[r1, 2 * u, w],
                    words[r0, 2 * u + 1, w], words[r1, 2 * u + 1, w]], axis=-1)   # [t,u,L,4]
    t8, u8, g8 = np.meshgrid(np.arange(TR), np.arange(T), np.arange(8), indexing="ij")
    s0, s1 = 16 * t8 + g8, 16 * t8 + g8 + 8
    scl = np.stack([sc[s0, 2 * u8], sc[s1, 2 * u8], sc[s0, 2 * u8 + 1], sc[s1, 2 * u8 + 1]],
                   axis=-1).astype("<u2")                                        # [t,u,8,4]
    tiles = np.zeros((TR, T, 576), np.uint8)
    tiles[:, :, :512] = nib.astype("<u4").view(np.uint8).reshape(TR, T, 512)
    tiles[:, :, 512:] = scl.view(np.uint8).reshape(TR, T, 64)
    out = np.zeros((TR * T, 576), np.uint8)
    for tt in range(TR):                 # the grouped order, as the header states it
        g0 = tt - tt % G
        n = min(G, TR - g0)
        for uu in range(T):
            out[g0 * T + uu * n + tt % G] = tiles[tt, uu]
    return out


@pytest.mark.parametrize("lead,rows,K,G", [((), 16, 64, 1), ((), 48, 320, 1), ((3,), 64, 1088, 1),
                                           ((5,), 1024, 4096, 1), ((2,), 4096, 1024, 16),
                                           ((3,), 1088, 320, 16), ((), 80, 128, 4)])
def test_tile_bytes_match_the_layout_definition(dsm, lead, rows, K, G):
    g = torch.Generator(device="cuda")
    g.manual_seed(rows * 7 + K + G)
    qs, sc = synth.q4_matrix(lead, rows, K, g, "cuda")
    tiles = dsm.q4_tile(qs, sc, G)
    torch.cuda.synchronize()
    n_mats = int(np.prod(lead)) if lead else 1
    got = tiles.cpu().numpy().reshape(n_mats, -1, 576)
    qs_h = qs.cpu().numpy().reshape(n_mats, rows, K // 2)
    sc_h = synth.to_numpy_bits(sc).reshape(n_mats, rows, K // 32)
    for m in range(n_mats):
        assert np.array_equal(got[m], expected_tiles(qs_h[m], sc_h[m], G)), m


def test_tile_preserves_every_byte(dsm):
    # a permutation of bytes: the multiset of nibble bytes and of scales is unchanged
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    qs, sc = synth.q4_matrix((), 256, 512, g, "cuda")
    tiles = dsm.q4_tile(qs, sc).cpu().numpy().reshape(-1, 576)
    assert np.array_equal(np.sort(tiles[:, :512].reshape(-1)), np.sort(qs.cpu().numpy().reshape(-1)))
    assert np.array_equal(np.sort(tiles[:, 512:].reshape(-1).view("<u2")),
                          np.sort(synth.to_numpy_bits(sc).reshape(-1)))
