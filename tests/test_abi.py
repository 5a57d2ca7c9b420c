"""The C-ABI library loads, exports every symbol include/dsmoe.h declares, and rejects bad
arguments on the host before anything reaches a GPU (no compute calls here)."""
import ctypes as C
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def lib():
    from q4_moe_speculative_gb300.build import build_library
    build_library()
    from q4_moe_speculative_gb300 import _native
    return _native.load()


def declared_functions():
    text = (ROOT / "include" / "dsmoe.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ds_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_api():
    names = declared_functions()
    for n in ("ds_moe_verify_forward", "ds_select_blocks", "ds_moe_workspace_size",
              "ds_select_workspace_size", "ds_workspace_status", "ds_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from q4_moe_speculative_gb300 import _native
    names = declared_functions()
    assert sorted(_native.EXPORTS) == names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    for code, name in {0: "DS_OK", 1: "DS_ERR_INVALID_ARG", 3: "DS_ERR_WORKSPACE",
                       5: "DS_ERR_TIMEOUT", 6: "DS_ERR_DEVICE_CHECK"}.items():
        assert lib.ds_status_string(code).decode() == name
    assert b"sm_103a" in lib.ds_version()


FAKE = 1 << 20  # a 256-aligned address that is never dereferenced: validation fails first


def fake_layer(H=4096, E=384, I=1024, k=8):
    from q4_moe_speculative_gb300 import _native as N
    q = N.DsQ4Tiled(FAKE)
    return N.DsMoeLayer(H, E, I, k, FAKE, q, q, q, q, q, q)


def test_moe_workspace_size_host_only(lib):
    st = fake_layer()
    s6 = lib.ds_moe_workspace_size(st, 6)
    s1 = lib.ds_moe_workspace_size(st, 1)
    assert s6 > s1 > 0
    # h [R][1+k][I] bf16 and fp32 partials [R][1+k][H] dominate
    assert s6 >= 6 * 9 * 1024 * 2 + 6 * 9 * 4096 * 4
    assert lib.ds_moe_workspace_size(st, 0) == 0
    assert lib.ds_moe_workspace_size(st, 7) == 0
    # sizes the call refuses (invalid, or valid but not run by this build) get no size
    assert lib.ds_moe_workspace_size(fake_layer(I=1056), 6) == 0
    assert lib.ds_moe_workspace_size(fake_layer(H=4010), 6) == 0


@pytest.mark.parametrize("mutate,R,expect", [
    (lambda s: None, 0, 1),
    (lambda s: None, 7, 1),
    (lambda s: setattr(s, "hidden", 4010), 6, 1),        # not a multiple of 32
    (lambda s: setattr(s, "inter", 1000), 6, 1),
    (lambda s: setattr(s, "inter", 1056), 6, 2),         # multiple of 32, not of 64
    (lambda s: setattr(s, "hidden", 4064), 6, 2),
    (lambda s: setattr(s.up, "tiles", FAKE + 8), 6, 1),  # tiles not 16-byte aligned
    (lambda s: setattr(s, "top_k", 0), 6, 1),
    (lambda s: setattr(s, "top_k", 17), 6, 1),
    (lambda s: setattr(s, "n_experts", 4), 6, 1),        # E < k
    (lambda s: setattr(s, "router_w", None), 6, 1),
    (lambda s: setattr(s.gate, "tiles", FAKE + 4), 6, 1),
    (lambda s: setattr(s.sh_down, "tiles", None), 6, 1),
])
def test_moe_forward_rejects_bad_arguments(lib, mutate, R, expect):
    st = fake_layer()
    mutate(st)
    r = lib.ds_moe_verify_forward(st, FAKE, R, FAKE, FAKE, FAKE, FAKE, 1 << 40, None)
    assert r == expect


def test_moe_forward_rejects_small_workspace(lib):
    st = fake_layer()
    need = lib.ds_moe_workspace_size(st, 6)
    assert lib.ds_moe_verify_forward(st, FAKE, 6, FAKE, FAKE, FAKE, FAKE, need - 1, None) == 3
    assert lib.ds_moe_verify_forward(st, FAKE, 6, FAKE, FAKE, FAKE, None, need, None) == 3
    assert lib.ds_moe_verify_forward(st, FAKE, 6, FAKE, FAKE, FAKE, FAKE + 16, need, None) == 3


def test_moe_forward_rejects_null_io(lib):
    st = fake_layer()
    assert lib.ds_moe_verify_forward(st, None, 6, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == 1
    assert lib.ds_moe_verify_forward(st, FAKE, 6, None, FAKE, FAKE, FAKE, 1 << 40, None) == 1
    assert lib.ds_moe_verify_forward(st, FAKE + 2, 6, FAKE, FAKE, FAKE, FAKE, 1 << 40, None) == 1


def fake_select(**kw):
    from q4_moe_speculative_gb300 import _native as N
    a = dict(n_layers=43, n_rows=6, n_heads=8, head_dim=128, n_blocks=75000, top_k=512,
             keys=FAKE, key_layer_stride=75000 * 128, q=FAKE, head_w=FAKE, mask=FAKE, limit=FAKE)
    a.update(kw)
    return N.DsSelectArgs(**a)


def test_select_workspace_size_host_only(lib):
    s = lib.ds_select_workspace_size(fake_select())
    LRN = 43 * 6 * 75000
    assert s >= LRN * 8  # compacted index + scores
    assert lib.ds_select_workspace_size(fake_select(head_dim=64)) == 0


@pytest.mark.parametrize("kw", [
    dict(head_dim=64), dict(n_rows=0), dict(n_rows=9), dict(n_heads=17), dict(n_blocks=0),
    dict(top_k=0), dict(top_k=4096), dict(key_layer_stride=100), dict(keys=FAKE + 8),
    dict(keys=None), dict(mask=None), dict(limit=None), dict(head_w=None), dict(q=None),
    dict(flags=4), dict(flags=-1),
])
def test_select_rejects_bad_arguments(lib, kw):
    a = fake_select(**kw)
    assert lib.ds_select_blocks(a, FAKE, FAKE, None, None, FAKE, 1 << 40, None) == 1


def test_select_rejects_half_compacted_outputs_and_small_workspace(lib):
    a = fake_select()
    assert lib.ds_select_blocks(a, FAKE, FAKE, FAKE, None, FAKE, 1 << 40, None) == 1
    need = lib.ds_select_workspace_size(a)
    assert lib.ds_select_blocks(a, FAKE, FAKE, None, None, FAKE, need - 1, None) == 3


def test_status_query_rejects_null(lib):
    assert lib.ds_workspace_status(None, None) == 1


def test_noalloc_scratch_limit_matches_header():
    from q4_moe_speculative_gb300 import _native as N
    text = (ROOT / "include" / "dsmoe.h").read_text()
    m = re.search(r"#define DS_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m, "DS_NOALLOC_SCRATCH_BYTES not found"
    assert int(m.group(1)) << int(m.group(2)) == N.DS_NOALLOC_SCRATCH_BYTES


def test_noalloc_rejects_on_the_host(lib):
    from q4_moe_speculative_gb300 import _native as N
    # The verify layer fits the scratch at every R; a larger one is refused before any
    # CUDA call (this machine may have no GPU at all).
    for R in range(1, 7):
        assert 0 < lib.ds_moe_workspace_size(fake_layer(), R) <= N.DS_NOALLOC_SCRATCH_BYTES
    big = fake_layer(H=16384, E=64, I=1024, k=16)
    assert lib.ds_moe_workspace_size(big, 6) > N.DS_NOALLOC_SCRATCH_BYTES
    assert lib.ds_moe_verify_forward_noalloc(big, FAKE, 6, FAKE, FAKE, FAKE, None) == 3
    assert lib.ds_moe_verify_forward_noalloc(fake_layer(), FAKE, 0, FAKE, FAKE, FAKE, None) == 1
    assert lib.ds_moe_verify_forward_noalloc(fake_layer(), FAKE, 7, FAKE, FAKE, FAKE, None) == 1
    assert lib.ds_moe_verify_forward_noalloc(fake_layer(I=1056), FAKE, 6, FAKE, FAKE, FAKE,
                                             None) == 2


def test_noalloc_status_without_a_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; the GPU tests cover the status query")
    assert lib.ds_noalloc_status(None) == 4   # DS_ERR_CUDA: no device to query
    assert lib.ds_moe_verify_forward_noalloc(None, FAKE, 1, FAKE, FAKE, FAKE, None) == 1


def test_q4_tiled_bytes_and_tile_argument_checks(lib):
    from q4_moe_speculative_gb300 import _native as N
    assert lib.ds_q4_tiled_bytes(1024, 4096) == 1024 * 4096 * 9 // 16
    assert lib.ds_q4_tiled_bytes(384 * 1024, 4096) == 384 * 1024 * 4096 * 9 // 16
    for rows, K in ((1000, 4096), (1024, 4064), (0, 64), (16, 0), (-16, 64)):
        assert lib.ds_q4_tiled_bytes(rows, K) == 0
    src = N.DsQ4(FAKE, FAKE)
    need = lib.ds_q4_tiled_bytes(64, 256)
    assert lib.ds_q4_tile(src, 1, 64, 256, 1, FAKE, need - 1, None) == 3
    assert lib.ds_q4_tile(src, 2, 64, 256, 16, FAKE, 2 * need - 1, None) == 3
    assert lib.ds_q4_tile(src, 1, 60, 256, 1, FAKE, 1 << 30, None) == 1
    assert lib.ds_q4_tile(src, 1, 64, 256, 1, FAKE + 8, need, None) == 1      # dst not 16-aligned
    assert lib.ds_q4_tile(N.DsQ4(FAKE + 2, FAKE), 1, 64, 256, 1, FAKE, need, None) == 1
    assert lib.ds_q4_tile(N.DsQ4(FAKE, None), 1, 64, 256, 1, FAKE, need, None) == 1
    assert lib.ds_q4_tile(None, 1, 64, 256, 1, FAKE, need, None) == 1
    assert lib.ds_q4_tile(src, 0, 64, 256, 1, FAKE, need, None) == 1          # no matrices
    assert lib.ds_q4_tile(src, 1, 64, 256, 0, FAKE, need, None) == 1          # group 0


def test_header_group_constant_matches_binding():
    from q4_moe_speculative_gb300 import _native as N
    text = (ROOT / "include" / "dsmoe.h").read_text()
    m = re.search(r"#define DS_Q4_DOWN_GROUP (\d+)", text)
    assert m and int(m.group(1)) == N.Q4_DOWN_GROUP


def test_verify_workspace_size_host_only(lib):
    s = lib.ds_verify_workspace_size(8, 6, 129280)
    assert s > 0 and s % 256 == 0
    assert lib.ds_verify_workspace_size(16, 6, 129280) > s
    for B, R, V in ((0, 6, 100), (4097, 6, 100), (1, 0, 100), (1, 17, 100), (1, 6, 0),
                    (1, 6, (1 << 24) + 1)):
        assert lib.ds_verify_workspace_size(B, R, V) == 0


@pytest.mark.parametrize("T", [0.0, -0.5, float("inf"), float("nan")])
def test_verify_sample_rejects_temperature(lib, T):
    ws = lib.ds_verify_workspace_size(1, 2, 100)
    st = lib.ds_verify_sample(FAKE, 1, 2, 100, T, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws,
                              None)
    assert st == 1


def test_verify_rejects_bad_arguments_on_the_host(lib):
    ws = lib.ds_verify_workspace_size(2, 6, 1000)
    g = lib.ds_verify_greedy
    assert g(None, 2, 6, 1000, FAKE, FAKE, FAKE, FAKE, ws, None) == 1      # logits
    assert g(FAKE, 2, 6, 1000, None, FAKE, FAKE, FAKE, ws, None) == 1      # drafts, R > 1
    assert g(FAKE, 2, 6, 1000, FAKE, None, FAKE, FAKE, ws, None) == 1      # out
    assert g(FAKE, 2, 6, 1000, FAKE, FAKE, None, FAKE, ws, None) == 1      # n_out
    assert g(FAKE, 0, 6, 1000, FAKE, FAKE, FAKE, FAKE, ws, None) == 1      # B
    assert g(FAKE, 2, 17, 1000, FAKE, FAKE, FAKE, FAKE, ws, None) == 1     # R
    assert g(FAKE, 2, 6, 1000, FAKE, FAKE, FAKE, FAKE, ws - 1, None) == 3  # workspace size
    assert g(FAKE, 2, 6, 1000, FAKE, FAKE, FAKE, FAKE + 8, ws, None) == 3  # alignment
    assert g(FAKE, 2, 6, 1000, FAKE, FAKE, FAKE, None, ws, None) == 3
    s = lib.ds_verify_sample
    assert s(FAKE, 2, 6, 1000, 1.0, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws, None) == 1
    assert s(FAKE, 2, 6, 1000, 1.0, FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, ws, None) == 1
    assert s(FAKE, 2, 6, 1000, 1.0, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, ws, None) == 1
    assert s(FAKE, 2, 6, 1000, 1.0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws - 1,
             None) == 3


def test_q8_sizes_and_argument_checks(lib):
    from q4_moe_speculative_gb300 import _native as N
    assert lib.ds_q8_tiled_bytes(4096, 4096) == 256 * 64 * 1088
    for rows, K in ((0, 64), (15, 64), (16, 32), (16, 0), (16, 96), ((1 << 24) + 16, 64)):
        assert lib.ds_q8_tiled_bytes(rows, K) == 0
    assert lib.ds_q8_workspace_size() == 256
    src = N.DsQ8(FAKE, FAKE)
    n = lib.ds_q8_tiled_bytes(64, 512)
    assert lib.ds_q8_tile(None, 64, 512, FAKE, n, None) == 1
    assert lib.ds_q8_tile(src, 60, 512, FAKE, n, None) == 1
    assert lib.ds_q8_tile(src, 64, 480, FAKE, n, None) == 1      # K % 64
    assert lib.ds_q8_tile(src, 64, 512, FAKE + 4, n, None) == 1  # alignment
    assert lib.ds_q8_tile(src, 64, 512, FAKE, n - 1, None) == 3
    w = N.DsQ8Tiled(FAKE)
    p = lib.ds_q8_project
    assert p(None, 64, 512, FAKE, 6, FAKE, FAKE, 256, None) == 1
    assert p(w, 64, 512, None, 6, FAKE, FAKE, 256, None) == 1
    assert p(w, 64, 512, FAKE, 0, FAKE, FAKE, 256, None) == 1
    assert p(w, 64, 512, FAKE, 9, FAKE, FAKE, 256, None) == 1
    assert p(w, 48, 512, FAKE, 6, FAKE + 8, FAKE, 256, None) == 1   # x alignment
    assert p(w, 64, 544, FAKE, 6, FAKE, FAKE, 256, None) == 2       # K % 512: unsupported
    assert p(w, 64, 1056, FAKE, 6, FAKE, FAKE, 256, None) == 2


def test_attention_argument_checks(lib):
    from q4_moe_speculative_gb300 import _native as N

    def args(**kw):
        d = dict(n_layers=2, n_rows=6, n_heads=16, head_dim=128, n_blocks=2048, block_tokens=4,
                 top_k=512, q=FAKE, k=FAKE, v=FAKE, kv_layer_stride=2048 * 4 * 128, sel=FAKE)
        d.update(kw)
        return N.DsAttnArgs(*[d[f] for f, _ in N.DsAttnArgs._fields_])

    good = args()
    ws = lib.ds_attn_workspace_size(good)
    assert ws > 0 and ws % 256 == 0
    for kw, code in (({"n_rows": 9}, 1), ({"n_heads": 17}, 1), ({"block_tokens": 3}, 1),
                     ({"top_k": 2049}, 1), ({"head_dim": 64}, 2), ({"q": None}, 1),
                     ({"k": FAKE + 8}, 1), ({"kv_layer_stride": 100}, 1), ({"n_blocks": 0}, 1)):
        a = args(**kw)
        assert lib.ds_attn_workspace_size(a) == 0
        assert lib.ds_sparse_attention(a, FAKE, FAKE, ws, None) == code, kw
    assert lib.ds_sparse_attention(good, None, FAKE, ws, None) == 1
    assert lib.ds_sparse_attention(good, FAKE, FAKE, ws - 1, None) == 3
    assert lib.ds_sparse_attention(good, FAKE, FAKE + 16, ws, None) == 3
