"""ctypes view of libdsmoe.so (declarations mirror include/dsmoe.h).

Loading fails loudly: there is no fallback implementation of any entry point.
"""
from __future__ import annotations

import ctypes as C
from pathlib import Path

LIB_PATH = Path(__file__).resolve().parent / "libdsmoe.so"

DS_OK = 0
DS_ERR_WORKSPACE = 3
STATUS_NAMES = {
    0: "DS_OK", 1: "DS_ERR_INVALID_ARG", 2: "DS_ERR_UNSUPPORTED", 3: "DS_ERR_WORKSPACE",
    4: "DS_ERR_CUDA", 5: "DS_ERR_TIMEOUT", 6: "DS_ERR_DEVICE_CHECK",
}

# Every symbol include/dsmoe.h declares.
EXPORTS = (
    "ds_moe_workspace_size", "ds_moe_verify_forward", "ds_select_workspace_size",
    "ds_select_blocks", "ds_workspace_status", "ds_status_string", "ds_version",
    "ds_moe_verify_forward_marked", "ds_select_blocks_marked", "ds_moe_workspace_h_offset",
    "ds_moe_verify_forward_noalloc", "ds_noalloc_status", "ds_q4_tiled_bytes", "ds_q4_tile",
    "ds_select_workspace_offset", "ds_verify_workspace_size", "ds_verify_greedy",
    "ds_verify_sample", "ds_q8_tiled_bytes", "ds_q8_tile", "ds_q8_workspace_size",
    "ds_q8_project", "ds_attn_workspace_size", "ds_sparse_attention",
)
SELECT_WS_PARTS = {"union": 0, "union_count": 1, "scores": 2, "key_norms": 3, "row_scales": 4}

DS_SELECT_CANONICAL_SCORES = 1
DS_SELECT_KEEP_WORKSPACE = 2
DS_NOALLOC_SCRATCH_BYTES = 4 << 20  # same value as the C header's macro


class DsQ4(C.Structure):
    _fields_ = [("qs", C.c_void_p), ("sc", C.c_void_p)]


class DsQ4Tiled(C.Structure):
    _fields_ = [("tiles", C.c_void_p)]


Q4_TILE_BYTES = 576   # 16 rows x 64 values: 512 bytes of nibbles + 64 bytes of scales
Q4_DOWN_GROUP = 16    # tile rows per group of the down matrices (same value as the header)


class DsQ8(C.Structure):
    _fields_ = [("qs", C.c_void_p), ("sc", C.c_void_p)]


class DsQ8Tiled(C.Structure):
    _fields_ = [("tiles", C.c_void_p)]


Q8_TILE_BYTES = 1088  # 16 rows x 64 int8 values + 32 fp16 scales


class DsMoeLayer(C.Structure):
    _fields_ = [
        ("hidden", C.c_int32), ("n_experts", C.c_int32), ("inter", C.c_int32),
        ("top_k", C.c_int32), ("router_w", C.c_void_p),
        ("gate", DsQ4Tiled), ("up", DsQ4Tiled), ("down", DsQ4Tiled),
        ("sh_gate", DsQ4Tiled), ("sh_up", DsQ4Tiled), ("sh_down", DsQ4Tiled),
    ]


class DsSelectArgs(C.Structure):
    _fields_ = [
        ("n_layers", C.c_int32), ("n_rows", C.c_int32), ("n_heads", C.c_int32),
        ("head_dim", C.c_int32), ("n_blocks", C.c_int32), ("top_k", C.c_int32),
        ("keys", C.c_void_p), ("key_layer_stride", C.c_int64),
        ("q", C.c_void_p), ("head_w", C.c_void_p),
        ("mask", C.c_void_p), ("limit", C.c_void_p), ("flags", C.c_int32),
    ]


class DsAttnArgs(C.Structure):
    _fields_ = [
        ("n_layers", C.c_int32), ("n_rows", C.c_int32), ("n_heads", C.c_int32),
        ("head_dim", C.c_int32), ("n_blocks", C.c_int32), ("block_tokens", C.c_int32),
        ("top_k", C.c_int32), ("q", C.c_void_p), ("k", C.c_void_p), ("v", C.c_void_p),
        ("kv_layer_stride", C.c_int64), ("sel", C.c_void_p),
    ]


class DsmoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what} failed: {STATUS_NAMES.get(status, status)}")


_lib = None


def load() -> C.CDLL:
    """Returns the loaded library; raises if it was not built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not LIB_PATH.exists():
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; "
            f"g.build()\"` (nvcc, sm_103a). There is no CPU fallback.")
    lib = C.CDLL(str(LIB_PATH))
    lib.ds_q4_tiled_bytes.argtypes = [C.c_int64, C.c_int32]
    lib.ds_q4_tiled_bytes.restype = C.c_size_t
    lib.ds_q4_tile.argtypes = [C.POINTER(DsQ4), C.c_int32, C.c_int64, C.c_int32, C.c_int32,
                               C.c_void_p, C.c_size_t, C.c_void_p]
    lib.ds_q4_tile.restype = C.c_int
    lib.ds_moe_workspace_size.argtypes = [C.POINTER(DsMoeLayer), C.c_int32]
    lib.ds_moe_workspace_size.restype = C.c_size_t
    lib.ds_moe_verify_forward.argtypes = [
        C.POINTER(DsMoeLayer), C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p,
        C.c_void_p, C.c_size_t, C.c_void_p]
    lib.ds_moe_verify_forward.restype = C.c_int
    lib.ds_moe_verify_forward_marked.argtypes = lib.ds_moe_verify_forward.argtypes + [C.c_void_p]
    lib.ds_moe_verify_forward_marked.restype = C.c_int
    lib.ds_moe_workspace_h_offset.argtypes = [C.POINTER(DsMoeLayer), C.c_int32]
    lib.ds_moe_workspace_h_offset.restype = C.c_size_t
    lib.ds_moe_verify_forward_noalloc.argtypes = [
        C.POINTER(DsMoeLayer), C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p,
        C.c_void_p]
    lib.ds_moe_verify_forward_noalloc.restype = C.c_int
    lib.ds_noalloc_status.argtypes = [C.c_void_p]
    lib.ds_noalloc_status.restype = C.c_int
    lib.ds_select_workspace_size.argtypes = [C.POINTER(DsSelectArgs)]
    lib.ds_select_workspace_size.restype = C.c_size_t
    lib.ds_select_workspace_offset.argtypes = [C.POINTER(DsSelectArgs), C.c_int32, C.c_int32]
    lib.ds_select_workspace_offset.restype = C.c_size_t
    lib.ds_select_blocks.argtypes = [
        C.POINTER(DsSelectArgs), C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
        C.c_size_t, C.c_void_p]
    lib.ds_select_blocks.restype = C.c_int
    lib.ds_select_blocks_marked.argtypes = lib.ds_select_blocks.argtypes + [C.c_void_p]
    lib.ds_select_blocks_marked.restype = C.c_int
    lib.ds_attn_workspace_size.argtypes = [C.POINTER(DsAttnArgs)]
    lib.ds_attn_workspace_size.restype = C.c_size_t
    lib.ds_sparse_attention.argtypes = [C.POINTER(DsAttnArgs), C.c_void_p, C.c_void_p,
                                        C.c_size_t, C.c_void_p]
    lib.ds_sparse_attention.restype = C.c_int
    lib.ds_q8_tiled_bytes.argtypes = [C.c_int64, C.c_int32]
    lib.ds_q8_tiled_bytes.restype = C.c_size_t
    lib.ds_q8_tile.argtypes = [C.POINTER(DsQ8), C.c_int64, C.c_int32, C.c_void_p, C.c_size_t,
                               C.c_void_p]
    lib.ds_q8_tile.restype = C.c_int
    lib.ds_q8_workspace_size.argtypes = []
    lib.ds_q8_workspace_size.restype = C.c_size_t
    lib.ds_q8_project.argtypes = [C.POINTER(DsQ8Tiled), C.c_int64, C.c_int32, C.c_void_p,
                                  C.c_int32, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]
    lib.ds_q8_project.restype = C.c_int
    lib.ds_verify_workspace_size.argtypes = [C.c_int32, C.c_int32, C.c_int32]
    lib.ds_verify_workspace_size.restype = C.c_size_t
    lib.ds_verify_greedy.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_void_p,
                                     C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]
    lib.ds_verify_greedy.restype = C.c_int
    lib.ds_verify_sample.argtypes = [C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_double,
                                     C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                     C.c_void_p, C.c_void_p, C.c_void_p, C.c_size_t, C.c_void_p]
    lib.ds_verify_sample.restype = C.c_int
    lib.ds_workspace_status.argtypes = [C.c_void_p, C.c_void_p]
    lib.ds_workspace_status.restype = C.c_int
    lib.ds_status_string.argtypes = [C.c_int]
    lib.ds_status_string.restype = C.c_char_p
    lib.ds_version.argtypes = []
    lib.ds_version.restype = C.c_char_p
    _lib = lib
    return lib
