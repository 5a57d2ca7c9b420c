"""GB300-native speculative-verify Q4 MoE layer and compressed-attention block selection.

Thin Python binding over libdsmoe.so (include/dsmoe.h). Every step of the computation runs
in the library's CUDA kernels; this module only checks tensors and passes pointers, sizes
and the current CUDA stream. PyTorch provides device memory and streams.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _native as N

__all__ = [
    "MoeLayer", "q4_tile", "moe_workspace_size", "moe_verify_forward", "select_workspace_size",
    "select_blocks", "workspace_status", "version", "DsmoeError", "verify_greedy",
    "verify_sample", "q8_tile", "q8_project", "sparse_attention",
]

DsmoeError = N.DsmoeError


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple | None = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype} (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)} (got {tuple(t.shape)})")


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def _check(status: int, what: str):
    if status != N.DS_OK:
        raise N.DsmoeError(status, what)


def q4_tile(qs: torch.Tensor, sc: torch.Tensor, group: int = 1, stream=None) -> torch.Tensor:
    """Tile-major form (include/dsmoe.h) of a planar Q4 matrix or expert stack, with tile
    rows in groups of `group`: qs uint8 [..., rows, K/2], sc fp16 [..., rows, K/32] ->
    uint8 [..., rows/16, K/64, 576] (the tile order inside each matrix is the grouped one),
    written on the device by ds_q4_tile (a rearrangement of bytes, done once at load)."""
    lib = N.load()
    _need(qs, "qs", torch.uint8)
    _need(sc, "sc", torch.float16)
    lead, rows, K = tuple(qs.shape[:-2]), qs.shape[-2], qs.shape[-1] * 2
    if tuple(sc.shape) != lead + (rows, K // 32):
        raise ValueError(f"sc must have shape {lead + (rows, K // 32)} (got {tuple(sc.shape)})")
    n_mats = 1
    for n in lead:
        n_mats *= n
    if rows % 16 or K % 64:
        raise ValueError(f"tile-major Q4 needs rows % 16 == 0 and K % 64 == 0 (got {rows}, {K})")
    out = torch.empty(lead + (rows // 16, K // 64, N.Q4_TILE_BYTES), dtype=torch.uint8,
                      device=qs.device)
    src = N.DsQ4(_ptr(qs), _ptr(sc))
    _check(lib.ds_q4_tile(src, n_mats, rows, K, group, _ptr(out), out.numel(), _stream(stream)),
           "ds_q4_tile")
    return out


def q8_tile(qs: torch.Tensor, sc: torch.Tensor, stream=None) -> torch.Tensor:
    """Tile-major form (include/dsmoe.h) of a planar Q8 matrix: qs int8 [rows, K], sc fp16
    [rows, K/32] -> uint8 [rows/16, K/64, 1088], written on the device by ds_q8_tile."""
    lib = N.load()
    _need(qs, "qs", torch.int8)
    rows, K = qs.shape
    _need(sc, "sc", torch.float16, (rows, K // 32))
    out = torch.empty((rows // 16, K // 64, N.Q8_TILE_BYTES), dtype=torch.uint8,
                      device=qs.device)
    src = N.DsQ8(_ptr(qs), _ptr(sc))
    _check(lib.ds_q8_tile(src, rows, K, _ptr(out), out.numel(), _stream(stream)), "ds_q8_tile")
    return out


def q8_project(tiles: torch.Tensor, x: torch.Tensor, *, y=None, workspace=None, stream=None):
    """R verify rows through one tile-major Q8 matrix: tiles uint8 [rows/16, K/64, 1088],
    x bf16 [R, K] -> y bf16 [R, rows] (ds_q8_project)."""
    lib = N.load()
    _need(tiles, "tiles", torch.uint8)
    _need(x, "x", torch.bfloat16)
    rows, K = tiles.shape[0] * 16, tiles.shape[1] * 64
    R = x.shape[0]
    if x.shape[1] != K:
        raise ValueError(f"x must be [R, {K}] (got {tuple(x.shape)})")
    y = torch.empty((R, rows), dtype=torch.bfloat16, device=x.device) if y is None else y
    _need(y, "y", torch.bfloat16, (R, rows))
    if workspace is None:
        workspace = torch.empty(lib.ds_q8_workspace_size(), dtype=torch.uint8, device=x.device)
    w = N.DsQ8Tiled(_ptr(tiles))
    _check(lib.ds_q8_project(w, rows, K, _ptr(x), R, _ptr(y), _ptr(workspace),
                             workspace.numel(), _stream(stream)), "ds_q8_project")
    return y


@dataclass
class MoeLayer:
    """One MoE layer on the device (include/dsmoe.h): router_w bf16 [E,H]; routed gate/up
    uint8 tiles [E, I/16, H/64, 576] (groups of 1), routed down [E, H/16, I/64, 576] (groups of
    16 tile rows); the shared expert the same without the E axis. Built from planar weights
    with `from_dict`."""
    router_w: torch.Tensor
    gate: torch.Tensor
    up: torch.Tensor
    down: torch.Tensor
    sh_gate: torch.Tensor
    sh_up: torch.Tensor
    sh_down: torch.Tensor
    top_k: int

    @property
    def hidden(self) -> int:
        return self.router_w.shape[1]

    @property
    def n_experts(self) -> int:
        return self.router_w.shape[0]

    @property
    def inter(self) -> int:
        return self.gate.shape[1] * 16

    def validate(self):
        E, H, I = self.n_experts, self.hidden, self.inter
        T = N.Q4_TILE_BYTES
        _need(self.router_w, "router_w", torch.bfloat16, (E, H))
        for nm, rows, K, stack in (("gate", I, H, True), ("up", I, H, True), ("down", H, I, True),
                                   ("sh_gate", I, H, False), ("sh_up", I, H, False),
                                   ("sh_down", H, I, False)):
            lead = (E,) if stack else ()
            _need(getattr(self, nm), nm, torch.uint8, lead + (rows // 16, K // 64, T))

    def struct(self) -> N.DsMoeLayer:
        t = lambda a: N.DsQ4Tiled(_ptr(a))  # noqa: E731
        return N.DsMoeLayer(
            self.hidden, self.n_experts, self.inter, self.top_k, _ptr(self.router_w),
            t(self.gate), t(self.up), t(self.down), t(self.sh_gate), t(self.sh_up),
            t(self.sh_down))

    @staticmethod
    def from_dict(d: dict, top_k: int) -> "MoeLayer":
        """From planar device tensors (router_w, and qs/sc of gate, up, down, sh_gate, sh_up,
        sh_down): the Q4 matrices are converted to the tile-major form on the device."""
        mats = {nm: q4_tile(d[nm + "_qs"], d[nm + "_sc"],
                            N.Q4_DOWN_GROUP if nm.endswith("down") else 1)
                for nm in ("gate", "up", "down", "sh_gate", "sh_up", "sh_down")}
        return MoeLayer(router_w=d["router_w"], **mats, top_k=top_k)


def version() -> str:
    return N.load().ds_version().decode()


def moe_workspace_size(layer: MoeLayer, R: int) -> int:
    st = layer.struct()
    return int(N.load().ds_moe_workspace_size(st, R))


def moe_verify_forward(layer: MoeLayer, x: torch.Tensor, *, y=None, topk_idx=None, topk_w=None,
                       workspace=None, stream=None, validate: bool = True):
    """One verify step of one MoE layer for R = x.shape[0] rows (1..6).
    Returns (y bf16 [R,H], topk_idx int32 [R,k], topk_w fp32 [R,k])."""
    lib = N.load()
    R, H = x.shape
    k = layer.top_k
    if validate:
        layer.validate()
        _need(x, "x", torch.bfloat16, (R, layer.hidden))
    dev = x.device
    y = torch.empty((R, H), dtype=torch.bfloat16, device=dev) if y is None else y
    topk_idx = torch.empty((R, k), dtype=torch.int32, device=dev) if topk_idx is None else topk_idx
    topk_w = torch.empty((R, k), dtype=torch.float32, device=dev) if topk_w is None else topk_w
    if validate:
        _need(y, "y", torch.bfloat16, (R, H))
        _need(topk_idx, "topk_idx", torch.int32, (R, k))
        _need(topk_w, "topk_w", torch.float32, (R, k))
    st = layer.struct()
    if workspace is None:
        workspace = torch.empty(int(lib.ds_moe_workspace_size(st, R)), dtype=torch.uint8, device=dev)
    status = lib.ds_moe_verify_forward(st, _ptr(x), R, _ptr(y), _ptr(topk_idx), _ptr(topk_w),
                                       _ptr(workspace), workspace.numel(), _stream(stream))
    _check(status, "ds_moe_verify_forward")
    return y, topk_idx, topk_w


def moe_verify_forward_noalloc(layer: MoeLayer, x: torch.Tensor, y: torch.Tensor,
                               topk_idx: torch.Tensor, topk_w: torch.Tensor, *, stream=None):
    """moe_verify_forward on the library's own per-device scratch array: no workspace and
    no allocation in the call (every output is the caller's). Calls that overlap on the
    GPU share the scratch and race. Raises when the layer needs more scratch than
    DS_NOALLOC_SCRATCH_BYTES."""
    lib = N.load()
    R, H = x.shape
    k = layer.top_k
    layer.validate()
    _need(x, "x", torch.bfloat16, (R, layer.hidden))
    _need(y, "y", torch.bfloat16, (R, H))
    _need(topk_idx, "topk_idx", torch.int32, (R, k))
    _need(topk_w, "topk_w", torch.float32, (R, k))
    st = layer.struct()
    status = lib.ds_moe_verify_forward_noalloc(st, _ptr(x), R, _ptr(y), _ptr(topk_idx),
                                               _ptr(topk_w), _stream(stream))
    if status == N.DS_ERR_WORKSPACE:
        need = int(lib.ds_moe_workspace_size(st, R))
        raise RuntimeError(f"ds_moe_verify_forward_noalloc: the layer needs {need} bytes of "
                           f"scratch at R={R}; the library holds {N.DS_NOALLOC_SCRATCH_BYTES}")
    _check(status, "ds_moe_verify_forward_noalloc")
    return y, topk_idx, topk_w


def _select_struct(keys, q, head_w, mask, limit, top_k, key_layer_stride=None,
                   canonical: bool = False, keep_workspace: bool = False) -> N.DsSelectArgs:
    L, Nb, D = keys.shape
    _, R, Hh, _ = q.shape
    stride = keys.stride(0) if key_layer_stride is None else key_layer_stride
    flags = (N.DS_SELECT_CANONICAL_SCORES if canonical else 0) | \
        (N.DS_SELECT_KEEP_WORKSPACE if keep_workspace else 0)
    return N.DsSelectArgs(L, R, Hh, D, Nb, top_k, _ptr(keys), stride, _ptr(q), _ptr(head_w),
                          _ptr(mask), _ptr(limit), flags)


def select_workspace_size(keys, q, head_w, mask, limit, top_k: int) -> int:
    return int(N.load().ds_select_workspace_size(_select_struct(keys, q, head_w, mask, limit, top_k)))


def select_blocks(keys, q, head_w, mask, limit, top_k: int = 512, *, sel=None, nsel=None,
                  cidx=None, ccount=None, want_compacted: bool = False, workspace=None,
                  stream=None, validate: bool = True, canonical: bool = False,
                  keep_workspace: bool = False):
    """Block selection for L layers x R rows.
    keys bf16 [L,N,128]; q bf16 [L,R,Hh,128]; head_w fp32 [L,R,Hh]; mask int32 [L,R,ceil(N/32)]
    (bit patterns); limit int32 [L,R]. Returns (sel [L,R,top_k], nsel [L,R], cidx, ccount),
    the last two None unless want_compacted or passed in. canonical=True scores every admitted
    block in the canonical order on CUDA cores (same selection, slower); keep_workspace=True
    leaves the scores, key norms and union lists in `workspace` for select_workspace_views."""
    lib = N.load()
    L, Nb, D = keys.shape
    R, Hh = q.shape[1], q.shape[2]
    W = (Nb + 31) // 32
    if validate:
        _need(keys, "keys", torch.bfloat16, (L, Nb, D))
        _need(q, "q", torch.bfloat16, (L, R, Hh, D))
        _need(head_w, "head_w", torch.float32, (L, R, Hh))
        _need(mask, "mask", torch.int32, (L, R, W))
        _need(limit, "limit", torch.int32, (L, R))
    dev = keys.device
    sel = torch.empty((L, R, top_k), dtype=torch.int32, device=dev) if sel is None else sel
    nsel = torch.empty((L, R), dtype=torch.int32, device=dev) if nsel is None else nsel
    if want_compacted and cidx is None:
        cidx = torch.empty((L, R, Nb), dtype=torch.int32, device=dev)
        ccount = torch.empty((L, R), dtype=torch.int32, device=dev)
    args = _select_struct(keys, q, head_w, mask, limit, top_k, canonical=canonical,
                          keep_workspace=keep_workspace)
    if workspace is None:
        workspace = torch.empty(int(lib.ds_select_workspace_size(args)), dtype=torch.uint8, device=dev)
    status = lib.ds_select_blocks(args, _ptr(sel), _ptr(nsel), _ptr(cidx), _ptr(ccount),
                                  _ptr(workspace), workspace.numel(), _stream(stream))
    _check(status, "ds_select_blocks")
    return sel, nsel, cidx, ccount


def select_workspace_views(keys, q, head_w, mask, limit, top_k: int, workspace: torch.Tensor,
                           with_compacted: bool = False) -> dict:
    """Views of what a completed tensor-core-mode select call with keep_workspace=True left
    in `workspace`
    (include/dsmoe.h): union [L,N] int32 and union_count [L]; scores [L,R,NS] fp32 by union
    entry (-inf where the row does not admit it); key_norms [L,NS]; row_scales [L,R]."""
    lib = N.load()
    L, Nb, _ = keys.shape
    R = q.shape[1]
    NS = (Nb + 31) & ~31
    args = _select_struct(keys, q, head_w, mask, limit, top_k)
    shapes = {"union": ((L, Nb), torch.int32), "union_count": ((L,), torch.int32),
              "scores": ((L, R, NS), torch.float32), "key_norms": ((L, NS), torch.float32),
              "row_scales": ((L, R), torch.float32)}
    out = {}
    for name, (shape, dt) in shapes.items():
        off = int(lib.ds_select_workspace_offset(args, 1 if with_compacted else 0,
                                                 N.SELECT_WS_PARTS[name]))
        n = 1
        for d in shape:
            n *= d
        out[name] = workspace[off:off + 4 * n].view(dt).view(shape)
    return out


# position of value v (0..7) of a group of 8 in the workspace's h: v0, v4, v1, v5, ...
_H_PAIR_POS = (0, 2, 4, 6, 1, 3, 5, 7)


def moe_workspace_h(layer: MoeLayer, R: int, workspace: torch.Tensor) -> torch.Tensor:
    """The bf16 SwiGLU activations h [R, 1+k, I] that the last call left in `workspace`
    (slot 0 = shared expert, slot j+1 = the row's rank-j expert), in natural order (the
    workspace keeps each group of 8 values in tensor-core operand order)."""
    off = int(N.load().ds_moe_workspace_h_offset(layer.struct(), R))
    n = R * (1 + layer.top_k) * layer.inter
    h = workspace[off: off + 2 * n].view(torch.bfloat16).view(R, 1 + layer.top_k, layer.inter)
    pos = torch.tensor(_H_PAIR_POS, device=h.device)
    idx = (torch.arange(layer.inter, device=h.device) & ~7) + pos[torch.arange(layer.inter, device=h.device) & 7]
    return h[..., idx]


def _verify_common(logits, draft, out, n_out, workspace):
    if logits.dim() != 3:
        raise ValueError("logits must be [B][R][V]")
    _need(logits, "logits", torch.float32)
    B, R, V = logits.shape
    if R > 1:
        _need(draft, "draft", torch.int32, (B, R - 1))
    dev = logits.device
    out = torch.empty((B, R), dtype=torch.int32, device=dev) if out is None else out
    n_out = torch.empty((B,), dtype=torch.int32, device=dev) if n_out is None else n_out
    _need(out, "out", torch.int32, (B, R))
    _need(n_out, "n_out", torch.int32, (B,))
    need = N.load().ds_verify_workspace_size(B, R, V)
    if need == 0:
        raise ValueError(f"unsupported verify sizes B={B} R={R} V={V}")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    return B, R, V, out, n_out, workspace


def verify_greedy(logits: torch.Tensor, draft: torch.Tensor | None, *, out=None, n_out=None,
                  workspace=None, stream=None):
    """Greedy acceptance of B verify steps: logits fp32 [B][R][V], draft int32 [B][R-1].
    Returns (out int32 [B][R], -1 padded; n_out int32 [B])."""
    B, R, V, out, n_out, workspace = _verify_common(logits, draft, out, n_out, workspace)
    st = N.load().ds_verify_greedy(logits.data_ptr(), B, R, V, _ptr(draft) if R > 1 else None,
                                   out.data_ptr(), n_out.data_ptr(), workspace.data_ptr(),
                                   workspace.numel(), _stream(stream))
    _check(st, "ds_verify_greedy")
    return out, n_out


def verify_sample(logits: torch.Tensor, T: float, qd: torch.Tensor | None,
                  draft: torch.Tensor | None, u_acc: torch.Tensor | None, u_res: torch.Tensor,
                  *, out=None, n_out=None, workspace=None, stream=None):
    """Exact speculative sampling for B verify steps at temperature T: logits fp32 [B][R][V],
    qd fp64 [B][R-1][V], draft int32 [B][R-1], u_acc fp64 [B][R-1], u_res fp64 [B][R].
    Returns (out int32 [B][R], -1 padded; n_out int32 [B])."""
    B, R, V, out, n_out, workspace = _verify_common(logits, draft, out, n_out, workspace)
    if R > 1:
        _need(qd, "qd", torch.float64, (B, R - 1, V))
        _need(u_acc, "u_acc", torch.float64, (B, R - 1))
    _need(u_res, "u_res", torch.float64, (B, R))
    st = N.load().ds_verify_sample(
        logits.data_ptr(), B, R, V, float(T), _ptr(qd) if R > 1 else None,
        _ptr(draft) if R > 1 else None, _ptr(u_acc) if R > 1 else None, u_res.data_ptr(),
        out.data_ptr(), n_out.data_ptr(), workspace.data_ptr(), workspace.numel(),
        _stream(stream))
    _check(st, "ds_verify_sample")
    return out, n_out


def sparse_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, sel: torch.Tensor,
                     block_tokens: int = 4, *, out=None, workspace=None, stream=None):
    """Attention of each row's query heads over the tokens of its selected blocks:
    q bf16 [L, R, Hq, 128], k and v bf16 [L, T, 128] (T = blocks x block_tokens), sel int32
    [L, R, K] (block ids, -1 for none) -> bf16 [L, R, Hq, 128] (ds_sparse_attention)."""
    lib = N.load()
    _need(q, "q", torch.bfloat16)
    L, R, Hq, D = q.shape
    _need(k, "k", torch.bfloat16)
    _need(v, "v", torch.bfloat16, tuple(k.shape))
    _need(sel, "sel", torch.int32)
    if k.shape[0] != L or k.shape[2] != D or sel.shape[:2] != (L, R):
        raise ValueError("k, v must be [L, T, D] and sel [L, R, K] for q [L, R, Hq, D]")
    T = k.shape[1]
    args = N.DsAttnArgs(L, R, Hq, D, T // block_tokens, block_tokens, sel.shape[2], _ptr(q),
                        _ptr(k), _ptr(v), T * D, _ptr(sel))
    out = torch.empty_like(q) if out is None else out
    _need(out, "out", torch.bfloat16, tuple(q.shape))
    need = lib.ds_attn_workspace_size(args)
    if need == 0:
        raise ValueError("invalid sparse attention arguments")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(lib.ds_sparse_attention(args, _ptr(out), _ptr(workspace), workspace.numel(),
                                   _stream(stream)), "ds_sparse_attention")
    return out


def noalloc_status(stream=None) -> int:
    """Synchronises the stream and returns the device status code that the last
    moe_verify_forward_noalloc call on the current device left in the library's scratch."""
    return int(N.load().ds_noalloc_status(_stream(stream)))


def workspace_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns the device status code left in the workspace."""
    return int(N.load().ds_workspace_status(_ptr(workspace), _stream(stream)))
