"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers and packs them into the input layouts; it holds none of
the method's arithmetic (no routing, no dequantisation, no scoring, no selection). Both the
oracle side and the CUDA side receive the same bytes from here.

Workloads (the pages' model is private; these stand in for it, with the shapes and value
distributions of the workload definitions):
  - MoE layer: router bf16 N(0, 0.02); Q4 values uniform in [-8, 7] (uniform random bytes:
    two uniform nibbles each); fp16 scales |N(0, 0.02)|; activations bf16 N(0, 1).
  - Block select: keys and queries bf16 N(0, 1); per-head fp32 weights N(0, 1); causal limit
    of row r at position T - R + r with T = 4N tokens (blocks of 4 tokens), i.e.
    limit_r = floor((T - R + r + 1) / 4); the last 32 blocks below the limit always
    admitted, the rest Bernoulli(0.7), drawn per (layer, block) and shared by the rows
    (default) or drawn per (layer, row, block). Mask bits at or above the limit are random
    too, so a consumer must honour the limit.
  - Paired Q8 projections: int8 values uniform in [-128, 127], fp16 scales
    uniform(0.5, 2) x 2^-7 (so |W| is about 0.5 at most, comparable to a trained layer's
    weights), verify rows bf16 N(0, 1).
  - Sparse attention over the selected blocks: queries bf16 N(0, sigma^2) [L][R][Hq][128]
    (sigma 1, or larger for peaked attention), keys and values bf16 N(0, 1) per token
    [L][T][128], T = 4 x blocks.
  - Speculative acceptance: Bernoulli(a) per draft, seeded (the sweep); and, for the
    acceptance step itself, target logits N(0, 1.5^2) per token with one planted strong
    token per row (its logit raised by `peak` x U(0.5, 1.5)), a drafter distribution that
    is the mixture alpha x (one-hot at the planted token) + (1 - alpha) x uniform, drafts
    drawn from that mixture, and uniforms in [0, 1). Vocabulary 129,280 tokens.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class MoeShape:
    H: int   # hidden
    E: int   # routed experts
    I: int   # expert intermediate
    k: int   # top-k


@dataclass(frozen=True)
class SelectShape:
    L: int     # layers
    R: int     # query rows
    Hh: int    # index heads
    N: int     # candidate blocks
    topk: int
    D: int = 128


# The workload sizes (one MoE layer of the tiny and of the single-layer verify case; the
# block-select cases at 64 blocks, 8k context and 300k context).
TINY_MOE = MoeShape(H=512, E=16, I=256, k=2)
VERIFY_MOE = MoeShape(H=4096, E=384, I=1024, k=8)
TINY_SELECT = SelectShape(L=1, R=1, Hh=1, N=64, topk=8)
SELECT_8K = SelectShape(L=1, R=6, Hh=8, N=2048, topk=512)
SELECT_64K = SelectShape(L=43, R=6, Hh=8, N=16000, topk=512)
SELECT_300K = SelectShape(L=43, R=6, Hh=8, N=75000, topk=512)

SLIDING_WINDOW = 32
P_ADMIT = 0.7


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def q4_matrix(lead: tuple, rows: int, K: int, g: torch.Generator, device):
    """Random Q4 matrix: qs uint8 [*lead, rows, K/2] (uniform bytes), sc fp16 |N(0,0.02)|.
    On the host the bytes come from numpy (PCG64 seeded from `g`), which is much faster
    than torch's host generator for gigabyte stacks; on a GPU from torch's device
    generator. Same distributions, different bytes."""
    shape = (*lead, rows, K // 2)
    if torch.device(device).type == "cpu":
        seed = int(torch.randint(0, 2**62, (1,), generator=g).item())
        n = int(np.prod(shape))
        words = np.random.PCG64(seed).random_raw((n + 7) // 8)   # uniform 64-bit outputs
        qs = torch.from_numpy(words.view(np.uint8)[:n].reshape(shape).copy())
    else:
        qs = torch.randint(0, 256, shape, dtype=torch.uint8, generator=g, device=device)
    sc = torch.randn((*lead, rows, K // 32), generator=g, device=device).mul_(0.02).abs_()
    return qs, sc.to(torch.float16)


def moe_layer(shape: MoeShape, seed: int = 0, device="cpu") -> dict:
    """Tensors of one MoE layer (routed experts stacked expert-major + shared expert)."""
    g = _gen(seed, device)
    H, E, I = shape.H, shape.E, shape.I
    d = {"router_w": torch.randn((E, H), generator=g, device=device).mul_(0.02).to(torch.bfloat16)}
    d["gate_qs"], d["gate_sc"] = q4_matrix((E,), I, H, g, device)
    d["up_qs"], d["up_sc"] = q4_matrix((E,), I, H, g, device)
    d["down_qs"], d["down_sc"] = q4_matrix((E,), H, I, g, device)
    d["sh_gate_qs"], d["sh_gate_sc"] = q4_matrix((), I, H, g, device)
    d["sh_up_qs"], d["sh_up_sc"] = q4_matrix((), I, H, g, device)
    d["sh_down_qs"], d["sh_down_sc"] = q4_matrix((), H, I, g, device)
    return d


def activations(R: int, H: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Verify rows: bf16 N(0, 1) [R, H]."""
    g = _gen(seed + 1_000_003, device)
    return torch.randn((R, H), generator=g, device=device).to(torch.bfloat16)


def causal_limits(N: int, R: int) -> np.ndarray:
    """limit_r = floor((p_r + 1) / 4) with p_r = 4N - R + r (row r's token position)."""
    T = 4 * N
    return np.array([(T - R + r + 1) // 4 for r in range(R)], dtype=np.int32)


def pack_bits(bits: np.ndarray) -> np.ndarray:
    """bool [..., n] -> uint32 [..., ceil(n/32)], bit b%32 of word b//32 (little-endian)."""
    n = bits.shape[-1]
    W = (n + 31) // 32
    pad = np.zeros(bits.shape[:-1] + (W * 32,), dtype=bool)
    pad[..., :n] = bits
    by = np.packbits(pad.reshape(bits.shape[:-1] + (W * 4, 8)), axis=-1, bitorder="little")
    return by.reshape(bits.shape[:-1] + (W * 4,)).view("<u4").astype(np.uint32)


def admission_mask(shape: SelectShape, seed: int = 0, shared: bool = True,
                   p: float = P_ADMIT, window: int = SLIDING_WINDOW):
    """(mask uint32 [L,R,W], limit int32 [L,R]) on the host."""
    rng = np.random.Generator(np.random.PCG64(seed + 7_000_001))
    L, R, N = shape.L, shape.R, shape.N
    lim = causal_limits(N, R)
    if shared:
        draw = rng.random((L, 1, N)) < p
        bits = np.repeat(draw, R, axis=1)
    else:
        bits = rng.random((L, R, N)) < p
    b = np.arange(N)
    for r in range(R):
        win = (b >= lim[r] - window) & (b < lim[r])
        bits[:, r, :] |= win[None, :]
    limit = np.broadcast_to(lim[None, :], (L, R)).astype(np.int32).copy()
    return pack_bits(bits), limit


def select_inputs(shape: SelectShape, seed: int = 0, device="cpu", shared_mask: bool = True) -> dict:
    """keys bf16 [L,N,D], q bf16 [L,R,Hh,D], head_w f32 [L,R,Hh], mask int32 [L,R,W]
    (uint32 bit patterns), limit int32 [L,R]."""
    g = _gen(seed + 5_000_011, device)
    L, R, Hh, N, D = shape.L, shape.R, shape.Hh, shape.N, shape.D
    keys = torch.empty((L, N, D), dtype=torch.bfloat16, device=device)
    for l in range(L):
        keys[l] = torch.randn((N, D), generator=g, device=device).to(torch.bfloat16)
    q = torch.randn((L, R, Hh, D), generator=g, device=device).to(torch.bfloat16)
    head_w = torch.randn((L, R, Hh), generator=g, device=device)
    mask, limit = admission_mask(shape, seed, shared=shared_mask)
    return {
        "keys": keys, "q": q, "head_w": head_w,
        "mask": torch.from_numpy(mask.view(np.int32).copy()).to(device),
        "limit": torch.from_numpy(limit).to(device),
    }


def draft_acceptance(n_steps: int, R: int, a: float, seed: int = 0) -> np.ndarray:
    """uint8 [n_steps, R-1]: 1 where draft j of step t is accepted (Bernoulli(a))."""
    rng = np.random.Generator(np.random.PCG64(seed + 9_000_007))
    return (rng.random((n_steps, max(R - 1, 0))) < a).astype(np.uint8)


def to_numpy_bits(t: torch.Tensor) -> np.ndarray:
    """Host copy of a tensor's raw bits (bf16/fp16 -> uint16, int32 mask -> uint32)."""
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.int32:
        return t.numpy()
    return t.numpy()


VOCAB = 129280   # tokens in the vocabulary of the acceptance workload


def verify_inputs(B: int, R: int, V: int, seed: int = 0, peak: float = 6.0,
                  alpha: float = 0.7) -> dict:
    """One batch of B verify steps of R rows: logits fp32 [B][R][V], the planted strong
    token of each row, the drafter's distributions qd fp64 [B][R-1][V] (alpha on the
    planted token plus (1 - alpha) / V everywhere), drafts int32 [B][R-1] drawn from qd,
    and the uniforms u_acc fp64 [B][R-1], u_res fp64 [B][R]."""
    rng = np.random.default_rng(seed)
    z = (rng.standard_normal((B, R, V)) * 1.5).astype(np.float32)
    strong = rng.integers(0, V, size=(B, R))
    lift = (peak * rng.uniform(0.5, 1.5, size=(B, R))).astype(np.float32)
    bi, ri = np.meshgrid(np.arange(B), np.arange(R), indexing="ij")
    z[bi, ri, strong] += lift
    n = max(R - 1, 0)
    qd = np.full((B, n, V), (1.0 - alpha) / V, dtype=np.float64)
    if n:
        qd[bi[:, :n], ri[:, :n], strong[:, :n]] += alpha
    # a draw from the mixture: the planted token with probability alpha, else uniform
    pick = rng.random((B, n)) < alpha
    draft = np.where(pick, strong[:, :n], rng.integers(0, V, size=(B, n))).astype(np.int32)
    return {"logits": z, "strong": strong.astype(np.int32), "qd": qd, "draft": draft,
            "u_acc": rng.random((B, n)), "u_res": rng.random((B, R))}


def greedy_inputs(B: int, R: int, V: int, seed: int = 0) -> dict:
    """Greedy verify steps with known row maxima: logits N(0, 1) with the row's top token
    planted at `top` (value 10); step b plants a tie for odd b (the same value at a second
    token `twin`, below `top` in id for b % 4 == 1, above it for b % 4 == 3); the drafts
    repeat `top` for the first b % R rows, then one different token, then random ones."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((B, R, V)).astype(np.float32)
    top = rng.integers(1, V - 1, size=(B, R)) if V > 2 else np.zeros((B, R), np.int64)
    twin = np.where((np.arange(B) % 4 == 1)[:, None], rng.integers(0, np.maximum(top, 1)),
                    top + 1 + rng.integers(0, np.maximum(V - 1 - top, 1)))
    twin = np.minimum(twin, V - 1)
    bi, ri = np.meshgrid(np.arange(B), np.arange(R), indexing="ij")
    z[bi, ri, top] = 10.0
    odd = (np.arange(B) % 2 == 1)[:, None] & (twin != top)
    z[bi[odd], ri[odd], twin[odd]] = 10.0
    n = max(R - 1, 0)
    draft = rng.integers(0, V, size=(B, n)).astype(np.int32)
    for b in range(B):
        k = b % R
        draft[b, :min(k, n)] = top[b, :min(k, n)]
        if k < n:
            draft[b, k] = (top[b, k] + 1) % V
    return {"logits": z, "draft": draft}


def q8_matrix(rows: int, K: int, seed: int = 0, device="cpu"):
    """Random Q8 matrix: qs int8 [rows, K] uniform in [-128, 127], sc fp16 [rows, K/32]
    uniform(0.5, 2) x 2^-7."""
    g = _gen(seed, device)
    qs = torch.randint(-128, 128, (rows, K), dtype=torch.int8, generator=g, device=device)
    sc = torch.rand((rows, K // 32), generator=g, device=device).mul_(1.5).add_(0.5)
    return qs, sc.mul_(2.0 ** -7).to(torch.float16)


def attention_inputs(L: int, R: int, Hq: int, T: int, seed: int = 0, sigma: float = 1.0,
                     device="cpu") -> dict:
    """Queries bf16 N(0, sigma^2) [L][R][Hq][128]; keys and values bf16 N(0, 1) [L][T][128]."""
    g = _gen(seed, device)
    q = torch.randn((L, R, Hq, 128), generator=g, device=device).mul_(sigma)
    k = torch.randn((L, T, 128), generator=g, device=device)
    v = torch.randn((L, T, 128), generator=g, device=device)
    return {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16)}
