"""Small workloads that run one kernel family a few times, for single-kernel ncu captures.

    python tests/profile_cases.py moe      # one verify layer (H 4096, 96 + 1 experts, I 1024, R 6)
    python tests/profile_cases.py select   # block select, 43 layers x 6 rows x 16,000 blocks
    python tests/profile_cases.py q8       # paired Q8 projection, 16384 x 4096, R 6
    python tests/profile_cases.py attn     # sparse attention, 43 layers x 6 rows x 512 blocks
    python tests/profile_cases.py accept   # acceptance, 8 steps x 6 rows x 129,280 tokens

Each case holds a few GB on the device at most, with weights / keys larger than L2, and
runs its call `--reps` times (default 4) on synthetic inputs, then checks the workspace
status. Not a test module (no test_ prefix); measurement infrastructure.
"""
from __future__ import annotations

import argparse
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402
import q4_moe_speculative_gb300 as dsm  # noqa: E402


def run(case: str, reps: int) -> None:
    dev = torch.device("cuda", 0)
    if case == "moe":
        shape = synth.MoeShape(H=4096, E=96, I=1024, k=8)
        layer = dsm.MoeLayer.from_dict(synth.moe_layer(shape, seed=1, device=dev), shape.k)
        x = synth.activations(6, shape.H, seed=2, device=dev)
        ws = torch.empty(dsm.moe_workspace_size(layer, 6), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            dsm.moe_verify_forward(layer, x, workspace=ws)
    elif case == "select":
        sh = synth.SELECT_64K
        d = synth.select_inputs(sh, seed=1, device=dev)
        args = (d["keys"], d["q"], d["head_w"], d["mask"], d["limit"], sh.topk)
        ws = torch.empty(dsm.select_workspace_size(*args), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            dsm.select_blocks(*args, workspace=ws)
    elif case == "q8":
        qs, sc = synth.q8_matrix(16384, 4096, seed=1, device=dev)
        tiles = dsm.q8_tile(qs, sc)
        x = synth.activations(6, 4096, seed=2, device=dev)
        ws = torch.empty(256, dtype=torch.uint8, device=dev)
        for _ in range(reps):
            dsm.q8_project(tiles, x, workspace=ws)
    elif case == "attn":
        T = 75000 * 4
        a = synth.attention_inputs(43, 6, 16, T, seed=1, device=dev)
        rng = np.random.default_rng(2)
        sel = np.sort(np.stack([rng.choice(75000, size=512, replace=False) for _ in range(258)]),
                      axis=1).astype(np.int32).reshape(43, 6, 512)
        st = torch.from_numpy(sel).to(dev)
        ws = None
        for _ in range(reps):
            dsm.sparse_attention(a["q"], a["k"], a["v"], st)
    elif case == "accept":
        d = synth.verify_inputs(8, 6, synth.VOCAB, seed=1)
        t = {k: torch.from_numpy(np.ascontiguousarray(d[k])).to(dev)
             for k in ("logits", "qd", "draft", "u_acc", "u_res")}
        ws = None
        for _ in range(reps):
            dsm.verify_greedy(t["logits"], t["draft"])
            dsm.verify_sample(t["logits"], 1.0, t["qd"], t["draft"], t["u_acc"], t["u_res"])
    else:
        raise SystemExit(f"unknown case {case}")
    torch.cuda.synchronize()
    if ws is not None:
        assert dsm.workspace_status(ws) == 0
    print(f"{case}: {reps} runs ok")


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("case")
    ap.add_argument("--reps", type=int, default=4)
    args = ap.parse_args()
    run(args.case, args.reps)
