#!/usr/bin/env python3
"""Benchmark of the verify-step hot path on GB300.

One step = one speculative-verify MoE layer call at R = 6 rows (hidden 4096, 384 routed +
1 shared experts, intermediate 1024, top-8, Q4 block-32 weights, ~2.7 GB per layer) plus
one block-select call over 43 layers x 6 rows x 75,000 candidate blocks (300k context,
top-512). The MoE call rotates over several distinct layers so that no weight byte is
served from L2 (an R = 6 call reads ~332 MB > 129 MB of L2; the 43-layer keys are 826 MB).

Prints one JSON line. `value` = algorithmic Q4 weight bytes of the R = 6 MoE calls divided
by their device time (CUDA events on the launching stream), in GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun every rank runs an independent replica ("replicas only": the path does not
shard), rank 0 prints whole-job throughput = sum of bytes / max over ranks of the time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

import numpy as np
import torch

ROOT = Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

import synth  # noqa: E402

# Kernels one step launches: the MoE verify call (a prologue that zeroes the workspace
# header, then one kernel: router, gate/up/SwiGLU, down projection, combine) and the
# tensor-core select (compact, score, top-k).
MOE_KERNELS = 2
SELECT_KERNELS = 3
METRIC = "Q4 MoE verify weight GB/s (% of HBM peak) at R=1/6; top-512 select µs @300k ctx"
UNIT = "GB/s"
Q4_BYTES_PER_WEIGHT = 0.5625          # 4 bits + one fp16 scale per 32 values
FALLBACK_HBM_GBS = 6800.0
R_VERIFY = 6

WORKLOAD = ("one Q4 MoE verify layer (hidden 4096, 384 routed + 1 shared experts, "
            "intermediate 1024, top-8 sigmoid, R=6 rows, block-32 int4 + fp16 scale) + "
            "block select at 300k context (43 layers x 6 rows x 75,000 blocks, 8 heads d=128, "
            "70% admission, top-512)")


# ------------------------------------------------------------------------- helpers --

def expert_bytes(shape: synth.MoeShape) -> float:
    return 3.0 * shape.H * shape.I * Q4_BYTES_PER_WEIGHT


def moe_weight_bytes(shape: synth.MoeShape, n_union: int) -> float:
    """Router (bf16) + shared expert + union of routed experts (gate, up, down in Q4)."""
    return 2.0 * shape.E * shape.H + (1 + n_union) * expert_bytes(shape)


def union_size(idx: np.ndarray) -> int:
    return len(np.unique(idx))


def select_bytes(inp_host: dict, shape: synth.SelectShape) -> dict:
    """Algorithmic bytes of one select call, per kernel (workspace traffic not counted)."""
    mask = inp_host["mask"].view(np.uint32)
    limit = inp_host["limit"]
    L, R, N = shape.L, shape.R, shape.N
    bits = np.unpackbits(mask.astype("<u4").view(np.uint8).reshape(L, R, -1), axis=-1,
                         bitorder="little")[..., :N].astype(bool)
    adm = bits & (np.arange(N)[None, None, :] < limit[..., None])
    key_union = int(adm.any(axis=1).sum())          # keys admitted by some row, all layers
    count = int(adm.sum())                          # admitted (layer, row, block)
    mask_b = mask.nbytes
    q_b = L * R * shape.Hh * shape.D * 2 + L * R * shape.Hh * 4 + L * R * 4
    return {
        "compact": mask_b + 4 * count + 4 * L * R,
        "score": key_union * shape.D * 2 + mask_b + q_b,
        "topk": 4 * L * R * shape.topk + 4 * L * R,
        "total": key_union * shape.D * 2 + mask_b + q_b + 4 * count + 4 * L * R * (shape.topk + 1),
        "key_union": key_union, "admitted": count,
    }


def measured_peaks() -> tuple[float, str]:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            for k in ("hbm_gbs", "hbm_GBs", "hbm_gb_s"):
                if k in d and isinstance(d[k], (int, float)):
                    return float(d[k]), "measured"
                if k in d and isinstance(d[k], dict):
                    v = d[k].get("burst") or d[k].get("value")
                    if v:
                        return float(v), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def traffic_for(kernel: str) -> tuple[float | None, str | None]:
    """DRAM bytes per launch from the committed ncu summary, if the kernel's source is
    unchanged since the counters were taken (sha256 of the source file)."""
    p = ROOT / "profiles" / "traffic.json"
    if not p.exists():
        return None, None
    try:
        d = json.loads(p.read_text()).get(kernel)
        if not d:
            return None, None
        src = ROOT / d["source"]
        if hashlib.sha256(src.read_bytes()).hexdigest() != d["source_sha256"]:
            return None, "stale"
        return float(d["dram_bytes_per_launch"]), d.get("note")
    except Exception:
        return None, None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which: str):
        setattr(self, which, time.time())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append({"t": ts, "sm": float(f[2]), "max": float(f[3]), "active": f[5],
                             "hw": f[6], "hwt": f[7], "swt": f[8], "pcap": f[9]})
            except Exception:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = [r for r in rows if self.t0 - 1 <= r["t"] <= self.t1 + 1] or rows
        reasons = set()
        for r in inside:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in inside),
                "sm_max_mhz": max(r["max"] for r in inside), "reasons": sorted(reasons),
                "samples": len(inside)}


# ------------------------------------------------------------------------ dist ------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce(v: float, world: int, op: str) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------- our arm --------

def run_ours(args, world, rank, local):
    import q4_moe_speculative_gb300 as dsm
    from q4_moe_speculative_gb300 import _native as N
    lib = N.load()                      # fails loudly if the CUDA library is missing
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream

    shape = synth.VERIFY_MOE
    nl = args.layers
    layers = [dsm.MoeLayer.from_dict(synth.moe_layer(shape, seed=args.seed + i, device=dev), shape.k)
              for i in range(nl)]
    structs = [l.struct() for l in layers]
    n_x = 16
    xs6 = [synth.activations(R_VERIFY, shape.H, seed=args.seed + 100 + i, device=dev) for i in range(n_x)]
    xs1 = [synth.activations(1, shape.H, seed=args.seed + 200 + i, device=dev) for i in range(n_x)]
    ws_moe = torch.empty(lib.ds_moe_workspace_size(structs[0], R_VERIFY), dtype=torch.uint8, device=dev)

    sshape = synth.SelectShape(L=args.select_layers, R=6, Hh=8, N=75000, topk=512)
    sel_host = synth.select_inputs(sshape, seed=args.seed, device="cpu")
    sel_in = {k: v.to(dev) for k, v in sel_host.items()}
    sargs = dsm._select_struct(sel_in["keys"], sel_in["q"], sel_in["head_w"], sel_in["mask"],
                               sel_in["limit"], sshape.topk)
    ws_sel = torch.empty(lib.ds_select_workspace_size(sargs), dtype=torch.uint8, device=dev)
    sel = torch.empty((sshape.L, sshape.R, sshape.topk), dtype=torch.int32, device=dev)
    nsel = torch.empty((sshape.L, sshape.R), dtype=torch.int32, device=dev)
    sbytes = select_bytes({"mask": sel_host["mask"].numpy(), "limit": sel_host["limit"].numpy()}, sshape)

    K, W = args.steps, args.warmup
    y = torch.empty((R_VERIFY, shape.H), dtype=torch.bfloat16, device=dev)
    idx_all = torch.empty((K, R_VERIFY, shape.k), dtype=torch.int32, device=dev)
    w_all = torch.empty((K, R_VERIFY, shape.k), dtype=torch.float32, device=dev)
    scratch_idx = torch.empty((R_VERIFY, shape.k), dtype=torch.int32, device=dev)
    scratch_w = torch.empty((R_VERIFY, shape.k), dtype=torch.float32, device=dev)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    # timed loop: start, after the MoE call, after the select call (no events between the
    # kernels of a call, so their programmatic launch overlap stays intact);
    # breakdown loop: start, moe marks (3), select marks (3)
    evm = [[ev() for _ in range(3)] for _ in range(K)]
    evs = [[ev() for _ in range(7)] for _ in range(K)]
    for lst in evm + evs:               # torch creates the CUDA event on first record
        for e in lst:
            e.record(stream)
    torch.cuda.synchronize()
    import ctypes as C
    Marks = C.c_void_p * 3

    def marks_of(lst):
        return Marks(*[e.cuda_event for e in lst])

    marks = [(marks_of(e[1:4]), marks_of(e[4:7])) for e in evs]

    def step(i, mode):
        """mode: "warm" (untimed), "main" (timed per call), "marked" (timed per kernel)."""
        li = i % nl
        x = xs6[i % n_x]
        ib = idx_all[i] if mode == "main" else scratch_idx
        wb = w_all[i] if mode == "main" else scratch_w
        mk = mode == "marked"
        if mode == "main":
            evm[i][0].record(stream)
        elif mk:
            evs[i][0].record(stream)
        st = lib.ds_moe_verify_forward_marked(
            structs[li], x.data_ptr(), R_VERIFY, y.data_ptr(), ib.data_ptr(), wb.data_ptr(),
            ws_moe.data_ptr(), ws_moe.numel(), sptr, marks[i][0] if mk else None)
        if st:
            raise N.DsmoeError(st, "ds_moe_verify_forward")
        if mode == "main":
            evm[i][1].record(stream)
        st = lib.ds_select_blocks_marked(sargs, sel.data_ptr(), nsel.data_ptr(), None, None,
                                         ws_sel.data_ptr(), ws_sel.numel(), sptr,
                                         marks[i][1] if mk else None)
        if st:
            raise N.DsmoeError(st, "ds_select_blocks")
        if mode == "main":
            evm[i][2].record(stream)

    for i in range(W):
        step(i, "warm")
    torch.cuda.synchronize()

    clk = ClockSampler(torch.cuda.current_device() if world == 1 else local)
    clk.start()
    barrier(world)
    torch.cuda.synchronize()
    t_begin, t_end = ev(), ev()
    clk.mark("t0")
    t_begin.record(stream)
    for i in range(K):
        step(i, "main")
    t_end.record(stream)
    torch.cuda.synchronize()
    clk.mark("t1")
    barrier(world)
    clocks = clk.stop()
    assert dsm.workspace_status(ws_moe) == 0 and dsm.workspace_status(ws_sel) == 0

    total_ms = t_begin.elapsed_time(t_end)
    moe_ms = [e[0].elapsed_time(e[1]) for e in evm]
    sel_ms = [e[1].elapsed_time(e[2]) for e in evm]
    # per-kernel breakdown (events after every kernel) in a second pass of the same steps
    for i in range(K):
        step(i, "marked")
    torch.cuda.synchronize()
    # marks: moe prologue, moe kernel (recorded twice), compact, score, top-k
    names = ["moe_prologue", "moe", "moe_end", "compact", "score", "topk"]
    per = {n: [] for n in names}
    marked_ms = []
    for e in evs:
        t = [e[0].elapsed_time(e[j]) for j in range(1, 7)]
        prev = [0.0] + t[:-1]
        for n, a, b in zip(names, prev, t):
            per[n].append(b - a)
        marked_ms.append(t[5])
    del per["moe_end"]
    names = [n for n in names if n != "moe_end"]
    idx_np = idx_all.cpu().numpy()
    unions = [union_size(idx_np[i]) for i in range(K)]
    moe_bytes = [moe_weight_bytes(shape, u) for u in unions]
    y0_sha = hashlib.sha256(y.view(torch.int16).cpu().numpy().tobytes()).hexdigest()[:16]

    if args.skip_extras:   # profiling runs: only the timed step
        r1_bytes, r1_ms, e2e_bytes, e2e_moe, e2e_sel, h2d, d2h = [1.0], [1.0], [1.0], [1.0], [1.0], 0, 0
    else:
        # R = 1 figure (same rotation, separate timed loop)
        y1 = torch.empty((1, shape.H), dtype=torch.bfloat16, device=dev)
        ws1 = torch.empty(lib.ds_moe_workspace_size(structs[0], 1), dtype=torch.uint8, device=dev)
        idx1 = torch.empty((K, 1, shape.k), dtype=torch.int32, device=dev)
        w1 = torch.empty((1, shape.k), dtype=torch.float32, device=dev)
        r1_ev = [(ev(), ev()) for _ in range(K)]
        for i in range(W + K):
            li = i % nl
            if i >= W:
                r1_ev[i - W][0].record(stream)
            lib.ds_moe_verify_forward(structs[li], xs1[i % n_x].data_ptr(), 1, y1.data_ptr(),
                                      idx1[(i - W) % K].data_ptr(), w1.data_ptr(), ws1.data_ptr(),
                                      ws1.numel(), sptr)
            if i >= W:
                r1_ev[i - W][1].record(stream)
        torch.cuda.synchronize()
        r1_ms = [a.elapsed_time(b) for a, b in r1_ev]
        idx1_np = idx1.cpu().numpy()
        r1_bytes = [moe_weight_bytes(shape, union_size(idx1_np[i])) for i in range(K)]

        # end to end through the C ABI with pinned host buffers, copies inside the timed region
        hx = [x.cpu().pin_memory() for x in xs6]
        hq = {k: sel_host[k].pin_memory() for k in ("q", "head_w", "mask", "limit")}
        dq = {k: torch.empty_like(sel_in[k]) for k in hq}
        hy = torch.empty((R_VERIFY, shape.H), dtype=torch.bfloat16).pin_memory()
        hidx = torch.empty((R_VERIFY, shape.k), dtype=torch.int32).pin_memory()
        hw_ = torch.empty((R_VERIFY, shape.k), dtype=torch.float32).pin_memory()
        hsel = torch.empty_like(sel, device="cpu").pin_memory()
        hnsel = torch.empty_like(nsel, device="cpu").pin_memory()
        dx = torch.empty_like(xs6[0])
        sargs_e = dsm._select_struct(sel_in["keys"], dq["q"], dq["head_w"], dq["mask"], dq["limit"],
                                     sshape.topk)
        e2e_moe, e2e_sel = [], []
        e2e_idx = []
        for i in range(W + K):
            a, b, c = ev(), ev(), ev()
            a.record(stream)
            dx.copy_(hx[i % n_x], non_blocking=True)
            st = lib.ds_moe_verify_forward(structs[i % nl], dx.data_ptr(), R_VERIFY, y.data_ptr(),
                                           scratch_idx.data_ptr(), scratch_w.data_ptr(),
                                           ws_moe.data_ptr(), ws_moe.numel(), sptr)
            hy.copy_(y, non_blocking=True)
            hidx.copy_(scratch_idx, non_blocking=True)
            hw_.copy_(scratch_w, non_blocking=True)
            b.record(stream)
            for k_ in hq:
                dq[k_].copy_(hq[k_], non_blocking=True)
            st |= lib.ds_select_blocks(sargs_e, sel.data_ptr(), nsel.data_ptr(), None, None,
                                       ws_sel.data_ptr(), ws_sel.numel(), sptr)
            hsel.copy_(sel, non_blocking=True)
            hnsel.copy_(nsel, non_blocking=True)
            c.record(stream)
            c.synchronize()
            if st:
                raise RuntimeError("e2e call failed")
            if i >= W:
                e2e_moe.append(a.elapsed_time(b))
                e2e_sel.append(b.elapsed_time(c))
                e2e_idx.append(hidx.numpy().copy())
        e2e_bytes = [moe_weight_bytes(shape, union_size(ix)) for ix in e2e_idx]
        h2d = hx[0].numel() * 2 + sum(v.numel() * v.element_size() for v in hq.values())
        d2h = hy.numel() * 2 + hidx.numel() * 4 + hw_.numel() * 4 + hsel.numel() * 4 + hnsel.numel() * 4

    # whole-job aggregation (replicas): sum of bytes / max of times
    moe_s = allreduce(sum(moe_ms) / 1e3, world, "max")
    bytes_all = allreduce(sum(moe_bytes), world, "sum")
    total_ms = allreduce(total_ms, world, "max")
    value = bytes_all / moe_s / 1e9
    r1_gbs = allreduce(sum(r1_bytes), world, "sum") / allreduce(sum(r1_ms) / 1e3, world, "max") / 1e9
    e2e_gbs = allreduce(sum(e2e_bytes), world, "sum") / allreduce(sum(e2e_moe) / 1e3, world, "max") / 1e9

    peak, peak_src = measured_peaks()
    kbytes = {
        "moe_prologue": [0.0] * K,
        "moe": moe_bytes,
        "compact": [sbytes["compact"]] * K, "score": [sbytes["score"]] * K,
        "topk": [sbytes["topk"]] * K,
    }
    kernels = {}
    for n in names:
        ms = float(np.mean(per[n]))
        gbs = float(np.sum(kbytes[n]) / (np.sum(per[n]) / 1e3) / 1e9)
        kernels[n] = {"ms": round(ms, 5), "bytes_per_launch": float(np.mean(kbytes[n])),
                      "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                      "share": round(float(np.sum(per[n]) / np.sum(marked_ms)), 4)}
    dom = max(kernels, key=lambda n: kernels[n]["share"])
    src_of = {"moe_prologue": "moe", "moe": "moe", "compact": "select", "score": "select",
              "topk": "select"}
    traffic, tnote = traffic_for(dom)
    roofline = {"kernel": dom, "bound": "hbm", "achieved": kernels[dom]["gbs"], "peak": peak,
                "unit": "GB/s", "frac": kernels[dom]["frac"], "traffic": traffic,
                "peak_source": f"{peak_src} hbm_gbs" + (" (burst)" if peak_src == "measured" else ""),
                "source_file": f"q4_moe_speculative_gb300/csrc/{src_of[dom]}.cu"}
    if tnote:
        roofline["traffic_note"] = tnote

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": round(total_ms / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "R": R_VERIFY, "moe_layers_rotated": nl,
                   "l2": "inputs larger than L2 (R=6 call reads ~332 MB; layers rotated; "
                         "select keys 826 MB)",
                   "parallelism": f"replicas x{world}", "seed": args.seed},
        "pct_of_hbm_peak": round(100.0 * value / peak, 1),
        "components": {
            "moe_r6_gbs": round(value, 1), "moe_r6_us_median": round(1e3 * statistics.median(moe_ms), 2),
            "moe_r6_us_p90": round(1e3 * float(np.percentile(moe_ms, 90)), 2),
            "moe_r6_union_mean": round(float(np.mean(unions)), 2),
            "moe_r6_weight_bytes_mean": float(np.mean(moe_bytes)),
            "moe_r1_gbs": round(r1_gbs, 1), "moe_r1_us_median": round(1e3 * statistics.median(r1_ms), 2),
            "moe_r1_pct_of_hbm_peak": round(100.0 * r1_gbs / peak, 1),
            "select_300k_us_median": round(1e3 * statistics.median(sel_ms), 2),
            "select_300k_us_p90": round(1e3 * float(np.percentile(sel_ms, 90)), 2),
            "select_300k_bytes": sbytes["total"],
            "select_300k_gbs": round(sbytes["total"] / (statistics.median(sel_ms) / 1e3) / 1e9, 1),
            "select_300k_pct_of_hbm_peak": round(
                100.0 * sbytes["total"] / (statistics.median(sel_ms) / 1e3) / 1e9 / peak, 1),
        },
        "kernels": kernels,
        "roofline": roofline,
        "clocks": clocks,
        "e2e": {"value": round(e2e_gbs, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "select_300k_us_median": round(1e3 * statistics.median(e2e_sel), 2),
                "api": "ds_moe_verify_forward + ds_select_blocks, pinned host buffers"},
        "gpu_launches": (MOE_KERNELS + SELECT_KERNELS) * K,
        "sha256": {"y_last_step": y0_sha},
    }
    out["config"]["select_layers"] = args.select_layers
    if args.skip_extras:
        out["e2e"] = None
        for k_ in ("moe_r1_gbs", "moe_r1_us_median", "moe_r1_pct_of_hbm_peak"):
            out["components"][k_] = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle reads the planar form: regenerate layer 0's (same seed) for the host
        planar = synth.moe_layer(shape, seed=args.seed, device=dev)
        host = {k: synth.to_numpy_bits(v) for k, v in planar.items()}
        del planar
        out["cpu_baseline"] = cpu_baseline(host, xs6, sel_host, shape, sshape)
    if not args.no_sweep and not args.skip_extras:
        del layers, structs
        torch.cuda.empty_cache()
        out["sweep"] = decode_step_sweep(args, lib, dsm, dev, stream)
    return out


def _timed(fn) -> float:
    t = time.perf_counter()
    fn()
    return time.perf_counter() - t


def cpu_baseline(host, xs, sel_host, shape, sshape) -> dict:
    """The oracle, as it stands, on a bounded sample of the same workload, on the host cores:
    one thread, and one thread per core over independent units (the oracle's C calls drop
    Python's lock, so threads run in parallel): rows of verify calls for the MoE, layers of
    the select."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    nproc = os.cpu_count() or 1
    x6 = [synth.to_numpy_bits(x) for x in xs]
    ref = oracle.moe_forward(host, x6[0], shape.k)            # warm-up, and the union size
    call_bytes = moe_weight_bytes(shape, union_size(ref["idx"]))
    t1 = _timed(lambda: oracle.moe_forward(host, x6[0], shape.k))
    gbs1 = call_bytes / t1 / 1e9
    # all cores: nproc one-row jobs (rows of several verify calls), credited 1/R of a call
    jobs = [x6[(j // R_VERIFY) % len(x6)][j % R_VERIFY:j % R_VERIFY + 1] for j in range(nproc)]
    with ThreadPoolExecutor(nproc) as ex:
        tp = _timed(lambda: list(ex.map(lambda xr: oracle.moe_forward(host, xr, shape.k), jobs)))
    gbsp = call_bytes * (nproc / R_VERIFY) / tp / 1e9
    keys = synth.to_numpy_bits(sel_host["keys"])
    q = synth.to_numpy_bits(sel_host["q"])
    hw = sel_host["head_w"].numpy()
    mask = sel_host["mask"].numpy().view(np.uint32)
    lim = sel_host["limit"].numpy()

    def sel_layer(l):
        oracle.select(keys[l:l + 1], q[l:l + 1], hw[l:l + 1], mask[l:l + 1], lim[l:l + 1], sshape.topk)

    ds1 = _timed(lambda: sel_layer(0))
    nl = min(nproc, sshape.L)
    with ThreadPoolExecutor(nproc) as ex:
        dsp = _timed(lambda: list(ex.map(sel_layer, range(nl))))
    return {"value": round(gbs1, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"MoE: one R=6 verify call of one layer ({t1:.1f} s); select: 1 of 43 "
                      f"layers at 300k ({ds1:.1f} s), scaled x43",
            "select_300k_us": round(ds1 * sshape.L * 1e6, 0),
            "all_cores": {"value": round(gbsp, 4), "unit": UNIT, "cores": nproc,
                          "sample": f"MoE: {nproc} one-row verify calls in parallel threads "
                                    f"({tp:.1f} s), credited 1/6 of an R=6 call each; select: "
                                    f"{nl} layers in parallel ({dsp:.1f} s), scaled to 43",
                          "select_300k_us": round(dsp * (sshape.L / nl) * 1e6, 0)},
            "nproc": nproc}


def decode_step_sweep(args, lib, dsm, dev, stream) -> dict:
    """The full decode step: 43 distinct MoE layers resident in HBM (the verify layer's
    shape, ~2.7 GB each) called back to back at R = 1, 2, 4, 6, the block select over 43
    layers at 8k / 64k / 300k context, and weight bytes per committed token at draft
    acceptance rates 0.5 / 0.7 / 0.9 (seeded Bernoulli draws). The 43-layer step is timed
    both as stream launches and as one captured CUDA graph."""
    from q4_moe_speculative_gb300 import _native as NB
    shape = synth.VERIFY_MOE
    per_layer = 2.0 * shape.E * shape.H + (shape.E + 1) * expert_bytes(shape)
    free = torch.cuda.mem_get_info()[0]
    L = int(min(43, max(1, (free - 24e9) // per_layer)))
    sptr = stream.cuda_stream
    t0 = time.perf_counter()
    layers = []
    for i in range(L):
        d = synth.moe_layer(shape, seed=args.seed + 1000 + i, device=dev)
        layers.append(dsm.MoeLayer.from_dict(d, shape.k))
        del d
    torch.cuda.synchronize()
    structs = [l.struct() for l in layers]
    gen_s = time.perf_counter() - t0
    out = {"moe_layers": L, "layer_bytes": per_layer, "setup_s": round(gen_s, 1), "moe": {},
           "select": {}}

    def ev():
        return torch.cuda.Event(enable_timing=True)

    reps, warm = 5, 2
    for R in (1, 2, 4, 6):
        xs = [synth.activations(R, shape.H, seed=args.seed + 3000 + 10 * R + i, device=dev)
              for i in range(L)]
        ws = torch.empty(lib.ds_moe_workspace_size(structs[0], R), dtype=torch.uint8, device=dev)
        ys = [torch.empty((R, shape.H), dtype=torch.bfloat16, device=dev) for _ in range(L)]
        idx = torch.empty((L, R, shape.k), dtype=torch.int32, device=dev)
        w = torch.empty((L, R, shape.k), dtype=torch.float32, device=dev)

        def step():
            for l in range(L):
                st = lib.ds_moe_verify_forward(structs[l], xs[l].data_ptr(), R, ys[l].data_ptr(),
                                               idx[l].data_ptr(), w[l].data_ptr(), ws.data_ptr(),
                                               ws.numel(), sptr)
                if st:
                    raise RuntimeError(f"ds_moe_verify_forward: status {st}")

        ts = []
        for i in range(warm + reps):
            a, b = ev(), ev()
            a.record(stream)
            step()
            b.record(stream)
            torch.cuda.synchronize()
            if i >= warm:
                ts.append(a.elapsed_time(b))
        idx_np = idx.cpu().numpy()
        step_bytes = sum(moe_weight_bytes(shape, union_size(idx_np[l])) for l in range(L))
        us = 1e3 * statistics.median(ts)
        entry = {"us_per_step": round(us, 1), "gbs": round(step_bytes / (us * 1e-6) / 1e9, 1),
                 "weight_bytes_per_step": step_bytes, "per_layer_us": round(us / L, 2)}
        # the same step captured as one CUDA graph
        try:
            g = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream()
            cap.wait_stream(stream)
            with torch.cuda.stream(cap):
                sptr_c = cap.cuda_stream
                with torch.cuda.graph(g, stream=cap):
                    for l in range(L):
                        lib.ds_moe_verify_forward(structs[l], xs[l].data_ptr(), R, ys[l].data_ptr(),
                                                  idx[l].data_ptr(), w[l].data_ptr(), ws.data_ptr(),
                                                  ws.numel(), sptr_c)
            stream.wait_stream(cap)
            tg = []
            for i in range(warm + reps):
                a, b = ev(), ev()
                a.record(stream)
                g.replay()
                b.record(stream)
                torch.cuda.synchronize()
                if i >= warm:
                    tg.append(a.elapsed_time(b))
            gus = 1e3 * statistics.median(tg)
            entry["graph_us_per_step"] = round(gus, 1)
            entry["graph_gbs"] = round(step_bytes / (gus * 1e-6) / 1e9, 1)
            del g
        except Exception as e:  # capture not available: say so
            entry["graph_us_per_step"] = None
            entry["graph_error"] = str(e)[:120]
        # weight bytes per committed token: 1 + leading accepted drafts among R - 1
        for a_ in (0.5, 0.7, 0.9):
            acc = synth.draft_acceptance(20000, R, a_, seed=args.seed)
            lead = np.cumprod(acc, axis=1).sum(axis=1) if R > 1 else np.zeros(len(acc))
            mean_c = float(np.mean(1 + lead))
            closed = (1 - a_ ** R) / (1 - a_)
            entry[f"a{a_}"] = {"committed_mean": round(mean_c, 4), "closed_form": round(closed, 4),
                               "weight_bytes_per_committed_token": round(step_bytes / mean_c, 0)}
        out["moe"][f"R{R}"] = entry
        del xs, ys, ws
    for name, N in (("8k", 2048), ("64k", 16000), ("300k", 75000)):
        sh = synth.SelectShape(L=43, R=6, Hh=8, N=N, topk=512)
        inp = synth.select_inputs(sh, seed=args.seed + 77, device=dev)
        sa = dsm._select_struct(inp["keys"], inp["q"], inp["head_w"], inp["mask"], inp["limit"], 512)
        ws = torch.empty(lib.ds_select_workspace_size(sa), dtype=torch.uint8, device=dev)
        sel = torch.empty((43, 6, 512), dtype=torch.int32, device=dev)
        nsel = torch.empty((43, 6), dtype=torch.int32, device=dev)
        ts = []
        for i in range(warm + 3 * reps):
            a, b = ev(), ev()
            a.record(stream)
            st = lib.ds_select_blocks(sa, sel.data_ptr(), nsel.data_ptr(), None, None, ws.data_ptr(),
                                      ws.numel(), sptr)
            b.record(stream)
            torch.cuda.synchronize()
            if st:
                raise RuntimeError(f"ds_select_blocks: status {st}")
            if i >= warm:
                ts.append(a.elapsed_time(b))
        out["select"][name] = {"blocks": N, "layers": 43, "us": round(1e3 * statistics.median(ts), 1)}
        del inp, ws
    # the single-layer 8k case
    sh = synth.SELECT_8K
    inp = synth.select_inputs(sh, seed=args.seed + 78, device=dev)
    sa = dsm._select_struct(inp["keys"], inp["q"], inp["head_w"], inp["mask"], inp["limit"], 512)
    ws = torch.empty(lib.ds_select_workspace_size(sa), dtype=torch.uint8, device=dev)
    sel = torch.empty((1, 6, 512), dtype=torch.int32, device=dev)
    nsel = torch.empty((1, 6), dtype=torch.int32, device=dev)
    ts = []
    for i in range(warm + 20):
        a, b = ev(), ev()
        a.record(stream)
        lib.ds_select_blocks(sa, sel.data_ptr(), nsel.data_ptr(), None, None, ws.data_ptr(), ws.numel(), sptr)
        b.record(stream)
        torch.cuda.synchronize()
        if i >= warm:
            ts.append(a.elapsed_time(b))
    out["select"]["8k_one_layer"] = {"blocks": 2048, "layers": 1, "us": round(1e3 * statistics.median(ts), 1)}
    # paired Q8 projections: 43 distinct 4096 x 4096 matrices (one per layer, 17.8 MB each,
    # 765 MB in all: past L2) for R = 1 and 6, back to back as one captured CUDA graph (the
    # per-call host cost of a small projection exceeds its GPU time, so single calls would
    # time the host), and one 65536 x 4096 matrix (285 MB) by itself
    out["q8"] = {}
    q8_list = []
    for l in range(43):
        qs, sc = synth.q8_matrix(4096, 4096, seed=args.seed + 500 + l, device=dev)
        q8_list.append(dsm.q8_tile(qs, sc))
        del qs, sc
    q8_ws = torch.empty(lib.ds_q8_workspace_size(), dtype=torch.uint8, device=dev)
    q8_structs = [NB.DsQ8Tiled(t.data_ptr()) for t in q8_list]
    for R in (1, 6):
        xq = synth.activations(R, 4096, seed=args.seed + 600 + R, device=dev)
        yq = [torch.empty((R, 4096), dtype=torch.bfloat16, device=dev) for _ in range(43)]
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                for l in range(43):
                    lib.ds_q8_project(q8_structs[l], 4096, 4096, xq.data_ptr(), R,
                                      yq[l].data_ptr(), q8_ws.data_ptr(), q8_ws.numel(),
                                      cap.cuda_stream)
        stream.wait_stream(cap)
        tg = []
        for i in range(warm + reps):
            a, b = ev(), ev()
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            if i >= warm:
                tg.append(a.elapsed_time(b))
        us = 1e3 * statistics.median(tg)
        by = 43 * 4096 * 4096 * 1.0625
        out["q8"][f"43x4096x4096_R{R}_graph"] = {
            "us": round(us, 1), "us_per_matrix": round(us / 43, 2),
            "gbs": round(by / (us * 1e-6) / 1e9, 1)}
        del g, yq
    st_ = lib.ds_q8_workspace_size()
    del q8_list, q8_structs
    qs, sc = synth.q8_matrix(65536, 4096, seed=args.seed + 700, device=dev)
    big = [dsm.q8_tile(qs, sc) for _ in range(2)]
    del qs, sc
    for R in (1, 6):
        xq = synth.activations(R, 4096, seed=args.seed + 800 + R, device=dev)
        yq = torch.empty((R, 65536), dtype=torch.bfloat16, device=dev)
        ts = []
        for i in range(warm + 20):
            a, b = ev(), ev()
            a.record(stream)
            st = lib.ds_q8_project(NB.DsQ8Tiled(big[i % 2].data_ptr()), 65536, 4096,
                                   xq.data_ptr(), R, yq.data_ptr(), q8_ws.data_ptr(),
                                   q8_ws.numel(), sptr)
            b.record(stream)
            torch.cuda.synchronize()
            if st:
                raise RuntimeError(f"ds_q8_project: status {st}")
            if i >= warm:
                ts.append(a.elapsed_time(b))
        us = 1e3 * statistics.median(ts)
        out["q8"][f"65536x4096_R{R}"] = {"us": round(us, 1),
                                         "gbs": round(65536 * 4096 * 1.0625 / (us * 1e-6) / 1e9, 1)}
    del big
    assert dsm.workspace_status(q8_ws) == 0 and st_ == 256
    # sparse attention over the selected blocks: 43 layers x 6 rows x 16 heads, 512 blocks
    # of 4 tokens per row (keys and values of the selected tokens: 1 MB per row), at 300k
    # context (75,000 blocks per layer; the selection is random, ascending)
    T = 75000 * 4
    ai = synth.attention_inputs(43, 6, 16, T, seed=args.seed + 900, device=dev)
    rng = np.random.default_rng(args.seed + 901)
    sel_np = np.sort(np.stack([rng.choice(75000, size=512, replace=False)
                               for _ in range(43 * 6)]), axis=1).astype(np.int32)
    sel_a = torch.from_numpy(sel_np.reshape(43, 6, 512)).to(dev)
    a_out = torch.empty_like(ai["q"])
    a_args = NB.DsAttnArgs(43, 6, 16, 128, 75000, 4, 512, ai["q"].data_ptr(), ai["k"].data_ptr(),
                           ai["v"].data_ptr(), T * 128, sel_a.data_ptr())
    a_ws = torch.empty(lib.ds_attn_workspace_size(a_args), dtype=torch.uint8, device=dev)
    ts = []
    for i in range(warm + 20):
        a, b = ev(), ev()
        a.record(stream)
        st = lib.ds_sparse_attention(a_args, a_out.data_ptr(), a_ws.data_ptr(), a_ws.numel(), sptr)
        b.record(stream)
        torch.cuda.synchronize()
        if st:
            raise RuntimeError(f"ds_sparse_attention: status {st}")
        if i >= warm:
            ts.append(a.elapsed_time(b))
    us = 1e3 * statistics.median(ts)
    a_bytes = 43 * 6 * 512 * 4 * 256 * 2 + 43 * 6 * 16 * 128 * 2 * 2
    out["attention"] = {"layers": 43, "rows": 6, "heads": 16, "blocks": 512, "us": round(us, 1),
                        "bytes": a_bytes, "gbs": round(a_bytes / (us * 1e-6) / 1e9, 1)}
    del ai, a_out, a_ws, sel_a
    # the acceptance step after the verify: R = 6 rows over the vocabulary, one step and a
    # batch of 64 independent steps, greedy and exact speculative sampling at T = 1
    out["accept"] = {}
    for B in (1, 64):
        d = synth.verify_inputs(B, 6, synth.VOCAB, seed=args.seed + 90 + B)
        t = {k: torch.from_numpy(np.ascontiguousarray(d[k])).to(dev)
             for k in ("logits", "qd", "draft", "u_acc", "u_res")}
        ws = torch.empty(lib.ds_verify_workspace_size(B, 6, synth.VOCAB), dtype=torch.uint8,
                         device=dev)
        o = torch.empty((B, 6), dtype=torch.int32, device=dev)
        n = torch.empty((B,), dtype=torch.int32, device=dev)
        for mode in ("greedy", "sample"):
            ts = []
            for i in range(warm + 20):
                a, b = ev(), ev()
                a.record(stream)
                if mode == "greedy":
                    st = lib.ds_verify_greedy(t["logits"].data_ptr(), B, 6, synth.VOCAB,
                                              t["draft"].data_ptr(), o.data_ptr(), n.data_ptr(),
                                              ws.data_ptr(), ws.numel(), sptr)
                else:
                    st = lib.ds_verify_sample(t["logits"].data_ptr(), B, 6, synth.VOCAB, 1.0,
                                              t["qd"].data_ptr(), t["draft"].data_ptr(),
                                              t["u_acc"].data_ptr(), t["u_res"].data_ptr(),
                                              o.data_ptr(), n.data_ptr(), ws.data_ptr(),
                                              ws.numel(), sptr)
                b.record(stream)
                torch.cuda.synchronize()
                if st:
                    raise RuntimeError(f"ds_verify_{mode}: status {st}")
                if i >= warm:
                    ts.append(a.elapsed_time(b))
            us = 1e3 * statistics.median(ts)
            read = B * 6 * synth.VOCAB * 4 + (B * 5 * synth.VOCAB * 8 if mode == "sample" else 0)
            out["accept"][f"{mode}_B{B}"] = {"us": round(us, 1), "vocab": synth.VOCAB, "rows": 6,
                                             "input_mb": round(read / 1e6, 1)}
        del t, ws, o, n
    del layers, structs
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------- reference arm ----

def run_reference(args, world, rank):
    """The oracle timed on the host cores, on the same config/metric; bounded samples."""
    import oracle
    shape = synth.VERIFY_MOE
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    layer = {k: synth.to_numpy_bits(v) for k, v in synth.moe_layer(shape, seed=args.seed, device=gen_dev).items()}
    x = synth.to_numpy_bits(synth.activations(R_VERIFY, shape.H, seed=args.seed + 100, device=gen_dev))
    idx_all, _, _ = oracle.router(x, layer["router_w"], shape.k)
    share = moe_weight_bytes(shape, union_size(idx_all)) / R_VERIFY
    # Each step is one row of the R = 6 verify (rows are independent in the oracle); it is
    # credited with 1/6 of the R = 6 call's weight bytes.
    times = []
    for i in range(args.warmup + args.steps):
        r = i % R_VERIFY
        t = time.perf_counter()
        oracle.moe_forward(layer, x[r:r + 1], shape.k)
        dt = time.perf_counter() - t
        if i >= args.warmup:
            times.append(dt)
    value = share * len(times) / sum(times) / 1e9
    sshape = synth.SelectShape(L=1, R=6, Hh=8, N=75000, topk=512)
    sin = synth.select_inputs(sshape, seed=args.seed, device="cpu")
    t = time.perf_counter()
    oracle.select(synth.to_numpy_bits(sin["keys"]), synth.to_numpy_bits(sin["q"]), sin["head_w"].numpy(),
                  sin["mask"].numpy().view(np.uint32), sin["limit"].numpy(), 512)
    ds = time.perf_counter() - t
    sample = (f"each step: one row of the R=6 verify of one layer, credited 1/6 of the call's "
              f"weight bytes; select: 1 of 43 layers at 300k ({ds:.1f} s) scaled x43")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * sum(times) / len(times), 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "R": R_VERIFY, "seed": args.seed},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "select_300k_us": round(ds * 43 * 1e6, 0),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=8, help="distinct MoE layers rotated")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--select-layers", type=int, default=43, help="layers of the 300k select")
    ap.add_argument("--skip-extras", action="store_true", help="no R=1 and end-to-end loops")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the 43-layer decode-step sweep (R=1/2/4/6, select 8k/64k/300k)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world, rank)), flush=True)
        return
    out = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
