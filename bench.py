"""Benchmark of one Medusa decode step (heads + top-s, tree build, tree attention through the
synthetic layer, verification, acceptance, KV compaction) on the Vicuna-13B-shaped batch of 8
(the headline), with the Vicuna-7B-shaped step and the Zephyr-7B-shaped GQA batch of 16
measured into the same line under "workloads".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--also NAME,NAME]

Prints one JSON line.  `value` is whole-job decode steps per second with inputs resident in
HBM; `e2e` is the same metric through the C ABI with the step's input copied from pinned
host memory and its result read back every step.  Each step streams > 1.8 GB of weights,
far more than the 129 MB L2, so no L2 flush is needed between steps.  Under torchrun every
rank runs an independent replica of the workload (sequences are independent: no
collective on the data path); timing is the max over ranks.  `--impl reference` times the
fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic as S  # noqa: E402

METRIC = "Medusa verify steps/s and tree-nodes/s on 1 GB300; HBM GB/s vs ~8 TB/s peak"
FALLBACK_HBM_GBS = 6800.0


FALLBACK_BF16_TFLOPS = 1700.0    # sustained figure of the fallback measurement


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 TFLOP/s for kernels timed inside a long step: the measured sustained
    figure (power-capped), else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def config_of(w: S.Workload, n1: int):
    return {"workload": w.name, "B": w.B, "d": w.d, "V": w.V, "K": w.K,
            "heads": f"{w.Hq}q/{w.Hkv}kv x {w.dh}", "prefix": list(sorted(set(w.lengths))),
            "tree_nodes": n1, "tree": f"{w.tree} top-{max(w.s)}", "mode": w.mode,
            "temperature": w.temperature, "paged": bool(w.page_size),
            "l2": "no flush: each step streams the weights (> 2 GB) through the 129 MB L2"}


# ----------------------------------------------------------------------- byte model
def kernel_bytes(w: S.Workload, n1: int, tc_heads: bool):
    """Algorithmic HBM bytes per launch of each kernel (weights and caches read once,
    activations and outputs at their stored widths)."""
    es = 4 if w.dtype == "f32" else 2
    B, d, V, K = w.B, w.d, w.V, w.K
    M = B * n1
    qd, kd = w.Hq * w.dh, w.Hkv * w.dh
    act = 4 if tc_heads else 0          # bf16 hi + lo copies written next to fp32
    kv_prefix = sum(w.lengths) * 2 * kd * es
    # CUDA-core heads (batch 1): the LM head's root pass shares the first launch
    lm = (V * d * es + B * V * 4) if not tc_heads else 0
    return {
        "heads_w1": K * d * d * es + B * d * 4 + B * K * d * (4 + act) + lm,
        "heads_vocab": (K + 1) * V * d * es + B * (K + 1) * d * 4 + B * (K + 1) * V * 4
                       - (lm + (B * d * 4 if lm else 0)),
        "layer_qkv": (qd + 2 * kd) * d * es + M * d * 2 + M * (qd + 2 * kd) * 4,
        "tree_attention": kv_prefix + M * (qd * 4 + 2 * kd * es),
        "layer_out": d * qd * es + M * qd * 4 + M * d * (2 + 4 + 4),
        "verify_logits": V * d * es + M * d * 4 + M * V * 4,
    }


def kernel_flops(w: S.Workload, n1: int, tc_heads: bool = True):
    """Algorithmic FLOPs per launch of the contractions (the method's products, counted
    once: the hi/lo activation halves that double the tensor-core work are not counted)."""
    B, d, V, K = w.B, w.d, w.V, w.K
    M = B * n1
    qd, kd = w.Hq * w.dh, w.Hkv * w.dh
    prefix = sum(w.lengths)
    lm = 0 if tc_heads else 2 * B * V * d
    return {
        "heads_w1": 2 * B * K * d * d + lm,
        "heads_vocab": 2 * B * (K + 1) * V * d - lm,
        "layer_qkv": 2 * M * (qd + 2 * kd) * d,
        "tree_attention": 4 * n1 * w.Hq * w.dh * prefix + 4 * B * n1 * n1 * w.Hq * w.dh // 2,
        "layer_out": 2 * M * d * qd,
        "verify_logits": 2 * M * V * d,
    }


def step_bytes(w: S.Workload, n1: int):
    """Bytes the method itself must move per step: head weights, LM head (for the root and
    for verification), the KV prefix, the tree nodes' K/V written and read, and the
    synthetic layer's weights."""
    es = 4 if w.dtype == "f32" else 2
    d, V, K = w.d, w.V, w.K
    qd, kd = w.Hq * w.dh, w.Hkv * w.dh
    heads = K * d * d * es + K * V * d * es
    lm = 2 * V * d * es
    kv = sum(w.lengths) * 2 * kd * es + w.B * n1 * 2 * kd * es * 2
    layer = (qd + 2 * kd + qd) * d * es + w.B * n1 * d * es
    return heads + lm + kv + layer


def steady_bytes(w: S.Workload, n1: int):
    """step_bytes of a decode-loop step whose root comes from the previous step: the LM
    head is read once (for verification)."""
    es = 4 if w.dtype == "f32" else 2
    return step_bytes(w, n1) - w.V * w.d * es


def steady_state(args, w: S.Workload, st, stream, barrier):
    """The decode loop's steady state: each step takes the previous step's root_next and
    h_next (so the LM head is not applied to h_t), as a CUDA graph of two ping-ponged
    steps.  The prefix length is held at the workload's (len_out goes to a side buffer),
    so every step sees the same context size."""
    from medusa_head_speculative_gb300 import binding as Bnd
    plan, o = st["plan"], st["out"]
    h_a = st["h"].clone()
    h_b = torch.empty_like(h_a)
    r_a = o["root_next"].clone()
    r_b = torch.empty_like(r_a)
    outs_a = Bnd.outputs_struct(o["out_tok"], o["n_acc"], o["path"], h_b, r_b)
    outs_b = Bnd.outputs_struct(o["out_tok"], o["n_acc"], o["path"], h_a, r_a)

    def pair():
        Bnd.step(plan, h_a, r_a, st["wstruct"], st["kv"], st["acc"], outs_a, st["ws"])
        Bnd.step(plan, h_b, r_b, st["wstruct"], st["kv"], st["acc"], outs_b, st["ws"])

    for _ in range(3):
        pair()
    run, mode = pair, "direct"
    if not args.no_graph:
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                pair()
            g.replay()
            run, mode = g.replay, "cuda_graph"
        except Exception as exc:                        # noqa: BLE001
            mode = f"direct (graph capture failed: {exc})"[:160]
    reps = max(1, args.steps // 2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for _ in range(reps):
        run()
    e1.record(stream)
    barrier()
    ms = e0.elapsed_time(e1) / (2 * reps)
    assert plan.status() == 0, "device status word set during the steady-state region"
    # accepted tokens per step along the same loop (outside the timed region)
    tot = torch.zeros(w.B, dtype=torch.int64, device=o["n_acc"].device)
    n_pairs = 100
    for _ in range(n_pairs):
        Bnd.step(plan, h_a, r_a, st["wstruct"], st["kv"], st["acc"], outs_a, st["ws"])
        tot += o["n_acc"]
        Bnd.step(plan, h_b, r_b, st["wstruct"], st["kv"], st["acc"], outs_b, st["ws"])
        tot += o["n_acc"]
    mean_tok = float(tot.sum()) / (2 * n_pairs * w.B)
    return {"value": round(1e3 / ms, 2), "unit": "steps/s", "ms_per_step": round(ms, 5),
            "steps": 2 * reps, "launch": mode,
            "mean_tokens_per_step": round(mean_tok, 3),
            "tokens_per_s": round(1e3 / ms * mean_tok * w.B, 1),
            "note": "root_in = previous root_next, h = previous h_next: the LM head is read "
                    "once per step; prefix length held fixed"}


def layers_bytes(w: S.Workload, n1: int, n_layers: int):
    """step_bytes through an n-layer backbone: every further layer adds its projections,
    its KV prefix, its tree K/V written and read, and the node activations."""
    es = 4 if w.dtype == "f32" else 2
    qd, kd = w.Hq * w.dh, w.Hkv * w.dh
    per = ((qd + 2 * kd + qd) * w.d * es + w.B * n1 * w.d * es
           + sum(w.lengths) * 2 * kd * es + w.B * n1 * 2 * kd * es * 2)
    return step_bytes(w, n1) + (n_layers - 1) * per


def multi_layer(args, w: S.Workload, st, device, stream, barrier):
    """medusa_step_layers through args.layers backbone layers (layer 0 = the workload's
    projections and cache, further layers seeded on their own), prefix held fixed, as a
    CUDA graph replayed back to back."""
    from medusa_head_speculative_gb300 import binding as Bnd
    n = args.layers
    plan = st["plan"]
    layers = [dict(wq=st["wts"]["wq"], wk=st["wts"]["wk"], wv=st["wts"]["wv"], wo=st["wts"]["wo"],
                   k=st["kc"], v=st["vc"])]
    for l in range(1, n):
        lw = S.layer_weights(w, l)
        kc, vc, _ = S.kv_cache(w, l)
        layers.append(dict(**{k: t.to(device) for k, t in lw.items()}, k=kc.to(device), v=vc.to(device)))
    arr = Bnd.layers_array(layers)
    ws = torch.empty(plan.workspace_size_layers(n), dtype=torch.uint8, device=device)
    kv = Bnd.kv_struct(None, None, st["length"], st["len_out"], st["pt"])

    def one():
        Bnd.step_layers(plan, st["h"], None, st["wstruct"], arr, kv, st["acc"], st["outs"], ws)

    for _ in range(3):
        one()
    run, mode = one, "direct"
    if not args.no_graph:
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                one()
            g.replay()
            run, mode = g.replay, "cuda_graph"
        except Exception as exc:                        # noqa: BLE001
            mode = f"direct (graph capture failed: {exc})"[:160]
    reps = max(1, min(args.steps, 1000))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for _ in range(reps):
        run()
    e1.record(stream)
    barrier()
    ms = e0.elapsed_time(e1) / reps
    assert plan.status() == 0, "device status word set during the multi-layer region"
    sb = layers_bytes(w, plan.n1, n)
    hbm, _ = peaks()
    return {"value": round(1e3 / ms, 2), "unit": "steps/s", "n_layers": n, "ms_per_step": round(ms, 5),
            "steps": reps, "launch": mode, "step_bytes": sb,
            "step_hbm_frac": round(sb / (ms * 1e-3) / 1e9 / hbm, 4),
            "note": "medusa_step_layers: every layer's projections, KV prefix and compaction; "
                    "prefix length held fixed"}


def tree_size(args, w: S.Workload, st, device, stream):
    """The tree size for this batch and context: trees of several sizes from the score table,
    built on the device (medusa_tree_greedy_device), each timed as a whole step (CUDA graph,
    prefix held fixed), and the size with the most expected tokens per unit time chosen
    (medusa_tree_size_choose) from the table's expected accepted length."""
    from medusa_head_speculative_gb300 import binding as Bnd
    sizes = [16, 32, 64, 128]
    smax = max(w.s)
    a = torch.from_numpy(S.score_table(w.K, smax)).to(device)
    nmax = max(sizes)
    par = torch.empty(nmax + 1, dtype=torch.int32, device=device)
    rnk = torch.empty_like(par)
    exp = torch.empty(nmax + 1, dtype=torch.float64, device=device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    Bnd.tree_greedy_device(list(w.s), a, nmax, par, rnk, exp)      # warm-up
    e0.record(stream)
    Bnd.tree_greedy_device(list(w.s), a, nmax, par, rnk, exp)
    e1.record(stream)
    torch.cuda.synchronize()
    build_us = e0.elapsed_time(e1) * 1e3
    expected = exp.cpu().numpy()
    dtype = Bnd.F32 if w.dtype == "f32" else Bnd.BF16
    ms_sizes = []
    for N in sizes:
        Bnd.tree_greedy_device(list(w.s), a, N, par, rnk)
        parent = par[:N + 1].cpu().numpy().astype(np.int32)
        rank = rnk[:N + 1].cpu().numpy().astype(np.int32)
        plan = Bnd.Plan(w.B, w.d, w.V, w.K, w.Hq, w.Hkv, w.dh, dtype, w.capacity, w.s, parent, rank,
                        rope_base=w.rope_base, page_size=w.page_size,
                        num_pages=w.B * w.pages_per_seq if w.page_size else 0)
        ws = torch.empty(plan.workspace_size, dtype=torch.uint8, device=device)

        def one():
            Bnd.step(plan, st["h"], None, st["wstruct"], st["kv"], st["acc"], st["outs"], ws)

        for _ in range(3):
            one()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            one()
        reps = max(1, min(args.steps, 200))
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        assert plan.status() == 0, "device status word set during the tree-size region"
        ms_sizes.append(e0.elapsed_time(e1) / reps)
        del g, ws
        plan.close()
    best = Bnd.tree_size_choose(expected, sizes, ms_sizes)
    return {"sizes": sizes, "ms_per_step": [round(x, 5) for x in ms_sizes],
            "expected_accepted": [round(float(expected[n]), 4) for n in sizes],
            "expected_tokens_per_s": [round(w.B * (1 + float(expected[n])) / (m * 1e-3), 1)
                                      for n, m in zip(sizes, ms_sizes)],
            "chosen": sizes[best], "builder_us": round(build_us, 1),
            "note": "trees built on the device from the fixed score table; expected tokens "
                    "per step = 1 + E[L] of the table (trained heads' accuracies would replace it)"}


def decode_loop(args, w: S.Workload, st, device):
    """The library's decode loop (medusa_loop_*): one captured step with root, h and the
    cache lengths carried in place, replayed back to back from the workload's prefix while
    the context grows by each step's kept tokens.  Own plan and cache, sized for the run."""
    import dataclasses
    from medusa_head_speculative_gb300 import binding as Bnd
    steps = max(2, min(args.steps, 1000))
    wl = dataclasses.replace(w, reserve=steps * (w.K + 1) + 128)
    parent, rank = st["parent"], st["rank"]
    dtype = Bnd.F32 if w.dtype == "f32" else Bnd.BF16
    plan = Bnd.Plan(w.B, w.d, w.V, w.K, w.Hq, w.Hkv, w.dh, dtype, wl.capacity, w.s, parent, rank,
                    rope_base=w.rope_base, page_size=w.page_size,
                    num_pages=w.B * wl.pages_per_seq if w.page_size else 0)
    kc, vc, pt = S.kv_cache(wl)
    kc, vc = kc.to(device), vc.to(device)
    pt = None if pt is None else pt.to(device)
    length = torch.tensor(w.lengths, dtype=torch.int32, device=device)
    ws = torch.empty(plan.workspace_size, dtype=torch.uint8, device=device)
    i32 = dict(dtype=torch.int32, device=device)
    h = st["h"].clone()
    root = torch.empty(w.B, **i32)
    kv = Bnd.kv_struct(kc, vc, length, length, pt)
    first = Bnd.outputs_struct(torch.empty(w.B, w.K + 1, **i32), torch.empty(w.B, **i32), None, h, root)
    Bnd.step(plan, h, None, st["wstruct"], kv, st["acc"], first, ws)       # root from the LM head
    tokens = torch.empty(steps, w.B, w.K + 1, **i32)
    n_acc = torch.empty(steps, w.B, **i32)
    loop = Bnd.Loop(plan, st["wstruct"], kv, st["acc"], h, root, tokens, n_acc, ws)
    stream = torch.cuda.current_stream(device)
    torch.cuda.synchronize(device)
    len0 = [int(x) for x in length.cpu()]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    loop.run(steps)
    e1.record(stream)
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / steps
    assert loop.steps() == steps and plan.status() == 0, "decode loop failed"
    mean_tok = float(n_acc.float().mean())
    res = {"value": round(1e3 / ms, 2), "unit": "steps/s", "ms_per_step": round(ms, 5),
           "steps": steps, "mean_tokens_per_step": round(mean_tok, 3),
           "tokens_per_s": round(1e3 / ms * mean_tok * w.B, 1),
           "context": [min(len0), int(length.max())], "launch": "cuda_graph (medusa_loop)"}
    loop.close()
    return res


# ----------------------------------------------------------------------- ranks
def max_over_ranks(x: float, dist, device) -> float:
    """The maximum of x over all ranks (x itself without a process group)."""
    if dist is None:
        return float(x)
    dev = device if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank: float, ms: float) -> float:
    """Units per second of the whole job when every rank processed units_per_rank in (at
    most) ms milliseconds: the replicas are independent, so their work adds up."""
    return world * units_per_rank / (ms / 1e3)


# ----------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            self.sel = vis.split(",")[device_index] if vis else str(device_index)

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.sel, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------------- setup
def setup(w: S.Workload, device, planted: bool = False):
    from medusa_head_speculative_gb300 import binding as Bnd
    if not os.path.exists(Bnd.LIB_PATH):
        from medusa_head_speculative_gb300 import build
        build.build()
    if w.tree == "cartesian":
        parent, rank = Bnd.tree_cartesian(w.s)
    else:
        parent, rank = Bnd.tree_greedy(w.s, S.score_table(w.K, max(w.s)), w.N)
    dtype = Bnd.F32 if w.dtype == "f32" else Bnd.BF16
    plan = Bnd.Plan(w.B, w.d, w.V, w.K, w.Hq, w.Hkv, w.dh, dtype, w.capacity, w.s, parent, rank,
                    rope_base=w.rope_base, page_size=w.page_size,
                    num_pages=w.B * w.pages_per_seq if w.page_size else 0)
    wts_cpu = S.planted_weights(w) if planted else S.weights(w)
    wts = {k: v.to(device) for k, v in wts_cpu.items()}
    # planted model: each sequence starts from the embedding of a token, as in decoding
    h_cpu = (wts_cpu["emb"][7:7 + w.B].float().clone() if planted else S.hidden(w))
    kc, vc, pt = S.kv_cache(w)
    st = dict(plan=plan, wts=wts, wts_cpu=wts_cpu, h_cpu=h_cpu, h=h_cpu.to(device),
              kc=kc.to(device), vc=vc.to(device), pt=None if pt is None else pt.to(device),
              length=torch.tensor(w.lengths, dtype=torch.int32, device=device),
              len_out=torch.empty(w.B, dtype=torch.int32, device=device),
              ws=torch.empty(plan.workspace_size, dtype=torch.uint8, device=device),
              parent=parent, rank=rank)
    i32 = dict(dtype=torch.int32, device=device)
    st["out"] = dict(out_tok=torch.empty(w.B, w.K + 1, **i32), n_acc=torch.empty(w.B, **i32),
                     path=torch.empty(w.B, w.K + 1, **i32),
                     h_next=torch.empty(w.B, w.d, dtype=torch.float32, device=device),
                     root_next=torch.empty(w.B, **i32))
    o = st["out"]
    st["wstruct"] = Bnd.weights_struct(wts)
    st["kv"] = Bnd.kv_struct(st["kc"], st["vc"], st["length"], st["len_out"], st["pt"])
    st["acc"] = Bnd.accept_struct(w.mode, w.temperature, w.eps, w.delta)
    st["outs"] = Bnd.outputs_struct(o["out_tok"], o["n_acc"], o["path"], o["h_next"], o["root_next"])
    return st


def run_ours(args, w: S.Workload):
    """The headline workload with every measurement, then the other workloads of
    args.also (the step, its kernels, roofline, steady state, e2e and CPU baseline) as
    sub-objects of the same line under "workloads"."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    res = measure(args, w, device, dist, world, rank, local, full=True)
    torch.cuda.empty_cache()
    subs = {}
    for name in [x for x in args.also.split(",") if x and x != w.name]:
        sub = measure(args, S.workload(name), device, dist, world, rank, local, full=False)
        torch.cuda.empty_cache()
        if sub is not None:
            subs[name] = {k: v for k, v in sub.items()
                          if k not in ("metric", "n_gpus", "higher_is_better", "scaling",
                                       "vs_baseline", "data", "launch")}
    if dist is not None:
        dist.destroy_process_group()
    if res is not None and subs:
        res["workloads"] = subs
    return res


def measure(args, w: S.Workload, device, dist, world: int, rank: int, local: int, full: bool):
    """One workload on this rank's GPU; the result dict on rank 0, None elsewhere.  With
    full, also the decode loop, the multi-layer step and the tree-size measurement."""
    from medusa_head_speculative_gb300 import binding as Bnd
    st = setup(w, device, planted=args.planted)
    plan = st["plan"]
    stream = torch.cuda.current_stream(device)

    def one_step():
        Bnd.step(plan, st["h"], None, st["wstruct"], st["kv"], st["acc"], st["outs"], st["ws"],
                 stream)

    def barrier():
        torch.cuda.synchronize(device)
        if dist is not None:
            dist.barrier()

    for _ in range(max(args.warmup, 3)):
        one_step()
    torch.cuda.synchronize(device)
    assert plan.status() == 0, "device status word set during warm-up"

    # launches per step, from one profiled step
    plan.profile_start(256)
    one_step()
    _, per_step = plan.profile_stop()

    # The step as a CUDA graph (the same kernels and arguments, replayed without per-launch
    # host overhead); direct calls if capture is not possible.
    graph, launch_mode = None, "direct"
    if not args.no_graph:
        try:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                Bnd.step(plan, st["h"], None, st["wstruct"], st["kv"], st["acc"], st["outs"],
                         st["ws"])
            g.replay()
            torch.cuda.synchronize(device)
            graph, launch_mode = g, "cuda_graph"
        except Exception as exc:                        # noqa: BLE001
            launch_mode = f"direct (graph capture failed: {exc})"[:160]
    run = graph.replay if graph is not None else one_step

    K = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier()
    clocks.start()
    time.sleep(0.3)                      # let the sampler attach before the region starts
    e0.record(stream)
    for _ in range(K):
        run()
    e1.record(stream)
    barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    launches = K * per_step
    # per-kernel times: CUDA events around every launch, in a second timed region
    kp = min(K, 300)
    plan.profile_start(kp * per_step + 16)
    for _ in range(kp):
        one_step()
    kernels, _ = plan.profile_stop()
    ms_max = max_over_ranks(ms, dist, device)
    assert plan.status() == 0, "device status word set during the timed region"
    n_acc_mean = float(st["out"]["n_acc"].float().mean())
    steady = steady_state(args, w, st, stream, barrier)
    loop = decode_loop(args, w, st, device) if full else None
    mlayer = multi_layer(args, w, st, device, stream, barrier) if full and args.layers > 1 else None
    tsize = tree_size(args, w, st, device, stream) if full and not args.no_tree_size else None

    # end to end: h_t from pinned host memory, result (tokens, counts) back, every step
    ke = min(K, 500)
    h_host = st["h_cpu"].pin_memory()
    tok_host = torch.empty(w.B, w.K + 1, dtype=torch.int32).pin_memory()
    nacc_host = torch.empty(w.B, dtype=torch.int32).pin_memory()
    h_dev = st["h"]

    def e2e_step():
        h_dev.copy_(h_host, non_blocking=True)
        Bnd.step(plan, st["h"], None, st["wstruct"], st["kv"], st["acc"], st["outs"], st["ws"])
        tok_host.copy_(st["out"]["out_tok"], non_blocking=True)
        nacc_host.copy_(st["out"]["n_acc"], non_blocking=True)

    # the copies and the step as one CUDA graph (pinned host buffers), one launch per step;
    # the host still waits for every step's result before the next
    e2e_run, e2e_mode = e2e_step, "direct"
    if graph is not None:
        try:
            ge = torch.cuda.CUDAGraph()
            with torch.cuda.graph(ge):
                e2e_step()
            ge.replay()
            torch.cuda.synchronize(device)
            e2e_run, e2e_mode = ge.replay, "cuda_graph"
        except Exception:                               # noqa: BLE001
            e2e_run, e2e_mode = e2e_step, "direct"
    barrier()
    t0 = time.perf_counter()
    e0.record(stream)
    for _ in range(ke):
        e2e_run()
        stream.synchronize()
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1)
    wall = time.perf_counter() - t0
    e2e_ms = max_over_ranks(max(e2e_ms, wall * 1e3), dist, device)
    steady_ms = max_over_ranks(steady["ms_per_step"], dist, device)
    steady.update(value=round(whole_job_rate(world, 1, steady_ms), 2), ms_per_step=round(steady_ms, 5),
                  tokens_per_s=round(whole_job_rate(world, steady["mean_tokens_per_step"] * w.B, steady_ms), 1))

    if rank != 0:
        return None

    n1 = plan.n1
    hbm, hbm_kind = peaks()
    kb = kernel_bytes(w, n1, plan_tc_heads(w))
    ktab = {}
    for name, (cnt, tot) in kernels.items():
        us = tot * 1e3 / cnt
        row = {"launches": cnt, "us_per_launch": round(us, 3),
               "share": round(tot / sum(v[1] for v in kernels.values()), 4)}
        if name in kb:
            row["gbs"] = round(kb[name] / (us * 1e-6) / 1e9, 1)
        ktab[name] = row
    kf = kernel_flops(w, n1, plan_tc_heads(w))
    tflops, tflops_kind = tensor_peak()
    ridge = tflops * 1e12 / (hbm * 1e9)                 # FLOP per byte where the bounds meet
    dom = max((n for n in kernels if n in kb), key=lambda n: kernels[n][1])
    dom_us = kernels[dom][1] * 1e3 / kernels[dom][0]
    traffic = load_traffic(w.name, dom)
    if kf.get(dom, 0) / kb[dom] > ridge:                # a dense contraction at this size
        roof = {"kernel": dom, "bound": "tensor", "achieved": round(kf[dom] / (dom_us * 1e-6) / 1e12, 1),
                "peak": tflops, "unit": "TFLOP/s",
                "frac": round(kf[dom] / (dom_us * 1e-6) / 1e12 / tflops, 4), "traffic": traffic,
                "algorithmic_flops": kf[dom],
                # fp32 activations enter the tensor cores as bf16 hi + lo halves: two MMAs
                # per product, of which only the method's one is counted above
                "issued_per_algorithmic": 2 if (dom in ("verify_logits", "layer_out")
                                                or (dom.startswith("heads") and plan_tc_heads(w))) else 1,
                "peak_source": f"{tflops_kind} (MEASURED_PEAKS.json bf16_tflops_sustained)"
                if tflops_kind == "measured" else "fallback 1.7 PFLOP/s sustained"}
    else:
        achieved = kb[dom] / (dom_us * 1e-6) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1),
                "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "traffic": traffic, "algorithmic_bytes": kb[dom],
                "peak_source": f"{hbm_kind} (MEASURED_PEAKS.json hbm_gbs)"
                if hbm_kind == "measured" else "fallback 6.8 TB/s"}
    # The whole step against its roofline: each modelled kernel bound by the slower of its
    # bytes at the HBM peak and its FLOPs at the tensor peak; the remaining kernels at zero.
    ideal_us = sum(max(kb[n] / (hbm * 1e9), kf.get(n, 0) / (tflops * 1e12)) * 1e6 for n in kb)
    steps_per_s = whole_job_rate(world, K, ms_max)
    sb = step_bytes(w, n1)
    res = {
        "metric": METRIC, "value": round(steps_per_s, 2), "unit": "steps/s", "n_gpus": world,
        "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_max / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": ("synthetic: planted weights (heads right ~70% per level), h_t = E[token], "
                 "N(0,1) KV prefix" if args.planted else
                 "synthetic: seeded N(0,1/d) weights, N(0,1) h_t and KV prefix (no trained weights)"),
        "config": config_of(w, n1),
        "tree_nodes_per_s": round(steps_per_s * w.B * n1, 1),
        "step_hbm_gbs": round(sb / (ms_max / K * 1e-3) / 1e9, 1),
        "step_hbm_frac": round(sb / (ms_max / K * 1e-3) / 1e9 / hbm, 4),
        "step_bytes": sb,
        "mean_tokens_per_step": round(n_acc_mean, 3),
        "roofline": roof,
        "step_roofline": {"ideal_us": round(ideal_us, 1), "frac": round(ideal_us / (ms_max / K * 1e3), 4),
                          "note": "per-kernel max(algorithmic bytes / HBM peak, FLOPs / bf16 "
                                  "sustained peak), summed over the modelled kernels"},
        "kernels": ktab,
        "e2e": {"value": round(whole_job_rate(world, ke, e2e_ms), 2), "unit": "steps/s",
                "h2d_bytes_per_step": int(h_host.numel() * 4),
                "d2h_bytes_per_step": int(tok_host.numel() * 4 + nacc_host.numel() * 4),
                "launch": e2e_mode, "sync": "host waits for every step's tokens"},
        "clocks": clk,
        "steady_state": dict(steady, step_hbm_frac=round(
            steady_bytes(w, n1) / (steady["ms_per_step"] * 1e-3) / 1e9 / hbm, 4),
            step_bytes=steady_bytes(w, n1)),
        "decode_loop": loop,
        "multi_layer": mlayer,
        "tree_size": tsize,
        "gpu_launches": int(launches),
        "launch": launch_mode,
    }
    for k in ("decode_loop", "multi_layer", "tree_size"):
        if res[k] is None:
            del res[k]
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, st, plan_spec=(st["parent"], st["rank"]))
    return res


def plan_tc_heads(w: S.Workload):
    return w.dtype == "bf16" and w.B >= 2


def load_traffic(workload: str, kernel: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary
    (profiles/<kernel>__<workload>.json), only while the kernel's source files still hash
    to what they were when the counters were taken; else None."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{kernel}__{workload}.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        src = b"".join(open(os.path.join(ROOT, x), "rb").read() for x in rec["source_files"])
        if hashlib.sha256(src).hexdigest()[:16] != rec["source_sha256_16"]:
            return None
        return rec.get("traffic_bytes_per_launch")
    except Exception:
        return None


# ----------------------------------------------------------------------- oracle (CPU)
def _oracle_sample_step(w, wts64, h_cpu, spec):
    import oracle as O
    k, v = S.kv_prefix(w, 0)
    dims = {"Hq": w.Hq, "Hkv": w.Hkv, "dh": w.dh, "rope_base": w.rope_base}
    acc = {"mode": w.mode, "temperature": w.temperature, "eps": w.eps, "delta": w.delta}
    t0 = time.perf_counter()
    O.medusa_step(wts64, h_cpu[0], k, v, spec, dims, acc, s=list(w.s))
    return time.perf_counter() - t0


def _oracle_spec(w):
    import oracle as O
    if w.tree == "cartesian":
        return O.cartesian_tree(w.s)
    return O.greedy_tree(S.score_table(w.K, max(w.s)), w.s, w.N)


def cpu_baseline(w, st, plan_spec=None):
    import oracle as O
    wts64 = O.oracle_weights(st["wts_cpu"])
    spec = _oracle_spec(w)
    secs = _oracle_sample_step(w, wts64, st["h_cpu"], spec)
    per_step = secs * w.B               # sequences are independent: one is 1/B of a step
    return {"value": round(1.0 / per_step, 5), "unit": "steps/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"one full oracle step of sequence 0 ({secs:.1f} s), scaled by B={w.B}"}


def run_reference(args, w: S.Workload):
    """The fp64 oracle on the host cores, on the same workload, metric and unit."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import oracle as O
    wts_cpu = S.weights(w)
    wts64 = O.oracle_weights(wts_cpu)
    h_cpu = S.hidden(w)
    spec = _oracle_spec(w)
    _oracle_sample_step(w, wts64, h_cpu, spec)          # one untimed warm-up step
    budget_s = 120.0
    times = []
    for _ in range(args.steps):
        times.append(_oracle_sample_step(w, wts64, h_cpu, spec))
        if sum(times) > budget_s:
            break
    per_step = sum(times) / len(times) * w.B
    v = 1.0 / per_step
    return {"metric": METRIC, "value": round(v, 5), "unit": "steps/s", "impl": "reference",
            "n_gpus": 0, "steps": len(times), "steps_requested": args.steps, "warmup": 1,
            "ms_per_step": round(per_step * 1e3, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic: seeded N(0,1/d) weights, N(0,1) h_t and KV prefix",
            "config": config_of(w, spec.N + 1),
            "cpu_baseline": {"value": round(v, 5), "unit": "steps/s", "cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": f"{len(times)} full oracle steps of sequence 0, scaled "
                                       f"by B={w.B}; timed steps capped at ~{budget_s:.0f} s"},
            "e2e": {"value": round(v, 5), "unit": "steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------- 33B sweep
def device_inputs(w: S.Workload, device):
    """Seeded synthetic weights, h_t and KV cache drawn on the device (torch's CUDA
    generator), with the same shapes and distributions as synthetic.inputs.  Used only for
    timing the large sweep points, where drawing tens of GB on the host would dominate."""
    gen = torch.Generator(device=device)
    dt = w.torch_dtype

    def normal(shape, std, tag):
        gen.manual_seed(w.seed * 1000003 + tag)
        return (torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
                * std).to(dt)

    d, V, K = w.d, w.V, w.K
    qd, kd = w.Hq * w.dh, w.Hkv * w.dh
    sd = 1.0 / math.sqrt(d)
    wts = {"w1": normal((K, d, d), sd, 1), "w2": normal((K, V, d), sd, 2),
           "lm": normal((V, d), sd, 3), "emb": normal((V, d), 1.0, 4),
           "wq": normal((qd, d), sd, 5), "wk": normal((kd, d), sd, 6),
           "wv": normal((kd, d), sd, 7), "wo": normal((d, qd), 1.0 / math.sqrt(qd), 8)}
    h = normal((w.B, d), 1.0, 9).float()
    kc = torch.zeros((w.B, w.capacity, w.Hkv, w.dh), dtype=dt, device=device)
    vc = torch.zeros_like(kc)
    for b in range(w.B):
        L = w.lengths[b]
        kc[b, :L] = normal((L, w.Hkv, w.dh), 1.0, 100 + 2 * b)
        vc[b, :L] = normal((L, w.Hkv, w.dh), 1.0, 101 + 2 * b)
    return wts, h, kc, vc


def run_sweep(args):
    """The Vicuna-33B-shaped grid: batch x prefix x tree size, one JSON line per point with
    steps/s and the heads' and tree attention's HBM GB/s (separately)."""
    from medusa_head_speculative_gb300 import binding as Bnd
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    hbm, _ = peaks()
    tflops, _ = tensor_peak()
    Bs = [int(x) for x in args.sweep_b.split(",")]
    Ls = [int(x) for x in args.sweep_l.split(",")]
    Ns = [int(x) for x in args.sweep_n.split(",")]
    wts = None
    for N in Ns:
        for B in Bs:
            for L in Ls:
                w = S.vicuna33b(B, L, N)
                parent, rank = Bnd.tree_greedy(w.s, S.score_table(w.K, max(w.s)), w.N)
                plan = Bnd.Plan(w.B, w.d, w.V, w.K, w.Hq, w.Hkv, w.dh, Bnd.BF16, w.capacity,
                                w.s, parent, rank, rope_base=w.rope_base)
                wp, h, kc, vc = device_inputs(w, device)
                if wts is None:
                    wts = wp
                else:
                    del wp
                length = torch.tensor(w.lengths, dtype=torch.int32, device=device)
                len_out = torch.empty_like(length)
                ws = torch.empty(plan.workspace_size, dtype=torch.uint8, device=device)
                i32 = dict(dtype=torch.int32, device=device)
                outs = Bnd.outputs_struct(torch.empty(B, w.K + 1, **i32), torch.empty(B, **i32),
                                          torch.empty(B, w.K + 1, **i32),
                                          torch.empty(B, w.d, dtype=torch.float32, device=device),
                                          torch.empty(B, **i32))
                wst = Bnd.weights_struct(wts)
                kv = Bnd.kv_struct(kc, vc, length, len_out, None)
                acc = Bnd.accept_struct("greedy", 0.0, 0.09, 0.3)

                def one():
                    Bnd.step(plan, h, None, wst, kv, acc, outs, ws)

                for _ in range(3):
                    one()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    one()
                g.replay()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                for _ in range(args.steps):
                    g.replay()
                e1.record()
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1) / args.steps
                plan.profile_start(8 * 32)
                for _ in range(8):
                    one()
                kern, _ = plan.profile_stop()
                status = plan.status()
                n1 = plan.n1
                kb = kernel_bytes(w, n1, plan_tc_heads(w))
                t = {k: v[1] / v[0] for k, v in kern.items()}          # ms per launch
                heads_ms = t.get("heads_w1", 0) + t.get("heads_vocab", 0) + t.get("split_h", 0)
                attn_ms = t.get("tree_attention", 0) + t.get("attn_combine", 0) + t.get("cast_q", 0)
                sb = step_bytes(w, n1)
                kf = kernel_flops(w, n1, plan_tc_heads(w))
                ideal_us = sum(max(kb[k] / (hbm * 1e9), kf.get(k, 0) / (tflops * 1e12)) * 1e6 for k in kb)
                row = {"sweep": "vicuna33b", "B": B, "prefix": L, "tree_nodes": n1,
                       "steps_per_s": round(1e3 / ms, 2), "ms_per_step": round(ms, 4),
                       "tree_nodes_per_s": round(1e3 / ms * B * n1, 1),
                       "step_hbm_gbs": round(sb / (ms * 1e-3) / 1e9, 1),
                       "step_hbm_frac": round(sb / (ms * 1e-3) / 1e9 / hbm, 4),
                       "medusa_heads_gbs": round((kb["heads_w1"] + kb["heads_vocab"])
                                                 / (heads_ms * 1e-3) / 1e9, 1),
                       "tree_attention_gbs": round(kb["tree_attention"] / (attn_ms * 1e-3) / 1e9, 1),
                       "step_roofline_frac": round(ideal_us / (ms * 1e3), 4),
                       "kernels_us": {k: round(v * 1e3, 1) for k, v in t.items()},
                       "status": status}
                print(json.dumps(row), flush=True)
                del g, plan, ws, kc, vc, h, kv
                torch.cuda.empty_cache()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="vicuna13b",
                    help="headline workload (default: the Vicuna-13B-shaped batch of 8)")
    ap.add_argument("--also", default="vicuna7b,zephyr7b",
                    help="further workloads measured into the same line ('' for none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="time direct calls, not a CUDA graph")
    ap.add_argument("--no-tree-size", action="store_true", help="skip the tree-size measurement")
    ap.add_argument("--layers", type=int, default=4,
                    help="backbone layers of the multi_layer measurement (1: skip it)")
    ap.add_argument("--planted", action="store_true",
                    help="planted weights whose heads are often right (long accepted paths)")
    ap.add_argument("--sweep", action="store_true",
                    help="Vicuna-33B-shaped grid instead of the default workload")
    ap.add_argument("--sweep-b", default="1,4,16,64")
    ap.add_argument("--sweep-l", default="1024,4096,16384")
    ap.add_argument("--sweep-n", default="16,64,128")
    args = ap.parse_args()
    if args.sweep:
        run_sweep(args)
        return
    w = S.workload(args.workload)
    res = run_reference(args, w) if args.impl == "reference" else run_ours(args, w)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
