#!/usr/bin/env python3
"""Benchmark of the speculative-decoding verify step on GB300.

One step = one verify pass of a 9B-class decoder at T = 32 drafted tokens:
36 layers of int4 asymmetric group-64 projections (fused q/k/v 4096->6144,
o 4096->4096, fused gate/up 4096->24576, down 12288->4096), the int4 LM head
(4096 -> 151936, fp32 logits), then the acceptance rule over 32 drafts on
V = 151936 (softmax, min(1, p/q) tests, residual resample / bonus token).
The synthetic draft distributions rotate over three acceptance levels
(~0.3, ~0.6, ~0.9).  Weights (4.08 GB) are drawn on the device from a seeded
generator; they exceed L2, so no step reuses another's cached weights.

Printed: one JSON line.  `value` is algorithmic HBM bytes per step / device
time per step (GB/s) with inputs resident; `e2e` is the same metric when
every step also copies its inputs from pinned host memory (double-buffered
against the previous step's compute) and reads its result back.  The GEMMs
run on the engine `--engine` names (default: the split engine, one launch
per GEMM); `stack_engine` times the step's GEMM stack and the 27B-class
stack on the persistent engine for comparison.  Sub-objects time, each on
its own graph: `t16` (the stack at T = 16 without head and acceptance),
`t16_unfused` (seven GEMMs per layer), `per_gemm_launches` (one
qgemm_w4a16 call per GEMM), `w4_rot32` (the T = 32 stack with the block-32
rotation), `w8_27b` (the 27B-class int8 stack with rotation),
`accept_gumbel` (shared-seed acceptance of the same blocks) and
`accept_tree` (greedy trees of 1 to 64 nodes).  `--impl reference` times the
fp64 CPU oracle on a bounded sample instead; `--kernel-case`,
`--kernel-case-w8`, `--stack-case`, `--accept-case`, `--gumbel-case` and
`--tree-case` time one kernel alone.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from bit_qgemm_w4_gb300 import inputs  # noqa: E402

T_MAIN, T_SMALL = 32, 16
VOCAB = inputs.VOCAB_9B
HIDDEN = 4096
GROUP = 64
ACCEPT_LEVELS = (0.3, 0.6, 0.9)
GUMBEL_SEED = 0x5EED0000   # seed shared by the drafter and the verifier in the timed runs
FALLBACK_HBM_GBS = 6800.0
METRIC = "verify-step HBM GB/s (% of peak) and draft tokens scored/s at T=16/32, int4 9B-class"
WORKLOAD = ("9B-class int4 g64 verify step, T=32: 36 layers (qkv 4096x6144, o 4096x4096, "
            "gate_up 4096x24576, down 12288x4096) + LM head 4096x151936 (fp32 logits) + "
            "softmax/accept over V=151936")


# ----------------------------------------------------------------------------
# algorithmic bytes
# ----------------------------------------------------------------------------

def w4_gemm_bytes(T: int, N: int, K: int, g: int = GROUP, out_bytes: int = 2) -> int:
    """Bytes a W4A16 GEMM must move: packed codes (0.5 B/weight), fp16 scales
    and uint4 zeros per group, bf16 activations in, outputs out."""
    return N * K // 2 + (K // g) * N * 2 + (K // g) * (N // 2) + T * K * 2 + T * N * out_bytes


def w8_gemm_bytes(T: int, N: int, K: int, out_bytes: int = 2) -> int:
    """Bytes a per-channel W8A16 GEMM must move: int8 codes, one fp16 scale per
    output channel, bf16 activations in, outputs out (a rotation pre-pass adds
    its own 4*T*K, counted separately)."""
    return N * K + N * 2 + T * K * 2 + T * N * out_bytes


def stack_bytes(T: int) -> int:
    return inputs.LAYERS_9B * sum(w4_gemm_bytes(T, N, K) for _, K, N in inputs.LAYER_9B)


def head_bytes(T: int) -> int:
    return w4_gemm_bytes(T, VOCAB, HIDDEN, out_bytes=4)


def accept_bytes(T: int, V: int = VOCAB) -> int:
    """Target logits of all T+1 rows once, plus the one draft-probability row
    the final draw needs."""
    return (T + 1) * V * 4 + V * 4


def accept_gumbel_bytes(T: int, V: int = VOCAB) -> int:
    """Shared-seed acceptance: the logits once plus the drafts and outputs."""
    return (T + 1) * V * 4 + T * 4 + (T + 2) * 4


def step_bytes(T: int = T_MAIN) -> int:
    return stack_bytes(T) + head_bytes(T) + accept_bytes(T)


# ----------------------------------------------------------------------------
# peaks, clocks, ncu traffic
# ----------------------------------------------------------------------------

def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for key in ("hbm_gbs_burst", "hbm_gbs", "hbm_GBps"):
                if key in d and isinstance(d[key], (int, float)):
                    return float(d[key]), "measured"
            if isinstance(d.get("hbm"), dict):
                for key in ("burst_gbs", "gbs"):
                    if key in d["hbm"]:
                        return float(d["hbm"][key]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the GPU works."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


ENGINES = {"auto": 0, "split": 1, "stack": 2}   # SPEC_GEMM_ENGINE_*


def open_ctx(args, device: int):
    """A context on `device` whose GEMMs run on the engine --engine names."""
    import bit_qgemm_w4_gb300 as sv
    ctx = sv.Context(device)
    sv.spec_set_gemm_engine(ctx, ENGINES[args.engine])
    return ctx


def kernel_source_hash(name: str = "qgemm_split.cu") -> str:
    p = os.path.join(ROOT, "bit_qgemm_w4_gb300", "csrc", name)
    return hashlib.sha256(open(p, "rb").read()).hexdigest()[:16]


def ncu_traffic(key: str):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, or None when the kernel source changed since the capture."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p)).get(key)
    except Exception:
        return None
    src = d.get("source") if d else None
    if not src or d.get("source_sha256_16") != kernel_source_hash(src):
        return None
    return d.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------
# distributed helpers (replicas only: each rank runs its own verify step)
# ----------------------------------------------------------------------------

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def dist_barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_gbs(world: int, bytes_per_step: int, ms_per_step: float) -> float:
    """Whole-job throughput of `world` replicas: every rank processes one
    step's bytes per step, and a step takes the slowest rank's time."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


def dist_max(world, value: float, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ----------------------------------------------------------------------------

def host_layer0(seed: int = 4242):
    """Layer-0 weights, activations and one acceptance input set on the host
    (numpy generators; value distributions as the device stack)."""
    import numpy as np
    rng = np.random.default_rng(seed)
    layer, xs = [], []
    for _, K, N in inputs.LAYER_9B:
        W = inputs.w4_weights(rng, N, K, GROUP, keep_raw=False)
        layer.append({"qcodes": W.qcodes, "scales": W.scales, "zeros": W.zeros})
        xs.append(inputs.activations(rng, T_MAIN, K))
    sigma = inputs.fit_noise_for_acceptance(0.6, VOCAB, 3.0, seed=60)
    acc = inputs.accept_inputs(rng, T_MAIN, VOCAB, logit_std=3.0, noise_std=sigma)
    return layer, xs, acc


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def run_gpu(args):
    import numpy as np
    import torch

    import bit_qgemm_w4_gb300 as sv
    from bit_qgemm_w4_gb300 import build as svbuild

    world, rank, local = dist_setup()
    svbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ctx = open_ctx(args, local)
    gen = torch.Generator(device=dev)
    gen.manual_seed(20240 + rank)

    # ---- weights and activations (device-resident)
    layers = [[inputs.w4_weights_device(gen, N, K, dev, GROUP) for _, K, N in inputs.LAYER_9B]
              for _ in range(inputs.LAYERS_9B)]
    head = inputs.w4_weights_device(gen, VOCAB, HIDDEN, dev, GROUP)
    # every activation of a step lives in one device buffer (views per GEMM),
    # so the end-to-end run stages a step's activations with one copy
    x_elems = inputs.LAYERS_9B * sum(T_MAIN * K for _, K, _ in inputs.LAYER_9B) + T_MAIN * HIDDEN
    x_flat = torch.empty(x_elems, dtype=torch.bfloat16, device=dev)

    def x_views(flat, fill):
        off, out = 0, []
        for _ in range(inputs.LAYERS_9B):
            row = []
            for _, K, _ in inputs.LAYER_9B:
                v = flat[off:off + T_MAIN * K].view(T_MAIN, K)
                if fill:
                    v.copy_(inputs.activations_device(gen, T_MAIN, K, dev))
                row.append(v)
                off += T_MAIN * K
            out.append(row)
        xh = flat[off:off + T_MAIN * HIDDEN].view(T_MAIN, HIDDEN)
        if fill:
            xh.copy_(inputs.activations_device(gen, T_MAIN, HIDDEN, dev))
        return out, xh

    xs, x_head = x_views(x_flat, True)
    ys = [torch.empty((T_MAIN, N), dtype=torch.bfloat16, device=dev) for _, _, N in inputs.LAYER_9B]
    logits_head = torch.empty((T_MAIN, VOCAB), dtype=torch.float32, device=dev)

    # ---- acceptance inputs: three sweep points (host-generated, seeded)
    acc_sets = []
    for i, level in enumerate(ACCEPT_LEVELS):
        sigma = inputs.fit_noise_for_acceptance(level, VOCAB, 3.0, seed=10 + i)
        rng = np.random.default_rng(77 + i)
        a = inputs.accept_inputs(rng, T_MAIN, VOCAB, logit_std=3.0, noise_std=sigma)
        acc_sets.append({
            "host": a, "sigma": sigma, "level": level,
            "logits": torch.from_numpy(a.logits).to(dev), "q": torch.from_numpy(a.q).to(dev),
            "drafts": torch.from_numpy(a.drafts).to(dev), "u": torch.from_numpy(a.u).to(dev),
            "n": torch.zeros(1, dtype=torch.int32, device=dev),
            "tok": torch.zeros(T_MAIN + 1, dtype=torch.int32, device=dev),
        })

    def w4_desc(w, x, y, T, wait_prev=1):
        return {"quant": sv.SPEC_QUANT_W4, "qcodes": w["qcodes"], "scales": w["scales"],
                "zeros": w["zeros"], "group_size": w["g"], "x": x, "y": y, "T": T, "N": w["N"],
                "K": w["K"], "wait_prev": wait_prev}

    def stack_descs(T, xs_b, xh_b, with_head):
        # every GEMM waits for its predecessor (the decoder's dependency chain)
        d = [w4_desc(layers[l][j], xs_b[l][j][:T], ys[j][:T], T)
             for l in range(inputs.LAYERS_9B) for j in range(len(inputs.LAYER_9B))]
        if with_head:
            d.append(w4_desc(head, xh_b, logits_head, T))
        return d

    st32 = sv.GemmStack(ctx, stack_descs(T_MAIN, xs, x_head, True))
    st16 = sv.GemmStack(ctx, stack_descs(T_SMALL, xs, x_head, False))

    def gemm_part():
        st32.run()

    def accept_part(i):
        a = acc_sets[i]
        sv.spec_accept(ctx, a["logits"], a["q"], a["drafts"], a["u"], T_MAIN, VOCAB, a["n"], a["tok"])

    side = torch.cuda.Stream(device=dev)

    def graph_of(fn):
        fn()
        sv.spec_sync_status(ctx)
        g = torch.cuda.CUDAGraph()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                fn()
        torch.cuda.synchronize()
        return g

    def time_graph(g, reps, warm=2):
        for _ in range(warm):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        sv.spec_sync_status(ctx)
        return e0.elapsed_time(e1) / reps

    # ---- eager warm-up (also checks the device error word), then graphs
    g_gemm = graph_of(gemm_part)
    g_acc = [graph_of(lambda i=i: accept_part(i)) for i in range(3)]
    g_t16 = graph_of(st16.run)

    K, W = args.steps, args.warmup
    for i in range(W):
        g_gemm.replay()
        g_acc[i % 3].replay()
        g_t16.replay()
    torch.cuda.synchronize()

    # ---- timed region: full verify steps, inputs resident
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    dist_barrier(world)
    torch.cuda.synchronize()
    for i in range(K):
        evs[i][0].record()
        g_gemm.replay()
        evs[i][1].record()
        g_acc[i % 3].replay()
        evs[i][2].record()
    torch.cuda.synchronize()
    dist_barrier(world)
    total_ms = evs[0][0].elapsed_time(evs[K - 1][2])
    gemm_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    acc_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    step_times = sorted(e[0].elapsed_time(e[2]) for e in evs)
    step_ms_med = statistics.median(step_times)
    step_ms_p10 = step_times[int(0.1 * (len(step_times) - 1))]
    step_ms_p90 = step_times[int(round(0.9 * (len(step_times) - 1)))]
    sv.spec_sync_status(ctx)

    # outputs of the last timed step, kept for the CPU-oracle leg's comparison
    check_layer = inputs.LAYERS_9B - 1
    kept = {"ys": [y.float().cpu().numpy() for y in ys], "logits": logits_head.cpu().numpy(),
            "acc": [(int(a["n"].item()), a["tok"].cpu().numpy()) for a in acc_sets]}

    # ---- T=16 stack (configs' T=16 verify GEMM pass)
    t16_ms = time_graph(g_t16, max(K, 10))

    # ---- the same T=32 GEMMs as 145 separate calls (one launch each)
    def per_gemm_part():
        for l in range(inputs.LAYERS_9B):
            for j in range(len(inputs.LAYER_9B)):
                w = layers[l][j]
                sv.qgemm_w4a16(ctx, w["qcodes"], w["scales"], w["zeros"], GROUP, xs[l][j], ys[j],
                               T_MAIN, w["N"], w["K"])
        sv.qgemm_w4a16(ctx, head["qcodes"], head["scales"], head["zeros"], GROUP, x_head, logits_head,
                       T_MAIN, VOCAB, HIDDEN)

    g_pg = graph_of(per_gemm_part)
    pg_ms = time_graph(g_pg, max(5, min(K, 20)))
    del g_pg

    # ---- the same T=32 stack (36 layers + LM head) with the block-32 random
    # Hadamard rotation of every GEMM's activations inside the launch
    s32 = {k_: torch.from_numpy(inputs.hadamard_signs(np.random.default_rng(400 + k_), k_)).to(dev)
           for k_ in sorted({k for _, k, _ in inputs.LAYER_9B} | {HIDDEN})}
    st32r = sv.GemmStack(ctx, [dict(d, signs=s32[d["K"]], hadamard_block=32)
                               for d in stack_descs(T_MAIN, xs, x_head, True)])
    g_r32 = graph_of(st32r.run)
    r32_ms = time_graph(g_r32, max(5, min(K, 20)))
    del g_r32, st32r

    # ---- config 1 as stated: q, k, v, o, gate, up, down as seven GEMMs per
    # layer at T=16 (q/k/v share their input, so k and v do not wait for q; up
    # does not wait for gate).  The codes are row ranges of the fused
    # matrices; their scales and zero points are copied into contiguous
    # per-projection arrays.
    def split_w(w, r0, r1):
        return {"N": r1 - r0, "K": w["K"], "g": w["g"], "qcodes": w["qcodes"][r0:r1],
                "scales": w["scales"][:, r0:r1].contiguous(),
                "zeros": w["zeros"][:, r0 // 2:r1 // 2].contiguous()}

    unf_descs, unf_keep = [], []
    y_unf = [torch.empty((T_SMALL, n), dtype=torch.bfloat16, device=dev)
             for n in (4096, 1024, 1024, 4096, 12288, 12288, 4096)]
    for l in range(inputs.LAYERS_9B):
        qkv, o, gu, down = layers[l]
        parts = [(split_w(qkv, 0, 4096), 0, 1), (split_w(qkv, 4096, 5120), 0, 0),
                 (split_w(qkv, 5120, 6144), 0, 0), (o, 1, 1), (split_w(gu, 0, 12288), 2, 1),
                 (split_w(gu, 12288, 24576), 2, 0), (down, 3, 1)]
        for p_i, (w, j, wp) in enumerate(parts):
            unf_keep.append(w)
            unf_descs.append(w4_desc(w, xs[l][j][:T_SMALL], y_unf[p_i], T_SMALL, wp))
    st_unf = sv.GemmStack(ctx, unf_descs)
    g_unf = graph_of(st_unf.run)
    unf_ms = time_graph(g_unf, max(K, 10))
    del g_unf, st_unf, unf_keep, y_unf

    # ---- shared-seed (Gumbel-max) acceptance of the same T=32 blocks: the
    # drafter's tokens are sampled on the GPU from log q with the same seed
    # and positions as the verification (one launch over the logits)
    gum = []
    for i, a in enumerate(acc_sets):
        logq = torch.from_numpy(np.log(a["host"].q).astype(np.float32)).to(dev)
        d = torch.zeros(T_MAIN, dtype=torch.int32, device=dev)
        sv.spec_gumbel_sample(ctx, logq, T_MAIN, VOCAB, GUMBEL_SEED + i, 0, d)
        gum.append({"drafts": d, "n": torch.zeros(1, dtype=torch.int32, device=dev),
                    "tok": torch.zeros(T_MAIN + 1, dtype=torch.int32, device=dev)})

    def gumbel_part(i):
        g = gum[i]
        sv.spec_accept_gumbel(ctx, acc_sets[i]["logits"], g["drafts"], T_MAIN, VOCAB,
                              GUMBEL_SEED + i, 0, g["n"], g["tok"])

    g_gum = [graph_of(lambda i=i: gumbel_part(i)) for i in range(3)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    KG = max(K, 30)
    e0.record()
    for i in range(KG):
        g_gum[i % 3].replay()
    e1.record()
    torch.cuda.synchronize()
    gum_ms = e0.elapsed_time(e1) / KG
    sv.spec_sync_status(ctx)

    # ---- greedy tree acceptance over V=151936: T in {1, 4, 8, 16, 32, 64}
    # nodes as max(1, T/8) branches of depth min(T, 8), drafts matching the
    # row argmax with p = 0.7
    tree_res = []
    for Tt in (1, 4, 8, 16, 32, 64):
        tin = inputs.tree_inputs(np.random.default_rng(500 + Tt), Tt, VOCAB, logit_std=3.0, p_match=0.7)
        tbuf = {"l": torch.from_numpy(tin.logits).to(dev), "d": torch.from_numpy(tin.drafts).to(dev),
                "p": torch.from_numpy(tin.parent).to(dev),
                "n": torch.zeros(1, dtype=torch.int32, device=dev),
                "t": torch.zeros(Tt + 1, dtype=torch.int32, device=dev),
                "k": torch.zeros(Tt, dtype=torch.int32, device=dev)}

        def tree_call(b=tbuf, T_=Tt):
            sv.spec_accept_tree(ctx, b["l"], b["d"], b["p"], T_, VOCAB, b["n"], b["t"], b["k"])

        g_tree = graph_of(tree_call)
        t_ms = time_graph(g_tree, max(K, 30), warm=3)
        tree_res.append({"T": Tt, "branches": max(1, Tt // 8), "depth": min(Tt, 8), "ms": round(t_ms, 5),
                         "logits_GB/s": round((Tt + 1) * VOCAB * 4 / (t_ms * 1e-3) / 1e9, 1),
                         "path_len": int(tbuf["n"].item())})
        del tbuf, g_tree

    # ---- 27B-class Large tier: 64 layers of per-channel int8 projections at
    # T=32, with and without the block-1024 random Hadamard rotation of every
    # GEMM's activations (rotated inside the same launch)
    L8 = inputs.LAYER_27B
    w8 = [[inputs.w8_weights_device(gen, N, K, dev) for _, K, N in L8] for _ in range(inputs.LAYERS_27B)]
    x8 = [inputs.activations_device(gen, T_MAIN, K, dev) for _, K, _ in L8]
    y8 = [torch.empty((T_MAIN, N), dtype=torch.bfloat16, device=dev) for _, _, N in L8]
    s8 = [torch.from_numpy(inputs.hadamard_signs(np.random.default_rng(300 + j), K)).to(dev)
          for j, (_, K, _) in enumerate(L8)]

    def w8_descs(rotate):
        return [{"quant": sv.SPEC_QUANT_W8, "qcodes": w8[l][j]["qcodes"], "scales": w8[l][j]["scales"],
                 "zeros": None, "group_size": 0, "x": x8[j], "y": y8[j], "T": T_MAIN, "N": N, "K": K,
                 "signs": s8[j] if rotate else None, "hadamard_block": 1024 if rotate else 0,
                 "wait_prev": 1}
                for l in range(inputs.LAYERS_27B) for j, (_, K, N) in enumerate(L8)]

    st8 = sv.GemmStack(ctx, w8_descs(True))
    st8n = sv.GemmStack(ctx, w8_descs(False))
    g_w8 = graph_of(st8.run)
    g_w8n = graph_of(st8n.run)
    K8 = max(5, min(K, 20))
    w8_ms = time_graph(g_w8, K8)
    w8n_ms = time_graph(g_w8n, K8)
    w8_bytes = inputs.LAYERS_27B * sum(w8_gemm_bytes(T_MAIN, N, K) for _, K, N in L8)
    # ---- the other engine on the same T=32 stack and 27B rotated stack
    other = "stack" if ENGINES[args.engine] != ENGINES["stack"] else "split"
    sv.spec_set_gemm_engine(ctx, ENGINES[other])
    g_o32 = graph_of(st32.run)
    o32_ms = time_graph(g_o32, max(5, min(K, 20)))
    g_o8 = graph_of(st8.run)
    o8_ms = time_graph(g_o8, K8)
    sv.spec_set_gemm_engine(ctx, ENGINES[args.engine])
    del g_o32, g_o8
    del g_w8, g_w8n, st8, st8n, w8
    clocks = sampler.stop()
    sv.spec_sync_status(ctx)

    # ---- end to end: inputs copied from pinned host memory every step,
    # result (accepted count + tokens) read back every step.  The device
    # inputs are double-buffered: step i+1's copy runs on a copy stream while
    # step i computes (each step still copies all of its own inputs inside
    # the timed region).
    pin = lambda t: t.detach().cpu().pin_memory()  # noqa: E731
    h_xflat = pin(x_flat)
    keys = ("logits", "q", "drafts", "u")
    h_acc = [{k: pin(a[k]) for k in keys} for a in acc_sets]
    h_out = [torch.empty(1, dtype=torch.int32).pin_memory(),
             torch.empty(T_MAIN + 1, dtype=torch.int32).pin_memory()]
    h2d = h_xflat.numel() * h_xflat.element_size() + \
        sum(v.numel() * v.element_size() for v in h_acc[0].values())
    d2h = 4 * (T_MAIN + 2)

    x_flat2 = torch.empty_like(x_flat)
    xs2, x_head2 = x_views(x_flat2, False)
    x_flat2.copy_(x_flat)
    stacks_e = [st32, sv.GemmStack(ctx, stack_descs(T_MAIN, xs2, x_head2, True))]
    ebuf = [{k: torch.empty_like(acc_sets[0][k]) for k in keys + ("n", "tok")} for _ in range(2)]

    def accept_on(b):
        e = ebuf[b]
        sv.spec_accept(ctx, e["logits"], e["q"], e["drafts"], e["u"], T_MAIN, VOCAB, e["n"], e["tok"])

    for b in range(2):
        for k in keys:
            ebuf[b][k].copy_(acc_sets[b][k])
    g_gemm_e = [graph_of(stacks_e[b].run) for b in range(2)]
    g_acc_e = [graph_of(lambda b=b: accept_on(b)) for b in range(2)]
    comp = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    result = torch.cuda.Event()
    for b in range(2):
        done[b].record(comp)
    K_e2e = max(10, min(K, 200))
    e2e_evs = [torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)]
    xbuf = [x_flat, x_flat2]

    def issue_copy(i):
        b = i % 2
        with torch.cuda.stream(copy_stream):
            if i == 0:
                copy_stream.wait_event(e2e_evs[0])
            copy_stream.wait_event(done[b])          # step i-2 has finished with buffer b
            xbuf[b].copy_(h_xflat, non_blocking=True)
            for k in keys:
                ebuf[b][k].copy_(h_acc[i % 3][k], non_blocking=True)
            copied[b].record(copy_stream)

    torch.cuda.synchronize()
    dist_barrier(world)
    e2e_evs[0].record(comp)
    issue_copy(0)
    for i in range(K_e2e):
        b = i % 2
        comp.wait_event(copied[b])
        g_gemm_e[b].replay()
        g_acc_e[b].replay()
        done[b].record(comp)
        h_out[0].copy_(ebuf[b]["n"], non_blocking=True)
        h_out[1].copy_(ebuf[b]["tok"], non_blocking=True)
        result.record(comp)
        if i + 1 < K_e2e:
            issue_copy(i + 1)
        result.synchronize()                       # the host reads the result
        _ = int(h_out[0][0])
    e2e_evs[1].record(comp)
    torch.cuda.synchronize()
    e2e_ms = e2e_evs[0].elapsed_time(e2e_evs[1]) / K_e2e
    sv.spec_sync_status(ctx)

    total_ms = dist_max(world, total_ms, dev)
    e2e_ms = dist_max(world, e2e_ms, dev)
    ms_per_step = total_ms / K
    nbytes = step_bytes()
    gemm_bytes = stack_bytes(T_MAIN) + head_bytes(T_MAIN)
    n_gemm = inputs.LAYERS_9B * len(inputs.LAYER_9B) + 1   # GEMM launches per step (split engine)
    peak, peak_kind = hbm_peak()
    achieved = gemm_bytes / (gemm_ms * 1e-3) / 1e9
    accepted = []
    for a in acc_sets:
        accepted.append({"level": a["level"], "sigma": round(a["sigma"], 4),
                         "n_accepted": int(a["n"].item())})

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_oracle_leg(layers[check_layer], xs[check_layer], head, x_head, acc_sets, kept,
                             args.cpu_budget)

    if rank == 0:
        out = {
            "metric": METRIC,
            "value": round(whole_job_gbs(world, nbytes, ms_per_step), 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": K,
            "warmup": W,
            "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "int4 weights x bf16 activations, fp32 accumulate",
            "data": "synthetic (seeded; weights drawn on device, value distributions of the "
                    "configs)",
            "config": {
                "workload": WORKLOAD,
                "T": T_MAIN, "layers": inputs.LAYERS_9B, "hidden": HIDDEN, "vocab": VOCAB,
                "group_size": GROUP, "bytes_per_step": nbytes,
                "acceptance_levels": list(ACCEPT_LEVELS),
                "l2": "inputs larger than L2 (4.08 GB of weights per step)",
                "parallelism": f"replicas x{world}",
                "engine": args.engine,
                "graph": ("one CUDA graph per step part: the GEMM stack (145 launches, one per "
                          "GEMM, each starting its weight stream while its predecessor ends and "
                          "reading its activations once that one has finished)"
                          if ENGINES[args.engine] != ENGINES["stack"] else
                          "one CUDA graph per step part: the GEMM stack (one persistent launch of "
                          "all 145 GEMMs, each waiting for its predecessor)") +
                         " and the acceptance (two launches)",
            },
            "pct_of_peak": round(100.0 * nbytes / (ms_per_step * 1e-3) / 1e9 / peak, 2),
            "draft_tokens_scored_per_s": round(world * T_MAIN / (ms_per_step * 1e-3), 1),
            "verify_step_ms_median": round(step_ms_med, 5),
            "verify_step_ms_p10": round(step_ms_p10, 5),
            "verify_step_ms_p90": round(step_ms_p90, 5),
            "acceptance_ms": round(acc_ms, 5),
            "acceptance_share": round(acc_ms / (gemm_ms + acc_ms), 4),
            "accepted": accepted,
            "per_gemm_launches": {
                "workload": "the same T=32 GEMMs (36 layers + head) as 145 separate qgemm_w4a16 "
                            "calls in one graph (no acceptance)",
                "ms": round(pg_ms, 5),
                "value": round(gemm_bytes / (pg_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "frac": round(gemm_bytes / (pg_ms * 1e-3) / 1e9 / peak, 4),
            },
            "accept_gumbel": {
                "workload": "shared-seed (Gumbel-max) acceptance of the same T=32 blocks over "
                            "V=151936: one launch reads the (T+1)xV fp32 logits once; the drafts "
                            "are sampled on the GPU from the same q with the same seed",
                "ms": round(gum_ms, 5),
                "share_if_used_in_step": round(gum_ms / (gemm_ms + gum_ms), 4),
                "logits_GB/s": round(accept_gumbel_bytes(T_MAIN) / (gum_ms * 1e-3) / 1e9, 1),
                "accepted": [{"level": a["level"], "n_accepted": int(g["n"].item())}
                             for a, g in zip(acc_sets, gum)],
            },
            "accept_tree": {
                "workload": "greedy tree acceptance over V=151936 (one launch; reads the (T+1)xV "
                            "fp32 logits once)",
                "cases": tree_res,
            },
            "t16": {
                "workload": "same 36-layer int4 stack at T=16 (no head, no acceptance), one stack "
                            "run",
                "ms_per_step": round(t16_ms, 5),
                "value": round(stack_bytes(T_SMALL) / (t16_ms * 1e-3) / 1e9, 2),
                "unit": "GB/s",
                "frac": round(stack_bytes(T_SMALL) / (t16_ms * 1e-3) / 1e9 / peak, 4),
                "draft_tokens_scored_per_s": round(T_SMALL / (t16_ms * 1e-3), 1),
            },
            "t16_unfused": {
                "workload": "the T=16 stack as the configuration states it: q, k, v, o, gate, up, "
                            "down as 7 GEMMs per layer (252 GEMMs, one stack run; on the stack "
                            "engine k, v and up do not wait for the GEMM before them)",
                "ms_per_step": round(unf_ms, 5),
                "value": round(stack_bytes(T_SMALL) / (unf_ms * 1e-3) / 1e9, 2),
                "unit": "GB/s",
                "frac": round(stack_bytes(T_SMALL) / (unf_ms * 1e-3) / 1e9 / peak, 4),
            },
            "w4_rot32": {
                "workload": "the T=32 verify GEMM stack (36 layers + LM head) with the block-32 "
                            "random Hadamard rotation of every GEMM's activations (split engine: "
                            "a rotation launch before each GEMM; stack engine: inside the launch)",
                "ms_per_step": round(r32_ms, 5),
                "value": round(gemm_bytes / (r32_ms * 1e-3) / 1e9, 2),
                "unit": "GB/s",
                "frac": round(gemm_bytes / (r32_ms * 1e-3) / 1e9 / peak, 4),
                "without_rotation_ms": round(gemm_ms, 5),
                "rotation_overhead": round(r32_ms / gemm_ms - 1.0, 4),
            },
            "w8_27b": {
                "workload": "27B-class int8 per-channel stack at T=32: 64 layers (qkv 5120x7168, "
                            "o 5120x5120, gate_up 5120x34816, down 17408x5120), block-1024 random "
                            "Hadamard rotation of every GEMM's activations (no head, no "
                            "acceptance)",
                "ms_per_step": round(w8_ms, 5),
                "bytes_per_step": w8_bytes,
                "value": round(w8_bytes / (w8_ms * 1e-3) / 1e9, 2),
                "unit": "GB/s",
                "frac": round(w8_bytes / (w8_ms * 1e-3) / 1e9 / peak, 4),
                "draft_tokens_scored_per_s": round(T_MAIN / (w8_ms * 1e-3), 1),
                "without_rotation_ms": round(w8n_ms, 5),
                "rotation_overhead": round(w8_ms / w8n_ms - 1.0, 4),
            },
            "stack_engine" if other == "stack" else "split_engine": {
                "workload": f"the same T=32 verify GEMM stack and 27B-class int8 rotated stack on "
                            f"the {other} engine",
                "t32_ms": round(o32_ms, 5),
                "t32_value": round(gemm_bytes / (o32_ms * 1e-3) / 1e9, 2),
                "t32_frac": round(gemm_bytes / (o32_ms * 1e-3) / 1e9 / peak, 4),
                "w8_27b_ms": round(o8_ms, 5),
                "w8_27b_value": round(w8_bytes / (o8_ms * 1e-3) / 1e9, 2),
                "unit": "GB/s",
            },
            "roofline": {
                "kernel": ("qgemm_split_kernel<W4, TPAD=32> (the step's 145 GEMM launches; "
                           "bytes and time are their sums)"
                           if ENGINES[args.engine] != ENGINES["stack"] else
                           "qgemm_kernel<W4, TPAD=32> (one launch: the step's 145 GEMMs)"),
                "bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                "peak_source": f"{peak_kind} HBM copy bandwidth" +
                               (" (of fallback)" if peak_kind == "fallback" else " (of measured)"),
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": ncu_traffic("qgemm_w4_t32_verify_step"
                                       if ENGINES[args.engine] != ENGINES["stack"] else
                                       "qgemm_w4_t32_verify_step_stack_engine"),
                "bytes_per_launch": gemm_bytes,
                "launch_ms": round(gemm_ms, 6),
                "launches_per_step": 1 if ENGINES[args.engine] == ENGINES["stack"] else n_gemm,
            },
            "cpu_baseline": cpu,
            "e2e": {
                "value": round(whole_job_gbs(world, nbytes, e2e_ms), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "steps": K_e2e,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "staging": "double-buffered device inputs: step i+1's host-to-device copy runs on a "
                           "copy stream while step i computes; every step reads its result back",
            },
            "gpu_launches": K * ((1 if ENGINES[args.engine] == ENGINES["stack"] else n_gemm) + 2),
            "clocks": clocks,
        }
        print(json.dumps(out), flush=True)
    ctx.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def cpu_oracle_leg(layer, xl, head, x_head, acc_sets, kept, budget_s):
    """The fp64 oracle on the host cores, on a bounded sample of the timed
    step: row samples of the last layer's four GEMMs and of the LM head (the
    same weights and activations the GPU used) and the three acceptance calls.
    Returns the CPU baseline (throughput of the sample) together with the
    GPU step's agreement with the oracle on that sample."""
    import numpy as np
    import torch

    import oracle

    def host_w4(w, rows):
        # output rows in pairs (zero points pack two rows per byte)
        pairs = rows[0::2] // 2
        return (w["qcodes"][torch.from_numpy(rows).to(w["qcodes"].device)].cpu().numpy(),
                w["scales"][:, torch.from_numpy(rows).to(w["scales"].device)].cpu().numpy(),
                w["zeros"][:, torch.from_numpy(pairs).to(w["zeros"].device)].cpu().numpy())

    def bits(x):
        return x.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    rng = np.random.default_rng(31)
    gemms = [(w, x, kept["ys"][j], False) for j, (w, x) in enumerate(zip(layer, xl))]
    gemms.append((head, x_head, kept["logits"], True))
    t0 = time.perf_counter()
    done_bytes, worst, checked = 0, 0.0, []
    n_pairs = 16
    while True:
        for w, x, y, f32 in gemms:
            N, K_ = w["N"], w["K"]
            p = np.sort(rng.choice(N // 2, size=n_pairs, replace=False))
            rows = np.stack([2 * p, 2 * p + 1], axis=1).reshape(-1)
            qc, sc, zr = host_w4(w, rows)
            ref = oracle.qgemm_w4a16(qc, sc, zr, GROUP, bits(x), T_MAIN, len(rows), K_)
            got = y[:, rows]
            allowed = 1e-2 * np.sqrt(np.mean(ref ** 2)) + (0.0 if f32 else 2.0 ** -8 * np.abs(ref))
            worst = max(worst, float(np.max(np.abs(got - ref) / allowed)))
            done_bytes += w4_gemm_bytes(T_MAIN, len(rows), K_, out_bytes=4 if f32 else 2)
            checked.append(f"{N}x{K_}")
        if time.perf_counter() - t0 > budget_s:
            break
        n_pairs = min(2 * n_pairs, 512)
    acc = []
    for a, (n_gpu, tok_gpu) in zip(acc_sets, kept["acc"]):
        h = a["host"]
        n_o, t_o, near = oracle.spec_accept(h.logits, h.q, h.drafts, h.u)
        evaluated = near[:min(n_o + 1, T_MAIN)].any() or near[T_MAIN]
        acc.append({"level": a["level"], "n_gpu": n_gpu, "n_oracle": int(n_o),
                    "match": bool(n_gpu == n_o and list(tok_gpu[:n_gpu + 1]) == list(t_o)),
                    "near_ties": int(near.sum()), "near_tie_decides": bool(evaluated)})
        done_bytes += accept_bytes(T_MAIN)
    dt = time.perf_counter() - t0
    sample = (f"oracle (numpy fp64) on row samples of the timed step's last layer (qkv, o, gate_up, "
              f"down) and LM head ({len(checked)} row-sampled GEMMs, up to {2 * n_pairs} rows each) "
              f"and its three spec_accept calls over V={VOCAB}: {done_bytes / 1e6:.1f} MB of the "
              f"step's {step_bytes() / 1e9:.2f} GB; {dt:.1f} s; numpy BLAS threads for the matmul, "
              f"the rest single-threaded")
    return {"value": round(done_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": os.cpu_count(),
            "threads": {"blas_matmul": os.cpu_count(), "everything_else": 1},
            "kind": "oracle", "sample": sample,
            "parity": {"gemm_max_err_over_bar": round(worst, 4), "gemm_pass": worst <= 1.0,
                       "accept": acc,
                       "accept_pass": all(x["match"] or x["near_tie_decides"] for x in acc)}}


# ----------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ----------------------------------------------------------------------------

def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    lay, xh, acc_h = host_layer0()
    levels = list(zip(inputs.LAYER_9B, lay, xh))

    def sub(w, rows):
        # output rows [r0, r1) of one int4 matrix (even bounds: zeros pack two rows)
        r0, r1 = rows
        return w["qcodes"][r0:r1], w["scales"][:, r0:r1], w["zeros"][:, r0 // 2:r1 // 2]

    def gemm_rows(i, nrows):
        (name, K, N), w, xb = levels[i % len(levels)]
        r0 = (i // len(levels) * nrows) % N
        r1 = min(N, r0 + nrows)
        qc, sc, zr = sub(w, (r0, r1))
        oracle.qgemm_w4a16(qc, sc, zr, GROUP, xb, T_MAIN, r1 - r0, K)
        return w4_gemm_bytes(T_MAIN, r1 - r0, K)

    # size each step so that warm-up + timed steps take about args.ref_seconds
    t0 = time.perf_counter()
    calib_bytes = gemm_rows(0, 512)
    calib_s = time.perf_counter() - t0
    per_step_s = args.ref_seconds / max(1, args.steps + args.warmup)
    nrows = int(512 * per_step_s / max(calib_s, 1e-6)) // 2 * 2
    nrows = max(32, min(nrows, 24576))

    def one_step(i):
        nbytes = gemm_rows(i, nrows)
        if i % 16 == 15:
            oracle.spec_accept(acc_h.logits, acc_h.q, acc_h.drafts, acc_h.u)
            nbytes += accept_bytes(T_MAIN)
        return nbytes

    for i in range(args.warmup):
        one_step(i)
    t0 = time.perf_counter()
    total = 0
    for i in range(args.steps):
        total += one_step(args.warmup + i)
    dt = time.perf_counter() - t0
    gbs = total / dt / 1e9
    sample = (f"each step: {nrows} output rows of one of layer 0's four int4 GEMMs at T=32, in "
              f"rotation (qkv, o, gate_up, down), plus spec_accept over V=151936 every 16th "
              f"step; throughput = algorithmic bytes of the sample / host time "
              f"(calibration: 512 rows = {calib_bytes / 1e6:.1f} MB in {calib_s:.2f} s)")
    out = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD, "T": T_MAIN, "sample": sample},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": os.cpu_count(),
                         "threads": {"blas_matmul": os.cpu_count(), "everything_else": 1},
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def run_kernel_case(args):
    """One W4A16 GEMM shape launched warm-up + steps times (for profiling one
    kernel in isolation); prints its device time and achieved bandwidth."""
    import torch

    import bit_qgemm_w4_gb300 as sv
    from bit_qgemm_w4_gb300 import build as svbuild
    svbuild.build()
    T, N, K = (int(v) for v in args.kernel_case.split(","))
    dev = torch.device("cuda", 0)
    ctx = open_ctx(args, 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    # enough distinct matrices that consecutive launches do not hit in L2
    copies = max(1, min(16, (256 << 20) // max(1, N * K // 2) + 1))
    ws = [inputs.w4_weights_device(gen, N, K, dev, GROUP) for _ in range(copies)]
    x = inputs.activations_device(gen, T, K, dev)
    y = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
    for i in range(args.warmup):
        w = ws[i % copies]
        sv.qgemm_w4a16(ctx, w["qcodes"], w["scales"], w["zeros"], GROUP, x, y, T, N, K)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        w = ws[(args.warmup + i) % copies]
        sv.qgemm_w4a16(ctx, w["qcodes"], w["scales"], w["zeros"], GROUP, x, y, T, N, K)
    e1.record()
    torch.cuda.synchronize()
    sv.spec_sync_status(ctx)
    ms = e0.elapsed_time(e1) / args.steps
    nbytes = w4_gemm_bytes(T, N, K)
    print(json.dumps({"kernel_case": [T, N, K], "copies": copies, "ms_per_launch": round(ms, 6),
                      "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1), "bytes": nbytes}), flush=True)
    ctx.close()


def run_kernel_case_w8(args):
    """One per-channel W8A16 GEMM shape (optionally with the block random
    Hadamard rotation of the activations, block B) launched warm-up + steps
    times; prints its device time and achieved bandwidth."""
    import numpy as np
    import torch

    import bit_qgemm_w4_gb300 as sv
    from bit_qgemm_w4_gb300 import build as svbuild
    svbuild.build()
    vals = [int(v) for v in args.kernel_case_w8.split(",")]
    T, N, K = vals[:3]
    B = vals[3] if len(vals) > 3 else 0
    dev = torch.device("cuda", 0)
    ctx = open_ctx(args, 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(9)
    copies = max(1, min(16, (256 << 20) // max(1, N * K) + 1))
    ws = [inputs.w8_weights_device(gen, N, K, dev) for _ in range(copies)]
    x = inputs.activations_device(gen, T, K, dev)
    y = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
    signs = torch.from_numpy(inputs.hadamard_signs(np.random.default_rng(5), K)).to(dev) if B else None

    def run(i):
        w = ws[i % copies]
        sv.qgemm_w8a16(ctx, w["qcodes"], w["scales"], 0, x, y, T, N, K, signs, B)

    for i in range(args.warmup):
        run(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        run(args.warmup + i)
    e1.record()
    torch.cuda.synchronize()
    sv.spec_sync_status(ctx)
    ms = e0.elapsed_time(e1) / args.steps
    nbytes = w8_gemm_bytes(T, N, K)
    print(json.dumps({"kernel_case_w8": [T, N, K, B], "copies": copies, "ms_per_launch": round(ms, 6),
                      "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1), "bytes": nbytes}), flush=True)
    ctx.close()


def run_fwht_case(args):
    """The standalone rotation fwht_rotate on a T x K bf16 block (block size
    B) launched warm-up + steps times; prints its device time and the
    bandwidth of its 4*T*K bytes (bf16 in and out)."""
    import numpy as np
    import torch

    import bit_qgemm_w4_gb300 as sv
    from bit_qgemm_w4_gb300 import build as svbuild
    svbuild.build()
    T, K, B = [int(v) for v in args.fwht_case.split(",")]
    dev = torch.device("cuda", 0)
    ctx = open_ctx(args, 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(13)
    x = inputs.activations_device(gen, T, K, dev)
    y = torch.empty_like(x)
    signs = torch.from_numpy(inputs.hadamard_signs(np.random.default_rng(5), K)).to(dev)
    for _ in range(args.warmup):
        sv.fwht_rotate(ctx, x, y, T, K, signs, B)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        sv.fwht_rotate(ctx, x, y, T, K, signs, B)
    e1.record()
    torch.cuda.synchronize()
    sv.spec_sync_status(ctx)
    ms = e0.elapsed_time(e1) / args.steps
    nbytes = 4 * T * K
    print(json.dumps({"fwht_case": [T, K, B], "ms_per_launch": round(ms, 6),
                      "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1), "bytes": nbytes}), flush=True)
    ctx.close()


def run_stack_case(args):
    """One GEMM stack alone, graph-replayed warm-up + steps times: `9b32[:L]`
    (L layers of the T=32 int4 stack plus the LM head), `9b32r32[:L]` (the same
    with the block-32 rotation of every GEMM's activations), `9b16[:L]` (the
    T=16 stack), `27b[:L]` / `27bnr[:L]` (the int8 Large-tier stack with /
    without rotation).  L defaults to the full depth.  Prints device time per launch
    and bandwidth."""
    import numpy as np
    import torch

    import bit_qgemm_w4_gb300 as sv
    from bit_qgemm_w4_gb300 import build as svbuild
    svbuild.build()
    name, _, depth = args.stack_case.partition(":")
    dev = torch.device("cuda", 0)
    ctx = open_ctx(args, 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(11)
    descs, keep, nbytes = [], [], 0
    if name in ("9b32", "9b32r32", "9b16"):
        T = 16 if name == "9b16" else 32
        rot = name == "9b32r32"
        sgn = {k: torch.from_numpy(inputs.hadamard_signs(np.random.default_rng(400 + k), k)).to(dev)
               for k in sorted({k for _, k, _ in inputs.LAYER_9B} | {HIDDEN})}
        L = int(depth) if depth else inputs.LAYERS_9B
        ys = [torch.empty((T, N), dtype=torch.bfloat16, device=dev) for _, _, N in inputs.LAYER_9B]
        for _ in range(L):
            for j, (_, K, N) in enumerate(inputs.LAYER_9B):
                w = inputs.w4_weights_device(gen, N, K, dev, GROUP)
                x = inputs.activations_device(gen, T, K, dev)
                keep += [w, x]
                descs.append({"quant": sv.SPEC_QUANT_W4, "qcodes": w["qcodes"], "scales": w["scales"],
                              "zeros": w["zeros"], "group_size": GROUP, "x": x, "y": ys[j], "T": T,
                              "N": N, "K": K, "wait_prev": 1,
                              "signs": sgn[K] if rot else None, "hadamard_block": 32 if rot else 0})
                nbytes += w4_gemm_bytes(T, N, K)
        if name != "9b16":
            w = inputs.w4_weights_device(gen, VOCAB, HIDDEN, dev, GROUP)
            x = inputs.activations_device(gen, T, HIDDEN, dev)
            y = torch.empty((T, VOCAB), dtype=torch.float32, device=dev)
            keep += [w, x, y]
            descs.append({"quant": sv.SPEC_QUANT_W4, "qcodes": w["qcodes"], "scales": w["scales"],
                          "zeros": w["zeros"], "group_size": GROUP, "x": x, "y": y, "T": T,
                          "N": VOCAB, "K": HIDDEN, "wait_prev": 1,
                          "signs": sgn[HIDDEN] if rot else None, "hadamard_block": 32 if rot else 0})
            nbytes += head_bytes(T)
    else:
        rot = name == "27b"
        L = int(depth) if depth else inputs.LAYERS_27B
        ys = [torch.empty((T_MAIN, N), dtype=torch.bfloat16, device=dev) for _, _, N in inputs.LAYER_27B]
        for _ in range(L):
            for j, (_, K, N) in enumerate(inputs.LAYER_27B):
                w = inputs.w8_weights_device(gen, N, K, dev)
                x = inputs.activations_device(gen, T_MAIN, K, dev)
                s = torch.from_numpy(inputs.hadamard_signs(np.random.default_rng(j), K)).to(dev)
                keep += [w, x, s]
                descs.append({"quant": sv.SPEC_QUANT_W8, "qcodes": w["qcodes"], "scales": w["scales"],
                              "zeros": None, "group_size": 0, "x": x, "y": ys[j], "T": T_MAIN, "N": N,
                              "K": K, "signs": s if rot else None, "hadamard_block": 1024 if rot else 0,
                              "wait_prev": 1})
                nbytes += w8_gemm_bytes(T_MAIN, N, K)
    st = sv.GemmStack(ctx, descs)
    st.run()
    sv.spec_sync_status(ctx)
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            st.run()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    sv.spec_sync_status(ctx)
    ms = e0.elapsed_time(e1) / args.steps
    peak, _ = hbm_peak()
    print(json.dumps({"stack_case": args.stack_case, "gemms": len(descs), "ms_per_launch": round(ms, 5),
                      "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1),
                      "frac": round(nbytes / (ms * 1e-3) / 1e9 / peak, 4), "bytes": nbytes,
                      "prefetch": [os.environ.get("SPEC_PREFETCH_LEAD"),
                                   os.environ.get("SPEC_PREFETCH_LEAD_FULL")]}), flush=True)
    del g, st
    ctx.close()


def run_accept_case(args):
    """spec_accept alone at T drafts over V tokens, launched warm-up + steps
    times eagerly (for profiling the acceptance kernels in isolation); prints
    its device time per call and the logits' read rate."""
    import numpy as np
    import torch

    import bit_qgemm_w4_gb300 as sv
    from bit_qgemm_w4_gb300 import build as svbuild
    svbuild.build()
    T, V = (int(v) for v in args.accept_case.split(","))
    dev = torch.device("cuda", 0)
    ctx = open_ctx(args, 0)
    a = inputs.accept_inputs(np.random.default_rng(11), T, V, logit_std=3.0, alpha=1.0, noise_std=0.5)
    logits = torch.from_numpy(a.logits).to(dev)
    q = torch.from_numpy(a.q).to(dev)
    d = torch.from_numpy(a.drafts).to(dev)
    u = torch.from_numpy(a.u).to(dev)
    n = torch.zeros(1, dtype=torch.int32, device=dev)
    tok = torch.zeros(T + 1, dtype=torch.int32, device=dev)
    for _ in range(args.warmup):
        sv.spec_accept(ctx, logits, q, d, u, T, V, n, tok)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        sv.spec_accept(ctx, logits, q, d, u, T, V, n, tok)
    e1.record()
    torch.cuda.synchronize()
    sv.spec_sync_status(ctx)
    ms = e0.elapsed_time(e1) / args.steps
    nbytes = (T + 1) * V * 4
    print(json.dumps({"accept_case": [T, V], "ms_per_call": round(ms, 6),
                      "logits_GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1), "logits_bytes": nbytes}),
          flush=True)
    ctx.close()


def run_gumbel_case(args):
    """spec_accept_gumbel alone at T drafts over V tokens, launched warm-up +
    steps times eagerly (for profiling the kernel in isolation); prints its
    device time per call and the logits' read rate."""
    import numpy as np
    import torch

    import bit_qgemm_w4_gb300 as sv
    from bit_qgemm_w4_gb300 import build as svbuild
    svbuild.build()
    T, V = (int(v) for v in args.gumbel_case.split(","))
    dev = torch.device("cuda", 0)
    ctx = open_ctx(args, 0)
    a = inputs.accept_inputs(np.random.default_rng(11), T, V, logit_std=3.0, alpha=1.0, noise_std=0.5)
    logits = torch.from_numpy(a.logits).to(dev)
    logq = torch.from_numpy(np.log(a.q).astype(np.float32)).to(dev)
    d = torch.zeros(max(T, 1), dtype=torch.int32, device=dev)
    n = torch.zeros(1, dtype=torch.int32, device=dev)
    tok = torch.zeros(T + 1, dtype=torch.int32, device=dev)
    if T > 0:
        sv.spec_gumbel_sample(ctx, logq, T, V, GUMBEL_SEED, 0, d)
    for _ in range(args.warmup):
        sv.spec_accept_gumbel(ctx, logits, d, T, V, GUMBEL_SEED, 0, n, tok)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        sv.spec_accept_gumbel(ctx, logits, d, T, V, GUMBEL_SEED, 0, n, tok)
    e1.record()
    torch.cuda.synchronize()
    sv.spec_sync_status(ctx)
    ms = e0.elapsed_time(e1) / args.steps
    nbytes = accept_gumbel_bytes(T, V)
    print(json.dumps({"gumbel_case": [T, V], "ms_per_call": round(ms, 6), "n_accepted": int(n.item()),
                      "logits_GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1), "bytes": nbytes}),
          flush=True)
    ctx.close()


def run_tree_case(args):
    """spec_accept_tree alone on a tree of T nodes over V tokens, launched
    warm-up + steps times eagerly (for profiling); prints its device time per
    call and the logits' read rate."""
    import numpy as np
    import torch

    import bit_qgemm_w4_gb300 as sv
    from bit_qgemm_w4_gb300 import build as svbuild
    svbuild.build()
    T, V = (int(v) for v in args.tree_case.split(","))
    dev = torch.device("cuda", 0)
    ctx = open_ctx(args, 0)
    tin = inputs.tree_inputs(np.random.default_rng(500 + T), T, V, logit_std=3.0, p_match=0.7)
    logits = torch.from_numpy(tin.logits).to(dev)
    d = torch.from_numpy(tin.drafts).to(dev)
    par = torch.from_numpy(tin.parent).to(dev)
    n = torch.zeros(1, dtype=torch.int32, device=dev)
    tok = torch.zeros(T + 1, dtype=torch.int32, device=dev)
    nodes = torch.zeros(T, dtype=torch.int32, device=dev)
    for _ in range(args.warmup):
        sv.spec_accept_tree(ctx, logits, d, par, T, V, n, tok, nodes)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        sv.spec_accept_tree(ctx, logits, d, par, T, V, n, tok, nodes)
    e1.record()
    torch.cuda.synchronize()
    sv.spec_sync_status(ctx)
    ms = e0.elapsed_time(e1) / args.steps
    nbytes = (T + 1) * V * 4
    print(json.dumps({"tree_case": [T, V], "ms_per_call": round(ms, 6), "path_len": int(n.item()),
                      "logits_GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1), "logits_bytes": nbytes}),
          flush=True)
    ctx.close()


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--engine", default="auto", choices=sorted(ENGINES),
                    help="GEMM engine: split (one launch per GEMM; auto), stack (one persistent "
                         "launch per call or stack)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle GEMM work in the CPU baseline sample")
    ap.add_argument("--ref-seconds", type=float, default=90.0,
                    help="host seconds the reference arm spends on warm-up + timed steps")
    ap.add_argument("--accept-case", default=None, metavar="T,V",
                    help="time spec_accept alone at T drafts over V tokens (eager launches)")
    ap.add_argument("--tree-case", default=None, metavar="T,V",
                    help="time spec_accept_tree alone on a T-node tree over V tokens (eager launches)")
    ap.add_argument("--gumbel-case", default=None, metavar="T,V",
                    help="time spec_accept_gumbel alone at T drafts over V tokens (eager launches)")
    ap.add_argument("--kernel-case-w8", default=None, metavar="T,N,K[,B]",
                    help="time one per-channel int8 GEMM shape (B > 0: rotation block)")
    ap.add_argument("--stack-case", default=None, metavar="NAME[:LAYERS]",
                    help="time one GEMM stack alone: 9b32, 9b32r32, 9b16, 27b or 27bnr, optionally fewer layers")
    ap.add_argument("--fwht-case", default=None, metavar="T,K,B",
                    help="time the standalone rotation on a T x K block")
    ap.add_argument("--kernel-case", default=None, metavar="T,N,K",
                    help="time one int4 GEMM shape in isolation instead of the verify step")
    args = ap.parse_args()
    if args.accept_case:
        run_accept_case(args)
        return
    if args.gumbel_case:
        run_gumbel_case(args)
        return
    if args.tree_case:
        run_tree_case(args)
        return
    if args.kernel_case_w8:
        run_kernel_case_w8(args)
        return
    if args.stack_case:
        run_stack_case(args)
        return
    if args.fwht_case:
        run_fwht_case(args)
        return
    if args.kernel_case:
        run_kernel_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
