"""Throughput of the encoder forward on GB300 (one JSON line on stdout).

A step is one forward pass of the whole encoder stack (every block, the
input norm and, for the text workload, the final-norm mean-pool) over one
packed batch of seeded synthetic input already resident in HBM.  The forward
is captured once in a CUDA graph and replayed; L2 is flushed (a 512 MiB
write) before every timed step and each step is timed with CUDA events on the
launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config c5|c4|c3|c2|c1|...]
                  [--impl ours|reference] [--op <one op of the workload>]

The default workload is the largest one that fits one GPU: the 30-block DiT
stack (d=3840, 30 heads x 128, SwiGLU 10240) over 2 x 4224 tokens (c5).  The
smaller workloads stay available with --config.

--impl reference times the CPU oracle (the plain f64 numpy restatement of
the method, test infrastructure) on a bounded sample of the same workload on
this machine's host cores; it is the slow baseline, not a target.

Multi-GPU: sequences are independent and the forward has no exchange step.
With N ranks the packed batch is N draws of the one-GPU batch, split along
sequence boundaries into N shares of near-equal work (shard.partition), one
per rank (weak scaling, no data-path collective); value = the work of all
ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from transformer_encoder_forward_gb300 import synth  # noqa: E402

METRIC = "encoder-block TFLOP/s and tokens/s at 1 GB300; % of dense bf16 tensor peak"


# ------------------------------------------------------------ work counting

def visible_pairs(lens, window):
    """(query, key) pairs the attention computes: same sequence and, with a
    window, |i - j| <= window."""
    tot = 0
    for n in lens:
        n = int(n)
        if window == 0 or window >= n - 1:
            tot += n * n
        else:
            i = np.arange(n)
            tot += int(np.sum(np.minimum(n - 1, i + window) - np.maximum(0, i - window) + 1))
    return tot


def layer_flops(cfg, lens, layer):
    T = int(np.sum(lens))
    d, hd, H, KV, F = cfg.d, cfg.hd, cfg.heads, cfg.kv_heads, cfg.ffn
    gemm = 2 * T * (d * (H + 2 * KV) * hd + H * hd * d + d * F * (2 if cfg.gated else 1) + F * d
                    + 3 * d * cfg.ple_dim)
    attn = 4 * hd * H * visible_pairs(synth.unit_lens(cfg, lens), cfg.window_of(layer))
    return gemm, attn


def forward_flops(cfg, lens, layers=None):
    n = cfg.layers if layers is None else layers
    g = a = 0
    for i in range(n):
        gi, ai = layer_flops(cfg, lens, i)
        g += gi
        a += ai
    return g, a


def launches_per_forward(cfg):
    """Kernels of this library one forward launches (what the graph replays)."""
    n = 1                                                     # input pre-norm
    for i in range(cfg.layers):
        n += 4                                                # q8 GEMMs: qkv, o, gate|up (+gate), down
        n += 1 if (cfg.qk_norm or cfg.rope or cfg.v_norm) else 0   # q/k (v) norm + RoPE
        n += 2                                                # attention, FFN pre-norm
        n += 1 if (cfg.form == "sandwich" or i + 1 < cfg.layers) else 0   # closing norm
        n += 7 if cfg.ple_dim else 0       # per-layer input: 3 GEMMs, norm, cast, gate, residual
    n += 1 if cfg.ple_dim else 0                              # the per-layer inputs' bf16 source
    return n + (1 if cfg.pool else 0)                         # final norm + pool


# ------------------------------------------------------------------ helpers

def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained", j["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def draw_layers(cfg, seed, n):
    """The first n layers' seeded weights.  Each layer has its own generator
    and numpy fills arrays without the GIL, so the draws run in threads (the
    30-layer DiT stack holds 5.3 GB of int8 weights)."""
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=min(n, os.cpu_count() or 1, 16)) as ex:
        return list(ex.map(lambda i: synth.draw_layer(cfg, i, seed, jitter=False), range(n)))


def build_stack(key, device, lens=None, x_seed_offset=0, layers=None):
    """The workload's stack on `device`; layers=n builds only its first n
    layers (one op timed alone needs one layer's weights)."""
    from transformer_encoder_forward_gb300.model import EncoderStack
    cfg = synth.CONFIGS[key]
    lens = synth.draw_lens(cfg) if lens is None else np.asarray(lens, dtype=np.int32)
    seed = synth.config_seed(key)
    ps = draw_layers(cfg, seed, cfg.layers if layers is None else layers)
    tables = synth.rope_tables(cfg, lens)
    fin = synth.draw_final_norm(cfg, seed) if cfg.pool else None
    ple = synth.draw_ple(cfg, seed) if cfg.ple_dim else None
    st = EncoderStack(cfg, ps, lens, tables, fin, device=device, ple=ple,
                      items=synth.attn_items(cfg, lens))
    del ps   # the device holds the weights now
    x0 = synth.draw_x(st.T, cfg.d, seed + x_seed_offset)
    return cfg, lens, st, x0, tables


def rank_lens(key, world, rank):
    """This rank's share of the packed batch of a `world`-GPU run."""
    from transformer_encoder_forward_gb300 import shard
    cfg = synth.CONFIGS[key]
    if world == 1 or cfg.cfg_pair:
        # a CFG pair is one program over its items' interleaved ranges: every
        # rank runs the whole one-GPU program (weak scaling)
        return synth.draw_lens(cfg)
    allv = shard.global_lens(cfg, world, lambda c, r: synth.draw_lens(c, synth.BASE_SEED + r))
    part = shard.partition(shard.sequence_costs(cfg, allv), world)
    return allv[part[rank]]


# --------------------------------------------------------------- GPU timing

OP_SOURCE = {"gemm": "q8_linear.cu", "attn": "attn.cu", "qk_prep": "rowops.cu",
             "add_norm": "rowops.cu", "rownorm": "rowops.cu"}


def workload_ops(cfg, st, torch):
    """Each op of one block with the workload's shapes, launched alone.
    Returns {name: (fn(stream), algorithmic flops, algorithmic bytes,
    launches per forward, bound)}."""
    import transformer_encoder_forward_gb300 as te
    T, d, hd, H, KV, F = st.T, cfg.d, cfg.hd, cfg.heads, cfg.kv_heads, cfg.ffn
    qw, kw = H * hd, KV * hd
    ldq = qw + 2 * kw
    dev = st.device
    L0 = st.layers[0]
    g = torch.Generator(device=dev).manual_seed(0)
    a = torch.randn(T, d, device=dev, generator=g).to(torch.bfloat16)
    qkv = torch.randn(T, ldq, device=dev, generator=g).to(torch.bfloat16)
    o = torch.randn(T, qw, device=dev, generator=g).to(torch.bfloat16)
    tmp = torch.randn(T, d, device=dev, generator=g)
    m = torch.randn(T, F, device=dev, generator=g).to(torch.bfloat16)
    x = torch.randn(T, d, device=dev, generator=g)
    w = lambda k: te.q8w(*L0.t[k])
    nl = cfg.layers
    ug = 2 if cfg.gated else 1
    g_keys = ["wg", "wu"] if cfg.gated else ["wg"]

    def items(keys, y, ldy, offs):
        return [{"w": w(k), "y": y[:, off:] if off else y, "ldy": ldy} for k, off in zip(keys, offs)]

    it_qkv = items(["wq", "wk", "wv"], qkv, ldq, [0, qw, qw + kw])
    act_code = te.TE_ACT_SILU if cfg.act == "silu" else te.TE_ACT_GELU_TANH

    def gate_up(s):
        # the block's FFN producer: gate|up with the gate in the epilogue
        # (ungated: up with the activation in the epilogue); writes m
        if cfg.gated:
            te.q8_gated_linear(a, w("wg"), w("wu"), act_code, m, stream=s)
        else:
            te.q8_linear(a, [{"w": w("wg"), "y": m, "ldy": F, "epilogue": act_code + 1}], stream=s)
    ops = {
        "gemm_qkv": (lambda s: te.q8_linear(a, it_qkv, stream=s), 2 * T * d * ldq,
                     T * d * 2 + ldq * d + T * ldq * 2, nl, "tensor"),
        "gemm_o": (lambda s: te.q8_linear(o, [{"w": w("wo"), "y": tmp, "ldy": d}], stream=s),
                   2 * T * qw * d, T * qw * 2 + qw * d + T * d * 4, nl, "tensor"),
        "gemm_gu": (gate_up, 2 * T * d * F * ug, T * d * 2 + ug * F * d + T * F * 2, nl, "tensor"),
        "gemm_down": (lambda s: te.q8_linear(m, [{"w": w("wd"), "y": tmp, "ldy": d}], stream=s),
                      2 * T * F * d, T * F * 2 + F * d + T * d * 4, nl, "tensor"),
    }
    for win in sorted({cfg.window_of(i) for i in range(nl)}):
        cnt = sum(1 for i in range(nl) if cfg.window_of(i) == win)
        pairs = visible_pairs(synth.unit_lens(cfg, st.lens), win)
        if st.items_host is not None:     # two-range items (the CFG pair)
            fn = lambda s, win=win: te.attn_items_fwd(qkv, ldq, 0, qw, qw + kw, st.items_host, st.items_dev,
                                                      T, H, KV, hd, win, cfg.scale, o, qw, stream=s)
        else:
            fn = lambda s, win=win: te.attn_varlen_fwd(qkv, ldq, 0, qw, qw + kw, st.cu_host, st.cu_dev, H,
                                                       KV, hd, win, cfg.scale, o, qw, stream=s)
        ops[f"attn_w{win}"] = (fn, 4 * hd * H * pairs, T * ldq * 2 + T * qw * 2, cnt, "tensor")
    if cfg.qk_norm or cfg.rope or cfg.v_norm:
        vw = kw if cfg.v_norm else 0
        ops["qk_prep"] = (lambda s: te.qkv_prep_rope(
            qkv, ldq, 0, qw, qw + kw, H, KV, hd, L0.t["q_norm"], L0.t["k_norm"], cfg.v_norm, cfg.eps,
            st.rope_cos, st.rope_sin, st.rope_pos, st.rope_sec, 1.0, T, stream=s), 0,
            2 * T * (qw + kw + vw) * 2, nl, "hbm")
    if cfg.adaln:   # with the gate on the branch and the scale on the next norm
        md = L0.t["mod"]
        ops["add_norm"] = (lambda s: te.add_norm_mod(x, tmp, L0.t["post_attn_w"], md[1], 1.0, L0.t["norm2_w"],
                                                     None, md[2], te.TE_NORM_RMS, cfg.eps, a, stream=s),
                           0, T * d * (4 * 3 + 2), 2 * nl, "hbm")
    elif cfg.form == "sandwich":
        ops["add_norm"] = (lambda s: te.add_norm(x, tmp, L0.t["post_attn_w"], 1.0, L0.t["norm2_w"], L0.t["norm2_b"],
                                                 te.TE_NORM_LN if cfg.norm == "ln" else te.TE_NORM_RMS, cfg.eps,
                                                 a, stream=s), 0, T * d * (4 * 3 + 2), 2 * nl, "hbm")
    else:
        # the plain form adds each projection into x in its GEMM's epilogue;
        # its row op is the norm of x into the next GEMM's bf16 input (the
        # FFN norm and the next block's norm, or the stack's input norm)
        ops["rownorm"] = (lambda s: te.rownorm(x, L0.t["norm2_w"], L0.t["norm2_b"],
                                               te.TE_NORM_LN if cfg.norm == "ln" else te.TE_NORM_RMS, cfg.eps,
                                               a, stream=s), 0, T * d * (4 + 2), 2 * nl, "hbm")
    return ops


def time_op(fn, torch, dev, reps=20):
    """Device time per launch: `reps` launches captured in one CUDA graph and
    replayed (no host gaps), timed with CUDA events on the replay stream."""
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(3):
            fn(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(reps):
            fn(stream)
    with torch.cuda.stream(stream):
        graph.replay()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        graph.replay()
        e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e) / reps


def time_kernels(cfg, st, torch):
    import transformer_encoder_forward_gb300 as te
    res = {}
    for name, (fn, flops, nbytes, count, bound) in workload_ops(cfg, st, torch).items():
        res[name] = (time_op(fn, torch, st.device), flops, nbytes, count, bound)
    te.check()
    return res


def source_sha(op):
    import hashlib
    key = next(k for k in OP_SOURCE if op.startswith(k))
    path = os.path.join(ROOT, "transformer_encoder_forward_gb300", "csrc", OP_SOURCE[key])
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def measured_traffic(config_key, op):
    """DRAM bytes per launch of `op` from the committed ncu summary, or None
    when there is none or the kernel source changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        j = json.load(f)
    rec = j.get(f"{op}@{config_key}")
    if not rec or rec.get("source_sha256") != source_sha(op):
        return None
    return rec.get("dram_bytes_per_launch")


def roofline_for(kern, config_key, peaks):
    """The op with the largest share of the forward, against its roof."""
    name = max(kern, key=lambda k: kern[k][0] * kern[k][3])
    ms, flops, nbytes, count, bound = kern[name]
    if bound == "tensor":
        ach = flops / (ms * 1e-3) / 1e12
        peak, unit, src = peaks["bf16_tflops"], "TFLOP/s", "bf16 burst (cuBLAS), timed alone"
    else:
        ach = nbytes / (ms * 1e-3) / 1e9
        peak, unit, src = peaks["hbm_gbs"], "GB/s", "HBM copy"
    return {"kernel": name, "bound": bound, "achieved": round(ach, 1), "peak": peak, "unit": unit,
            "frac": round(ach / peak, 4), "traffic": measured_traffic(config_key, name),
            "algorithmic_per_launch": flops if bound == "tensor" else nbytes,
            "ms_per_launch": round(ms, 4), "peak_source": f"{peaks['source']} {src}"}


def run_op(args):
    """One op of the workload alone (for profiling): W warm-up launches, then
    K launches; prints one JSON line with its per-launch device time."""
    import torch
    import transformer_encoder_forward_gb300 as te
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    te.lib()
    cfg, lens, st, _, _ = build_stack(args.config, dev, layers=1)
    ops = workload_ops(cfg, st, torch)
    if args.op not in ops:
        raise SystemExit(f"--op {args.op}: not an op of {cfg.name}'s forward (ops: {', '.join(sorted(ops))})")
    fn, flops, nbytes, count, bound = ops[args.op]
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        fn(stream)
    torch.cuda.synchronize()
    for _ in range(args.steps):
        fn(stream)
    torch.cuda.synchronize()
    te.check()
    ms = time_op(fn, torch, dev)
    out = {"op": args.op, "config": cfg.name, "ms_per_launch": round(ms, 4),
           "launches_per_forward": count, "bound": bound}
    if flops:
        out["tflops"] = round(flops / (ms * 1e-3) / 1e12, 1)
    out["gbs_algorithmic"] = round(nbytes / (ms * 1e-3) / 1e9, 1)
    print(json.dumps(out), flush=True)


def run_mma_peak(args):
    """The q8 GEMM's MMA form issued back to back with no loads (te_mma_peak)
    at each token-tile width: the tensor ceiling its pipeline could reach,
    one JSON line per width."""
    import torch
    import transformer_encoder_forward_gb300 as te
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    pairs = te.sm_count(dev.index) // 2
    peaks = read_peaks()
    for bn in (64, 128, 192, 256):
        stages = 4000
        for _ in range(args.warmup):
            te.mma_peak(bn, stages)
        ms = min(te.mma_peak(bn, stages) for _ in range(max(args.steps, 1)))
        flops = pairs * stages * 8 * 2 * 256 * bn * 16
        tf = flops / (ms * 1e-3) / 1e12
        print(json.dumps({"op": "mma_peak", "n": bn, "m": 256, "k_per_mma": 16, "sm_pairs": pairs,
                          "ms": round(ms, 4), "tflops": round(tf, 1),
                          "of_measured_bf16": round(tf / peaks["bf16_tflops"], 4)}), flush=True)


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import transformer_encoder_forward_gb300 as te
    from transformer_encoder_forward_gb300 import shard
    te.lib()
    cfg, lens, st, x0_np, _ = build_stack(args.config, dev, rank_lens(args.config, world, rank),
                                             x_seed_offset=rank)
    T = st.T
    gflops, aflops = forward_flops(cfg, lens)
    total_flops = gflops + aflops
    all_flops = shard.sum_over_ranks(total_flops, dist)
    all_tokens = shard.sum_over_ranks(T, dist)
    x0 = torch.from_numpy(x0_np).to(dev)
    x, a, out = st.buffers()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    # capture one forward in a CUDA graph (warm the launch path first)
    with torch.cuda.stream(stream):
        x.copy_(x0)
        st.forward_device(x, a, out, stream=stream)
    torch.cuda.synchronize()
    te.check(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        st.forward_device(x, a, out, stream=stream)
    torch.cuda.synchronize()

    def step():
        x.copy_(x0)
        flush.fill_(1)
        graph.replay()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    te.check(stream)

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for s, e in evs:
                x.copy_(x0)
                flush.fill_(1)
                s.record(stream)
                graph.replay()
                e.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    if world > 1:
        dist.barrier()
    te.check(stream)
    step_ms = [s.elapsed_time(e) for s, e in evs]
    ms = shard.max_over_ranks(sum(step_ms) / len(step_ms), dist)
    clk = clocks.summary()

    # end to end through the public API from pinned host memory (the first
    # calls run eagerly and capture the graph that later calls replay)
    x_host = torch.from_numpy(x0_np).pin_memory()
    res_host = torch.empty((len(lens) if cfg.pool else T, cfg.d), dtype=torch.float32).pin_memory()
    with torch.cuda.stream(stream):
        for _ in range(2):
            st.forward_host(x_host, res_host, x, a, out, stream=stream)
    torch.cuda.synchronize()
    e2e = []
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            flush.fill_(1)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            st.forward_host(x_host, res_host, x, a, out, stream=stream)
            e.record(stream)
            e2e.append((s, e))
    torch.cuda.synchronize()
    e2e_serial_ms = shard.max_over_ranks(statistics.mean(s.elapsed_time(e) for s, e in e2e), dist)
    te.check(stream)

    # the same through forward_host_stream: the K forwards in sequence, each
    # step's copy in and copy out overlapping the neighbouring forwards (the L2
    # flush runs ahead of each forward, inside the timed region)
    res2 = [res_host, torch.empty_like(res_host).pin_memory()]
    st.forward_host_stream([x_host] * 2, res2, stream=stream, before=lambda: flush.fill_(1))
    torch.cuda.synchronize()
    s0, s1 = st.forward_host_stream([x_host] * args.steps, [res2[i & 1] for i in range(args.steps)],
                                    stream=stream, before=lambda: flush.fill_(1))
    torch.cuda.synchronize()
    e2e_ms = shard.max_over_ranks(s0.elapsed_time(s1) / args.steps, dist)
    te.check(stream)

    # per-kernel device times with the workload's shapes -> roofline
    kern = time_kernels(cfg, st, torch)
    peaks = read_peaks()
    roofline = roofline_for(kern, args.config, peaks)
    attn_ms = sum(v[0] * v[3] for k, v in kern.items() if k.startswith("attn"))
    attn_fl = sum(v[1] * v[3] for k, v in kern.items() if k.startswith("attn"))
    gemm_ms = sum(v[0] * v[3] for k, v in kern.items() if k.startswith("gemm"))
    gemm_fl = sum(v[1] * v[3] for k, v in kern.items() if k.startswith("gemm"))
    kernels = {k: {"ms_per_launch": round(v[0], 4), "launches_per_forward": v[3],
                   "ms_per_forward": round(v[0] * v[3], 3),
                   **({"tflops": round(v[1] / (v[0] * 1e-3) / 1e12, 1)} if v[1] else {}),
                   "gbs": round(v[2] / (v[0] * 1e-3) / 1e9, 1)} for k, v in kern.items()}

    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(cfg, args.config, budget_s=args.cpu_seconds)

    tflops = all_flops / (ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random-init q8_row weights of the named shape)",
        "config": {"workload": cfg.name, "layers": cfg.layers, "tokens": T, "seqs": len(lens),
                   "d": cfg.d, "heads": cfg.heads, "head_dim": cfg.hd, "ffn": cfg.ffn,
                   "l2": "flushed before every step (512 MiB write)", "graph": "one CUDA graph per forward",
                   "parallelism": (f"data-parallel x{world}: sequences split by work, "
                                   f"{int(all_tokens)} tokens in all") if world > 1 else "single GPU"},
        "tokens_per_s": round(all_tokens / (ms * 1e-3), 1),
        "pct_bf16_peak": round(100 * tflops / world / peaks["bf16_tflops"], 2),
        "flops_per_step": {"gemm": gflops, "attention": aflops},
        "e2e": {"value": round(all_flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 3), "h2d_bytes_per_step": x_host.numel() * 4,
                "d2h_bytes_per_step": res_host.numel() * 4,
                "path": "EncoderStack.forward_host_stream: per step a pinned H2D of the input on one copy "
                        "stream, the L2 flush and the forward's CUDA-graph replay on the compute stream, a "
                        "D2H of the result on another copy stream; neighbouring steps' copies overlap the "
                        "forward (two device buffer sets alternate)",
                "serial": {"value": round(all_flops / (e2e_serial_ms * 1e-3) / 1e12, 2),
                           "ms_per_step": round(e2e_serial_ms, 3),
                           "path": "EncoderStack.forward_host: H2D, graph replay, D2H in order, one step "
                                   "at a time (L2 flushed before each step, outside its time)"}},
        "roofline": roofline,
        "kernels": kernels,
        "attention_tflops": round(attn_fl / (attn_ms * 1e-3) / 1e12, 1) if attn_ms else None,
        "gemm_tflops": round(gemm_fl / (gemm_ms * 1e-3) / 1e12, 1) if gemm_ms else None,
        "gpu_launches": launches_per_forward(cfg) * args.steps,
        "clocks": clk,
        "wall_s_timed": round(wall, 3),
        "cpu_baseline": cpu,
    }
    if os.environ.get("TEFWD_PROF"):
        # the pages' per-op-class switch: one eager forward with the blocks'
        # step-boundary events, GPU ms a class over the whole stack
        x.copy_(x0)
        cls = st.profile_forward(x, a, stream=stream)
        te.check(stream)
        line["step_classes_ms"] = {k: round(v, 4) for k, v in cls.items()}
        if rank == 0:
            tot = sum(cls.values()) or 1.0
            for k, v in cls.items():
                print(f"[TEFWD_PROF] {k:10s} {v:9.3f} ms {100 * v / tot:5.1f} %", file=sys.stderr)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------- CPU oracle

def cpu_sample(key):
    """A bounded sample of the workload for the oracle: one layer of the stack
    over the first sequences (about a second of numpy f64 work)."""
    cfg = synth.CONFIGS[key]
    lens = synth.draw_lens(cfg)
    seed = synth.config_seed(key)
    take = {"c1": 2, "c2": 6, "c3": 1, "c4": 1, "c5": 1, "c4m": 1, "c5m": 1, "c3q8": 1, "c3q4": 1, "c4f": 1,
            "c2v": 6, "c2p": 6, "c4c": 1}[key]
    if cfg.cfg_pair:
        # the first item's rows (image and caption) attended as one sequence,
        # which is what an item is
        import dataclasses
        cfg = dataclasses.replace(cfg, cfg_pair=False)
        sl = np.asarray([int(synth.unit_lens(synth.CONFIGS[key], lens)[0])], dtype=np.int32)
        return cfg, sl, seed
    sl = lens[:take]
    if key in ("c4", "c5", "c4m", "c5m", "c4f"):
        sl = np.asarray([min(int(sl[0]), 1056)], dtype=np.int32)
    return cfg, sl, seed


def oracle_layer(cfg, lens, layer, p, x, tables, seed=0):
    from oracle import encoder as O
    cu = synth.cu_seqlens(lens)
    mod = p.get("mod")
    a = O.round_bf16(O.norm(cfg.norm, x, p["norm1_w"], p["norm1_b"], cfg.eps,
                            mod_scale=None if mod is None else mod[0]))
    ple = None
    if cfg.ple_dim:
        ple = dict(synth.draw_ple(cfg, seed), x_in=x)
    return O.block_forward(cfg, p, x, a, cu, layer, tables, None, mod=mod, ple=ple)


def cpu_baseline(cfg_full, key, budget_s=15.0):
    cfg, sl, seed = cpu_sample(key)
    tables = synth.rope_tables(cfg, sl)
    T = int(np.sum(sl))
    x = synth.draw_x(T, cfg.d, seed).astype(np.float64)
    ps = {}
    done, flops, t_used = 0, 0.0, 0.0
    layer = 0
    while t_used < budget_s and done < 2 * max(1, cfg.layers):
        li = layer % cfg.layers
        if li not in ps:
            ps[li] = synth.draw_layer(cfg, li, seed, jitter=False)
        t0 = time.perf_counter()
        oracle_layer(cfg, sl, li, ps[li], x, tables, seed)
        t_used += time.perf_counter() - t0
        g, a = layer_flops(cfg, sl, li)
        flops += g + a
        done += 1
        layer += 1
    return {"value": round(flops / t_used / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{done} layer(s) of {cfg.name} over the first {len(sl)} sequence(s) "
                      f"({T} tokens), numpy f64, {t_used:.1f} s",
            "tokens_per_s": round(T * done / t_used / cfg.layers, 2)}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg, sl, seed = cpu_sample(args.config)
    tables = synth.rope_tables(cfg, sl)
    T = int(np.sum(sl))
    x = synth.draw_x(T, cfg.d, seed).astype(np.float64)
    ps = [synth.draw_layer(cfg, i, seed, jitter=False) for i in range(min(2, cfg.layers))]
    for i in range(args.warmup):
        oracle_layer(cfg, sl, i % len(ps), ps[i % len(ps)], x, tables, seed)
    times, flops = [], 0.0
    for i in range(args.steps):
        li = i % len(ps)
        t0 = time.perf_counter()
        oracle_layer(cfg, sl, li, ps[li], x, tables, seed)
        times.append(time.perf_counter() - t0)
        g, a = layer_flops(cfg, sl, li)
        flops += g + a
    tot = sum(times)
    val = flops / tot / 1e12
    full_cfg = synth.CONFIGS[args.config]
    sample = (f"each step: one layer of {cfg.name} over the first {len(sl)} sequence(s) "
              f"({T} tokens), numpy f64 oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": "TFLOP/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot / len(times), 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": full_cfg.name, "sample": sample},
        "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "cores": os.cpu_count(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="c5", choices=sorted(synth.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--op", default=None,
                    help="time one op of the workload alone (gemm_qkv, gemm_o, gemm_gu (gate fused), "
                         "gemm_down, attn_w<window>, qk_prep, add_norm or rownorm) instead of the forward; "
                         "mma_peak: the GEMM's MMA form without loads, its tensor ceiling")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "mma_peak":
        run_mma_peak(args)
    elif args.op:
        run_op(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
