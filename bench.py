#!/usr/bin/env python
"""Benchmark of the joint audio-video attention sub-block forward on GB300.

One step = one fused sub-block forward (modulate -> QKV projection + 3D RoPE
-> joint attention -> output projection + gated residual) over the full-size
packed sequence: L = 58,758 tokens (358 text + 57,600 video + 800 audio),
d = 5120, 40 heads x 128, full attention, batch 1.  Reports block TFLOP/s
(algorithmic FLOPs 6Ld^2 + 4L^2d + 2Ld^2 over device time), tokens/s, the
attention kernel against the bf16 tensor roofline, an end-to-end number
through the public API with host buffers, and the CPU fp64 oracle timed on a
bounded sample of the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs an independent replica (the block does not
shard: replicas only); the printed value is the aggregate over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attn-block fwd TFLOP/s & tokens/s at L=58,758; % of GB300 dense BF16 peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def _workload(cfg) -> str:
    return (f"joint A/V DiT attention sub-block, L={cfg.L} ({cfg.n_text} text + {cfg.n_video} "
            f"video + {cfg.n_audio} audio), d={cfg.d}, {cfg.n_heads}x{cfg.head_dim} heads, "
            f"full attention, batch 1")


L2_BYTES = 129e6   # GB300 L2


def _config(cfg, world: int = 1) -> dict:
    """The workload description both arms print (same keys, same values)."""
    x_b, qkv_b = cfg.L * cfg.d * 2, cfg.L * 3 * cfg.d * 2
    sizes = f"x {x_b / 1e6:.0f} MB, qkv {qkv_b / 1e9:.2f} GB per step"
    l2 = (f"inputs larger than L2 ({sizes})" if x_b + qkv_b > L2_BYTES else
          f"working set fits in the 129 MB L2 ({sizes}): steps run L2-warm, no flush")
    return {"workload": _workload(cfg), "L": cfg.L, "d": cfg.d, "heads": cfg.n_heads,
            "causal": False, "l2": l2, "parallelism": f"replicas x{world}"}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return FALLBACK_PEAKS, "fallback"


# ---------------------------------------------------------------------------- ranks
def max_over_ranks(value: float, world: int, device) -> float:
    """The largest per-rank value (the slowest replica sets the job's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(per_rank_work: float, world: int, max_ms: float) -> float:
    """Whole-job rate: the work every replica did, over the slowest replica's time."""
    return world * per_rank_work / (max_ms * 1e-3)


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------- oracle sample
def oracle_sample(cfg, inp, scale_factor: float = 1.0):
    """Time the CPU fp64 oracle on a bounded sample of the block workload.

    Stages and sample sizes: modulate on R1 rows, QKV projection + RoPE on R2
    rows, attention for R3 query rows of H3 heads against all L keys (random
    workload-shaped qkv), output projection + gated residual on R2 rows.
    Each stage's time is scaled to the full block by its work ratio.
    Returns (extrapolated full-block seconds, sample description, cores).
    """
    import numpy as np
    import oracle as orc
    from h3inputs import attention_qkv

    L, d, H = cfg.L, cfg.d, cfg.n_heads
    R1 = min(L, int(4096 * scale_factor))
    R2 = min(L, int(384 * scale_factor))
    R3, H3 = min(L, int(128 * scale_factor)), 4
    f64 = lambda t: t.float().double().numpy()
    mod, pos = orc.packed_layout(cfg.n_text, cfg.video_t, cfg.video_h, cfg.video_w,
                                 cfg.audio_channels, cfg.audio_steps)
    rows1 = np.linspace(0, L - 1, R1).astype(np.int64)
    rows2 = np.linspace(0, L - 1, R2).astype(np.int64)
    x1, x2 = f64(inp["x"][rows1]), f64(inp["x"][rows2])
    shift, scale, gate = f64(inp["shift"]), f64(inp["scale"]), f64(inp["gate"])
    wqkv, wo = f64(inp["Wqkv"]), f64(inp["Wo"])
    qkv_s = f64(attention_qkv(L, H3, seed=99))
    rows3 = np.linspace(0, L - 1, R3).astype(np.int64)

    t = time.perf_counter()
    orc.adaln_modulate(x1, mod[rows1], shift, scale, cfg.ln_eps)
    t_mod = time.perf_counter() - t
    t = time.perf_counter()
    y2 = orc.adaln_modulate(x2, mod[rows2], shift, scale, cfg.ln_eps)
    q = orc.mrope(orc.linear(y2, wqkv), pos[rows2], H)
    t_qkv = time.perf_counter() - t
    t = time.perf_counter()
    o, _ = orc.attention(qkv_s, H3, 128, rows=rows3)
    t_att = time.perf_counter() - t
    t = time.perf_counter()
    orc.gated_residual(x2, orc.linear(q[:, :d], wo), mod[rows2], gate)
    t_out = time.perf_counter() - t
    full = (t_mod * L / R1 + t_qkv * L / R2 + t_att * (L / R3) * (H / H3) + t_out * L / R2)
    sample = (f"oracle (numpy fp64) on {R1} rows of modulate, {R2} rows of QKV projection + "
              f"RoPE and of output projection + gated residual, {R3} query rows x {H3} heads "
              f"of attention over all {L} keys; scaled to the full block by work ratio "
              f"(sample {t_mod + t_qkv + t_att + t_out:.1f} s)")
    cores = len(os.sched_getaffinity(0))
    return full, sample, cores, t_mod + t_qkv + t_att + t_out


# ---------------------------------------------------------------------------- reference arm
def run_reference(args, cfg):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from h3inputs import block_inputs
    inp = block_inputs(cfg)
    flops = cfg.flops()
    times, sample_s = [], []
    for i in range(args.warmup + args.steps):
        full, sample, cores, s = oracle_sample(cfg, inp, scale_factor=2.0)
        if i >= args.warmup:
            times.append(full)
            sample_s.append(s)
    full = statistics.mean(times)
    value = flops / full / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": full * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(cfg, args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "tokens_per_s": cfg.L / full,
        "note": "each step is a bounded oracle sample; ms_per_step is the extrapolated "
                "full-block CPU time",
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------- GPU arm
def run_gpu(args, cfg):
    import torch
    import torch.distributed as dist
    import joint_audio_video_gb300 as h3
    from joint_audio_video_gb300 import build as h3build
    from h3inputs import block_inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0 or world == 1:
        h3build.build()
    if world > 1:
        dist.barrier()
    h3.load()
    dev = torch.device("cuda", local)

    def barrier():
        if world > 1:
            dist.barrier()

    L, d, H = cfg.L, cfg.d, cfg.n_heads
    inp = block_inputs(cfg)
    mod, pos = h3.h3_build_packed_layout(cfg.n_text, cfg.video_t, cfg.video_h, cfg.video_w,
                                         cfg.audio_channels, cfg.audio_steps)
    x = inp["x"].to(dev)
    wqkv, wo = inp["Wqkv"].to(dev), inp["Wo"].to(dev)
    shift, scale, gate = inp["shift"].to(dev), inp["scale"].to(dev), inp["gate"].to(dev)
    mod_d, pos_d = torch.from_numpy(mod).to(dev), torch.from_numpy(pos).to(dev)
    desc = h3.BlockDesc.make(L=L, d=d, n_heads=H, rope_sec=cfg.rope_sections,
                             rope_base=cfg.rope_base, ln_eps=cfg.ln_eps, n_mod=cfg.n_mod)
    nbytes = h3.h3_workspace_size(desc)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = torch.empty(L, d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(events=None):
        h3.h3_attn_block_fwd_profiled(desc, x, mod_d, pos_d, shift, scale, gate, wqkv, wo, ws,
                                      nbytes, out, events, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = h3.h3_sync_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {h3.h3_status_string(st)}")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    barrier()
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.start()
        time.sleep(0.3)
    wall0 = time.perf_counter()
    t0.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    barrier()
    clocks = sampler.stop() if sampler else None
    st = h3.h3_sync_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after timed steps: {h3.h3_status_string(st)}")
    ms = t0.elapsed_time(t1) / args.steps
    names = ["modulate", "qkv_rope_gemm", "attention", "out_gemm"]
    per = {n: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs)
           for i, n in enumerate(names)}
    ms = max_over_ranks(ms, world, dev)

    # ---- end to end through the public API with host buffers: every step uploads
    # its input x and modulation vectors from pinned host memory and downloads its
    # output.  Copies run on a second stream, double-buffered, so step k's
    # compute overlaps step k+1's upload and step k-1's download.
    x_host = inp["x"].pin_memory()
    mod_host = {k: inp[k].pin_memory() for k in ("shift", "scale", "gate")}
    out_host = [torch.empty(L, d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h2d = x_host.numel() * 2 + sum(v.numel() * 4 for v in mod_host.values())
    d2h = out_host[0].numel() * 2
    xb = [x, torch.empty_like(x)]
    ob = [out, torch.empty_like(out)]
    mb = [{k: v for k, v in (("shift", shift), ("scale", scale), ("gate", gate))},
          {k: torch.empty_like(v) for k, v in (("shift", shift), ("scale", scale), ("gate", gate))}]
    cs = torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]

    def upload(b):
        with torch.cuda.stream(cs):
            xb[b].copy_(x_host, non_blocking=True)
            for k in ("shift", "scale", "gate"):
                mb[b][k].copy_(mod_host[k], non_blocking=True)
            ev_in[b].record(cs)

    def download(b, k):
        with torch.cuda.stream(cs):
            cs.wait_event(ev_done[b])
            out_host[k % 2].copy_(ob[b], non_blocking=True)

    def e2e_run(n):
        upload(0)
        for k in range(n):
            b = k % 2
            stream.wait_event(ev_in[b])
            h3.h3_attn_block_fwd(desc, xb[b], mod_d, pos_d, mb[b]["shift"], mb[b]["scale"],
                                 mb[b]["gate"], wqkv, wo, ws, nbytes, ob[b], stream=stream)
            ev_done[b].record(stream)
            if k >= 1:
                download(1 - b, k - 1)
            if k + 1 < n:
                if k >= 1:
                    cs.wait_event(ev_done[1 - b])   # step k-1 no longer reads xb[1-b]
                upload(1 - b)
        download((n - 1) % 2, n - 1)

    e2e_run(2)
    torch.cuda.synchronize(dev)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cs)
    e2e_run(args.steps)
    e1.record(cs)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / args.steps
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    st = h3.h3_sync_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after e2e steps: {h3.h3_status_string(st)}")

    # ---- the 50-step denoising sweep: step k uses its own seeded modulation set
    # and the previous step's output (in place) as its input
    from h3inputs import sweep_modulation
    sweep_mods = [{k: v.to(dev) for k, v in sweep_modulation(cfg, s).items()}
                  for s in range(1, 51)]
    xs = x.clone()
    sev = [torch.cuda.Event(enable_timing=True) for _ in range(51)]
    torch.cuda.synchronize(dev)
    barrier()
    sev[0].record(stream)
    for s_i in range(50):
        m = sweep_mods[s_i]
        h3.h3_attn_block_fwd(desc, xs, mod_d, pos_d, m["shift"], m["scale"], m["gate"], wqkv, wo,
                             ws, nbytes, xs, stream=stream)
        sev[s_i + 1].record(stream)
    torch.cuda.synchronize(dev)
    st = h3.h3_sync_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after the sweep: {h3.h3_status_string(st)}")
    sweep_steps = [sev[i].elapsed_time(sev[i + 1]) for i in range(50)]
    sweep_total = sev[0].elapsed_time(sev[50])
    del xs

    # ---- block-diagonal attention over the modality segments (cu_seqlens
    # [0, T, T+V, L]) on this step's rotated qkv, timed on its own
    cu = [0, cfg.n_text, cfg.n_text + cfg.n_video, L]
    qkv_ws = ws[(L * d * 2 + 255) // 256 * 256:][:L * 3 * d * 2].view(torch.bfloat16).view(L, 3 * d)
    o_var = torch.empty(L, d, dtype=torch.bfloat16, device=dev)
    h3.h3_joint_attn_varlen_fwd(qkv_ws, cu, L, H, 128, 0, None, o_var, stream=stream)
    vev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    vev[0].record(stream)
    for _ in range(5):
        h3.h3_joint_attn_varlen_fwd(qkv_ws, cu, L, H, 128, 0, None, o_var, stream=stream)
    vev[1].record(stream)
    torch.cuda.synchronize(dev)
    varlen_ms = vev[0].elapsed_time(vev[1]) / 5
    varlen_flops = 4.0 * d * sum((cu[i + 1] - cu[i]) ** 2 for i in range(3))

    # ---- the causal option of the same attention call (key index <= query
    # index in packed order) on the same rotated qkv, timed on its own
    h3.h3_joint_attn_fwd(qkv_ws, L, H, 128, 1, None, o_var, stream=stream)
    cev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    cev[0].record(stream)
    for _ in range(5):
        h3.h3_joint_attn_fwd(qkv_ws, L, H, 128, 1, None, o_var, stream=stream)
    cev[1].record(stream)
    torch.cuda.synchronize(dev)
    causal_ms = cev[0].elapsed_time(cev[1]) / 5
    causal_flops = 4.0 * d * L * (L + 1) / 2.0
    del o_var

    # ---- the standalone 3D RoPE call (h3_mrope_apply, in place on Q and K of the
    # workspace's qkv; the fused block applies RoPE in the QKV epilogue instead).
    # Its 2.4 GB of traffic per call exceed L2, so no flush is needed.
    for _ in range(2):
        h3.h3_mrope_apply(qkv_ws, pos_d, L, H, stream=stream)
    rev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    rev[0].record(stream)
    for _ in range(10):
        h3.h3_mrope_apply(qkv_ws, pos_d, L, H, stream=stream)
    rev[1].record(stream)
    torch.cuda.synchronize(dev)
    mrope_ms = rev[0].elapsed_time(rev[1]) / 10
    mrope_bytes = 8.0 * L * d + 12.0 * L

    # ---- the modulate kernel on its own.  In the step it starts while the L2
    # still holds the previous output projection's dirty lines, whose write-back
    # shares DRAM with it; here the L2 is flushed by reading a 256 MB buffer
    # before each timed call (clean lines, x in DRAM)
    y_sa = torch.empty_like(x)
    flush_r = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    mts = []
    for it in range(6):
        flush_r.sum()
        ma, mb_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ma.record(stream)
        h3.h3_adaln_modulate(x, mod_d, shift, scale, L, d, cfg.n_mod, cfg.ln_eps, y_sa,
                             stream=stream)
        mb_.record(stream)
        torch.cuda.synchronize(dev)
        if it > 0:
            mts.append(ma.elapsed_time(mb_))
    mod_sa_ms = statistics.median(mts)
    # yardstick: a plain device copy of x (the same bytes read and written)
    # after the same flush
    cts = []
    for it in range(6):
        flush_r.sum()
        ma, mb_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ma.record(stream)
        with torch.cuda.stream(stream):
            y_sa.copy_(x)
        mb_.record(stream)
        torch.cuda.synchronize(dev)
        if it > 0:
            cts.append(ma.elapsed_time(mb_))
    mod_copy_ms = statistics.median(cts)
    del y_sa, flush_r

    # ---- the MLP sub-block of the same layer (hidden 4d), timed on its own
    hid = 4 * d
    gmlp = torch.Generator(device="cpu").manual_seed(11)
    w1m = (torch.randn(hid, d, generator=gmlp) / d ** 0.5).to(torch.bfloat16).to(dev)
    w2m = (torch.randn(d, hid, generator=gmlp) / hid ** 0.5).to(torch.bfloat16).to(dev)
    mdesc = h3.MlpDesc.make(L=L, d=d, hidden=hid, ln_eps=cfg.ln_eps, n_mod=cfg.n_mod)
    mbytes = h3.h3_mlp_workspace_size(mdesc)
    mws = torch.empty(mbytes, dtype=torch.uint8, device=dev)
    mout = torch.empty(L, d, dtype=torch.bfloat16, device=dev)
    for _ in range(2):
        h3.h3_mlp_block_fwd(mdesc, x, mod_d, shift, scale, gate, w1m, w2m, mws, mbytes, mout,
                            stream=stream)
    mev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    mev[0].record(stream)
    for _ in range(5):
        h3.h3_mlp_block_fwd(mdesc, x, mod_d, shift, scale, gate, w1m, w2m, mws, mbytes, mout,
                            stream=stream)
    mev[1].record(stream)
    torch.cuda.synchronize(dev)
    mlp_ms = mev[0].elapsed_time(mev[1]) / 5
    mlp_flops = 4.0 * L * d * hid
    del w1m, w2m, mws, mout

    # ---- the fp8 (E4M3) variants: both projections of the attention block and of
    # the MLP in fp8 (weights quantised per output channel once, activations per
    # token on every call); the attention block's scores from E4M3 Q and K
    # (per-token / per-key-block scales), P.V in bf16
    def quant(w):
        q = torch.empty(w.shape, dtype=torch.uint8, device=dev)
        sc8 = torch.empty(w.shape[0], dtype=torch.float32, device=dev)
        h3.h3_quantize_rows_fp8(w, w.shape[0], w.shape[1], q, sc8, stream=stream)
        return q, sc8

    wqkv8, wqkv8s = quant(wqkv)
    wo8, wo8s = quant(wo)
    f8bytes = h3.h3_workspace_size_fp8(desc)
    ws8 = torch.empty(f8bytes, dtype=torch.uint8, device=dev)
    out8 = torch.empty(L, d, dtype=torch.bfloat16, device=dev)

    def fp8_block():
        h3.h3_attn_block_fwd_fp8(desc, x, mod_d, pos_d, shift, scale, gate, wqkv8, wqkv8s, wo8,
                                 wo8s, ws8, f8bytes, out8, stream=stream)

    def timed(fn, n=5):
        fn()
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record(stream)
        for _ in range(n):
            fn()
        eb.record(stream)
        torch.cuda.synchronize(dev)
        return ea.elapsed_time(eb) / n

    fp8_block_ms = timed(fp8_block)
    # the fp8-score attention on its own (its Q/K quantisation included), on the
    # rotated qkv the fp8 block left in its workspace
    r256 = lambda n: (n + 255) // 256 * 256
    qkv8 = ws8[r256(L * d * 2):r256(L * d * 2) + L * 3 * d * 2].view(torch.bfloat16).view(L, 3 * d)
    a8bytes = h3.h3_attn_workspace_size_fp8(L, H)
    aws8 = torch.empty(a8bytes, dtype=torch.uint8, device=dev)
    o8 = torch.empty(L, d, dtype=torch.bfloat16, device=dev)
    attn_fp8_ms = timed(lambda: h3.h3_joint_attn_fwd_fp8(qkv8, L, H, 128, 0, None, aws8, a8bytes,
                                                         o8, stream=stream))
    sq8 = aws8[r256(L * 2 * d):r256(L * 2 * d) + H * L * 4].view(torch.float32)
    sk_off = r256(L * 2 * d) + r256(H * L * 4)
    sk8 = aws8[sk_off:sk_off + H * ((L + 127) // 128) * 4].view(torch.float32)
    quant_qk_ms = timed(lambda: h3.h3_quantize_qk_fp8(qkv8, L, H, 128, aws8, sq8, sk8,
                                                      stream=stream))
    del ws8, out8, wqkv8, wo8, aws8, o8
    g8 = torch.Generator(device="cpu").manual_seed(11)
    w1f = (torch.randn(4 * d, d, generator=g8) / d ** 0.5).to(torch.bfloat16).to(dev)
    w2f = (torch.randn(d, 4 * d, generator=g8) / (4 * d) ** 0.5).to(torch.bfloat16).to(dev)
    w1q, w1qs = quant(w1f)
    w2q, w2qs = quant(w2f)
    del w1f, w2f
    m8desc = h3.MlpDesc.make(L=L, d=d, hidden=4 * d, ln_eps=cfg.ln_eps, n_mod=cfg.n_mod)
    m8bytes = h3.h3_mlp_workspace_size_fp8(m8desc)
    mws8 = torch.empty(m8bytes, dtype=torch.uint8, device=dev)
    mout8 = torch.empty(L, d, dtype=torch.bfloat16, device=dev)
    fp8_mlp_ms = timed(lambda: h3.h3_mlp_block_fwd_fp8(m8desc, x, mod_d, shift, scale, gate, w1q,
                                                        w1qs, w2q, w2qs, mws8, m8bytes, mout8,
                                                        stream=stream))
    del mws8, mout8, w1q, w2q
    st = h3.h3_sync_status(stream)
    if st != 0:
        raise RuntimeError(f"device status after the fp8 runs: {h3.h3_status_string(st)}")

    # ---- one denoising-step update of the packed latent (C = 96 channels per
    # token: 24 latent channels x 1x2x2 patch), HBM-bound; L2 flushed between runs
    # by reading a 256 MB buffer (twice the L2): the update's inputs come from
    # DRAM, and the L2 holds clean lines when it starts, so the timed launch does
    # not also pay for writing back a flush's dirty lines
    C_lat = 96
    zl = torch.randn(L, C_lat, device=dev)
    vl = torch.randn(L, C_lat, device=dev).to(torch.bfloat16)
    x0l = torch.empty_like(zl)
    flush = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    dts = []
    for it in range(6):
        flush.sum()
        e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_a.record(stream)
        h3.h3_denoise_step(zl, x0l, vl, mod_d, None, None, L, C_lat, [0.0, 0.6, 0.4],
                           [0.0, 0.5, 0.3], [0, 1, 1], stream=stream)
        e_b.record(stream)
        torch.cuda.synchronize(dev)
        if it > 0:
            dts.append(e_a.elapsed_time(e_b))
    denoise_ms = statistics.median(dts)
    lat_rows = L - cfg.n_text
    denoise_bytes = lat_rows * C_lat * (4 + 2 + 4 + 4) + cfg.n_text * C_lat * 8
    # yardstick for a launch this short: a plain device copy that moves the
    # same number of bytes (half read, half written) after the same flush
    src = torch.ones(denoise_bytes // 8, dtype=torch.float32, device=dev)
    dst = torch.empty_like(src)
    cts = []
    for it in range(6):
        flush.sum()
        e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_a.record(stream)
        with torch.cuda.stream(stream):
            dst.copy_(src)
        e_b.record(stream)
        torch.cuda.synchronize(dev)
        if it > 0:
            cts.append(e_a.elapsed_time(e_b))
    copy_same_ms = statistics.median(cts)
    del zl, vl, x0l, flush, src, dst

    flops = cfg.flops()
    value = job_throughput(flops, world, ms) / 1e12
    attn_flops = 4.0 * L * L * d
    peaks, peak_kind = _peaks()
    peak = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    achieved = attn_flops / (per["attention"] * 1e-3) / 1e12
    traffic = None
    tf = os.path.join(ROOT, "profiles", "attention_traffic.json")
    if os.path.exists(tf) and cfg.name == "full":
        import hashlib
        with open(tf) as f:
            rec = json.load(f)
        with open(os.path.join(ROOT, rec["source"]), "rb") as f:
            same = hashlib.sha256(f.read()).hexdigest() == rec.get("source_sha256")
        # counters taken on another version of the kernel do not describe this one
        traffic = rec.get("bytes_per_launch_full") if same else None

    # the peak's own clock: the sustained GEMM loop ran under the power cap at a
    # lower SM clock than a kernel inside this step, so the fraction is also
    # given against that peak scaled to the kernel's clock
    peak_mhz = None
    if isinstance(peaks.get("clocks_under_load"), dict):
        peak_mhz = peaks["clocks_under_load"].get("sm_mhz_median")
    run_mhz = clocks.get("sm_mhz") if clocks else None
    frac_clk = (achieved / (peak * run_mhz / peak_mhz)
                if peak_mhz and run_mhz else None)
    mcycles = ({n: t * run_mhz / 1e3 for n, t in per.items()} if run_mhz else None)
    hbm = float(peaks["hbm_gbs"])
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": _config(cfg, world),
        "tokens_per_s": job_throughput(L, world, ms),
        "pct_of_bf16_peak_block": flops / (ms * 1e-3) / 1e12 / peak,
        "kernel_ms": per,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "frac_at_kernel_clock": frac_clk,
                     "peak_sm_mhz": peak_mhz, "kernel_sm_mhz": run_mhz,
                     "kernel": "attention (attn_fwd_kernel)",
                     "peak_kind": f"{peak_kind} bf16 sustained (kernel inside a long step)"},
        "kernel_mcycles": mcycles,
        "e2e": {"value": job_throughput(flops, world, e2e_ms) / 1e12, "unit": UNIT,
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "sweep50": {"steps": 50, "total_ms": sweep_total,
                    "per_step_ms": {"median": statistics.median(sweep_steps),
                                    "min": min(sweep_steps), "max": max(sweep_steps)},
                    "sustained_tflops": 50 * flops / (sweep_total * 1e-3) / 1e12,
                    "frac_of_sustained_bf16_peak":
                        50 * flops / (sweep_total * 1e-3) / 1e12 / peak},
        "attn_varlen_modality": {"cu_seqlens": cu, "ms": varlen_ms,
                                 "tflops": varlen_flops / (varlen_ms * 1e-3) / 1e12,
                                 "frac_of_sustained_bf16_peak":
                                     varlen_flops / (varlen_ms * 1e-3) / 1e12 / peak},
        "attn_causal": {"ms": causal_ms, "flops": causal_flops,
                        "tflops": causal_flops / (causal_ms * 1e-3) / 1e12,
                        "frac_of_sustained_bf16_peak":
                            causal_flops / (causal_ms * 1e-3) / 1e12 / peak,
                        "note": "unmasked pairs only: 4 d L (L + 1) / 2 FLOPs"},
        "mlp_block": {"hidden": hid, "ms": mlp_ms,
                      "tflops": mlp_flops / (mlp_ms * 1e-3) / 1e12,
                      "frac_of_sustained_bf16_peak": mlp_flops / (mlp_ms * 1e-3) / 1e12 / peak},
        "fp8": {"attn_block_ms": fp8_block_ms,
                "attn_block_tflops": cfg.flops() / (fp8_block_ms * 1e-3) / 1e12,
                "attention_ms": attn_fp8_ms,
                "attention_tflops": 4.0 * L * L * d / (attn_fp8_ms * 1e-3) / 1e12,
                "quantize_qk_ms": quant_qk_ms,
                "mlp_block_ms": fp8_mlp_ms,
                "mlp_block_tflops": mlp_flops / (fp8_mlp_ms * 1e-3) / 1e12,
                "note": "projections in E4M3 (tcgen05 kind::f8f6f4); attention scores from "
                        "E4M3 Q and K, P.V in bf16; attention_ms includes the Q/K "
                        "quantisation; FLOPs counted as for the bf16 block"},
        "mrope_standalone": {"ms": mrope_ms, "bytes": mrope_bytes,
                             "gbs": mrope_bytes / (mrope_ms * 1e-3) / 1e9,
                             "frac_of_hbm_peak": mrope_bytes / (mrope_ms * 1e-3) / 1e9 / hbm},
        "modulate_hbm": {"ms": per["modulate"], "bytes": 4.0 * L * d,
                         "gbs": 4.0 * L * d / (per["modulate"] * 1e-3) / 1e9,
                         "frac_of_hbm_peak": 4.0 * L * d / (per["modulate"] * 1e-3) / 1e9 / hbm},
        "modulate_standalone": {"ms": mod_sa_ms, "bytes": 4.0 * L * d,
                                "gbs": 4.0 * L * d / (mod_sa_ms * 1e-3) / 1e9,
                                "frac_of_hbm_peak": 4.0 * L * d / (mod_sa_ms * 1e-3) / 1e9 / hbm,
                                "copy_same_bytes_ms": mod_copy_ms,
                                "frac_of_same_size_copy": mod_copy_ms / mod_sa_ms,
                                "note": "alone, L2 flushed by a read before each call; "
                                        "modulate_hbm is the same kernel inside the step"},
        "denoise_step": {"L": L, "C": C_lat, "ms": denoise_ms,
                         "gbs": denoise_bytes / (denoise_ms * 1e-3) / 1e9,
                         "frac_of_hbm_peak": denoise_bytes / (denoise_ms * 1e-3) / 1e9 / hbm,
                         "copy_same_bytes_ms": copy_same_ms,
                         "frac_of_same_size_copy": copy_same_ms / denoise_ms},
        "gpu_launches": 4 * args.steps,
        "clocks": clocks,
        "wall_s_timed": wall,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        full, sample, cores, _ = oracle_sample(cfg, inp, scale_factor=24.0)
        line["cpu_baseline"] = {"value": flops / full / 1e12, "unit": UNIT, "cores": cores,
                                "kind": "oracle", "sample": sample,
                                "extrapolated_block_s": full}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_library_context(args, cfg):
    """Context, not the contract line: this library's block (full and causal)
    next to PyTorch's fused attention (its cuDNN / flash / memory-efficient
    backends, whichever run) and cuBLAS on the same shapes and the same rotated
    Q, K, V, one GPU, CUDA events, 3 warm-up and `steps` timed calls each."""
    import torch
    import torch.nn.functional as F
    import joint_audio_video_gb300 as h3
    from joint_audio_video_gb300 import build as h3build
    from h3inputs import block_inputs

    h3build.build()
    h3.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    L, d, H = cfg.L, cfg.d, cfg.n_heads
    inp = block_inputs(cfg)
    mod, pos = h3.h3_build_packed_layout(cfg.n_text, cfg.video_t, cfg.video_h, cfg.video_w,
                                         cfg.audio_channels, cfg.audio_steps)
    x = inp["x"].to(dev)
    wqkv, wo = inp["Wqkv"].to(dev), inp["Wo"].to(dev)
    shift, scale, gate = inp["shift"].to(dev), inp["scale"].to(dev), inp["gate"].to(dev)
    mod_d, pos_d = torch.from_numpy(mod).to(dev), torch.from_numpy(pos).to(dev)
    n = max(args.steps, 3)

    def timed(fn):
        for _ in range(3):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / n

    res = {"context": "library", "config": {"workload": _workload(cfg), "L": L, "d": d,
                                            "heads": H}, "steps": n, "h3": {}, "torch_sdpa": {},
           "cublas": {}, "torch": torch.__version__}
    qkv = None
    for causal in (0, 1):
        desc = h3.BlockDesc.make(L=L, d=d, n_heads=H, rope_sec=cfg.rope_sections,
                                 rope_base=cfg.rope_base, ln_eps=cfg.ln_eps, n_mod=cfg.n_mod,
                                 causal=causal)
        nbytes = h3.h3_workspace_size(desc)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        out = torch.empty(L, d, dtype=torch.bfloat16, device=dev)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        step = lambda: h3.h3_attn_block_fwd_profiled(desc, x, mod_d, pos_d, shift, scale, gate,
                                                     wqkv, wo, ws, nbytes, out, evs, stream=stream)
        block_ms = timed(step)
        step()
        torch.cuda.synchronize(dev)
        attn_ms = evs[2].elapsed_time(evs[3])
        flops = cfg.flops(causal=bool(causal))
        attn_flops = 4.0 * d * (L * (L + 1) / 2.0 if causal else float(L) * L)
        res["h3"]["causal" if causal else "full"] = {
            "block_ms": block_ms, "block_tflops": flops / (block_ms * 1e-3) / 1e12,
            "attention_ms_last_call": attn_ms,
            "attention_tflops": attn_flops / (attn_ms * 1e-3) / 1e12}
        if qkv is None:
            off = (L * d * 2 + 255) // 256 * 256
            qkv = ws[off:off + L * 3 * d * 2].view(torch.bfloat16).view(L, 3, H, 128).clone()
        if h3.h3_sync_status(stream) != 0:
            raise RuntimeError("device status after the block runs")
        del ws, out
    q, k, v = (qkv[:, i].permute(1, 0, 2).unsqueeze(0).contiguous() for i in range(3))
    del qkv
    try:
        from torch.nn.attention import SDPBackend, sdpa_kernel
        backends = {"cudnn": SDPBackend.CUDNN_ATTENTION, "flash": SDPBackend.FLASH_ATTENTION,
                    "efficient": SDPBackend.EFFICIENT_ATTENTION}
    except ImportError:
        backends = {}
    for name, be in backends.items():
        for causal in (False, True):
            key = f"{name}_{'causal' if causal else 'full'}"
            try:
                with sdpa_kernel([be]):
                    ms = timed(lambda: F.scaled_dot_product_attention(q, k, v, is_causal=causal))
                attn_flops = 4.0 * d * (L * (L + 1) / 2.0 if causal else float(L) * L)
                res["torch_sdpa"][key] = {"ms": ms,
                                          "tflops": attn_flops / (ms * 1e-3) / 1e12}
            except Exception as e:   # a backend that does not support the shape or the GPU
                res["torch_sdpa"][key] = {"unavailable": str(e).splitlines()[0][:160]}
    del q, k, v
    y = torch.randn(L, d, device=dev).to(torch.bfloat16)
    for name, w in (("qkv_proj", wqkv), ("out_proj", wo)):
        ms = timed(lambda: torch.matmul(y, w.t()))
        res["cublas"][name] = {"ms": ms, "tflops": 2.0 * L * d * w.shape[0] / (ms * 1e-3) / 1e12}
    print(json.dumps(res), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="h3", choices=["h3", "reference"])
    ap.add_argument("--config", default="full", help="block workload (default: full, L=58758)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--library-context", action="store_true",
                    help="print this library's block next to PyTorch SDPA and cuBLAS on the "
                         "same shapes (context; not the benchmark line)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)        # at least 3 untimed warm-up steps
    from h3inputs import CONFIGS
    cfg = CONFIGS[args.config]
    if args.impl == "reference":
        return run_reference(args, cfg)
    if args.library_context:
        return run_library_context(args, cfg)
    return run_gpu(args, cfg)


if __name__ == "__main__":
    sys.exit(main())
