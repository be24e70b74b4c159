"""Benchmark of the DLite draft-and-verify round on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload NAME]

One step = one whole round (draft: staging, backbone, sequential head, LM head
with fused sampling; verify: speculative sampling with residual resampling;
RNG-position bookkeeping) over one batch of synthetic requests, replayed from
a captured CUDA graph. Inputs are resident in HBM when the timed region
starts; each round streams all 2.4 GB of weights (> L2), and the per-round
inputs cycle through a ring of 4 batches.

--impl reference times the CPU oracle (float64, numpy) on the host cores on a
bounded sample of the same workload. Under torchrun only rank 0 runs it.
"""
import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from history_free_speculative_gb300 import reporter as rp  # noqa: E402
from history_free_speculative_gb300 import workload as wk  # noqa: E402

METRIC = "draft+verify rounds/s & committed tok/s, Qwen3-8B-shape drafter B=32; %roofline"
RING = 4


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def shard_round_index(k, rank):
    """Input slot k of rank `rank`: every replica drafts its own requests (weak scaling)."""
    return k + 1000 * rank


def reduce_over_ranks(t_s, committed, device):
    """The job's time (the slowest rank) and its committed tokens (all ranks)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return t_s, committed
    tt = torch.tensor([t_s], device=device, dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    cc = torch.tensor([committed], device=device, dtype=torch.int64)
    dist.all_reduce(cc)
    return float(tt.item()), int(cc.item())


KERNEL_SOURCES = ["lm_head.cu", "tc_device.cuh", "tc_gemm.h", "internal.h", "common.cuh"]


def lm_head_traffic():
    """DRAM bytes per LM-head launch from the committed ncu summary, or None when
    the kernel sources changed since that capture."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", "lm_head_kernel_qwen3-8b-b32.md")
    if not os.path.exists(prof):
        return None
    vals = {}
    for line in open(prof):
        if ":" in line and line.strip().split(":")[0] in ("traffic_bytes_per_launch", "kernel_sources_sha256"):
            k, v = line.strip().split(":", 1)
            vals[k] = v.strip()
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "history_free_speculative_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    if vals.get("kernel_sources_sha256") != h.hexdigest():
        return None
    return int(vals["traffic_bytes_per_launch"])


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        """Start sampling; returns once the sampler is up (its start-up is kept out of the timed region)."""
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            t0 = time.time()
            while len(self.lines) < 2 and time.time() - t0 < 10:
                time.sleep(0.02)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if not self.proc:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()

    def summary(self, t_begin, t_end):
        """Summarise the samples taken between t_begin and t_end (wall clock)."""
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, l in list(self.lines):
            if not (t_begin <= ts <= t_end):
                continue
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                pw.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(pw) if pw else None,
                "window_s": round(t_end - t_begin, 3)}


# ---------------------------------------------------------------- GPU arm

N_ACCEPT_TABLES = 64   # per-round agreement tables of the greedy workloads, cycled by the device round counter


def accept_tables(wl, B, K, device):
    """Agreement probabilities of the synthetic target, [n_tables, B, K] float32:
    two request classes (Beta(6, 4) / Beta(18, 2), alternating) or one constant c."""
    if wl.accept_classes:
        c = wk.make_beta_accept(B, K, wl.input_seed + 7, n_tables=N_ACCEPT_TABLES)
    else:
        c = wk.make_const_accept(B, K, wl.accept_c)
    return c.to(device=device, dtype=torch.float32).contiguous()


class Rig:
    """One drafter's rounds over B requests, captured as one CUDA graph per input
    slot (draft; greedy: synthetic target; verification; position advance)."""

    def __init__(self, dr, wl, B, dev, stream, rank, match=False, nv=None, grp=1):
        from history_free_speculative_gb300 import binding
        cfg = dr.cfg
        self.dr, self.wl, self.B, self.stream = dr, wl, B, stream
        T = 0.0 if match else wl.temperature
        sampling = T > 0
        self.T, self.sampling, self.match, self.grp = T, sampling, match, grp
        ring = []
        for k in range(RING):
            hidden, _, _ = wk.make_round_inputs(wl, B=B, round_index=shard_round_index(k, rank), device=dev)
            item = {"hidden": hidden}
            if sampling or match:
                item["probs"] = wk.make_target_probs(B, cfg.K, cfg.V, wl.rng_seed + 17 * k + 1000 * rank, device=dev)
            ring.append(item)
        self.ring = ring
        _, anchor, pos = wk.make_round_inputs(wl, B=B, round_index=shard_round_index(999, rank), device=dev)
        self.anchor, self.pos = anchor, pos
        if grp > 1:   # the group [B, G] (anchor last); the verification writes its next anchor aside
            self.group = torch.randint(0, cfg.V, (B, grp), device=dev, dtype=torch.int32)
            self.next_tok = torch.empty(B, device=dev, dtype=torch.int32)
        self.out = dr.new_outputs(B, dev)
        self.stub = not sampling and not match   # greedy: the target's choices come from the synthetic target
        self.tgt = torch.empty(B, cfg.K + 1, device=dev, dtype=torch.int32)
        self.accept = accept_tables(wl, B, cfg.K, dev) if self.stub else None
        self.round_ctr = torch.zeros(1, device=dev, dtype=torch.int32)
        out, nxt = self.out, (self.next_tok if grp > 1 else anchor)

        def enqueue(k):
            it = ring[k]
            dr.draft_round(it["hidden"], self.group if grp > 1 else anchor, T, wl.rng_seed, pos, out["cand"],
                           out["qstats"], stream=stream)
            if self.stub:
                binding.synthetic_target(out["cand"], self.accept, wl.rng_seed, pos, self.tgt, cfg.V,
                                         round_counter=self.round_ctr, stream=stream)
            if match:
                dr.verify_ex(binding.VERIFY_MATCH, out["cand"], out["accepted"], out["commits"], out["n_commit"],
                             nxt, n_verify=nv, probs=it["probs"], seed=wl.rng_seed, pos=pos, stream=stream)
            elif nv is not None:
                dr.verify_ex(binding.VERIFY_SAMPLE if sampling else binding.VERIFY_GREEDY, out["cand"],
                             out["accepted"], out["commits"], out["n_commit"], nxt, n_verify=nv,
                             target_tokens=None if sampling else self.tgt,
                             qstats=out["qstats"] if sampling else None,
                             probs=it.get("probs") if sampling else None, temperature=T, seed=wl.rng_seed,
                             pos=pos, stream=stream)
            elif sampling:
                dr.verify_sample(out["cand"], out["qstats"], None, it["probs"], T, wl.rng_seed, pos,
                                 out["accepted"], out["commits"], out["n_commit"], nxt, stream=stream)
            else:
                dr.verify(out["cand"], self.tgt, out["accepted"], out["commits"], out["n_commit"], nxt,
                          stream=stream)
            if grp > 1:
                dr.shift_group(out["commits"], out["n_commit"], self.group, stream=stream)
            dr.advance(out["n_commit"], pos, stream=stream)

        self.enqueue = enqueue
        with torch.cuda.stream(stream):   # eager warm-up (also sets kernel attributes before capture)
            enqueue(0)
        stream.synchronize()
        self.graphs = []
        for k in range(RING):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(g, stream=stream):
                    enqueue(k)
            self.graphs.append(g)
        self.launches_per_step = (dr.launch_count(B, T) + 1 + (1 if match else 0) + (1 if grp > 1 else 0)
                                  + (1 if self.stub else 0))
        self.ncommit_total = torch.zeros((), dtype=torch.int64, device=dev)

    def replay(self, n, count=True, events=None):
        """n graph replays on the rig's stream (committed tokens summed on the device)."""
        with torch.cuda.stream(self.stream):
            for i in range(n):
                self.graphs[i % RING].replay()
                if count:
                    self.ncommit_total += self.out["n_commit"].sum()
                if events is not None:
                    events[i + 1].record(self.stream)

    def close(self):
        self.graphs = []


def replay_seconds(rig, steps, warmup):
    """Device-timed seconds of `steps` replays after `warmup`, and the tokens they committed."""
    rig.replay(warmup)
    rig.stream.synchronize()
    rig.ncommit_total.zero_()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(rig.stream)
    rig.replay(steps)
    ev1.record(rig.stream)
    rig.stream.synchronize()
    return ev0.elapsed_time(ev1) / 1e3, int(rig.ncommit_total.item())


def concurrency_sweep(dev, stream, rank, steps, warmup):
    """The two-class concurrency sweep on the Qwen3-8B-shaped drafter: greedy rounds
    with the synthetic target (c ~ Beta(6, 4) / Beta(18, 2), alternating requests),
    one captured graph per input slot and batch, B in wk.SWEEP_BATCHES."""
    from history_free_speculative_gb300 import binding
    wl = wk.WORKLOADS["qwen3-8b-sweep"]
    cfg = wl.cfg
    hbm, _, tf_sus, _ = measured_peaks()
    W = wk.make_weights(cfg, wl.weight_seed, device=dev)
    dr = binding.Drafter(cfg, W, B_max=max(wk.SWEEP_BATCHES))
    del W
    res = []
    launches = 0
    for B in wk.SWEEP_BATCHES:
        rig = Rig(dr, wl, B, dev, stream, rank)
        t_s, committed = replay_seconds(rig, steps, warmup)
        launches += rig.launches_per_step * steps
        floor = rp.roofline_floor_s(rp.round_bytes(cfg, B), rp.round_flops(cfg, B), hbm, tf_sus)
        ms = t_s * 1e3 / steps
        res.append({"B": B, "rounds_s": round(steps / t_s, 2), "committed_tok_s": round(committed / t_s, 1),
                    "mean_commit_per_request": round(committed / (steps * B), 4), "ms_per_round": round(ms, 4),
                    "round_roofline_frac": round(floor / (ms / 1e3), 4)})
        rig.close()
    dr.close()
    return res, launches


def run_gpu(args):
    from history_free_speculative_gb300 import binding

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(dev))
    wl = wk.WORKLOADS[args.workload]
    if args.batch:
        wl = dataclasses.replace(wl, B=args.batch, name=f"{wl.name}-B{args.batch}")
    match = args.verify == "match"
    nv = None if args.n_verify < 0 else args.n_verify
    if match:   # greedy draft against the target's own samples at the workload's temperature
        wl = dataclasses.replace(wl, name=f"{wl.name}-match")
    if nv is not None:
        wl = dataclasses.replace(wl, name=f"{wl.name}-nv{nv}")
    if args.head == "gated":   # the official gated token-feedback head
        wl = dataclasses.replace(wl, cfg=dataclasses.replace(wl.cfg, head="gated"), name=f"{wl.name}-gated")
    grp = max(1, args.group)
    if grp > 1:   # a local token group of G tokens ending at the anchor
        wl = dataclasses.replace(wl, cfg=dataclasses.replace(wl.cfg, G=grp), name=f"{wl.name}-G{grp}")
    if args.act_planes == 2:   # fp32-class backbone activations (two bf16 planes)
        wl = dataclasses.replace(wl, cfg=dataclasses.replace(wl.cfg, act_planes=2), name=f"{wl.name}-act2")
    if args.history > 0:   # the history-KV control: a ring of the last H draft K/V rows per layer
        wl = dataclasses.replace(wl, cfg=dataclasses.replace(wl.cfg, history=args.history),
                                 name=f"{wl.name}-H{args.history}")
    cfg = wl.cfg
    B = wl.B
    stream = torch.cuda.Stream(device=dev)
    clocks = ClockSampler(local) if not args.no_clock_sampler else None
    if clocks:
        clocks.start()

    W = wk.make_weights(cfg, wl.weight_seed, device=dev)
    dr = binding.Drafter(cfg, W, B_max=B)
    rig = Rig(dr, wl, B, dev, stream, rank, match=match, nv=nv, grp=grp)
    T, sampling, out = rig.T, rig.sampling, rig.out
    rig.replay(args.warmup)
    stream.synchronize()

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    # the same replays for >= 1 s right before the timed region, so that the clock
    # samples (every 50 ms) describe the load the timed steps ran under
    barrier()
    t_load = time.time()
    while time.time() - t_load < args.clock_window:
        rig.replay(RING, count=False)
        stream.synchronize()
    rig.ncommit_total.zero_()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier()
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with torch.cuda.stream(stream):
        ev0.record(stream)
        step_ev[0].record(stream)
    rig.replay(args.steps, events=step_ev)
    with torch.cuda.stream(stream):
        ev1.record(stream)
    stream.synchronize()
    t_end = time.time()
    clk = clocks.summary(t_load, t_end) if clocks else {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["not sampled"]}
    if clocks:
        clk["window"] = "the timed steps and the >= %.1f s of the same replays right before them" % args.clock_window
    step_ms = sorted(step_ev[i].elapsed_time(step_ev[i + 1]) for i in range(args.steps))
    barrier()
    ms = ev0.elapsed_time(ev1)
    t_s = ms / 1e3
    committed = int(rig.ncommit_total.item())
    t_s, committed = reduce_over_ranks(t_s, committed, dev)
    rounds_s = ws * args.steps / t_s
    tok_s = committed / t_s
    counters = dr.counters(reset=True)

    # ---- per-kernel CUDA-event times (eager, same inputs) for the roofline
    per = {}
    nprof = 5
    for r in range(nprof):
        it = rig.ring[r % RING]
        times = dr.stage_times(it["hidden"], rig.group if grp > 1 else rig.anchor, T, wl.rng_seed, rig.pos, out,
                               target_tokens=None if sampling else rig.tgt,
                               target_probs=it.get("probs"), stream=stream)
        for name, t in times:
            per.setdefault(name, []).append(t)
    per_launch = {n: sum(v) / len(v) for n, v in per.items()}   # ms per launch (mean over a name's launches)
    hbm, tf_burst, tf_sus, peak_src = measured_peaks()
    lm_ms = per_launch.get("lm_head", float("nan"))
    gated = getattr(cfg, "head", "rnn") == "gated"   # one W_o projection per step
    lm_bytes = rp.gated_lm_bytes(cfg, B) if gated else rp.lm_head_bytes(cfg, B)
    lm_flops = rp.gated_lm_flops(cfg, B) if gated else rp.lm_head_flops(cfg, B)
    achieved_gbs = lm_bytes / (lm_ms / 1e3) / 1e9
    achieved_tf = lm_flops / (lm_ms / 1e3) / 1e12
    t_bytes = lm_bytes / (hbm * 1e9)
    t_flops = lm_flops / (tf_sus * 1e12)
    bound = "hbm" if t_bytes >= t_flops else "tensor"
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": round(achieved_gbs, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved_gbs / hbm, 4)}
    else:
        roof = {"bound": "tensor", "achieved": round(achieved_tf, 1), "peak": tf_sus, "unit": "TFLOP/s",
                "frac": round(achieved_tf / tf_sus, 4)}
    traffic = lm_head_traffic() if (cfg.D == 4096 and B == 32 and not cfg.history and not gated) else None
    roof.update({"kernel": "lm_head", "traffic": traffic, "peak_source": peak_src,
                 "algorithmic_bytes_per_launch": lm_bytes, "algorithmic_flops_per_launch": lm_flops,
                 "ms_per_launch": round(lm_ms, 4), "tensor_tflops": round(achieved_tf, 1)})
    if cfg.history:   # the control's dominant kernel: the history attention (one launch per layer)
        h_ms = per_launch.get("hist_attn", float("nan"))
        h_bytes = rp.hist_attn_bytes(cfg, B)
        h_gbs = h_bytes / (h_ms / 1e3) / 1e9
        lm_roof = roof
        roof = {"bound": "hbm", "achieved": round(h_gbs, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(h_gbs / hbm, 4), "kernel": "hist_attn", "traffic": None, "peak_source": peak_src,
                "algorithmic_bytes_per_launch": h_bytes, "ms_per_launch": round(h_ms, 4), "lm_head": lm_roof}
    round_bytes = rp.round_bytes(cfg, B)
    round_flops = rp.round_flops(cfg, B)
    floor = rp.roofline_floor_s(round_bytes, round_flops, hbm, tf_sus)
    ms_step = t_s * 1e3 / args.steps
    gpu_launches = rig.launches_per_step * args.steps

    # ---- end to end through the public host-buffer call
    e2e = None
    if (rank == 0 or ws > 1) and not match and nv is None and grp == 1:   # the host call: default verification
        e2e = run_e2e(dr, wl, rig.ring, rig.anchor, rig.pos, stream, max(3, min(args.steps, 20)))

    result = {
        "metric": METRIC, "value": round(rounds_s, 2), "unit": "rounds/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": cfg.dtype,
        "data": "synthetic (seeded random weights and inputs of the workload's shapes)",
        "config": {"workload": wl.name, "B_per_gpu": B, "D": cfg.D, "m": cfg.m, "K": cfg.K,
                   "L_D": cfg.L_D, "F": cfg.F, "R": cfg.R, "V": cfg.V, "temperature": T,
                   "parallelism": f"replicas x{ws}", "l2": "inputs larger than L2 (2.4 GB of weights "
                   "streamed per round, 4-batch input ring)", "history": cfg.history,
                   "draft_kv_bytes": 2 * cfg.L_D * cfg.history * cfg.n_kv * cfg.d_h * 2 * B,
                   "target": ("synthetic target tokens drawn in the graph: " +
                              ("c ~ Beta(6,4) / Beta(18,2) per alternating request" if wl.accept_classes
                               else f"agreement c = {wl.accept_c}")) if rig.stub else
                             "target probability rows of the workload (sampling / match)"},
        "committed_tok_s": round(tok_s, 1),
        "round_roofline": {"floor_ms": round(floor * 1e3, 4), "frac": round(floor / (ms_step / 1e3), 4),
                           "bytes": round_bytes, "flops": round_flops, "peak_source": peak_src},
        "roofline": roof,
        "per_kernel_ms": {n: round(v, 4) for n, v in per_launch.items()},
        "counters": counters,
        "step_ms": {"min": round(step_ms[0], 4), "median": round(step_ms[len(step_ms) // 2], 4),
                    "max": round(step_ms[-1], 4)},
        "clocks": clk,
        "e2e": e2e,
    }
    rig.close()
    dr.close()
    torch.cuda.synchronize()
    default_line = args.workload == "qwen3-8b-b32" and not (args.batch or match or nv is not None or grp > 1 or
                                                             gated or cfg.history or args.act_planes == 2)
    if default_line and not args.no_sweep:   # the concurrency sweep (its B = 1 entry is the latency regime)
        t0 = time.time()
        sweep, sw_launches = concurrency_sweep(dev, stream, rank, args.sweep_steps, 3)
        t1 = time.time()
        sw_clk = clocks.summary(t0, t1) if clocks else None
        result["sweep"] = {"workload": "qwen3-8b-shape-sweep (greedy, synthetic target, two classes)",
                           "steps_per_batch": args.sweep_steps, "points": sweep, "clocks": sw_clk}
        b1 = next(p for p in sweep if p["B"] == 1)
        result["b1"] = {"workload": "qwen3-8b-shape-b1 (greedy, synthetic target)", **b1}
    result["gpu_launches"] = gpu_launches
    if clocks:
        clocks.stop()
    if rank == 0:
        if ws == 1 and not args.no_cpu_baseline and not cfg.history:
            result["cpu_baseline"] = cpu_baseline(wl, W, rig.ring, rig.anchor, rig.pos)
        print(json.dumps(result), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(dr, wl, ring, anchor, pos, stream, steps):
    cfg, B, T = wl.cfg, wl.B, wl.temperature
    host = []
    for it in ring:
        h = {"hidden": it["hidden"].cpu().pin_memory()}
        if T > 0:
            h["probs"] = it["probs"].cpu().pin_memory()
            h["tgt"] = None
        else:
            h["probs"] = None
            h["tgt"] = torch.randint(0, cfg.V, (B, cfg.K + 1), dtype=torch.int32).pin_memory()
        host.append(h)
    a_h = anchor.cpu().pin_memory()
    p_h = pos.cpu().pin_memory()
    out_h = {k: v.pin_memory() for k, v in dr.new_outputs(B, "cpu").items()}
    for i in range(2):
        hh = host[i % RING]
        dr.round_host(hh["hidden"], a_h, p_h, hh["tgt"], hh["probs"], T, wl.rng_seed, out_h, stream=stream)
    t0 = time.perf_counter()
    for i in range(steps):
        hh = host[i % RING]
        dr.round_host(hh["hidden"], a_h, p_h, hh["tgt"], hh["probs"], T, wl.rng_seed, out_h, stream=stream)
        a_h.copy_(out_h["next_anchor"])
        p_h += out_h["n_commit"].to(torch.int64)
    dt = time.perf_counter() - t0
    hb = host[0]
    h2d = hb["hidden"].numel() * hb["hidden"].element_size() + B * 4 + B * 8
    out = {}
    if T > 0:   # pinned probabilities are read in place: each request's K draft entries and one full row
        h2d += B * cfg.K * 4 + B * cfg.V * 4
        out["target_probs"] = (f"read in place from pinned host memory by the verification "
                               f"({hb['probs'].numel() * 4} B per step resident on the host; "
                               f"counted: the K entries and the one row each request reads)")
    else:
        h2d += B * (cfg.K + 1) * 4
    d2h = B * 4 * 3 + B * (cfg.K + 1) * 4
    return {"value": round(steps / dt, 2), "unit": "rounds/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": steps, **out}


# ---------------------------------------------------------------- oracle (CPU) arm

def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


def oracle_request_seconds(wl, W64, hidden, anchor, pos, probs, b):
    """Oracle time of ONE request's round (draft + verify)."""
    from oracle import dlite_oracle as O
    cfg, T = wl.cfg, wl.temperature
    t0 = time.perf_counter()
    r = O.draft_request(hidden, int(anchor), W64, cfg, temperature=T, seed=wl.rng_seed,
                        pos=int(pos), request=b)
    if T > 0:
        w_q = W64["W_o"] if getattr(cfg, "head", "rnn") == "gated" else W64["E"]   # q(v) weights
        O.verify_sample(r["cand"], r["logit_d"], r["lse"], r["h"], w_q, probs, T, wl.rng_seed,
                        int(pos), b)
    else:
        O.verify_greedy(r["cand"], list(r["cand"]) + [0])
    return time.perf_counter() - t0


def _w64(W):
    from oracle import dlite_oracle as O
    out = {k: O.f64(v) for k, v in W.items() if k != "layers"}
    out["layers"] = [{k: O.f64(v) for k, v in l.items()} for l in W["layers"]]
    return out


def cpu_baseline(wl, W, ring, anchor, pos):
    """The oracle on the host cores over one whole round of the workload (every request
    drafted and verified; no extrapolation)."""
    W64 = _w64(W)
    it = ring[0]
    t0 = time.perf_counter()
    for b in range(wl.B):
        probs = it["probs"][b].cpu().numpy() if wl.temperature > 0 else None
        oracle_request_seconds(wl, W64, it["hidden"][b].cpu(), anchor[b].item(), pos[b].item(), probs, b)
    t_round = time.perf_counter() - t0
    return {"value": round(1.0 / t_round, 6), "unit": "rounds/s", "cores": _blas_threads(),
            "kind": "oracle",
            "sample": f"one whole round of the {wl.B} requests (float64 numpy oracle, draft + verify), "
                      f"{t_round:.1f} s"}


def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return
    wl = wk.WORKLOADS[args.workload]
    cfg, B = wl.cfg, wl.B
    W = wk.make_weights(cfg, wl.weight_seed, device="cpu")
    W64 = _w64(W)
    del W
    hidden, anchor, pos = wk.make_round_inputs(wl, round_index=1000)
    probs = None
    if wl.temperature > 0:
        probs = wk.make_target_probs(B, cfg.K, cfg.V, wl.rng_seed, device="cpu")
    for i in range(args.warmup):
        b = i % B
        oracle_request_seconds(wl, W64, hidden[b], anchor[b], pos[b],
                               None if probs is None else probs[b].numpy(), b)
    ts = []
    for i in range(args.steps):
        b = i % B
        ts.append(oracle_request_seconds(wl, W64, hidden[b], anchor[b], pos[b],
                                         None if probs is None else probs[b].numpy(), b))
    t_req = sum(ts) / len(ts)
    value = 1.0 / (t_req * B)
    sample = (f"each step = one of the {B} requests of a round through the float64 oracle "
              f"(draft + verify); rounds/s = 1 / (mean seconds per request x {B})")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "rounds/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t_req * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "B_per_gpu": B, "D": cfg.D, "V": cfg.V,
                   "temperature": wl.temperature},
        "cpu_baseline": {"value": round(value, 6), "unit": "rounds/s", "cores": _blas_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "rounds/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def spawn_replicas(n):
    """`--gpus N` without a launcher: run this command as N ranks, one per GPU."""
    import socket
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="qwen3-8b-b32", choices=sorted(wk.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clock-sampler", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the concurrency sweep of the default line")
    ap.add_argument("--sweep-steps", type=int, default=100, help="timed rounds per batch size of the sweep")
    ap.add_argument("--clock-window", type=float, default=1.2,
                    help="seconds of the same replays right before the timed steps, sampled for clocks")
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (exploration)")
    ap.add_argument("--verify", default="default", choices=["default", "match"],
                    help="match: greedy draft verified against the target's own samples")
    ap.add_argument("--n-verify", type=int, default=-1, help="verification window (candidates verified; -1: all)")
    ap.add_argument("--group", type=int, default=1, help="local token group size G (anchor last)")
    ap.add_argument("--head", default="rnn", choices=["rnn", "gated"], help="sequential head")
    ap.add_argument("--act-planes", type=int, default=1, choices=[1, 2],
                    help="backbone activations: 1 = bf16, 2 = fp32-class (two bf16 planes)")
    ap.add_argument("--history", type=int, default=0,
                    help="history-KV control: ring of the last H draft K/V rows per layer (0: history-free)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(spawn_replicas(args.gpus))
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != ws:
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE is {ws}")
    if args.impl == "reference":
        run_reference(args)
        return
    run_gpu(args)


if __name__ == "__main__":
    main()
