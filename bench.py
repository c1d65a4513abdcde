"""Throughput of the batched 80 ms lockstep decode tick on GB300.

Default workload: the full PersonaPlex shape (Helium 4096-d / 32 layers, depformer
1024-d / 6 layers) at B=64 with every slot's 3000-frame ring already full (KV prefilled
with seeded bf16 N(0,1)), steady-state greedy ticks.  A step is one tick for all 64
sessions; the metric is session-frames/s.  Also reported: p50/p99 tick latency against
the 80 ms budget, the tick's HBM roofline fraction, a B=1 latency line, the dominant
kernel's roofline (timed live through event nodes inside the step graph), the same
metric end to end through host buffers, and the CPU oracle on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Multi-GPU: replicas only (the tick has no cross-session exchange); each rank runs the
same workload on its own GPU, value = all ranks' session-frames / max wall time.
"""
import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "session-frames/s at B=1..64; p50 tick latency vs 80 ms; % HBM roofline"
UNIT = "session-frames/s"
SEED = 5
HBM_NOMINAL_GBS = 8000.0

# DRAM traffic of the attention kernel from one ncu capture (the --set full capture of one
# launch at B=32 with a full 3000-position ring, two temporal layers): dram__bytes_read +
# dram__bytes_write of that launch per (slot, valid position).  Traffic grows in
# proportion to the slots, so a full launch's traffic is this times slots x positions.
# Valid only while k_attn_tc.cu is the source that was captured (its hash below).
ATTN_TRAFFIC = {"bytes_per_slot_position": (1574.919e6 + 5.621248e6) / (32 * 3000),
                "source_sha256_16": "dac474ff910b713b"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--batch", type=int, default=64)
    ap.add_argument("--pos", type=int, default=3000, help="slot position at start (3000 = full ring)")
    ap.add_argument("--profile-steps", type=int, default=10)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--b1-steps", type=int, default=100)
    ap.add_argument("--cpu-ticks", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--shape", default="full", choices=["tiny", "small", "full"])
    ap.add_argument("--engine-flags", type=int, default=0, help="pp_config.flags (PP_FLAG_*)")
    ap.add_argument("--rvq-iters", type=int, default=50,
                    help="timed calls of the Mimi RVQ dequantisation (0 = skip that line)")
    ap.add_argument("--skip-user-steps-steps", type=int, default=50,
                    help="ticks of the secondary measurement with PP_FLAG_SKIP_USER_STEPS "
                         "(0 = skip it)")
    ap.add_argument("--sampling-steps", type=int, default=50,
                    help="ticks of the secondary measurement with every slot sampled "
                         "(0 = skip it)")
    ap.add_argument("--latency-ticks", type=int, default=500,
                    help="ticks of the fixed latency sample (after 20 warm-up ticks) that "
                         "p50/p99 tick latency are taken over (0 = skip)")
    ap.add_argument("--staggered-ticks", type=int, default=3750,
                    help="ticks per session of the staggered B=8 workload (slot i opens at "
                         "tick 400*i; 3750 = 5 minutes of audio, every ring wraps; 0 = skip)")
    ap.add_argument("--layers", type=int, default=0,
                    help="temporal layers (0 = the shape's own); fewer layers give a small "
                         "case with full-size kernels for profiling")
    return ap.parse_args()


# ---- helpers ---------------------------------------------------------------------------

def weight_bytes_streamed(s):
    """Bytes of weights one tick streams once: temporal layers, text head, per-codebook
    depformer in-projections and heads, and the shared depformer layers once."""
    d, F, dd, Fd = s.d, s.ffn, s.dep_d, s.dep_ffn
    layer = 3 * d * d + d * d + 2 * F * d + d * F
    dep_layer = 3 * dd * dd + dd * dd + 2 * Fd * dd + dd * Fd
    params = (s.n_layers * layer + s.text_vocab * d + s.n_q * dd * d + s.dep_layers * dep_layer
              + s.n_q * s.audio_card * dd)
    return 2 * params


def kv_bytes_per_position(s):
    """Ring bytes per (slot, position) over all layers, K and V, bf16."""
    return s.n_layers * 2 * s.d * 2


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu):
        self.gpu = gpu
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "200"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(ws, v):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(ws, v):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---- CPU oracle baseline -----------------------------------------------------------------

def cpu_oracle_sample(shape, pos, ticks):
    """Time the CPU oracle on one session of the bench workload (a full ring at `pos`):
    returns (session-frames/s, seconds, cores, sample description)."""
    import oracle
    import synth
    w = synth.make_weights_host(shape, SEED)
    L = shape.n_layers
    rk = np.stack([synth.ring_kv_host(shape, SEED, 0, l, 0) for l in range(L)])
    rv = np.stack([synth.ring_kv_host(shape, SEED, 0, l, 1) for l in range(L)])
    orc = oracle.Oracle(shape, w)
    sess = orc.new_session(pos=pos, ring_k=rk, ring_v=rv)
    col = oracle.initial_column(shape)
    user = synth.uniform_i32(ticks * 8, SEED, 300, 0, shape.audio_card).reshape(ticks, 8)
    t0 = time.perf_counter()
    for t in range(ticks):
        col, _, _ = orc.step(sess, col, user[t], want_logits=False)
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    sample = ("%d tick(s) of one session of the bench workload (%s shape, ring full at "
              "position %d), fp64 oracle, OpenMP over matrix rows" % (ticks, "full" if shape.d == 4096 else "reduced", pos))
    return ticks / dt, dt, cores, sample


def run_reference(a):
    ws, rank, _ = dist_setup()
    if rank != 0:
        return
    import synth
    shape = synth.PRESETS[a.shape]
    pos = min(a.pos, 2 ** 31 - 2)
    # each step: one session-tick of the B=64 workload on the CPU oracle
    import oracle
    w = synth.make_weights_host(shape, SEED)
    L = shape.n_layers
    rk = np.stack([synth.ring_kv_host(shape, SEED, 0, l, 0) for l in range(L)])
    rv = np.stack([synth.ring_kv_host(shape, SEED, 0, l, 1) for l in range(L)])
    orc = oracle.Oracle(shape, w)
    sess = orc.new_session(pos=pos, ring_k=rk, ring_v=rv)
    col = oracle.initial_column(shape)
    n = a.warmup + a.steps
    user = synth.uniform_i32(n * 8, SEED, 300, 0, shape.audio_card).reshape(n, 8)
    for t in range(a.warmup):
        col, _, _ = orc.step(sess, col, user[t], want_logits=False)
    t0 = time.perf_counter()
    for t in range(a.warmup, n):
        col, _, _ = orc.step(sess, col, user[t], want_logits=False)
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    v = a.steps / dt
    sample = "one session-tick of the B=%d full-ring workload per step" % a.batch
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": a.gpus,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1000 * dt / a.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded random-init weights and ring KV)",
            "config": {"workload": "full PersonaPlex shape, ring full at position %d, CPU oracle" % pos,
                       "global_batch": 1, "seq_len": shape.window, "parallelism": "replicas"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---- GPU arm -----------------------------------------------------------------------------

def fill_rings(eng, shape, B, pos):
    import torch
    import synth
    stream = torch.cuda.current_stream().cuda_stream
    for slot in range(B):
        for l in range(shape.n_layers):
            for kv in range(2):
                synth.ring_kv_fill_device(eng.ring_block(l, slot, kv), shape, SEED, slot, l, kv,
                                          stream)
        eng.import_session(slot, pos)
    torch.cuda.synchronize()


def time_ticks(eng, B, shape, steps, warmup, seed_stream):
    """Run warmup + steps ticks feeding each tick's column back; returns (total ms,
    per-tick ms list)."""
    import torch
    import synth
    n = warmup + steps
    user = torch.from_numpy(synth.uniform_i32(n * B * 8, SEED, seed_stream, 0, shape.audio_card)
                            .reshape(n, B, 8)).cuda()
    init = torch.tensor([shape.text_vocab] + [shape.audio_card] * shape.n_q, dtype=torch.int32)
    prev = init.repeat(B, 1).cuda()
    cols = [torch.empty((B, 17), dtype=torch.int32, device="cuda") for _ in range(2)]
    for t in range(warmup):
        prev = eng.step(prev, user[t], out=cols[t % 2])
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    evs[0].record()
    for t in range(steps):
        prev = eng.step(prev, user[warmup + t], out=cols[(warmup + t) % 2])
        evs[t + 1].record()
    torch.cuda.synchronize()
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
    return evs[0].elapsed_time(evs[-1]), per


def staggered_line(pp, shape, w_dev, flags, ticks, B=8, stride=400):
    """The staggered B=8 workload at full length: slot i opens at tick stride*i and runs
    `ticks` ticks of greedy decoding on run/silence user codes, then closes; every tick
    of the whole schedule is timed with CUDA events on its stream.  Returns the
    session-frames/s over the schedule and the tick latency percentiles."""
    import torch
    from synth import schedules
    sessions = schedules.staggered_sessions(shape, 3, n_slots=B, stride=stride, T=ticks)
    horizon = stride * (B - 1) + ticks
    user = np.zeros((horizon, B, 8), np.int32)
    for slot, start, u, _, _ in sessions:
        user[start:start + ticks, slot] = u
    d_user = torch.from_numpy(user).cuda()
    eng = pp.Engine(shape, B, w_dev, flags=flags)
    init = torch.tensor([shape.text_vocab] + [shape.audio_card] * shape.n_q, dtype=torch.int32)
    prev = init.repeat(B, 1).cuda()
    cols = [torch.empty((B, 17), dtype=torch.int32, device="cuda") for _ in range(2)]
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(horizon + 1)]
    live_ticks = 0
    torch.cuda.synchronize()
    evs[0].record()
    for t in range(horizon):
        for slot, start, _, _, _ in sessions:
            if start + ticks == t:
                eng.close(slot)
            if start == t:
                eng.open(slot)
                prev[slot] = init.cuda()   # a fresh session's first column
        live_ticks += sum(1 for _, start, _, _, _ in sessions if start <= t < start + ticks)
        prev = eng.step(prev, d_user[t], out=cols[t % 2])
        evs[t + 1].record()
    torch.cuda.synchronize()
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(horizon)]
    total = evs[0].elapsed_time(evs[-1])
    status = eng.status()
    eng.close_engine()
    return {"value": live_ticks / (total / 1000.0), "unit": "session-frames/s",
            "ticks": horizon, "session_ticks": live_ticks, "ms_total": total,
            "p50_tick_ms": float(np.percentile(per, 50)),
            "p99_tick_ms": float(np.percentile(per, 99)),
            "max_tick_ms": float(np.max(per)), "status_bits": status,
            "note": "B=8, slot i opens at tick %d*i and runs %d ticks (every ring wraps past "
                    "%d), greedy, run/silence user codes; includes the host's open/close "
                    "calls between ticks" % (stride, ticks, shape.window)}


def rvq_line(pp, B, iters):
    """pp_rvq_dequantize timed with CUDA events: once on a [B][17] tick column (the
    per-tick use: 8 codebooks of 2048 x 512 fp32) and once on a 65536-frame batch.  The
    32 MB of codebooks stay in L2, so the batch figure is an L2-bound throughput."""
    import torch
    import synth
    n_books, card, dim = 8, 2048, 512
    cb = torch.from_numpy(synth.normal_f32(n_books * card * dim, SEED, 31, 1.0)).cuda()
    res = {}
    for name, n in (("tick_column", B), ("batch_65536", 65536)):
        stride = 17 if name == "tick_column" else n_books
        codes = torch.from_numpy(synth.uniform_i32(n * stride, SEED, 32, 0, card)).cuda()
        ptr = codes.data_ptr() + (4 if stride == 17 else 0)
        out = torch.empty((n, dim), dtype=torch.float32, device="cuda")
        s = torch.cuda.current_stream()
        call = lambda: pp.pp_rvq_dequantize(ptr, stride, n, n_books, cb.data_ptr(), card, dim,
                                            out.data_ptr(), None, s.cuda_stream)
        for _ in range(3):
            call()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        for _ in range(iters):
            call()
        e1.record(s)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / iters
        nbytes = n * (n_books * dim * 4 + dim * 4 + n_books * 4)   # entries read + latent + codes
        res[name] = {"frames": n, "us_per_call": ms * 1e3, "frames_per_s": n / (ms / 1e3),
                     "GBps": nbytes / (ms / 1e3) / 1e9}
    res["note"] = ("8 codebooks x 2048 x 512 fp32 (32 MB, L2-resident); bytes = selected "
                   "entries read + latent written + codes")
    return res


def main():
    a = parse()
    if a.impl == "reference":
        return run_reference(a)
    import torch
    ws, rank, local = dist_setup()
    torch.cuda.set_device(local)
    import full_duplex_speech_lockstep_gb300 as pp
    import synth
    shape = synth.PRESETS[a.shape]
    if a.layers:
        import dataclasses
        shape = dataclasses.replace(shape, n_layers=a.layers)
    B = a.batch
    pos = a.pos
    props = torch.cuda.get_device_properties(local)

    w_dev = synth.make_weights_device(shape, SEED)
    eng = pp.Engine(shape, B, w_dev, flags=a.engine_flags)
    fill_rings(eng, shape, B, pos)
    kernels_per_tick = eng.kernel_count()

    # -- timed region: K ticks through the captured graph --------------------------------
    clocks = ClockSampler(local)
    barrier(ws)
    torch.cuda.synchronize()
    clocks.start()
    total_ms, per = time_ticks(eng, B, shape, a.steps, a.warmup, 400 + rank)
    clk = clocks.stop()
    barrier(ws)
    total_ms = max_over_ranks(ws, total_ms)
    frames = sum_over_ranks(ws, B * a.steps)
    value = frames / (total_ms / 1000.0)
    ms_per_step = total_ms / a.steps
    p50 = float(np.percentile(per, 50))
    p99 = float(np.percentile(per, 99))

    n_valid = min(pos + a.warmup + a.steps, shape.window)  # steady state once the ring is full
    wbytes = weight_bytes_streamed(shape)
    kv_read = B * n_valid * kv_bytes_per_position(shape)
    tick_bytes = wbytes + kv_read + B * kv_bytes_per_position(shape)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    tick_gbs = tick_bytes / (ms_per_step / 1000.0) / 1e9

    # -- tick latency over a fixed sample: 20 warm-up ticks, then `latency_ticks` ----------
    latency = None
    if a.latency_ticks > 0:
        _, perl = time_ticks(eng, B, shape, a.latency_ticks, 20, 450 + rank)
        latency = {"ticks": a.latency_ticks, "warmup": 20,
                   "p50_ms": float(np.percentile(perl, 50)),
                   "p99_ms": float(np.percentile(perl, 99)),
                   "max_ms": float(np.max(perl)), "budget_ms": 80.0}

    # -- per-kernel profile through the event-instrumented graph --------------------------
    kind_ms = (ctypes.c_double * len(pp.KERNEL_KINDS))()
    kind_n = (ctypes.c_int64 * len(pp.KERNEL_KINDS))()
    init = torch.tensor([shape.text_vocab] + [shape.audio_card] * shape.n_q, dtype=torch.int32)
    prev = init.repeat(B, 1).cuda()
    user = torch.from_numpy(synth.uniform_i32(a.profile_steps * B * 8, SEED, 500, 0,
                                              shape.audio_card).reshape(-1, B, 8)).cuda()
    cols = [torch.empty((B, 17), dtype=torch.int32, device="cuda") for _ in range(2)]
    for t in range(a.profile_steps):
        prev = eng.profile_step(prev, user[t], kind_ms, kind_n, out=cols[t % 2])
    prof = {k: {"ms_total": kind_ms[i], "launches": int(kind_n[i]),
                "ms_per_launch": (kind_ms[i] / kind_n[i]) if kind_n[i] else 0.0}
            for i, k in enumerate(pp.KERNEL_KINDS)}
    ia = pp.KERNEL_KINDS.index("attn")
    attn_ms = kind_ms[ia] / kind_n[ia] if kind_n[ia] else float("nan")
    # algorithmic bytes of one attention launch (one layer): K and V of every valid
    # ring position of every head, plus q in and o out (fp32)
    n_prof = min(pos + a.warmup + a.steps + a.profile_steps, shape.window)
    attn_bytes = B * n_prof * 2 * shape.d * 2 + 2 * B * shape.d * 4
    attn_gbs = attn_bytes / (attn_ms / 1000.0) / 1e9 if kind_n[ia] else None
    traffic = None
    import hashlib
    src = os.path.join(ROOT, "full_duplex_speech_lockstep_gb300", "csrc", "k_attn_tc.cu")
    if hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] == ATTN_TRAFFIC["source_sha256_16"]:
        traffic = ATTN_TRAFFIC["bytes_per_slot_position"] * B * n_prof
    roofline = {"kernel": "k_attn_tc (tensor-core split-K ring attention)", "bound": "hbm",
                "achieved": attn_gbs, "peak": hbm_peak, "unit": "GB/s",
                "frac": attn_gbs / hbm_peak if attn_gbs else None, "traffic": traffic,
                "peak_source": peak_src, "bytes_per_launch": attn_bytes,
                "ms_per_launch": attn_ms}

    # -- end to end through host buffers (pp_step_host) -----------------------------------
    h2d = B * 17 * 4 + B * 8 * 4
    d2h = B * 17 * 4
    e2e_val = None
    if a.e2e_steps > 0:
        prev_h = torch.empty((B, 17), dtype=torch.int32).pin_memory()
        prev_h.copy_(init.repeat(B, 1))
        user_h = torch.from_numpy(synth.uniform_i32(a.e2e_steps * B * 8, SEED, 600, 0,
                                                    shape.audio_card).reshape(-1, B, 8)).pin_memory()
        col_h = torch.empty((B, 17), dtype=torch.int32).pin_memory()
        eng.step_host(prev_h, user_h[0], None, None, col_h)   # warm
        barrier(ws)
        t0 = time.perf_counter()
        for t in range(a.e2e_steps):
            eng.step_host(prev_h, user_h[t], None, None, col_h)
            prev_h.copy_(col_h)
        dt = time.perf_counter() - t0
        dt = max_over_ranks(ws, dt)
        e2e_val = sum_over_ranks(ws, B * a.e2e_steps) / dt
    # -- the same engine with every slot sampled (the pages' generation parameters) --------
    samp = None
    if a.sampling_steps > 0:
        params = dict(text_temperature=0.7, text_top_p=0.9, repetition_penalty=1.2,
                      penalty_window=64, audio_temperature=0.3)
        for slot in range(B):
            eng.set_sampling(slot, seed=1000 + slot, **params)
        ms3, per3 = time_ticks(eng, B, shape, a.sampling_steps, max(3, a.warmup // 4), 900)
        ms3 = max_over_ranks(ws, ms3)
        samp = {"value": sum_over_ranks(ws, B * a.sampling_steps) / (ms3 / 1000.0),
                "unit": UNIT, "ms_per_step": ms3 / a.sampling_steps,
                "p50_tick_ms": float(np.percentile(per3, 50)), "params": params,
                "note": "every slot sampled: text temperature + nucleus + repetition penalty, "
                        "audio temperature"}
        for slot in range(B):
            eng.set_sampling(slot)
    status = eng.status()
    eng.close_engine()
    del eng
    torch.cuda.empty_cache()

    # -- the same workload with depformer steps 8..15 elided (user rows, same columns) -----
    skip = None
    if a.skip_user_steps_steps > 0:
        e2 = pp.Engine(shape, B, w_dev, flags=a.engine_flags | pp.PP_FLAG_SKIP_USER_STEPS)
        fill_rings(e2, shape, B, pos)
        ms2, per2 = time_ticks(e2, B, shape, a.skip_user_steps_steps, max(3, a.warmup // 4), 800)
        ms2 = max_over_ranks(ws, ms2)
        skip = {"value": sum_over_ranks(ws, B * a.skip_user_steps_steps) / (ms2 / 1000.0),
                "unit": UNIT, "ms_per_step": ms2 / a.skip_user_steps_steps,
                "p50_tick_ms": float(np.percentile(per2, 50)),
                "note": "PP_FLAG_SKIP_USER_STEPS: identical columns; user-row logits not computed"}
        e2.close_engine()
        del e2
        torch.cuda.empty_cache()

    # -- Mimi RVQ dequantisation of the tick's agent codes (the first step after the tick) --
    rvq = None
    if a.rvq_iters > 0:
        rvq = rvq_line(pp, B, a.rvq_iters)

    # -- B=1 latency line (full shape, fresh session) ---------------------------------------
    b1 = None
    if a.b1_steps > 0:
        e1 = pp.Engine(shape, 1, w_dev, flags=a.engine_flags)
        e1.open(0)
        ms1, per1 = time_ticks(e1, 1, shape, a.b1_steps, max(3, a.warmup), 700)
        b1 = {"session_frames_s": a.b1_steps / (ms1 / 1000.0),
              "p50_ms": float(np.percentile(per1, 50)), "p99_ms": float(np.percentile(per1, 99)),
              "positions": [max(3, a.warmup), max(3, a.warmup) + a.b1_steps]}
        if a.profile_steps > 0:   # per-kind kernel times of the B=1 tick (event-instrumented)
            km = (ctypes.c_double * len(pp.KERNEL_KINDS))()
            kn = (ctypes.c_int64 * len(pp.KERNEL_KINDS))()
            p1 = init.repeat(1, 1).cuda()
            c1 = [torch.empty((1, 17), dtype=torch.int32, device="cuda") for _ in range(2)]
            u1 = torch.from_numpy(synth.uniform_i32(a.profile_steps * 8, SEED, 510, 0,
                                                    shape.audio_card).reshape(-1, 1, 8)).cuda()
            for t in range(a.profile_steps):
                p1 = e1.profile_step(p1, u1[t], km, kn, out=c1[t % 2])
            b1["kernels_profile_ms_per_tick"] = {
                k: km[i] / a.profile_steps for i, k in enumerate(pp.KERNEL_KINDS) if kn[i]}
        e1.close_engine()
        # the low-latency variant: all 16 depformer steps in one persistent kernel
        e1 = pp.Engine(shape, 1, w_dev, flags=a.engine_flags | pp.PP_FLAG_LOW_LATENCY)
        e1.open(0)
        ms1, per1 = time_ticks(e1, 1, shape, a.b1_steps, max(3, a.warmup), 700)
        b1["low_latency"] = {"session_frames_s": a.b1_steps / (ms1 / 1000.0),
                             "p50_ms": float(np.percentile(per1, 50)),
                             "p99_ms": float(np.percentile(per1, 99)),
                             "note": "PP_FLAG_LOW_LATENCY: the 16 depformer steps in one "
                                     "persistent kernel (CUDA cores, grid barriers)"}
        if a.profile_steps > 0:
            km = (ctypes.c_double * len(pp.KERNEL_KINDS))()
            kn = (ctypes.c_int64 * len(pp.KERNEL_KINDS))()
            p1 = init.repeat(1, 1).cuda()
            c1 = [torch.empty((1, 17), dtype=torch.int32, device="cuda") for _ in range(2)]
            u1 = torch.from_numpy(synth.uniform_i32(a.profile_steps * 8, SEED, 520, 0,
                                                    shape.audio_card).reshape(-1, 1, 8)).cuda()
            for t in range(a.profile_steps):
                p1 = e1.profile_step(p1, u1[t], km, kn, out=c1[t % 2])
            b1["low_latency"]["kernels_profile_ms_per_tick"] = {
                k: km[i] / a.profile_steps for i, k in enumerate(pp.KERNEL_KINDS) if kn[i]}
        e1.close_engine()
        if a.skip_user_steps_steps > 0:   # the low-B variant beside the literal 16 steps
            e1 = pp.Engine(shape, 1, w_dev, flags=a.engine_flags | pp.PP_FLAG_SKIP_USER_STEPS)
            e1.open(0)
            ms1, per1 = time_ticks(e1, 1, shape, a.b1_steps, max(3, a.warmup), 700)
            b1["skip_user_steps"] = {"session_frames_s": a.b1_steps / (ms1 / 1000.0),
                                     "p50_ms": float(np.percentile(per1, 50)),
                                     "p99_ms": float(np.percentile(per1, 99))}
            e1.close_engine()

    # -- the staggered B=8 workload at full length (every ring wraps) ----------------------
    staggered = None
    if a.staggered_ticks > 0 and a.shape == "full":
        staggered = staggered_line(pp, shape, w_dev, a.engine_flags, a.staggered_ticks)
        torch.cuda.empty_cache()

    # -- CPU oracle baseline (rank 0, N=1 only) -------------------------------------------
    cpu = None
    if rank == 0 and ws == 1 and not a.no_cpu_baseline:
        v, dt, cores, sample = cpu_oracle_sample(shape, min(pos, shape.window), a.cpu_ticks)
        cpu = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
               "seconds": dt}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded random-init weights N(0,0.02), ring KV N(0,1), uniform user codes)",
            "config": {"workload": "full PersonaPlex shape (4096-d/32L temporal, 1024-d/6L depformer), "
                                   "B=%d sessions, ring full at position %d of window %d, greedy"
                                   % (B, pos, shape.window) if a.shape == "full" else a.shape,
                       "global_batch": B * ws, "seq_len": shape.window,
                       "parallelism": "replicas x%d" % ws,
                       "l2": "inputs larger than L2 (%.0f GB ring + %.1f GB weights per GPU)"
                             % (B * shape.window * kv_bytes_per_position(shape) / 1e9, wbytes / 1e9)},
            "p50_tick_ms": p50, "p99_tick_ms": p99, "realtime_budget_ms": 80.0,
            "latency": latency,
            "tick_roofline": {"bytes_per_tick": tick_bytes, "achieved_gbs": tick_gbs,
                              "frac_of_8tbs": tick_gbs / HBM_NOMINAL_GBS,
                              "frac_of_measured": tick_gbs / hbm_peak},
            "roofline": roofline,
            "kernels_profile": prof,
            "b1": b1,
            "staggered_b8": staggered,
            "skip_user_steps": skip,
            "sampling": samp,
            "rvq": rvq,
            "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "cpu_baseline": cpu,
            "gpu_launches": kernels_per_tick * a.steps,
            "kernels_per_tick": kernels_per_tick,
            "clocks": clk,
            "status_bits": status,
            "device": props.name,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
