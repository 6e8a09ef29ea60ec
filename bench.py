#!/usr/bin/env python3
"""Benchmark: one step = one pass of the whole hot path over one synthetic batch.

Step (all on the GPU, through the C ABI):
  zigzag-shard q, k, v -> positions -> ring attention forward over C virtual
  ranks (C batched partial-attention launches + C-1 LSE merges, K/V rotation
  prefetched on a side stream) -> zigzag-unshard the output -> Ulysses
  sequence-to-head relayout of the q, k, v shards (global order).
Metric: algorithmic causal-attention TFLOP/s of the step (4*D FLOPs per visible
(query, key) pair), plus per-kernel TFLOP/s and GB/s from CUDA events recorded
on the launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload s32k]

Under torchrun (N > 1) every rank runs an independent replica (the C virtual
ranks of the method live on one GPU; nothing is exchanged between GPUs).
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal attn fwd TFLOP/s & % bf16 tensor peak; LSE-merge/relayout HBM GB/s"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def _code_only(text):
    """C/C++ source without comments and whitespace (string literals kept)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            i = text.find("\n", i)
            i = n if i < 0 else i
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            if not c.isspace():
                out.append(c)
            i += 1
    return "".join(out)


def attn_source_hash():
    """Hash of the attention kernel's code (comments and whitespace ignored), so
    a recorded traffic figure stays valid across comment edits only."""
    h = hashlib.sha256()
    for f in ("attn.cu", "cp_ptx.cuh", "cp_sched.cuh"):
        with open(os.path.join(ROOT, "context_causal_attention_gb300", "csrc", f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload, fused=False):
    """Per-launch DRAM bytes of the attention kernel (the ring's launches with the
    merge fused into the epilogue, or with the standalone merge) from the
    machine-readable record profiles/attn_traffic.json, if it was taken on the
    current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "attn_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    ent = rec.get("workloads", {}).get(workload, {}).get("fused_merge" if fused else "separate_merge")
    if not ent or ent.get("source") != attn_source_hash():
        return None
    return float(ent["bytes_per_launch"])


def tensor_peak(peaks, wall_s, clk):
    """The bf16 tensor peak a kernel timed in this run is held to: the burst
    figure (cuBLAS timed alone, at full clock) when the timed region is short
    and the SM clock stayed at its maximum; the sustained figure (cuBLAS back to
    back for seconds under the power cap) otherwise.  Returns (peak, which)."""
    sm, mx = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    at_max = sm is not None and mx and sm >= 0.97 * mx
    if wall_s < 5.0 and at_max:
        return peaks["bf16_tflops"], "bf16_tflops (burst)"
    return peaks["bf16_tflops_sustained"], "bf16_tflops_sustained"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons, sampled every 50 ms while running.

    Each sample carries nvidia-smi's own timestamp; `window(t0, t1)` (host
    wall-clock seconds) marks the timed region, and the summary keeps the
    samples taken inside it (all samples when none fell inside)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index, interval_ms=50):
        self.index = index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []
        self.t = None
        self.win = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", str(self.interval_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def window(self, t0, t1):
        self.win = (t0, t1)

    @staticmethod
    def parse(lines):
        """[(epoch seconds or None, sm MHz, max sm MHz, {reason: active})] from the csv lines."""
        out = []
        for ln in lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm, mx = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                if "." in parts[0]:
                    ts += float("0." + parts[0].split(".")[1])
            except (ValueError, OverflowError):
                ts = None
            act = {nm: val.lower().startswith("active") for nm, val in zip(ClockSampler.REASONS, parts[6:10])}
            out.append((ts, sm, mx, act))
        return out

    @staticmethod
    def summarise(samples, win):
        inside = [x for x in samples if win and x[0] is not None and win[0] <= x[0] <= win[1]]
        use = inside if inside else samples
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "samples_in_timed_region": 0}
        reasons = sorted({nm for x in use for nm, on in x[3].items() if on})
        return {"sm_mhz": statistics.median(x[1] for x in use), "sm_max_mhz": max(x[2] for x in use),
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside)}

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        return self.summarise(self.parse(self.lines), self.win)


def dist_setup(n_gpus):
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cuda"):
    """Largest value of x over all ranks (the slowest replica sets the job time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, ms_max):
    """Whole-job throughput: the units all ranks processed over the max-over-ranks time."""
    return units_per_rank * world / (ms_max * 1e-3)


# --------------------------------------------------------------------------
# CPU oracle timing (the reported baseline and the reference arm)
# --------------------------------------------------------------------------
def oracle_sample_run(w, q, k, v, rows, nthreads):
    """Time the fp64 oracle on the given query rows (all heads); returns
    (seconds, algorithmic flops of those rows)."""
    import numpy as np
    import oracle as O
    gp = np.arange(w.S, dtype=np.int32)
    t0 = time.perf_counter()
    O.attn_rows(q, k, v, gp, gp, rows, nthreads=nthreads)
    dt = time.perf_counter() - t0
    flops = 4.0 * w.B * w.N * w.D * float(np.sum(rows + 1))
    return dt, flops


def prepare_oracle_inputs(w, q, k, v):
    import numpy as np
    return tuple(t.float().numpy().astype(np.float64) for t in (q, k, v))


def cpu_rows(w, n, seed):
    import numpy as np
    rng = np.random.default_rng(seed)
    return np.sort(rng.integers(0, w.S, size=n)).astype(np.int64)


CPU_ROWS_PER_BATCH = 256  # query rows (x all heads) per oracle call, in the cpu_baseline and the reference arm


def cpu_baseline(w, qkv64, target_s=12.0):
    """The oracle on batches of CPU_ROWS_PER_BATCH random query rows (all heads),
    the same batch the reference arm times per step, until target_s of CPU time."""
    import oracle as O
    cores = O.default_threads()
    rows_total, secs, flops = 0, 0.0, 0.0
    seed = 100
    while secs < target_s and rows_total < 1 << 16:
        rows = cpu_rows(w, CPU_ROWS_PER_BATCH, seed)
        dt, fl = oracle_sample_run(w, *qkv64, rows, cores)
        secs += dt
        flops += fl
        rows_total += CPU_ROWS_PER_BATCH
        seed += 1
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "extrapolated_full_workload_s": w.flops / (flops / secs),
            "sample": "%d batches of %d random query rows x all %d heads of the %s workload (fp64 C oracle, "
                      "%d threads; the reference arm times the same batch per step), %.1f s"
                      % (rows_total // CPU_ROWS_PER_BATCH, CPU_ROWS_PER_BATCH, w.N, w.name, cores, secs)}


def run_reference(args, w):
    """The oracle, as it stands, timed on the host cores (rank 0 only)."""
    import cp_synth as SY
    import oracle as O
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    q, k, v, _ = SY.make_qkv(w)
    qkv64 = prepare_oracle_inputs(w, q, k, v)
    cores = O.default_threads()
    rows_per_step = CPU_ROWS_PER_BATCH
    for i in range(args.warmup):
        oracle_sample_run(w, *qkv64, cpu_rows(w, rows_per_step, 1000 + i), cores)
    secs, flops = 0.0, 0.0
    for i in range(args.steps):
        dt, fl = oracle_sample_run(w, *qkv64, cpu_rows(w, rows_per_step, 2000 + i), cores)
        secs += dt
        flops += fl
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": line_config(w, 1 if args.prefetch else 0, bool(args.fused_merge)),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": "%d random query rows x all %d heads per step of the %s workload (fp64 C "
                                   "oracle, %d threads; the same batch as the cpu_baseline of our arm)"
                                   % (rows_per_step, w.N, w.name, cores)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


L2_BYTES = 129e6
FLUSH_BYTES = 256 << 20


def input_bytes(w):
    return w.B * w.S * (w.N + 2 * w.Nkv) * w.D * 2


def needs_l2_flush(w):
    """q, k, v together within 1.5x of L2: flush L2 between timed steps."""
    return input_bytes(w) < 1.5 * L2_BYTES


def workload_config(w, prefetch, device_timing=True):
    cfg = {"workload": "%s: B=%d S=%d N=%d Nkv=%d D=%d, C=%d %s ring%s" % (
        w.name, w.B, w.S, w.N, w.Nkv, w.D, w.C, w.layout, ", RoPE" if w.rope else ""),
        "B": w.B, "S": w.S, "N": w.N, "Nkv": w.Nkv, "D": w.D, "C": w.C, "layout": w.layout}
    if device_timing:
        cfg["l2"] = ("L2 flushed between timed steps (%d MB write, outside each step's events); q, k, v %.1f MB in all"
                     % (FLUSH_BYTES >> 20, input_bytes(w) / 1e6) if needs_l2_flush(w)
                     else "inputs larger than L2 (q, k, v %.0f MB each)" % (w.B * w.S * w.N * w.D * 2 / 1e6))
    if prefetch is not None:
        cfg["prefetch"] = prefetch
    return cfg


def line_config(w, prefetch, fused):
    """The `config` of the JSON line, the same for both arms (the reference arm
    times the oracle on this workload; the GPU-side keys describe our arm's run)."""
    return dict(workload_config(w, prefetch),
                merge="fused into the attention epilogue (standalone merge kernel timed separately)"
                if fused else "standalone merge kernel per ring step")


def graph_replay_times(args, torch, F, step, inputs, flush_buf, parts):
    """Median time of >= 20 replays of one CUDA graph of `step(*inputs, None)` and
    of each permutation in `parts` (name -> (callable, algorithmic bytes)), each
    beside the same work launched eagerly; L2 flushed between runs when
    flush_buf is given (outside the events)."""
    reps = max(20, args.steps)

    def median_ms(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            if flush_buf is not None:
                flush_buf.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    def capture(fn):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g

    eager_step = lambda: step(*inputs, None)
    g = capture(eager_step)
    out = {"reps": reps, "statistic": "median", "step_ms_graph": median_ms(g.replay),
           "step_ms_eager": median_ms(eager_step)}
    for name, (fn, nbytes) in parts.items():
        gp = capture(fn)
        tg, te = median_ms(gp.replay), median_ms(fn)
        out[name + "_gbs_graph"] = nbytes / (tg * 1e-3) / 1e9
        out[name + "_gbs_eager"] = nbytes / (te * 1e-3) / 1e9
    return out


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------
class StepRig:
    """Resident device buffers and the step of one workload: zigzag-shard q, k,
    v -> positions -> ring forward -> unshard o -> Ulysses relayout of the
    shards.  Per-kernel CUDA events are recorded on the launching stream."""

    def __init__(self, w, dev, prefetch, fused, q, k, v):
        import torch
        from context_causal_attention_gb300 import ops as F
        self.F, self.torch, self.w = F, torch, w
        self.prefetch, self.fused = prefetch, fused
        C, S, B, N, Nkv, D = w.C, w.S, w.B, w.N, w.Nkv, w.D
        s = S // C
        self.lay = F.CP_ZIGZAG if w.layout == "zigzag" else F.CP_CONTIGUOUS
        self.qd, self.kd, self.vd = (t.to(dev) for t in (q, k, v))
        self.qs = torch.empty((C, B, s, N, D), dtype=torch.bfloat16, device=dev)
        self.ks = torch.empty((C, B, s, Nkv, D), dtype=torch.bfloat16, device=dev)
        self.vs = torch.empty_like(self.ks)
        self.pos = torch.empty((C, s), dtype=torch.int32, device=dev)
        self.o_sh = torch.empty((C, B, s, N, D), dtype=torch.float32, device=dev)
        self.lse_sh = torch.empty((C, B, N, s), dtype=torch.float32, device=dev)
        self.o_full = torch.empty((B, S, N, D), dtype=torch.float32, device=dev)
        self.ws = torch.empty(max(256, F.cp_ring_workspace_size(B, S, N, Nkv, D, C, prefetch, F.CP_F32, fused)),
                              dtype=torch.uint8, device=dev)
        self.qh = torch.empty((C, B, S, N // C, D), dtype=torch.bfloat16, device=dev)
        self.kh = torch.empty((C, B, S, Nkv // C, D), dtype=torch.bfloat16, device=dev)
        self.vh = torch.empty_like(self.kh)
        # long shards: each attention launch is preceded by the two plan kernels
        nt = -(-s // 128)
        plan = 0 if (C * 2 * nt <= 2048 and C * ((nt + 1) // 2) <= 1024) else 2
        self.launches_per_step = 3 + 1 + C * (1 + plan) + (0 if fused else C - 1) + 1 + 3

    def events(self):
        torch = self.torch

        def mk(n):
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
            for e in evs:
                e.record()
            return evs
        return {"ring": mk(4 * self.w.C), "shard": mk(2), "unshard": mk(2), "relayout": mk(2)}

    def step(self, qin, kin, vin, ev, o_out=None):
        """One pass of the hot path.  ev: dict of event lists or None.  qin, kin,
        vin may be pinned host tensors (the shard reads them across the host
        link); o_out (default: the device o_full) may be a pinned host tensor."""
        F, w, lay = self.F, self.w, self.lay
        C, S = w.C, w.S

        def mark(name, i):
            if ev is not None:
                ev[name][i].record()
        mark("shard", 0)
        F.cp_zigzag_shard(qin, C, lay, out=self.qs)
        F.cp_zigzag_shard(kin, C, lay, out=self.ks)
        F.cp_zigzag_shard(vin, C, lay, out=self.vs)
        mark("shard", 1)
        F.cp_zigzag_positions(S, C, lay, out=self.pos)
        F.cp_ring_attention_fwd(self.qs, self.ks, self.vs, self.pos, layout=lay, prefetch=self.prefetch,
                                o_dtype=F.CP_F32, workspace=self.ws, o=self.o_sh, lse=self.lse_sh,
                                events=ev["ring"] if ev is not None else None, fused_merge=self.fused)
        mark("unshard", 0)
        F.cp_zigzag_unshard(self.o_sh, lay, out=self.o_full if o_out is None else o_out)
        mark("unshard", 1)
        mark("relayout", 0)
        F.cp_ulysses_relayout(self.qs, C, F.CP_SEQ_TO_HEAD, F.CP_GLOBAL_ORDER, out=self.qh)
        F.cp_ulysses_relayout(self.ks, C, F.CP_SEQ_TO_HEAD, F.CP_GLOBAL_ORDER, out=self.kh)
        F.cp_ulysses_relayout(self.vs, C, F.CP_SEQ_TO_HEAD, F.CP_GLOBAL_ORDER, out=self.vh)
        mark("relayout", 1)


def ring_step_pairs(w):
    """Exact visible pairs per (b, h) of each ring step, all ranks together."""
    C, s, t = w.C, w.S // w.C, w.S // (2 * w.C)
    if w.layout == "zigzag":
        return [C * (t * t + t * (t + 1))] + [C * 2 * t * t] * (C - 1)
    return [C * s * (s + 1) // 2] + [(C - st) * s * s for st in range(1, C)]


def merge_bytes_per_step(w):
    """Algorithmic bytes of the merge of each ring step >= 1: rows whose tile
    lse is finite move 3*4*D + 12 bytes, the others 4."""
    C, B, N, D, s = w.C, w.B, w.N, w.D, w.S // w.C
    rows = C * B * N * s
    out = []
    for st in range(1, C):
        if w.layout == "zigzag":
            fr = sum(B * N * (s if (rr - st) % C < rr else s // 2) for rr in range(C))
        else:
            fr = B * N * s * (C - st)
        out.append(fr * (12 * D + 12) + (rows - fr) * 4)
    return out


def kernel_metrics(rig, evsets, peaks):
    """Per-kernel times and rates from the events of the timed steps."""
    w = rig.w
    C, B, N, Nkv, D, S = w.C, w.B, w.N, w.Nkv, w.D, w.S
    n = len(evsets)
    attn_ms, merge_ms = [0.0] * C, [0.0] * C
    shard_ms = unshard_ms = relayout_ms = 0.0
    for e in evsets:
        r = e["ring"]
        for st in range(C):
            attn_ms[st] += r[4 * st].elapsed_time(r[4 * st + 1]) / n
            if st > 0:
                merge_ms[st] += r[4 * st + 2].elapsed_time(r[4 * st + 3]) / n
        shard_ms += e["shard"][0].elapsed_time(e["shard"][1]) / n
        unshard_ms += e["unshard"][0].elapsed_time(e["unshard"][1]) / n
        relayout_ms += e["relayout"][0].elapsed_time(e["relayout"][1]) / n
    if rig.fused:
        # the step merges inside the attention epilogue; time the standalone merge
        # kernel on the same ring (separate-merge mode, traced) for its GB/s
        torch, F = rig.torch, rig.F
        ws2 = torch.empty(max(256, F.cp_ring_workspace_size(B, S, N, Nkv, D, C, rig.prefetch, F.CP_F32, False)),
                          dtype=torch.uint8, device=rig.qs.device)
        o2, l2 = torch.empty_like(rig.o_sh), torch.empty_like(rig.lse_sh)
        merge_ms = [0.0] * C
        reps = 2
        for rep_i in range(reps + 1):
            ev2 = rig.events()["ring"]
            F.cp_ring_attention_fwd(rig.qs, rig.ks, rig.vs, rig.pos, layout=rig.lay, prefetch=rig.prefetch,
                                    o_dtype=F.CP_F32, workspace=ws2, o=o2, lse=l2, events=ev2, fused_merge=False)
            torch.cuda.synchronize()
            if rep_i == 0:
                continue  # warm-up
            for st in range(1, C):
                merge_ms[st] += ev2[4 * st + 2].elapsed_time(ev2[4 * st + 3]) / reps
        del ws2, o2, l2
    attn_flops = [4.0 * B * N * D * p for p in ring_step_pairs(w)]
    attn_tflops = sum(attn_flops) / (sum(attn_ms) * 1e-3) / 1e12
    per_step_tflops = [f / (t * 1e-3) / 1e12 for f, t in zip(attn_flops, attn_ms)]
    mb = merge_bytes_per_step(w)
    merge_gbs = sum(mb) / (sum(merge_ms) * 1e-3) / 1e9 if C > 1 else None
    merge_gbs_steps = [b / (t * 1e-3) / 1e9 for b, t in zip(mb, merge_ms[1:])]
    qkv_bytes = (B * S * N * D + 2 * B * S * Nkv * D) * 2
    hbm = peaks["hbm_gbs"]
    shard_gbs = 2 * qkv_bytes / (shard_ms * 1e-3) / 1e9
    relayout_gbs = 2 * qkv_bytes / (relayout_ms * 1e-3) / 1e9
    return {
        "attn_ms_per_ring_step": attn_ms, "attn_tflops_per_ring_step": per_step_tflops, "attn_tflops": attn_tflops,
        "merge_ms_per_ring_step": merge_ms[1:], "merge_gbs": merge_gbs, "merge_gbs_per_ring_step": merge_gbs_steps,
        "merge_frac_hbm_per_ring_step": [x / hbm for x in merge_gbs_steps],
        "merge_measured_in": "separate-merge ring calls after the timed region" if rig.fused else "the timed step",
        "shard_gbs": shard_gbs, "unshard_gbs": 2 * (B * S * N * D * 4) / (unshard_ms * 1e-3) / 1e9,
        "relayout_gbs": relayout_gbs, "hbm_peak_gbs": hbm,
        "merge_frac_hbm": (merge_gbs / hbm) if merge_gbs else None,
        "shard_frac_hbm": shard_gbs / hbm, "relayout_frac_hbm": relayout_gbs / hbm,
    }


def time_device_steps(rig, steps, warmup, world=1, clocks=None):
    """W untimed steps, then K timed steps bracketed by a barrier and a
    synchronize on both sides, per-kernel events inside.  Workloads within
    1.5x of L2 get an L2 flush between steps, outside each step's events.
    Returns (ms per step, max over ranks), the event sets and the wall time."""
    torch = rig.torch
    w = rig.w
    for _ in range(warmup):
        rig.step(rig.qd, rig.kd, rig.vd, None)
    torch.cuda.synchronize()
    evsets = [rig.events() for _ in range(steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush = needs_l2_flush(w)
    flush_buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=rig.qs.device) if flush else None
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    if clocks is not None:
        clocks.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    t_start.record()
    for i in range(steps):
        if flush:
            flush_buf.zero_()  # evicts the previous step's data from L2 (outside the step's events)
        step_ev[i][0].record()
        rig.step(rig.qd, rig.kd, rig.vd, evsets[i])
        step_ev[i][1].record()
    t_end.record()
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    if clocks is not None:
        now = time.time()
        # nvidia-smi stamps whole milliseconds; widen the window by one interval
        clocks.window(now - wall - 0.05, now + 0.05)
    ms_total = (sum(a.elapsed_time(b) for a, b in step_ev) if flush else t_start.elapsed_time(t_end))
    return max_over_ranks(ms_total, world) / steps, evsets, wall, flush_buf


def secondary_step_line(w, dev, steps, warmup, peaks, prefetch, fused, graph=False):
    """The device step (same rig, same timing rules) on another workload, for
    the secondary keys of the default line; with `graph`, also the median of
    >= 20 CUDA-graph replays of the whole step beside the same step launched
    eagerly (L2 flushed between runs when the workload needs it)."""
    import types
    import cp_synth as SY
    q, k, v, _ = SY.make_qkv(w)
    rig = StepRig(w, dev, prefetch, fused, q, k, v)
    del q, k, v
    ms, evsets, wall, flush_buf = time_device_steps(rig, steps, warmup)
    km = kernel_metrics(rig, evsets, peaks)
    out = {"workload": workload_config(w, prefetch)["workload"], "l2": workload_config(w, prefetch)["l2"],
           "ms_per_step": ms, "value": w.flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
           "attn_tflops": km["attn_tflops"], "attn_tflops_per_ring_step": km["attn_tflops_per_ring_step"],
           "attn_frac_of_burst_bf16": km["attn_tflops"] / peaks["bf16_tflops"],
           "merge_gbs": km["merge_gbs"], "merge_frac_hbm": km["merge_frac_hbm"],
           "merge_gbs_per_ring_step": km["merge_gbs_per_ring_step"],
           "merge_frac_hbm_per_ring_step": km["merge_frac_hbm_per_ring_step"],
           "merge_measured_in": km["merge_measured_in"],
           "shard_gbs": km["shard_gbs"], "unshard_gbs": km["unshard_gbs"], "relayout_gbs": km["relayout_gbs"],
           "relayout_frac_hbm": km["relayout_frac_hbm"], "shard_frac_hbm": km["shard_frac_hbm"],
           "steps": steps, "warmup": warmup, "wall_s_timed": wall}
    if graph:
        g = graph_replay_times(types.SimpleNamespace(steps=steps), rig.torch, rig.F, rig.step,
                               (rig.qd, rig.kd, rig.vd), flush_buf, {})
        g["step_value_graph_tflops"] = w.flops / (g["step_ms_graph"] * 1e-3) / 1e12
        g["step_value_eager_tflops"] = w.flops / (g["step_ms_eager"] * 1e-3) / 1e12
        out["graph"] = g
    del rig
    return out


def run_secondary(args, dev, peaks, prefetch, fused):
    """Secondary keys of the default line: the S=4096 and S=131072 workloads'
    device steps (step TFLOP/s, relayout and per-step merge GB/s with their
    fraction of HBM; S=4096 also as CUDA-graph replays), and the S=65536 sweep point for C in {2, 4, 8},
    contiguous against zigzag (per-rank issued key tiles and per-rank time,
    max / mean over ranks)."""
    import cp_synth as SY
    torch = __import__("torch")
    out = {}
    for name in ("s4k", "s128k"):
        # the small workload also as CUDA-graph replays (its launches are short)
        out[name] = secondary_step_line(SY.WORKLOADS[name], dev, args.steps, args.warmup, peaks, prefetch, fused,
                                        graph=(name == "s4k"))
        torch.cuda.empty_cache()
    sw = []
    for w in SY.sweep_workloads():
        if w.S != 65536:
            continue
        m = sweep_measure(w, dev, reps=3, device_inputs=True)
        sw.append({k: m[k] for k in ("S", "C", "layout", "ring_ms", "ring_tflops", "pairs_max_over_mean",
                                     "issued_tiles_max_over_mean", "rank_ms_max_over_mean")})
        torch.cuda.empty_cache()
    out["sweep_S65536"] = {"what": "B=1 N=16 D=128 ring with prefetch; per-rank figures are max / mean over the C "
                                   "virtual ranks (rank time: each rank's C partials launched on their own)",
                           "runs": sw}
    return out


def run_ours(args, w):
    import numpy as np
    import torch

    import cp_synth as SY
    from context_causal_attention_gb300 import build as cuda_build
    from context_causal_attention_gb300 import ops as F

    rank, world, local = dist_setup(args.gpus)
    cuda_build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    q, k, v, _ = SY.make_qkv(w)
    C, S, B, N, Nkv, D = w.C, w.S, w.B, w.N, w.Nkv, w.D
    s = S // C
    lay = F.CP_ZIGZAG if w.layout == "zigzag" else F.CP_CONTIGUOUS
    prefetch = 1 if args.prefetch else 0
    fused = bool(args.fused_merge)
    rig = StepRig(w, dev, prefetch, fused, q, k, v)
    qd, kd, vd = rig.qd, rig.kd, rig.vd
    qs, o_sh, lse_sh, o_full, qh = rig.qs, rig.o_sh, rig.lse_sh, rig.o_full, rig.qh
    step = rig.step
    launches_per_step = rig.launches_per_step

    # ---- timed region (device time), per-kernel events inside
    clocks = ClockSampler(local)
    ms_step, evsets, wall, flush_buf = time_device_steps(rig, args.steps, args.warmup, world, clocks)
    clk = clocks.stop()
    flops_step = w.flops
    value = job_throughput(flops_step, world, ms_step) / 1e12

    # ---- per-kernel numbers from the events
    km = kernel_metrics(rig, evsets, peaks)
    attn_ms, attn_tflops, per_step_tflops = km["attn_ms_per_ring_step"], km["attn_tflops"], \
        km["attn_tflops_per_ring_step"]
    merge_gbs = km["merge_gbs"]
    qkv_bytes = (B * S * N * D + 2 * B * S * Nkv * D) * 2
    peak_tc, peak_name = tensor_peak(peaks, wall, clk)
    traffic = recorded_traffic(w.name, fused)

    # ---- end to end through the public API from pinned host memory.  The
    # shard kernels read q, k, v across the host link and the unshard writes o
    # into host memory (copy and permutation in one pass each); lse comes back
    # with one copy.  The same step with copy-engine transfers around the
    # device step is timed beside it.
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    ho = torch.empty((B, S, N, D), dtype=torch.float32).pin_memory()
    hl = torch.empty((C, B, N, s), dtype=torch.float32).pin_memory()

    def e2e_direct():
        step(hq, hk, hv, None, o_out=ho)
        hl.copy_(lse_sh, non_blocking=True)

    def e2e_copies():
        qd.copy_(hq, non_blocking=True)
        kd.copy_(hk, non_blocking=True)
        vd.copy_(hv, non_blocking=True)
        step(qd, kd, vd, None)
        ho.copy_(o_full, non_blocking=True)
        hl.copy_(lse_sh, non_blocking=True)

    def time_e2e(fn):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(e0.elapsed_time(e1), world) / args.steps

    # pipelined: step i+1's inputs are copied in (copy engine, own stream) and
    # step i-1's output copied out (own stream) while step i computes; inputs
    # and output double-buffered, ordered by events.  Every step still moves
    # all of its inputs and its result across the host link, and the timed
    # region includes the pipeline's fill and drain.
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    inbuf = [(qd, kd, vd), tuple(torch.empty_like(t) for t in (qd, kd, vd))]
    obuf = [o_full, torch.empty_like(o_full)]

    def e2e_pipelined(nsteps):
        ev_in = [torch.cuda.Event(), torch.cuda.Event()]
        ev_step = [torch.cuda.Event(), torch.cuda.Event()]
        ev_out = [torch.cuda.Event(), torch.cuda.Event()]

        def copy_in(b, after):
            with torch.cuda.stream(s_in):
                if after is not None:
                    s_in.wait_event(after)  # the buffer's previous step has read it
                for t, h in zip(inbuf[b], (hq, hk, hv)):
                    t.copy_(h, non_blocking=True)
                ev_in[b].record(s_in)

        copy_in(0, None)
        for i in range(nsteps):
            b = i & 1
            if i + 1 < nsteps:
                copy_in(b ^ 1, ev_step[b ^ 1] if i >= 1 else None)
            comp.wait_event(ev_in[b])
            if i >= 2:
                comp.wait_event(ev_out[b])  # the output buffer's previous copy-out is done
            step(*inbuf[b], None, o_out=obuf[b])
            hl.copy_(lse_sh, non_blocking=True)
            ev_step[b].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_step[b])
                ho.copy_(obuf[b], non_blocking=True)
                ev_out[b].record(s_out)
        comp.wait_stream(s_out)
        comp.wait_stream(s_in)

    def time_pipelined(reps):
        # the host link's speed varies from run to run, so
        # the pipelined figure is the median of `reps` timed runs of K steps
        e2e_pipelined(2)
        torch.cuda.synchronize()
        runs = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier(world)
            e0.record()
            e2e_pipelined(args.steps)
            e1.record()
            torch.cuda.synchronize()
            barrier(world)
            runs.append(max_over_ranks(e0.elapsed_time(e1), world) / args.steps)
        return runs

    e2e_direct_ms = time_e2e(e2e_direct)
    e2e_copy_ms = time_e2e(e2e_copies)
    e2e_runs = time_pipelined(3)
    e2e_ms = statistics.median(e2e_runs)
    h2d = qkv_bytes
    d2h = B * S * N * D * 4 + C * B * N * s * 4

    # ---- CUDA-graph replay: the whole step and each permutation alone, each
    # beside the same work launched eagerly (median of the replays)
    graph_info = None
    if args.graph:
        graph_info = graph_replay_times(args, torch, F, step, (qd, kd, vd), flush_buf, dict(
            shard=(lambda: F.cp_zigzag_shard(qd, C, lay, out=qs), 2 * B * S * N * D * 2),
            unshard=(lambda: F.cp_zigzag_unshard(o_sh, lay, out=o_full), 2 * B * S * N * D * 4),
            relayout=(lambda: F.cp_ulysses_relayout(qs, C, F.CP_SEQ_TO_HEAD, F.CP_GLOBAL_ORDER, out=qh),
                      2 * B * S * N * D * 2)))
        graph_info["step_value_graph_tflops"] = flops_step / (graph_info["step_ms_graph"] * 1e-3) / 1e12
        graph_info["step_value_eager_tflops"] = flops_step / (graph_info["step_ms_eager"] * 1e-3) / 1e12

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": line_config(w, prefetch, fused),
        "roofline": {"bound": "tensor", "achieved": attn_tflops, "peak": peak_tc, "unit": "TFLOP/s",
                     "frac": attn_tflops / peak_tc, "traffic": traffic,
                     "kernel": "attn_fwd_kernel<%d>" % D + (" (ring steps >= 1 also merge into the accumulator in "
                                                            "the epilogue)" if fused else ""),
                     "peak_note": "%s of %s peaks (timed region %.2f s, median SM clock %s of %s MHz); frac of "
                                  "sustained %.1f: %.3f" % (peak_name, peaks["source"], wall, clk.get("sm_mhz"),
                                                             clk.get("sm_max_mhz"), peaks["bf16_tflops_sustained"],
                                                             attn_tflops / peaks["bf16_tflops_sustained"])},
        "e2e": {"value": flops_step * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "runs_ms_per_step": e2e_runs,
                "how": "%d steps pipelined: each step's q, k, v copied in from pinned host memory and its o, lse "
                       "copied out, on their own streams while the neighbouring steps compute (double-buffered, "
                       "event-ordered; fill and drain inside the timed region); median of %d such timed runs"
                       % (args.steps, len(e2e_runs)),
                "serial_host_direct": {"value": flops_step * world / (e2e_direct_ms * 1e-3) / 1e12,
                                       "ms_per_step": e2e_direct_ms,
                                       "how": "one step at a time: q, k, v sharded straight from pinned host memory, "
                                              "o unsharded straight into it (the kernels cross the host link)"},
                "serial_copy_engine": {"value": flops_step * world / (e2e_copy_ms * 1e-3) / 1e12,
                                       "ms_per_step": e2e_copy_ms,
                                       "how": "one step at a time: cudaMemcpyAsync of q, k, v in and o, lse out "
                                              "around the device step"}},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "kernels": km,
        "wall_s_timed": wall,
    }
    if graph_info is not None:
        line["graph"] = graph_info
    if world == 1 and not args.no_secondary:
        # the other configurations, same device-step timing (after the main
        # timed region and its end-to-end runs, with their buffers freed)
        del rig, inbuf, obuf, qd, kd, vd, qs, o_sh, lse_sh, o_full, qh, step, flush_buf
        torch.cuda.empty_cache()
        line["secondary"] = run_secondary(args, dev, peaks, prefetch, fused)
    if rank == 0 and not args.no_cpu_baseline:
        qkv64 = prepare_oracle_inputs(w, q, k, v)
        line["cpu_baseline"] = cpu_baseline(w, qkv64, target_s=args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# --------------------------------------------------------------------------
# sweep: work balance per virtual rank, contiguous vs zigzag
# --------------------------------------------------------------------------
def tile_counts_per_rank(pos, q_block=256, k_tile=128, q_tile=128):
    """Per virtual rank, over all ring steps, the attention kernel's key-tile
    work under its per-tile causal rule: for every (256-row query block, 128-key
    tile) pair, `issued` if the tile's smallest key position is <= the block's
    largest query position, else `skipped`; issued pairs counted again per
    128-row query tile as `unmasked` (tile's largest key position <= the query
    tile's smallest position) or `masked`.  pos: int [C][s] global positions.
    Returns a list of dicts (one per rank)."""
    import numpy as np
    pos = np.asarray(pos)
    C, s = pos.shape

    def ranges(p, n):
        t = [p[i:i + n] for i in range(0, len(p), n)]
        return np.array([x.min() for x in t]), np.array([x.max() for x in t])

    out = []
    for r in range(C):
        bmin, bmax = ranges(pos[r], q_block)
        tmin, tmax = ranges(pos[r], q_tile)
        c = {"issued": 0, "skipped": 0, "unmasked": 0, "masked": 0}
        for st in range(C):
            kmin, kmax = ranges(pos[(r - st) % C], k_tile)
            iss = kmin[None, :] <= bmax[:, None]            # [blocks, key tiles]
            c["issued"] += int(iss.sum())
            c["skipped"] += int((~iss).sum())
            for qb in range(len(bmin)):
                for qt in range(2 * qb, min(2 * qb + 2, len(tmin))):
                    un = iss[qb] & (kmax <= tmin[qt])
                    c["unmasked"] += int(un.sum())
                    c["masked"] += int((iss[qb] & ~un).sum())
        out.append(c)
    return out


def exact_pairs_per_rank(S, C, layout):
    """Visible (query, key) pairs per rank (per batch and head), closed forms."""
    s = S // C
    if layout == "zigzag":
        t = S // (2 * C)
        return [(2 * C - 1) * t * t + t * (t + 1)] * C
    return [r * s * s + s * (s + 1) // 2 for r in range(C)]


def sweep_measure(w, dev, reps, device_inputs=False):
    """One sweep workload: ring TFLOP/s (prefetch on), per-rank pairs, issued
    key tiles and time (each rank's C partials launched on their own, timed
    with events), merge / shard / unshard / prefetch-copy GB/s.  Inputs are
    N(0, 1) bf16 drawn with seed 0 (on the device when device_inputs)."""
    import torch

    from context_causal_attention_gb300 import ops as F
    C, S, B, N, D = w.C, w.S, w.B, w.N, w.D
    s = S // C
    lay = F.CP_ZIGZAG if w.layout == "zigzag" else F.CP_CONTIGUOUS
    if device_inputs:
        g = torch.Generator(device=dev).manual_seed(0)
        q, k, v = (torch.randn(B, S, N, D, generator=g, device=dev).to(torch.bfloat16) for _ in range(3))
    else:
        g = torch.Generator("cpu").manual_seed(0)
        q, k, v = (torch.randn(B, S, N, D, generator=g).to(torch.bfloat16).to(dev) for _ in range(3))
    qs, ks, vs = (F.cp_zigzag_shard(t, C, lay) for t in (q, k, v))
    pos = F.cp_zigzag_positions(S, C, lay, device=dev)
    o = torch.empty((C, B, s, N, D), dtype=torch.float32, device=dev)
    lse = torch.empty((C, B, N, s), dtype=torch.float32, device=dev)
    ws = torch.empty(max(256, F.cp_ring_workspace_size(B, S, N, N, D, C, 1, F.CP_F32)), dtype=torch.uint8,
                     device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4 * C)]
    for e in ev:
        e.record()

    def ring(events=None):
        F.cp_ring_attention_fwd(qs, ks, vs, pos, layout=lay, prefetch=1, workspace=ws, o=o, lse=lse,
                                events=events)

    for _ in range(3):
        ring()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        ring()
    e1.record()
    torch.cuda.synchronize()
    ring_ms = e0.elapsed_time(e1) / reps
    ring(ev)
    torch.cuda.synchronize()
    merge_ms = sum(ev[4 * st + 2].elapsed_time(ev[4 * st + 3]) for st in range(1, C))
    attn_ms = sum(ev[4 * st].elapsed_time(ev[4 * st + 1]) for st in range(C))
    # per-rank diagnostic: rank r's C partials launched on their own
    o1 = torch.empty((B, s, N, D), dtype=torch.float32, device=dev)
    l1 = torch.empty((B, N, s), dtype=torch.float32, device=dev)
    rank_ms = []
    for r in range(C):
        def partials():
            for st in range(C):
                j = (r - st) % C
                F.cp_attn_partial(qs[r], ks[j], vs[j], pos[r], pos[j], o=o1, lse=l1)
        partials()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        for _ in range(2):
            partials()
        a1.record()
        torch.cuda.synchronize()
        rank_ms.append(a0.elapsed_time(a1) / 2)
    # permutations and the prefetch copy (one K rotation = the bytes the ring exchange moves per step)
    x = torch.empty_like(q)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(5):
        F.cp_zigzag_shard(q, C, lay, out=qs)
    t1.record()
    torch.cuda.synchronize()
    shard_gbs = 2 * q.numel() * 2 / (t0.elapsed_time(t1) / 5 * 1e-3) / 1e9
    t0.record()
    for _ in range(5):
        F.cp_zigzag_unshard(qs, lay, out=x)
    t1.record()
    torch.cuda.synchronize()
    unshard_gbs = 2 * q.numel() * 2 / (t0.elapsed_time(t1) / 5 * 1e-3) / 1e9
    kbuf = torch.empty_like(ks)
    t0.record()
    for _ in range(5):
        kbuf.copy_(ks)
    t1.record()
    torch.cuda.synchronize()
    copy_gbs = 2 * ks.numel() * 2 / (t0.elapsed_time(t1) / 5 * 1e-3) / 1e9
    pairs = exact_pairs_per_rank(S, C, w.layout)
    flops = 4.0 * B * N * D * S * (S + 1) / 2
    tiles = tile_counts_per_rank(pos.cpu().numpy())
    issued = [t["issued"] for t in tiles]
    return {
        "sweep": w.name, "S": S, "C": C, "layout": w.layout,
        "ring_ms": ring_ms, "ring_tflops": flops / (ring_ms * 1e-3) / 1e12,
        "attn_ms_in_ring": attn_ms, "merge_ms_in_ring": merge_ms,
        "pairs_per_rank": pairs, "pairs_max_over_mean": max(pairs) / (sum(pairs) / C),
        "rank_ms": rank_ms, "rank_ms_max_over_mean": max(rank_ms) / (sum(rank_ms) / C),
        "issued_tiles_max_over_mean": max(issued) / (sum(issued) / C),
        "shard_gbs": shard_gbs, "unshard_gbs": unshard_gbs, "kv_rotation_copy_gbs": copy_gbs,
        "merge_rows_per_step": C * B * N * s,
        "key_tiles_per_rank": tiles,
    }


def run_sweep(args):
    """One JSON line per sweep workload (see sweep_measure)."""
    import torch

    import cp_synth as SY
    from context_causal_attention_gb300 import build as cuda_build

    cuda_build.build()
    dev = torch.device("cuda", 0)
    peaks = load_peaks()
    names = args.sweep_only.split(",") if args.sweep_only else None
    for w in SY.sweep_workloads():
        if names and w.name not in names:
            continue
        line = sweep_measure(w, dev, reps=max(3, args.steps))
        line["hbm_peak_gbs"] = peaks["hbm_gbs"]
        print(json.dumps(line), flush=True)
        torch.cuda.empty_cache()
    return 0


def run_strategies(args):
    """One JSON line per (workload, strategy): the forward of the ring, the
    all-gather, the all-to-all (Ulysses) and the A2A x P2P mesh on the same
    zigzag shards, timed with CUDA events (3 warm-up calls, then the mean of
    `--steps` calls), TFLOP/s on the algorithmic causal FLOPs."""
    import torch

    import cp_synth as SY
    from context_causal_attention_gb300 import build as cuda_build
    from context_causal_attention_gb300 import ops as F

    cuda_build.build()
    dev = torch.device("cuda", 0)
    names = args.strategies.split(",")
    for wname in names:
        w = SY.WORKLOADS[wname]
        q, k, v, _ = SY.make_qkv(w)
        qs, ks, vs = (F.cp_zigzag_shard(t.to(dev), w.C) for t in (q, k, v))
        del q, k, v
        pos = F.cp_zigzag_positions(w.S, w.C, device=dev)
        runs = [("ring", lambda: F.cp_ring_attention_fwd(qs, ks, vs, pos, prefetch=1)),
                ("allgather", lambda: F.cp_allgather_attention_fwd(qs, ks, vs, pos))]
        if w.N % w.C == 0 and w.Nkv % w.C == 0:
            runs.append(("ulysses", lambda: F.cp_ulysses_attention_fwd(qs, ks, vs)))
        for A in range(2, w.C):
            if w.C % A == 0 and w.N % A == 0 and w.Nkv % A == 0:
                runs.append(("mesh_a%d_r%d" % (A, w.C // A),
                             lambda A=A: F.cp_mesh_attention_fwd(qs, ks, vs, pos, A, w.C // A, prefetch=1)))
        for name, fn in runs:
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = max(3, args.steps)
            e0.record()
            for _ in range(reps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / reps
            print(json.dumps({"strategy": name, "workload": w.name, "S": w.S, "C": w.C, "N": w.N, "D": w.D,
                              "ms": ms, "tflops": w.flops / (ms * 1e-3) / 1e12,
                              "note": "forward only, inputs already sharded on the device; includes the "
                                      "strategy's own relayouts / gathers"}), flush=True)
            torch.cuda.empty_cache()
        del qs, ks, vs, pos
        torch.cuda.empty_cache()
    return 0


def run_backward(args):
    """One JSON line per workload: the ring backward (statistics, then per ring
    step one dK/dV and one dQ launch) on the full workload, after a ring
    forward that supplies o and lse.  TFLOP/s on the algorithmic backward
    FLOPs, 10 D per visible (query, key) pair per head (five products: S, dP,
    dV, dK, dQ; 2.5x the forward); the kernels also recompute S and dP in the
    dQ pass (14 D per pair executed), reported as well."""
    import torch

    import cp_synth as SY
    from context_causal_attention_gb300 import build as cuda_build
    from context_causal_attention_gb300 import ops as F

    cuda_build.build()
    dev = torch.device("cuda", 0)
    peaks = load_peaks()
    sweep = {x.name: x for x in SY.sweep_workloads()}
    for wname in args.backward.split(","):
        w = SY.WORKLOADS.get(wname) or sweep[wname]
        q, k, v, _ = SY.make_qkv(w)
        g = torch.Generator("cpu").manual_seed(1)
        do = torch.randn(w.B, w.S, w.N, w.D, generator=g).to(torch.bfloat16)
        qs, ks, vs, dos = (F.cp_zigzag_shard(t.to(dev), w.C) for t in (q, k, v, do))
        del q, k, v, do
        pos = F.cp_zigzag_positions(w.S, w.C, device=dev)
        o_sh, lse_sh = F.cp_ring_attention_fwd(qs, ks, vs, pos, prefetch=1)
        ws = torch.empty(max(256, F.cp_ring_bwd_workspace_size(w.B, w.S, w.N, w.C)), dtype=torch.uint8, device=dev)
        dq, dk, dv = (torch.empty(t.shape, dtype=torch.float32, device=dev) for t in (qs, ks, vs))

        def bwd():
            F.cp_ring_attention_bwd(qs, ks, vs, o_sh, lse_sh, dos, pos, workspace=ws, dq=dq, dk=dk, dv=dv)

        for _ in range(max(3, args.warmup)):
            bwd()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(3, args.steps)
        e0.record()
        for _ in range(reps):
            bwd()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        pairs = w.S * (w.S + 1) / 2 * w.B * w.N
        alg = 10.0 * w.D * pairs
        print(json.dumps({"backward": w.name, "S": w.S, "C": w.C, "N": w.N, "D": w.D, "ms": ms,
                          "tflops_algorithmic": alg / (ms * 1e-3) / 1e12,
                          "tflops_executed": 1.4 * alg / (ms * 1e-3) / 1e12,
                          "frac_of_burst_bf16": alg / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                          "frac_of_sustained_bf16": alg / (ms * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"],
                          "status": F.cp_device_status()}), flush=True)
        del qs, ks, vs, dos, o_sh, lse_sh, ws, dq, dk, dv
        torch.cuda.empty_cache()
    return 0


def run_tf32(args):
    """One JSON line per workload: the ring forward over fp32 shards with the
    tensor cores in tf32 (CP_RING_TF32, zero copy), TFLOP/s on the algorithmic
    causal FLOPs against the tf32 peak (the measured bf16 burst peak -- the
    runs are short and at full clock -- x the nominal tf32 / bf16 ratio
    1.1 / 2.25; the sustained-based figure beside it)."""
    import torch

    import cp_synth as SY
    from context_causal_attention_gb300 import build as cuda_build
    from context_causal_attention_gb300 import ops as F

    cuda_build.build()
    dev = torch.device("cuda", 0)
    peaks = load_peaks()
    ratio = 1.1 / 2.25
    sweep = {x.name: x for x in SY.sweep_workloads()}
    for wname in args.tf32.split(","):
        w = SY.WORKLOADS.get(wname) or sweep[wname]
        g = torch.Generator("cpu").manual_seed(0)
        qs, ks, vs = (F.cp_zigzag_shard(torch.randn(w.B, w.S, n, w.D, generator=g).to(dev), w.C)
                      for n in (w.N, w.Nkv, w.Nkv))
        pos = F.cp_zigzag_positions(w.S, w.C, device=dev)
        ws = torch.empty(max(256, F.cp_ring_workspace_size(w.B, w.S, w.N, w.Nkv, w.D, w.C, tf32=True)),
                         dtype=torch.uint8, device=dev)

        def fwd():
            F.cp_ring_attention_fwd(qs, ks, vs, pos, tf32=True, workspace=ws)

        for _ in range(max(3, args.warmup)):
            fwd()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(3, args.steps)
        e0.record()
        for _ in range(reps):
            fwd()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        tf = w.flops / (ms * 1e-3) / 1e12
        print(json.dumps({"tf32_ring": w.name, "S": w.S, "C": w.C, "N": w.N, "D": w.D, "ms": ms, "tflops": tf,
                          "tf32_peak_burst": peaks["bf16_tflops"] * ratio,
                          "frac_of_tf32_burst": tf / (peaks["bf16_tflops"] * ratio),
                          "tf32_peak_sustained": peaks["bf16_tflops_sustained"] * ratio,
                          "frac_of_tf32_sustained": tf / (peaks["bf16_tflops_sustained"] * ratio),
                          "note": "includes the per-call transpose of v (fp32) for the K-major P V operand",
                          "status": F.cp_device_status()}), flush=True)
        del qs, ks, vs, ws
        torch.cuda.empty_cache()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="s32k")
    ap.add_argument("--no-prefetch", dest="prefetch", action="store_false")
    ap.add_argument("--fused-merge", dest="fused_merge", action="store_true",
                    help="merge ring steps >= 1 in the attention epilogue instead of with the standalone merge kernel "
                         "(about 3%% faster whole steps; the attention kernel then also moves the merge's bytes)")
    ap.add_argument("--separate-merge", dest="fused_merge", action="store_false", help="the default")
    ap.set_defaults(fused_merge=False)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the secondary workloads (S=4096, S=131072, the S=65536 sweep point) of the default line")
    ap.add_argument("--graph", action="store_true",
                    help="also time CUDA-graph replays of the step and of each permutation (with the eager times)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--sweep", action="store_true", help="run the contiguous-vs-zigzag sweep instead")
    ap.add_argument("--strategies", default="",
                    help="comma-separated workloads: time ring / all-gather / Ulysses / mesh forwards instead")
    ap.add_argument("--backward", default="",
                    help="comma-separated workloads: time the ring backward instead")
    ap.add_argument("--tf32", default="",
                    help="comma-separated workloads: time the ring forward over fp32 shards in tf32 instead")
    ap.add_argument("--sweep-only", default="", help="comma-separated sweep workload names")
    args = ap.parse_args()
    if args.sweep:
        return run_sweep(args)
    if args.strategies:
        return run_strategies(args)
    if args.backward:
        return run_backward(args)
    if args.tf32:
        return run_tf32(args)
    import cp_synth as SY
    w = SY.WORKLOADS.get(args.workload)
    if w is None:
        w = {x.name: x for x in SY.sweep_workloads()}[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
