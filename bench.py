"""Benchmark of the H2O budgeted eviction hot path on GB300.

One step = one whole generation job of the workload through the C ABI: the prefill score pass +
heavy-hitter selection over the prompts (h2o_prefill_select), then every decode step
(h2o_decode_step), all units of all layers. Inputs are seeded synthetic Q/K/V already resident in
HBM when the timed region starts; the KV cache (856 MB for the default workload) and every step's
inputs are larger than the 129 MB L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload opt-6.7b] [--impl h2o|reference]

Prints one JSON line. `value` is generated tokens/s (batch x decode steps per job / job time,
prefill + decode, as the H2O post §3.1.3 defines token throughput); `roofline` is the decode
kernel's algorithmic HBM bytes per launch over its average CUDA-event duration. `--impl reference`
times the CPU oracle (the plain restatement of the method used as the parity reference) on a
bounded sample of the same workload on this host's cores.
"""

from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
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

import synth  # noqa: E402

METRIC = "H2O decode tokens/s (batch x steps, 1 GB300) and KV-read GB/s vs HBM"
CSRC = os.path.join(ROOT, "kv_cache_eviction_step_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic.json")
GRAPH_STEPS = 1024  # decode launches per captured CUDA graph


def decode_bytes_per_unit(n: int, head_dim: int, elem_bytes: int) -> int:
    """Algorithmic HBM bytes of one unit's decode step with n valid cached slots: K and V rows read
    (2 n D eb), score read + write and position read (12 n); new q/k/v read, the victim's K/V row
    written and the output row (6 D eb); written score, position and the two eviction indices (16)."""
    return n * (2 * head_dim * elem_bytes + 12) + 6 * head_dim * elem_bytes + 16


def decode_bytes_per_unit_e4m3(n: int, head_dim: int) -> int:
    """The same for the E4M3 cache: K and V codes (2 n D), row scales read (8 n), score read + write
    and position read (12 n); bf16 q/k_new/v_new read and the output written (8 D); the victim's
    codes (2 D) and scales (8); written score, position and the two eviction indices (16)."""
    return n * (2 * head_dim + 20) + 10 * head_dim + 24


class Calls:
    """The library calls of one job, for the bf16 or the E4M3 cache. A decode step is launched once
    per layer (a model's forward pass has to: layer l + 1's query needs layer l's output) over that
    layer's B x H units, the slice [l B H, (l + 1) B H) of every array; with a bf16 cache each launch
    names the next launch's layer (the next step's layer 0 after the last layer) as the L2 prefetch
    hint of h2o_decode_step_prefetch. decode_all_layers is the same step as one launch over all
    units."""

    def __init__(self, h2o, dims, cache, e4m3: bool, layers: int = 1):
        self.h2o, self.dims, self.cache, self.e4m3 = h2o, dims, cache, e4m3
        self.L = layers
        self.ul = dims.units // layers
        self.dl = type(dims)(units_b=dims.units_b // layers, heads=dims.heads, head_dim=dims.head_dim,
                             budget=dims.budget, k_heavy=dims.k_heavy, k_local=dims.k_local, dtype=dims.dtype)
        self.sl = [slice(l * self.ul, (l + 1) * self.ul) for l in range(layers)]
        c = cache
        self.nxt = [None if e4m3 else h2o.next_cache(c.k_cache[self.sl[(l + 1) % layers]], c.v_cache[self.sl[(l + 1) % layers]],
                                                     c.scores[self.sl[(l + 1) % layers]], c.slot_pos[self.sl[(l + 1) % layers]])
                    for l in range(layers)]

    def prefill(self, P, q, k, v, stream):
        c = self.cache
        if self.e4m3:
            self.h2o.h2o_prefill_select_e4m3(self.dims, None, P, q, k, v, c.k_cache, c.v_cache, c.k_scale,
                                             c.v_scale, c.scores, c.slot_pos, c.workspace, stream)
        else:
            self.h2o.h2o_prefill_select(self.dims, P, q, k, v, c.k_cache, c.v_cache, c.scores, c.slot_pos,
                                        c.workspace, stream)

    def decode(self, t, q, k_new, v_new, out, evs, evp, stream, last: bool = False, hint: bool = True):
        """One decode step at position t, one launch per layer; ``last``: no later step follows (the
        last launch names no next cache); ``hint``: name the next launch's cache."""
        if self.L == 1:
            return self.decode_all_layers(t, q, k_new, v_new, out, evs, evp, stream)
        c, h2o = self.cache, self.h2o
        for l, sl in enumerate(self.sl):
            args = (q[sl], k_new[sl], v_new[sl], c.k_cache[sl], c.v_cache[sl])
            if self.e4m3:
                h2o.h2o_decode_step_e4m3(self.dl, None, t, *args, c.k_scale[sl], c.v_scale[sl], c.scores[sl],
                                         c.slot_pos[sl], out[sl], evs[sl], evp[sl], stream)
            elif hint:
                nxt = None if (last and l == self.L - 1) else self.nxt[l]
                h2o.h2o_decode_step_prefetch(self.dl, None, t, *args, c.scores[sl], c.slot_pos[sl], out[sl], evs[sl],
                                             evp[sl], nxt, stream)
            else:
                h2o.h2o_decode_step(self.dl, t, *args, c.scores[sl], c.slot_pos[sl], out[sl], evs[sl], evp[sl],
                                    stream)

    def decode_all_layers(self, t, q, k_new, v_new, out, evs, evp, stream):
        c = self.cache
        if self.e4m3:
            self.h2o.h2o_decode_step_e4m3(self.dims, None, t, q, k_new, v_new, c.k_cache, c.v_cache,
                                          c.k_scale, c.v_scale, c.scores, c.slot_pos, out, evs, evp, stream)
        else:
            self.h2o.h2o_decode_step(self.dims, t, q, k_new, v_new, c.k_cache, c.v_cache, c.scores,
                                     c.slot_pos, out, evs, evp, stream)


def measured_peaks() -> tuple[dict, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def source_sha(path: str) -> str:
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def decode_kernel(w: synth.Workload, sms: int, e4m3: bool = False) -> tuple[str, str]:
    """Which decode kernel the library launches for this workload (the C ABI's dispatch rule:
    persistent tcgen05 for >= 4 bf16 units of D = 128 per SM with budgets up to 512, the resident
    one-CTA-per-unit kernel for 1 to 4 such units per SM with budgets up to 208, the cluster-split
    tcgen05 kernel for other bf16 D = 128 caches up to 8192 slots, the CUDA-core kernel otherwise;
    the E4M3 cache always runs its persistent tcgen05 kernel)."""
    if e4m3:
        return "h2o_decode_e4m3_kernel", os.path.join(CSRC, "h2o_decode_e4m3.cu")
    if w.dtype == "bf16" and w.head_dim == 128 and w.budget <= 512 and w.units >= 4 * sms:
        return "h2o_decode_tc_kernel", os.path.join(CSRC, "h2o_decode_tc.cu")
    if w.dtype == "bf16" and w.head_dim == 128 and w.budget <= 208 and w.units >= sms:
        return "h2o_decode_resident_kernel", os.path.join(CSRC, "h2o_decode_resident.cu")
    if w.dtype == "bf16" and w.head_dim == 128 and w.budget <= 8192:
        return "h2o_decode_tc_split_kernel", os.path.join(CSRC, "h2o_decode_tc.cu")
    return "h2o_decode_step_kernel", os.path.join(CSRC, "h2o_decode.cu")


def prefill_launches(w: synth.Workload, sms: int) -> int:
    """Launches of one H2O prefill (h2o_prefill_select / _e4m3): the score pass, then the selection.
    The score pass is one launch (the one-pass column sums) for bf16 prompts of at most four 128-token
    tiles with at least one unit per SM, else two (row statistics, then column sums)."""
    one_pass = w.dtype == "bf16" and -(-w.prompt_len // 128) <= 4 and w.units >= sms
    return (1 if one_pass else 2) + 1


def recorded_traffic(workload: str, kernel: str, src: str, units_per_launch: int):
    """DRAM bytes per decode launch from the committed ncu records, if one was taken on the current
    source of this kernel, on this workload and with this many units per launch; otherwise None."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        recs = json.load(f)
    for rec in recs.get("records", [recs]):
        if (rec.get("kernel") == kernel and rec.get("kernel_sha") == source_sha(src)
                and rec.get("workload") == workload and rec.get("units_per_launch") == units_per_launch):
            return rec.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples every 50 ms while the timed region runs. The sampler is
    started first and the region is entered only once its first sample is written, so every sample
    kept falls inside the region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.skip = 0  # samples written before the region

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return self
        t0 = time.time()
        while time.time() - t0 < 5.0 and self.proc.poll() is None:
            with open(self.path) as f:
                n = sum(1 for _ in f)
            if n:
                self.skip = n
                break
            time.sleep(0.01)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for i, line in enumerate(open(self.path)):
            parts = [p.strip() for p in line.split(",")]
            if i >= self.skip and len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        pw = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------------------------
# CPU oracle baseline (the reference arm and the cpu_baseline key)


def _oracle_run(w: synth.Workload, inp: synth.Inputs, i: int, steps: int) -> None:
    """The oracle over sample unit ``i`` of ``inp``: prefill, then ``steps`` decode steps."""
    import oracle
    orc = oracle.Oracle(w.budget, w.k_heavy, w.k_local)
    st = orc.new_state(1, w.head_dim, synth.storage_dtype(w))
    orc.run_unit(inp.q_prompt[i], inp.k_prompt[i], inp.v_prompt[i], inp.q_dec[:steps],
                 inp.k_dec[:steps], inp.v_dec[:steps], st, unit=i)


def cpu_oracle_baseline(w: synth.Workload, seed: int, target_s: float = 12.0) -> dict:
    """Oracle throughput on a bounded sample of the workload: whole units (prefill + every decode
    step), one unit per task over all host cores, sized to about ``target_s`` seconds of wall time.
    Input generation happens before the timed region."""
    cores = os.cpu_count() or 1
    probe_inp = synth.generate(w, seed, units=np.array([0]))
    t0 = time.perf_counter()
    _oracle_run(w, probe_inp, 0, w.decode_steps)
    probe = time.perf_counter() - t0
    per_core = max(1, int(target_s / max(probe, 1e-3)))
    n_units = int(min(w.units, per_core * cores))
    units = np.linspace(0, w.units - 1, n_units).astype(np.int64)
    inp = synth.generate(w, seed, units=units)
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(cores) as ex:  # ctypes releases the GIL inside the oracle
        list(ex.map(lambda i: _oracle_run(w, inp, i, w.decode_steps), range(n_units)))
    wall = time.perf_counter() - t0
    # tokens/s of the whole job extrapolated from the sample: the job has w.units units.
    job_s = wall * w.units / n_units
    tokens = w.batch * w.decode_steps
    return {"value": tokens / job_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n_units} of {w.units} units (prefill + {w.decode_steps} decode steps each), "
                      f"{wall:.1f} s wall on {cores} threads, extrapolated to the whole job"}


# ---------------------------------------------------------------------------------------------


def run_reference(args, w, world, rank):
    if rank != 0:
        return
    seed = synth.DEFAULT_SEED
    steps_out = []
    for i in range(args.warmup + args.steps):
        b = cpu_oracle_baseline(w, seed, target_s=max(2.0, 30.0 / (args.warmup + args.steps)))
        if i >= args.warmup:
            steps_out.append(b)
    value = statistics.median(b["value"] for b in steps_out)
    tokens = w.batch * w.decode_steps
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * tokens / value, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, args),
            "cpu_baseline": dict(steps_out[-1], value=value),
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def config_of(w: synth.Workload, args) -> dict:
    return {"workload": f"{w.name}: {w.note}", "layers": w.layers, "batch": w.batch, "heads": w.heads,
            "head_dim": w.head_dim, "prompt_len": w.prompt_len, "decode_steps": w.decode_steps,
            "budget": w.budget, "k_heavy": w.k_heavy, "k_local": w.k_local, "units": w.units,
            "parallelism": f"replicas x{args.gpus} (units independent, no collective)",
            "kv_cache": ("E4M3 codes + float32 row scales (bf16 q/k/v/out)" if args.kv_cache == "e4m3"
                         else w.dtype),
            "l2": "no flush: KV cache and per-step inputs exceed the 129 MB L2",
            "timing": "CUDA events between replays of CUDA graphs per job (the prefill's launches, then the "
                      "decode launches)",
            "decode_launch": (f"one launch per layer and step ({w.layers} launches per step of {w.batch} x "
                              f"{w.heads} = {w.units // w.layers} units each"
                              + ("" if args.kv_cache == "e4m3" else
                                 ", each naming the next launch's layer as the L2 prefetch hint of "
                                 "h2o_decode_step_prefetch")
                              + "); all layers in one launch per step is timed separately as "
                                "decode_all_layers" if w.layers > 1 else
                              f"one launch per step over all {w.units} units")}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="opt-6.7b", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="h2o", choices=["h2o", "reference"])
    ap.add_argument("--layers", type=int, default=None,
                    help="override the workload's layer count (smaller cases for profiling)")
    ap.add_argument("--decode-steps", type=int, default=None,
                    help="override the workload's decode steps (shorter jobs for profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-prefill-forward", action="store_true")
    ap.add_argument("--no-per-layer", action="store_true",
                    help="skip the decode timings in the other launch shapes (all layers in one launch "
                         "per step; one launch per layer without the prefetch hint)")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip the other workloads' decode / prefill timings in the default line")
    ap.add_argument("--kv-cache", default="bf16", choices=["bf16", "e4m3"],
                    help="cache format: the workload's dtype, or E4M3 codes with per-row scales")
    args = ap.parse_args()
    w = synth.WORKLOADS[args.workload]
    if args.layers is not None:
        w = w.with_(layers=args.layers)
    if args.decode_steps is not None:
        w = w.with_(decode_steps=args.decode_steps)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, w, world, rank)
        return

    import torch

    import kv_cache_eviction_step_gb300 as h2o

    assert torch.cuda.is_available(), "bench.py needs a GPU"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    seed = synth.DEFAULT_SEED + 7919 * rank  # each rank: its own sequences (weak scaling)
    U, D, P, S = w.units, w.head_dim, w.prompt_len, w.decode_steps
    eb = w.elem_bytes
    tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    dims = h2o.Dims(units_b=w.units_b, heads=w.heads, head_dim=D, budget=w.budget,
                    k_heavy=w.k_heavy, k_local=w.k_local, dtype=h2o.F32 if w.dtype == "f32" else h2o.BF16)

    # Inputs: generated on the host (seeded), pinned, then resident in HBM.
    t_gen = time.perf_counter()
    inp = synth.generate(w, seed)
    t_gen = time.perf_counter() - t_gen

    def pinned(a):
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        t = t.pin_memory()
        return t.view(tdt) if a.dtype == np.uint16 else t

    host = {k: pinned(getattr(inp, k)) for k in ("q_prompt", "k_prompt", "v_prompt", "q_dec", "k_dec", "v_dec")}
    del inp
    dv = {k: v.to(dev) for k, v in host.items()}
    e4m3 = args.kv_cache == "e4m3"
    if e4m3 and (w.dtype != "bf16" or D != 128):
        raise SystemExit("--kv-cache e4m3 needs a bf16 workload with head_dim 128")
    cache = h2o.H2OCache(dims, P, device=dev, e4m3=e4m3)
    L = w.layers
    calls = Calls(h2o, dims, cache, e4m3, layers=L)
    out = torch.empty((S, U, D), dtype=tdt, device=dev)
    evs = torch.empty((S, U), dtype=torch.int32, device=dev)
    evp = torch.empty((S, U), dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sp_ptr = stream.cuda_stream

    def prefill():
        calls.prefill(P, dv["q_prompt"], dv["k_prompt"], dv["v_prompt"], sp_ptr)

    def decode_range(s0, s1):
        for s in range(s0, s1):
            calls.decode(P + s, dv["q_dec"][s], dv["k_dec"][s], dv["v_dec"][s], out[s], evs[s], evp[s], sp_ptr,
                         last=s == S - 1)

    # One direct run initialises the library's per-device state (kernel attributes, launch plans,
    # error word) outside any capture; then the job is captured as two CUDA graphs (the prefill
    # launches and the S decode launches) so host-side call overhead is out of the timed region.
    with torch.cuda.stream(stream):
        prefill()
        decode_range(0, S)
    torch.cuda.synchronize(dev)
    g_pre = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_pre, stream=stream):
        prefill()
    g_dec = []  # decode launches in graphs of at most GRAPH_STEPS launches
    steps_per_graph = max(1, GRAPH_STEPS // L)
    for s0 in range(0, S, steps_per_graph):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            decode_range(s0, min(S, s0 + steps_per_graph))
        g_dec.append(g)

    def job(marks=None):
        with torch.cuda.stream(stream):
            if marks is not None:
                marks[0].record(stream)
            g_pre.replay()
            if marks is not None:
                marks[1].record(stream)
            for g in g_dec:
                g.replay()
            if marks is not None:
                marks[2].record(stream)

    for _ in range(args.warmup):
        job()
    torch.cuda.synchronize(dev)
    if h2o.h2o_get_device_error(sp_ptr) != 0:
        raise RuntimeError("device error word set during warm-up")

    K = args.steps
    rec = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        for i in range(K):
            job(rec[i])
        torch.cuda.synchronize(dev)
    barrier(world)
    total_ms = rec[0][0].elapsed_time(rec[K - 1][2])
    total_ms = max_over_ranks(total_ms, world)
    if h2o.h2o_get_device_error(sp_ptr) != 0:
        raise RuntimeError("device error word set during the timed region")

    # Per decode step: the decode graphs' duration over the S steps (L launches each; includes the
    # short launch-to-launch gaps inside the graphs, so it slightly understates the kernel's own rate).
    decode_ms = [rec[i][1].elapsed_time(rec[i][2]) / S for i in range(K) for _ in range(S)]
    prefill_ms = [rec[i][0].elapsed_time(rec[i][1]) for i in range(K)]
    ms_per_step = total_ms / K
    tokens_per_job = w.batch * S
    value = world * tokens_per_job * K / (total_ms / 1000.0)

    # Roofline of the decode kernel (the dominant kernel): one launch = one layer's B x H units.
    peaks, peak_kind = measured_peaks()
    bytes_per_launch = [U // L * (decode_bytes_per_unit_e4m3(min(P + s, w.budget), D) if e4m3 else
                                  decode_bytes_per_unit(min(P + s, w.budget), D, eb)) for s in range(S)]
    avg_bytes = float(np.mean(bytes_per_launch))
    avg_decode_s = float(np.mean(decode_ms)) / 1000.0 / L
    achieved = avg_bytes / avg_decode_s / 1e9
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    n_pre = prefill_launches(w, sms)
    kname, ksrc = decode_kernel(w.with_(layers=1), sms, e4m3)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": recorded_traffic(w.name, kname, ksrc, U // L),
                "kernel": kname, "peak_source": f"{peak_kind} hbm_gbs (burst copy)",
                "algorithmic_bytes_per_launch": avg_bytes, "avg_launch_us": avg_decode_s * 1e6,
                "units_per_launch": U // L}

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if e4m3 else w.dtype,
            "data": "synthetic", "config": config_of(w, args), "roofline": roofline,
            "kv_read_gbs": achieved,
            "decode_tokens_per_s": world * tokens_per_job / (sum(decode_ms) / K / 1000.0),
            "prefill_ms": float(np.mean(prefill_ms)),
            "decode_ms_per_token_step": float(np.mean(decode_ms)),
            "gpu_launches": K * (n_pre + S * L),
            "clocks": clocks.summary(),
            "input_generation_s": t_gen}

    # The same decode steps in the other launch shapes: all layers in one launch per step, and one
    # launch per layer without the prefetch hint.
    if not args.no_per_layer and w.layers > 1:
        line.update(other_launch_shapes(h2o, w, dv, calls, out, evs, evp, stream, dev, g_pre, args.warmup, K,
                                        e4m3))

    # The prompt pass with the attention output (h2o_prefill_forward), timed on its own: not part of
    # the step above, which builds the cache only.
    if not args.no_prefill_forward and not e4m3:
        line["prefill_forward"] = prefill_forward_timing(h2o, dims, w, dv, cache, stream, dev, args.warmup, K)
    # The score pass of the prefill alone (its tensor-core rate), outside the step as well.
    if w.dtype == "bf16" and not e4m3:
        line["prefill_scores"] = prefill_scores_timing(h2o, dims, w, dv["q_prompt"], dv["k_prompt"], stream, dev,
                                                       args.warmup, K)

    # The other workloads of the method's configurations, each timed on this GPU in the same run
    # (decode kernel rate with its roofline, prefill time, clocks), and the E4M3 cache on this one.
    if (not args.no_workloads and world == 1 and not e4m3 and args.layers is None
            and args.decode_steps is None and w.name == "opt-6.7b"):
        line["workloads"] = other_workloads(h2o, dv, dev, args.warmup, K)

    # End to end through the public API with host buffers: every job copies its prompt and decode
    # inputs host->device (pinned) and the outputs and eviction indices device->host.
    if not args.no_e2e:
        line["e2e"] = e2e(args, w, calls, host, stream, dev, world, tokens_per_job)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not e4m3:
        line["cpu_baseline"] = cpu_oracle_baseline(w, seed)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def workload_timing(h2o, w: synth.Workload, dev, warmup: int, reps: int, e4m3: bool = False,
                    dv=None, fill: int = 0, window: int | None = None, copies: int = 1) -> dict:
    """One workload timed on its own: the prefill (h2o_prefill_select) and a window of ``window``
    decode steps (default: all of them) after ``fill`` untimed steps, each launch over all of the
    workload's units, captured in CUDA graphs. Every replay rebuilds the cache from the prompt and
    replays the fill steps (untimed), then CUDA events on the launching stream bracket the prefill
    and the window. ``dv``: device inputs to reuse (else generated here). ``copies`` > 1: for a
    workload whose cache fits in L2, that many independent instances (as the layers of one model),
    each step one launch of the workload's units per instance in turn, so that an instance's cache
    has left L2 when its next step reads it; the per-launch figures are the workload's own."""
    import torch
    w1 = w
    w = w.with_(layers=w.layers * copies)
    U, D, P = w.units, w.head_dim, w.prompt_len
    window = w.decode_steps - fill if window is None else window
    S = fill + window
    assert S <= w.decode_steps
    tdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    dims = h2o.Dims(units_b=w.units_b, heads=w.heads, head_dim=D, budget=w.budget,
                    k_heavy=w.k_heavy, k_local=w.k_local, dtype=h2o.F32 if w.dtype == "f32" else h2o.BF16)
    t_gen = 0.0
    if dv is None:
        t_gen = time.perf_counter()
        inp = synth.generate(w, synth.DEFAULT_SEED, steps=S)

        def to_dev(a):
            t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
            return (t.view(tdt) if a.dtype == np.uint16 else t).to(dev)

        dv = {k: to_dev(getattr(inp, k)) for k in ("q_prompt", "k_prompt", "v_prompt", "q_dec", "k_dec", "v_dec")}
        del inp
        t_gen = time.perf_counter() - t_gen
    cache = h2o.H2OCache(dims, P, device=dev, e4m3=e4m3)
    calls = Calls(h2o, dims, cache, e4m3, layers=copies)
    out = torch.empty((S, U, D), dtype=tdt, device=dev)
    evs = torch.empty((S, U), dtype=torch.int32, device=dev)
    evp = torch.empty((S, U), dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream

    def prefill():
        calls.prefill(P, dv["q_prompt"], dv["k_prompt"], dv["v_prompt"], sp)

    def decode_range(s0, s1):
        for s in range(s0, s1):
            calls.decode(P + s, dv["q_dec"][s], dv["k_dec"][s], dv["v_dec"][s], out[s], evs[s], evp[s], sp)

    with torch.cuda.stream(stream):  # one direct pass sets up the per-shape launch plans
        prefill()
        decode_range(0, S)
    torch.cuda.synchronize(dev)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    g_pre = capture(prefill)
    g_fill = [capture(lambda a=a: decode_range(a, min(fill, a + GRAPH_STEPS))) for a in range(0, fill, GRAPH_STEPS)]
    g_win = [capture(lambda a=a: decode_range(a, min(S, a + GRAPH_STEPS))) for a in range(fill, S, GRAPH_STEPS)]
    pre_ms, win_ms = [], []
    with ClockSampler(dev.index or 0) as clocks:
        for i in range(warmup + reps):
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            with torch.cuda.stream(stream):
                ev[0].record(stream)
                g_pre.replay()
                ev[1].record(stream)
                for g in g_fill:
                    g.replay()
                ev[2].record(stream)
                for g in g_win:
                    g.replay()
                ev[3].record(stream)
            torch.cuda.synchronize(dev)
            if i >= warmup:
                pre_ms.append(ev[0].elapsed_time(ev[1]))
                win_ms.append(ev[2].elapsed_time(ev[3]))
    if h2o.h2o_get_device_error(sp) != 0:
        raise RuntimeError(f"device error word set during the {w.name} timing")
    eb = w.elem_bytes
    step_bytes = [U * (decode_bytes_per_unit_e4m3(min(P + s, w.budget), D) if e4m3 else
                       decode_bytes_per_unit(min(P + s, w.budget), D, eb)) for s in range(fill, S)]
    avg_bytes = float(np.mean(step_bytes))
    us = float(np.median(win_ms)) * 1000.0 / window / copies  # per launch (one instance's step)
    avg_bytes /= copies
    peaks, peak_kind = measured_peaks()
    achieved = avg_bytes / (us * 1e-6) / 1e9
    kname, ksrc = decode_kernel(w1, torch.cuda.get_device_properties(dev).multi_processor_count, e4m3)
    scores = (prefill_scores_timing(h2o, dims, w, dv["q_prompt"], dv["k_prompt"], stream, dev, warmup, reps)
              if w.dtype == "bf16" and not e4m3 else None)
    res = {"workload": f"{w.name}: {w.note}", "units_per_launch": U // copies,
           "kv_cache": "E4M3 codes + float32 row scales" if e4m3 else w.dtype,
           "decode_steps_timed": window, "first_timed_position": P + fill,
           "decode_us_per_step": us,
           "decode_tokens_per_s": w.batch * copies * window / (float(np.median(win_ms)) / 1000.0),
           "prefill_ms": float(np.median(pre_ms)),
           **({"prefill_scores": scores} if scores else {}),
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": achieved / peaks["hbm_gbs"],
                        "traffic": recorded_traffic(w.name, kname, ksrc, U // copies), "kernel": kname,
                        "peak_source": f"{peak_kind} hbm_gbs (burst copy)",
                        "algorithmic_bytes_per_launch": avg_bytes, "avg_launch_us": us},
           "clocks": clocks.summary(),
           "gpu_launches_per_rep": prefill_launches(w, torch.cuda.get_device_properties(dev).multi_processor_count) + S * copies,
           "how": "median over the timed replays; CUDA events around the prefill graph and around the "
                  "window's decode graphs on the launching stream" +
                  (f"; {fill} untimed decode steps before the window fill the cache" if fill else "") +
                  (f"; {copies} independent instances stepped in turn, one launch each, so that each "
                   f"instance's {U // copies * decode_bytes_per_unit(w.budget, D, w.elem_bytes) / 1e6:.1f} MB "
                   f"cache has left the L2 before its next step (prefill_ms: one call over all of them)"
                   if copies > 1 else "")}
    if t_gen:
        res["input_generation_s"] = t_gen
    del dv, cache, out, evs, evp
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return res


def other_workloads(h2o, dv_main, dev, warmup: int, reps: int) -> dict:
    """The method's other configurations, each on this GPU in the same run: the LLaMA-7B-shaped
    decode (one layer of 2048 units per launch, the layer the configuration times), the OPT-30B-shaped
    decode with its prefill (the configuration also times h2o_prefill_select), the streaming workload
    over 2048 steps at its full 4096-slot cache, and the OPT-6.7B job with the E4M3 cache."""
    W = synth.WORKLOADS
    out = {}
    out["llama-7b"] = workload_timing(h2o, W["llama-7b"], dev, warmup, reps)
    out["opt-30b"] = workload_timing(h2o, W["opt-30b"], dev, warmup, reps)
    st = W["streaming"]
    fill = st.budget - st.prompt_len  # the cache is full from position 4096 on
    # Its 68.7 MB cache fits in the L2: four instances stepped in turn keep every read in HBM (the
    # line's figures); the configuration as written (one layer, its cache resident in L2 from step to
    # step) is reported beside them.
    out["streaming"] = workload_timing(h2o, st, dev, warmup, reps, fill=fill, window=2048, copies=4)
    one = workload_timing(h2o, st, dev, warmup, reps, fill=fill, window=2048)
    out["streaming"]["single_instance"] = {
        "decode_us_per_step": one["decode_us_per_step"], "decode_tokens_per_s": one["decode_tokens_per_s"],
        "kv_read_gbs_incl_l2": one["roofline"]["achieved"],
        "note": "one instance: each step finds part of the 68.7 MB cache in L2 from the step before, so "
                "the rate is not comparable with the HBM roofline"}
    out["opt-6.7b-e4m3"] = workload_timing(h2o, W["opt-6.7b"], dev, warmup, reps, e4m3=True, dv=dv_main)
    return out


def other_launch_shapes(h2o, w, dv, calls, out, evs, evp, stream, dev, g_pre, warmup: int, reps: int,
                        e4m3: bool) -> dict:
    """The main timing's decode steps in the other launch shapes, each captured in CUDA graphs of at
    most GRAPH_STEPS launches and timed with CUDA events around the decode graphs (the cache rebuilt
    by the prefill graph before each replay, untimed): all layers' units in one launch per step (the
    multi-layer decode), and, for bf16 caches, one launch per layer without the prefetch hint."""
    import torch
    L, P, S, D, U = w.layers, w.prompt_len, w.decode_steps, w.head_dim, w.units
    sp = stream.cuda_stream
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak = measured_peaks()[0]["hbm_gbs"]
    eb = 2 if w.dtype == "bf16" else 4
    unit_bytes = float(np.mean([decode_bytes_per_unit_e4m3(min(P + s, w.budget), D) if e4m3 else
                                decode_bytes_per_unit(min(P + s, w.budget), D, eb) for s in range(S)]))

    def timed(step, launches_per_step):
        with torch.cuda.stream(stream):  # one direct pass sets up the per-shape launch plans
            g_pre.replay()
            for s in range(S):
                step(s)
        torch.cuda.synchronize(dev)
        graphs = []
        per_graph = max(1, GRAPH_STEPS // launches_per_step)
        for s0 in range(0, S, per_graph):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for s in range(s0, min(S, s0 + per_graph)):
                    step(s)
            graphs.append(g)
        ms = []
        for i in range(warmup + reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                g_pre.replay()
                e0.record(stream)
                for g in graphs:
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize(dev)
            if i >= warmup:
                ms.append(e0.elapsed_time(e1))
        if h2o.h2o_get_device_error(sp) != 0:
            raise RuntimeError("device error word set during the launch-shape timings")
        return float(np.median(ms))

    def entry(ms, launches_per_step, kernel, call, traffic=None):
        us_launch = ms * 1000.0 / S / launches_per_step
        gbs = U / launches_per_step * unit_bytes / (us_launch * 1e-6) / 1e9
        return {"kernel": kernel, "call": call, "launches_per_step": launches_per_step,
                "units_per_launch": U // launches_per_step, "us_per_launch": us_launch,
                "decode_tokens_per_s": w.batch * S / (ms / 1000.0), "kv_read_gbs": gbs, "frac": gbs / peak,
                "traffic": traffic}

    def io(s):
        return dv["q_dec"][s], dv["k_dec"][s], dv["v_dec"][s], out[s], evs[s], evp[s], sp

    res = {}
    kname, ksrc = decode_kernel(w, sms, e4m3)
    res["decode_all_layers"] = entry(
        timed(lambda s: calls.decode_all_layers(P + s, *io(s)), 1), 1, kname,
        "h2o_decode_step_e4m3" if e4m3 else "h2o_decode_step", recorded_traffic(w.name, kname, ksrc, U))
    if not e4m3:
        res["decode_per_layer_plain"] = entry(
            timed(lambda s: calls.decode(P + s, *io(s), hint=False), L), L,
            decode_kernel(w.with_(layers=1), sms)[0], "h2o_decode_step")
    for v in res.values():
        v["how"] = ("CUDA graphs of the decode launches, CUDA events around them; median over the timed "
                    "replays; cache rebuilt by the prefill between replays (untimed)")
    return res


def prefill_score_kernels(w: synth.Workload, sms: int) -> str:
    """The score kernel(s) h2o_prefill_scores launches for this workload (see prefill_launches)."""
    if w.dtype != "bf16":
        return "prefill_row_stats_kernel, prefill_colsum_kernel (CUDA cores)"
    if prefill_launches(w, sms) == 2:
        return "prefill_tc_kernel<D, one pass>"
    return "prefill_tc_kernel<D, row stats>, prefill_tc_kernel<D, column sums>"


def prefill_scores_timing(h2o, dims, w, q, k, stream, dev, warmup: int, reps: int) -> dict:
    """h2o_prefill_scores (P1-P2, the tensor-core score pass) alone: one CUDA graph of the call replayed
    back to back, CUDA events on the launching stream. Its rate counts the causal QK^T the method needs
    once (P (P + 1) / 2 keys x D x 2 flops per unit, whatever the kernels issue) against the measured
    bf16 peak, and its DRAM rate the algorithmic bytes Q + K (the prompts exceed L2 on every workload
    this is reported for)."""
    import torch
    U, P, D = w.units, w.prompt_len, w.head_dim
    colsum = torch.empty((U, P), dtype=torch.float32, device=dev)
    ws = torch.empty(h2o.h2o_prefill_workspace_bytes(dims, P), dtype=torch.uint8, device=dev)
    sp = stream.cuda_stream

    def fn():
        h2o.h2o_prefill_scores(dims, P, q, k, colsum, ws, sp)

    with torch.cuda.stream(stream):
        fn()
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
        ev[0].record(stream)
        for _ in range(reps):
            g.replay()
        ev[1].record(stream)
    torch.cuda.synchronize(dev)
    if h2o.h2o_get_device_error(sp) != 0:
        raise RuntimeError("device error word set during the prefill score timing")
    us = ev[0].elapsed_time(ev[1]) * 1000.0 / reps
    peaks, peak_kind = measured_peaks()
    flops = float(U) * P * (P + 1) / 2 * D * 2
    qk_bytes = 2.0 * U * P * D * w.elem_bytes
    tflops = flops / (us * 1e-6) / 1e12
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    del colsum, ws
    return {"us": us, "kernels": prefill_score_kernels(w, sms), "causal_qk_gflop": flops / 1e9,
            "tflops": tflops, "bf16_peak_tflops": peaks["bf16_tflops"], "frac_of_bf16_peak": tflops / peaks["bf16_tflops"],
            "dram_gbs": qk_bytes / (us * 1e-6) / 1e9, "frac_of_hbm": qk_bytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"],
            "peak_source": f"{peak_kind} bf16_tflops (burst) and hbm_gbs",
            "how": f"CUDA graph of one h2o_prefill_scores call, {reps} replays after {warmup}, CUDA events"}


def prefill_forward_timing(h2o, dims, w, dv, cache, stream, dev, warmup: int, reps: int) -> dict:
    """h2o_prefill_forward (cache + the prompt's attention output) against h2o_prefill_select,
    replayed from CUDA graphs and timed with CUDA events on the launching stream."""
    import torch
    P, D, U = w.prompt_len, w.head_dim, w.units
    out = torch.empty((U, P, D), dtype=dv["q_prompt"].dtype, device=dev)
    sp = stream.cuda_stream

    def fwd():
        h2o.h2o_prefill_forward(dims, None, P, dv["q_prompt"], dv["k_prompt"], dv["v_prompt"], out,
                                cache.k_cache, cache.v_cache, cache.scores, cache.slot_pos,
                                cache.workspace, sp)

    def sel():
        h2o.h2o_prefill_select(dims, P, dv["q_prompt"], dv["k_prompt"], dv["v_prompt"], cache.k_cache,
                               cache.v_cache, cache.scores, cache.slot_pos, cache.workspace, sp)

    times = {}
    for name, fn in (("forward", fwd), ("select", sel)):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                g.replay()
            ev[0].record(stream)
            for _ in range(reps):
                g.replay()
            ev[1].record(stream)
        torch.cuda.synchronize(dev)
        times[name] = ev[0].elapsed_time(ev[1]) / reps
    if h2o.h2o_get_device_error(sp) != 0:
        raise RuntimeError("device error word set during the prefill-forward timing")
    flops = 2.0 * D * P * (P + 1) * U  # causal Q K^T and P V: 2 D flops per (query, key <= query) each
    return {"ms": times["forward"], "prefill_select_ms": times["select"],
            "output_extra_ms": times["forward"] - times["select"],
            "attention_tflops": flops / (times["forward"] / 1e3) / 1e12,
            "kernels": "prefill_tc_kernel<D, row stats + output>, prefill_tc_kernel<D, column sums>, "
                       "prefill_select_kernel" if w.dtype == "bf16" else "CUDA-core prefill kernels",
            "output_bytes": U * P * D * w.elem_bytes}


def e2e(args, w, calls, host, stream, dev, world, tokens_per_job):
    """The job end to end through the public API from pinned host buffers. Three streams: host->device
    copies, the library calls, device->host copies. Device inputs and outputs are double-buffered,
    so job j + 1's inputs are copied while job j decodes; each copy waits only for the launches that
    last used its buffer (events), and each decode chunk waits only for its own inputs. The library
    calls of each buffer set (the prefill, and each chunk's steps of one launch per layer) are
    captured once into CUDA graphs, as a serving loop would, and replayed every job: the 16,384
    per-layer calls of a job would otherwise be bound by the host."""
    import torch
    U, D, P, S = w.units, w.head_dim, w.prompt_len, w.decode_steps
    tdt = calls.cache.dtype
    chunk = 64
    chunks = list(range(0, S, chunk))
    h2d_s = torch.cuda.Stream(device=dev)
    d2h_s = torch.cuda.Stream(device=dev)
    prompt_keys, dec_keys = ("q_prompt", "k_prompt", "v_prompt"), ("q_dec", "k_dec", "v_dec")
    sets = [{"in": {k: torch.empty_like(host[k], device=dev) for k in prompt_keys + dec_keys},
             "out": torch.empty((S, U, D), dtype=tdt, device=dev),
             "evs": torch.empty((S, U), dtype=torch.int32, device=dev),
             "evp": torch.empty((S, U), dtype=torch.int32, device=dev),
             "inputs_free": None, "outputs_free": None} for _ in range(2)]
    h_out = torch.empty((S, U, D), dtype=tdt, pin_memory=True)
    h_evs = torch.empty((S, U), dtype=torch.int32, pin_memory=True)
    h_evp = torch.empty((S, U), dtype=torch.int32, pin_memory=True)
    sp = stream.cuda_stream
    h2d = sum(host[k].numel() * host[k].element_size() for k in host)
    d2h = h_out.numel() * h_out.element_size() + 2 * h_evs.numel() * 4

    def event(on):
        e = torch.cuda.Event()
        e.record(on)
        return e

    def issue_prefill(b):
        d = b["in"]
        calls.prefill(P, d["q_prompt"], d["k_prompt"], d["v_prompt"], sp)

    def issue_chunk(b, c0):
        d = b["in"]
        for s in range(c0, min(S, c0 + chunk)):
            calls.decode(P + s, d["q_dec"][s], d["k_dec"][s], d["v_dec"][s], b["out"][s], b["evs"][s], b["evp"][s],
                         sp, last=s == S - 1)

    for b in sets:  # real inputs in both sets, one direct run each, then the graphs
        for k in host:
            b["in"][k].copy_(host[k])
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            issue_prefill(b)
            for c0 in chunks:
                issue_chunk(b, c0)
        torch.cuda.synchronize(dev)
        b["g_pre"] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(b["g_pre"], stream=stream):
            issue_prefill(b)
        b["g_chunks"] = []
        for c0 in chunks:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                issue_chunk(b, c0)
            b["g_chunks"].append(g)

    def job(j):
        b = sets[j % 2]
        d = b["in"]
        if b["inputs_free"] is not None:
            h2d_s.wait_event(b["inputs_free"])
        with torch.cuda.stream(h2d_s):
            for k in prompt_keys:
                d[k].copy_(host[k], non_blocking=True)
            prompt_ready = event(h2d_s)
            ready = []
            for c0 in chunks:
                for k in dec_keys:
                    d[k][c0:c0 + chunk].copy_(host[k][c0:c0 + chunk], non_blocking=True)
                ready.append(event(h2d_s))
        stream.wait_event(prompt_ready)
        if b["outputs_free"] is not None:
            stream.wait_event(b["outputs_free"])
        with torch.cuda.stream(stream):
            b["g_pre"].replay()
        for ci, c0 in enumerate(chunks):
            stream.wait_event(ready[ci])
            with torch.cuda.stream(stream):
                b["g_chunks"][ci].replay()
            done = event(stream)
            d2h_s.wait_event(done)
            with torch.cuda.stream(d2h_s):
                sl = slice(c0, min(S, c0 + chunk))
                h_out[sl].copy_(b["out"][sl], non_blocking=True)
                h_evs[sl].copy_(b["evs"][sl], non_blocking=True)
                h_evp[sl].copy_(b["evp"][sl], non_blocking=True)
        b["inputs_free"] = done
        b["outputs_free"] = event(d2h_s)

    for j in range(args.warmup):
        job(j)
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = time.perf_counter()
    for j in range(args.steps):
        job(args.warmup + j)
    torch.cuda.synchronize(dev)
    dt = time.perf_counter() - t0
    dt = max_over_ranks(dt, world)
    return {"value": world * tokens_per_job * args.steps / dt, "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": 1000.0 * dt / args.steps,
            "how": "pinned host inputs copied per job on a host-to-device stream in 64-step chunks, the "
                   "outputs and eviction indices back per chunk on a device-to-host stream; device "
                   "buffers double-buffered so the next job's inputs arrive during this job's decode; "
                   "the library calls of each buffer set captured once into CUDA graphs (prefill, and "
                   "per chunk the steps' per-layer launches) and replayed per job; host wall clock "
                   "around the jobs, synchronised at both ends"}

if __name__ == "__main__":
    main()
