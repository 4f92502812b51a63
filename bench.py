"""Relay-pass HBM throughput of the sharded relay collectives on GB300.

Default workload: allreduce with A=2 active ranks of R=8 (6 helpers), bf16 payload
with fp32 accumulation, scale 1/2 (AVG), 1 GiB per rank (2^29 elements), on the
relay schedule the planner picks at that size (numChunks = H+2 = 8, reduce at the
helpers). One step is one relay_allreduce call: every pass of the schedule.

`value` = algorithmic bytes (read + written, summed over the schedule's passes, as
`relay_plan_passes` reports them) of all steps on all GPUs / the slowest rank's time.
Inputs are 1 GiB per rank, far above the 126 MiB L2, so no flush is needed between
steps. `e2e` is the same metric through the same public call with the inputs copied
in from pinned host memory and the outputs copied back inside the timed region.

`python bench.py [--gpus N --steps K --warmup W] [--impl reference]`. Under
torchrun each rank runs an independent replica (the path has no cross-GPU step).
`--impl reference` times the CPU oracle (the plain C restatement of the collective's
result) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

A, R = 2, 8
COUNT = 1 << 29              # elements per rank (bf16: 1 GiB)
SCALE = 0.5
WORKLOAD = "allreduce A=2 of R=8, bf16 (fp32 accumulate), 1 GiB per rank, scale 1/2"
CPU_SAMPLE = 1 << 24         # elements per rank in one step of the reference arm
CPU_BASELINE_SAMPLE = 1 << 27  # elements per rank of the bench's own CPU-baseline leg
PROFILE = os.path.join(ROOT, "profiles", "relay_pass_kernel_allreduce_a2_bf16_1g.json")
KERNEL_SRC = os.path.join(ROOT, "pack_virtual_rank_gb300", "csrc", "passes.cu")
KERNEL_HDR = os.path.join(ROOT, "pack_virtual_rank_gb300", "csrc", "program.h")
KERNEL_DEV = os.path.join(ROOT, "pack_virtual_rank_gb300", "csrc", "device.cuh")
HOST_SIDE_MARK = "// ------------------------------------------------------------------- host side --"


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _theoretical_hbm_gbs(dev):
    """The device's own figure: 2 transfers per memory clock x bus width (None where this
    PyTorch does not expose the clock or the width)."""
    import ctypes
    import torch
    pr = torch.cuda.get_device_properties(dev)
    khz, bits = getattr(pr, "memory_clock_rate", 0), getattr(pr, "memory_bus_width", 0)
    if not khz or not bits:
        # older PyTorch: ask the CUDA runtime (memory clock in kHz = attribute 36, global
        # memory bus width in bits = attribute 37)
        for name in ("libcudart.so", "/usr/local/cuda/lib64/libcudart.so"):
            try:
                rt = ctypes.CDLL(name)
            except OSError:
                continue
            v36, v37 = ctypes.c_int(0), ctypes.c_int(0)
            idx = dev.index if hasattr(dev, "index") and dev.index is not None else 0
            if rt.cudaDeviceGetAttribute(ctypes.byref(v36), 36, idx) == 0 and \
                    rt.cudaDeviceGetAttribute(ctypes.byref(v37), 37, idx) == 0:
                khz, bits = v36.value, v37.value
            break
    if not khz or not bits:
        return None
    return round(2 * khz * 1e3 * bits / 8 / 1e9, 1)


def kernel_code_sha() -> str:
    """First 16 hex digits of the SHA-256 of the per-pass kernels' code: the segment layout
    and tile constants (program.h), the shared device primitives (device.cuh) and the device
    part of passes.cu (everything before its host-side section), with comments removed and
    every run of whitespace folded to one space. An edit to a comment, to the host-side
    launch code or to another kernel's file keeps the recorded counters; any change to what
    these kernels execute voids them."""
    src = open(KERNEL_SRC).read()
    cut = src.find(HOST_SIDE_MARK)
    if cut >= 0:
        src = src[:cut]
    text = open(KERNEL_HDR).read() + "\n" + open(KERNEL_DEV).read() + "\n" + src
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    text = " ".join(text.split())
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def _profiled_traffic():
    """Per-launch DRAM bytes of each pass of the bench workload from the committed ncu
    counters (a small JSON file beside the profile summary), or None when the kernels'
    code changed since the counters were taken."""
    sha = kernel_code_sha()
    try:
        with open(PROFILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None, sha
    if rec.get("kernel_code_sha256_16") != sha:
        return None, sha
    return {k: int(v) for k, v in rec.get("traffic_bytes_per_launch", {}).items()}, sha


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region.
    summary() covers every sample; window(t0, t1) only those taken between two
    time.time() readings (each sample carries nvidia-smi's local-time timestamp)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, enabled: bool = True, period_ms: int = 100):
        self.proc = None
        self.enabled = enabled
        self.gpu = gpu_index
        self.period_ms = period_ms
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        if not self.enabled:
            return self
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def _samples(self):
        """(unix time, sm MHz, max MHz, active reasons) of every sample so far."""
        import datetime
        if self.proc is None:
            return []
        self.out.flush()
        with open(self.out.name) as f:
            text = f.read()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for line in text.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, mx = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            rows.append((ts, sm, mx, {nm for nm, v in zip(names, parts[6:10])
                                      if v.lower() == "active"}))
        return rows

    @staticmethod
    def _stats(rows):
        if not rows:
            return None
        return {"sm_mhz": statistics.median(r[1] for r in rows),
                "sm_max_mhz": max(r[2] for r in rows), "samples": len(rows),
                "reasons": sorted(set().union(*(r[3] for r in rows)))}

    def window(self, t0, t1):
        """Clock summary of the samples taken between unix times t0 and t1."""
        return self._stats([r for r in self._samples() if t0 <= r[0] <= t1])

    def summary(self):
        rows = self._samples()
        self.out.close()
        try:
            os.unlink(self.out.name)
        except OSError:
            pass
        return self._stats(rows)


def _cpu_oracle(sample: int, seed_config: int = 2, inputs=None):
    """Time the oracle's allreduce on `sample` elements per rank (host cores). `inputs`:
    host copies of the workload's own inputs, of which the first `sample` are used."""
    import oracle as orc
    import synth
    if inputs is None:
        xs = [synth.to_numpy(synth.rank_input(seed_config, r, sample, "bf16")) for r in range(A)]
    else:
        xs = [synth.to_numpy(x[:sample]) for x in inputs]
    t0 = time.perf_counter()
    orc.allreduce(orc.BF16, xs, SCALE)
    return time.perf_counter() - t0


def _host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _cpu_model():
    """The host CPU as /proc/cpuinfo names it (x86: model name; Arm: implementer/part)."""
    import platform
    try:
        info = open("/proc/cpuinfo").read().split("\n")
    except OSError:
        return platform.machine()
    for key in ("model name", "Model"):
        for ln in info:
            if ln.split(":")[0].strip() == key:
                return ln.split(":", 1)[1].strip()
    parts = {ln.split(":")[0].strip(): ln.split(":", 1)[1].strip() for ln in info if ":" in ln}
    return f"{platform.machine()} implementer {parts.get('CPU implementer', '?')} " \
           f"part {parts.get('CPU part', '?')}"


def _cpu_oracle_all_cores(sample: int, seed_config: int = 2, inputs=None):
    """The same oracle call on every host core at once: each thread runs the unchanged
    oracle allreduce on its own contiguous range of the sample's elements (elementwise
    collectives split by element without changing any result; the C call releases the
    GIL). Returns (seconds, threads)."""
    import concurrent.futures as cf
    import oracle as orc
    import synth
    if inputs is None:
        xs = [synth.to_numpy(synth.rank_input(seed_config, r, sample, "bf16")) for r in range(A)]
    else:
        xs = [synth.to_numpy(x[:sample]) for x in inputs]
    nt = _host_cores()
    cuts = [sample * t // nt for t in range(nt + 1)]
    orc.lib()
    with cf.ThreadPoolExecutor(nt) as ex:
        t0 = time.perf_counter()
        list(ex.map(lambda t: orc.allreduce(orc.BF16, xs, SCALE, cuts[t], cuts[t + 1]), range(nt)))
        dt = time.perf_counter() - t0
    return dt, nt


def _bind_near_gpu(dev):
    """Pin this process to the host cores the GPU's PCI function reports as local (sysfs
    local_cpulist), so that pinned host buffers allocated next sit in the memory next to
    the GPU's host link (the caller restores the affinity afterwards). Returns what was
    done, for the JSON line."""
    import torch
    pr = torch.cuda.get_device_properties(dev)
    dom, bus, slot = (getattr(pr, k, None) for k in ("pci_domain_id", "pci_bus_id", "pci_device_id"))
    if bus is not None and slot is not None:
        addr = f"{dom or 0:04x}:{bus:02x}:{slot:02x}.0"
    else:
        # older PyTorch: find the GPU by UUID in nvidia-smi's PCI listing
        try:
            out = subprocess.run(["nvidia-smi", "--query-gpu=uuid,pci.bus_id", "--format=csv,noheader"],
                                 capture_output=True, text=True, timeout=30).stdout
        except (OSError, subprocess.SubprocessError):
            return {"bound": False, "why": "no PCI location (nvidia-smi unavailable)"}
        want = str(getattr(pr, "uuid", "")).lower().replace("gpu-", "")
        addr = None
        for ln in out.splitlines():
            u, _, b = (x.strip() for x in ln.partition(","))
            if want and u.lower().replace("gpu-", "") == want:
                d, rest = b.split(":", 1)
                addr = f"{int(d, 16):04x}:{rest}".lower()
        if addr is None:
            return {"bound": False, "why": "GPU not found in nvidia-smi's PCI listing"}
    path = f"/sys/bus/pci/devices/{addr}/local_cpulist"
    try:
        spec = open(path).read().strip()
    except OSError:
        return {"bound": False, "why": f"no {path}"}
    cpus = set()
    for part in spec.split(","):
        if "-" in part:
            lo, hi = part.split("-")
            cpus.update(range(int(lo), int(hi) + 1))
        elif part:
            cpus.add(int(part))
    allowed = cpus & set(os.sched_getaffinity(0))
    if not allowed:
        return {"bound": False, "why": f"local cpus {spec} not in this process's set"}
    if allowed != set(os.sched_getaffinity(0)):
        os.sched_setaffinity(0, allowed)
    return {"bound": True, "local_cpulist": spec, "cpus": len(allowed)}


def _calibrate_link(rv, host_in, dev_in, dev_out, host_out, ctas):
    """Host-link rates on this GPU for the copy engines (torch copies) and for relay_copy
    with `ctas` CTAs, on the end-to-end leg's own transfers (every active's whole input in,
    every active's whole output out): each direction alone, then every pairing of the two
    directions running at once on two streams, as the leg runs them (median of 3). Returns
    (rates in GB/s, the fastest pairing)."""
    import torch
    pairs_in = list(zip(host_in, dev_in))
    pairs_out = list(zip(dev_out, host_out))

    def eng_in():
        for h, d in pairs_in:
            d.copy_(h, non_blocking=True)

    def ker_in():
        for h, d in pairs_in:
            rv.relay_copy(d, h, max_ctas=ctas)

    def eng_out():
        for d, h in pairs_out:
            h.copy_(d, non_blocking=True)

    def ker_out():
        for d, h in pairs_out:
            rv.relay_copy(h, d, max_ctas=ctas)

    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fin, fout):
        ts = []
        for rep in range(4):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            cur = torch.cuda.current_stream()
            e0.record(cur)
            for st, fn in ((s_in, fin), (s_out, fout)):
                if fn is None:
                    continue
                st.wait_event(e0)
                with torch.cuda.stream(st):
                    fn()
                cur.wait_stream(st)
            e1.record(cur)
            torch.cuda.synchronize()
            if rep:
                ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    gb_in = sum(h.numel() * h.element_size() for h in host_in) / 1e6
    gb_out = sum(h.numel() * h.element_size() for h in host_out) / 1e6
    out = {"h2d_engine_gbs": round(gb_in / timed(eng_in, None), 1),
           "h2d_kernel_gbs": round(gb_in / timed(ker_in, None), 1),
           "d2h_engine_gbs": round(gb_out / timed(None, eng_out), 1),
           "d2h_kernel_gbs": round(gb_out / timed(None, ker_out), 1)}
    pairs = {"torch": (eng_in, eng_out), "library-in": (ker_in, eng_out),
             "library-out": (eng_in, ker_out), "library": (ker_in, ker_out)}
    both = {m: timed(*fns) for m, fns in pairs.items()}
    for m, t in both.items():
        out[f"both_{m}_gbs_each"] = round(max(gb_in, gb_out) / t, 1)
    return out, min(both, key=both.get)


def _bytes_per_step(plan, rv, count=None):
    if count is not None and count != plan.count:
        plan = rv.relay_plan(rv.ALLREDUCE, count, rv.BF16, A, R)
    ps = rv.relay_plan_passes(plan)
    return sum(p["bytes_read"] + p["bytes_written"] for p in ps), ps


def slowest_rank(times_ms, world):
    """Max over ranks of each timing (replicas finish when the slowest one does)."""
    if world <= 1:
        return list(times_ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(times_ms), dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def whole_job_gbs(bytes_per_step, steps, world, ms):
    """Whole-job throughput: every replica's bytes over the slowest replica's time."""
    return bytes_per_step * steps * world / (ms / 1e3) / 1e9


def relay_allreduce_a2_bytes(g, esize):
    """Algorithmic bytes (read + written) of the 2-active relay allreduce's passes, from
    the oracle's plan `g` (chunk c, direct regions dirA and dirB, H helpers):
      group 1: each active sends H relay chunks and dirA: 2(H*c + dirA) read and written;
      group 2: each helper reads two slots and writes the reduced chunk to both actives
               (2c + 2c), each active sends dirB: 4*H*c + 4*dirB;
      active reduce: each active reads its own and the received dirA + dirB and writes
               the result: 6 (dirA + dirB).
    With dirA = dirB = c and H = 6 that is 68 c elements per call."""
    assert g["kind"] == 0 and g["A"] == 2, "relay schedule, 2 actives"
    H, c, da, db = g["H"], g["chunk"], g["dirA"], g["dirB"]
    elems = 4 * (H * c + da) + 4 * H * c + 4 * db + 6 * (da + db)
    return elems * esize


def run_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    g, _ = oracle.plan(oracle.AR, A, R, CPU_SAMPLE, 2)
    nbytes = relay_allreduce_a2_bytes(g, 2)
    for _ in range(args.warmup):
        _cpu_oracle(CPU_SAMPLE)
    ts = [_cpu_oracle(CPU_SAMPLE) for _ in range(args.steps)]
    total = sum(ts)
    value = nbytes * args.steps / total / 1e9
    t_all, cores = _cpu_oracle_all_cores(CPU_SAMPLE)
    sample = (f"oracle allreduce (bf16, A=2, fp32 sum, scale 1/2) on {CPU_SAMPLE} elements per "
              f"rank per step; GB/s counts the relay schedule's algorithmic bytes for that count")
    line = {"impl": "reference", "metric": "relay-pass HBM GB/s (allreduce A=2 of R=8, bf16)",
            "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16)",
            "config": {"workload": WORKLOAD, "sample_count": CPU_SAMPLE, "A": A, "R": R},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", "sample": sample, "cpu_model": _cpu_model(),
                             "all_cores": {"value": round(nbytes / t_all / 1e9, 3),
                                           "cores": cores,
                                           "how": "one step's sample split into one contiguous "
                                                  "element range per host thread, each running "
                                                  "the unchanged oracle"}},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def run_ours(args):
    rank, world, local = _dist()
    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("gloo")
    import pack_virtual_rank_gb300.build as b
    if rank == 0 or world == 1:
        b.build()
    if world > 1:
        dist.barrier()
    import pack_virtual_rank_gb300 as rv
    import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    count = args.count
    plan = rv.relay_plan(rv.ALLREDUCE, count, rv.BF16, A, R)
    nbytes, passes = _bytes_per_step(plan, rv)
    npass = len(passes)
    launches_per_step = sum((p["num_segments"] + 383) // 384 for p in passes)

    xs = [synth.rank_input(2, r, count, "bf16", device=dev) for r in range(A)]
    ys = [torch.empty_like(x) for x in xs]
    scratch = rv.alloc_scratch(plan, dev)
    send = xs + [None] * (R - A)
    recv = ys + [None] * (R - A)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()

    # per-pass events of every timed step; the warm-up steps run the same call (pass events
    # and all), so that everything the timed steps launch is loaded and warm beforehand
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(npass + 1)]
          for _ in range(args.steps)]
    opts = [rv.make_opts(pass_events=e) for e in ev]
    for k in range(args.warmup):
        rv.relay_allreduce(send, recv, scratch, count, rv.BF16, A, R, SCALE, opts[k % args.steps])
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with Clocks(local, enabled=not args.kernel_only) as clk:
        barrier()
        start.record(stream)
        for k in range(args.steps):
            rv.relay_allreduce(send, recv, scratch, count, rv.BF16, A, R, SCALE, opts[k])
        stop.record(stream)
        barrier()
    ms = start.elapsed_time(stop)
    clocks = clk.summary()
    per_pass = [statistics.mean(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(args.steps))
                for i in range(npass)]

    # the same steps under the library's default launch policy (no pass events: one chained
    # launch per call, each CTA running a tile's producers and consumers in pass order)
    for _ in range(args.warmup):
        rv.relay_allreduce(send, recv, scratch, count, rv.BF16, A, R, SCALE)
    default_form = rv.last_launch()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with Clocks(local, enabled=not args.kernel_only) as clk_d:
        barrier()
        d0.record(stream)
        for k in range(args.steps):
            rv.relay_allreduce(send, recv, scratch, count, rv.BF16, A, R, SCALE)
        d1.record(stream)
        barrier()
    default_ms = d0.elapsed_time(d1)
    default_clocks = clk_d.summary()

    # and once more with every scratch line written back to memory (RELAY_FLAG_KEEP_SCRATCH):
    # what dropping the chained launch's dead scratch lines from L2 saves
    keep = rv.make_opts(flags=rv.FLAG_KEEP_SCRATCH)
    for _ in range(args.warmup):
        rv.relay_allreduce(send, recv, scratch, count, rv.BF16, A, R, SCALE, keep)
    keep_form = rv.last_launch()
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with Clocks(local, enabled=not args.kernel_only) as clk_k:
        barrier()
        k0.record(stream)
        for k in range(args.steps):
            rv.relay_allreduce(send, recv, scratch, count, rv.BF16, A, R, SCALE, keep)
        k1.record(stream)
        barrier()
    keep_ms = k0.elapsed_time(k1)
    keep_clocks = clk_k.summary()

    # every other workload of the metric at one size, timed the same way with its own
    # clock record (rank 0 only: replicas add nothing to a per-collective table)
    per_wl = None
    if rank == 0 and count == COUNT and not args.kernel_only and not args.no_per_workload:
        with Clocks(local) as clk_wl:
            per_wl = run_per_workload(rv, synth, dev, args.steps, args.warmup, _peaks()[0], clk_wl)
        clk_wl.summary()

    # end to end: every step copies its inputs in from pinned host memory, runs the same
    # public call, and copies its results back to pinned host memory. Two device buffer
    # sets let step k+1's input copy and step k-1's result copy overlap step k's passes
    # (copy-in, compute and copy-out each on their own stream, ordered by events).
    # as many end-to-end steps as timed steps: the pipeline's first input copy and last
    # output copy run alone, and more steps spread that over more work
    e2e_ms, e2e_steps, calib = None, max(2, args.steps), None
    host_numa = None
    if not args.kernel_only:
        cpus_before = os.sched_getaffinity(0)
        host_numa = _bind_near_gpu(dev)
        hx = [x.cpu().pin_memory() for x in xs]
        hy = [torch.empty(count, dtype=torch.bfloat16).pin_memory() for _ in range(A)]
        os.sched_setaffinity(0, cpus_before)   # the buffers stay where they were placed
        sets = [(xs, ys), ([torch.empty_like(x) for x in xs], [torch.empty_like(y) for y in ys])]
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        # host-link copies: the library's kernel with half a CTA per SM (it reaches the
        # link's rate and leaves the other CTA slots to the passes), or the copy engines
        link_ctas = args.e2e_ctas or max(1, torch.cuda.get_device_properties(dev).multi_processor_count // 2)
        e2e_mode, calib = args.e2e_copy, None
        if e2e_mode == "auto":
            calib, e2e_mode = _calibrate_link(rv, hx, xs, ys, hy, link_ctas)
        def pipeline(mode, steps):
            """`steps` end-to-end steps, copies done the `mode` way; returns ms."""
            ev = lambda: torch.cuda.Event()
            done_in = [ev() for _ in range(steps)]
            done_comp = [ev() for _ in range(steps)]
            done_out = [ev() for _ in range(steps)]
            barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            s_in.wait_stream(stream)
            s_out.wait_stream(stream)
            for k in range(steps):
                bx, by = sets[k % 2]
                with torch.cuda.stream(s_in):
                    if k >= 2:
                        s_in.wait_event(done_comp[k - 2])   # set k%2's inputs are free again
                    for a in range(A):
                        if mode in ("torch", "library-out"):
                            bx[a].copy_(hx[a], non_blocking=True)
                        else:
                            rv.relay_copy(bx[a], hx[a], max_ctas=link_ctas, stream=s_in)
                    done_in[k].record(s_in)
                stream.wait_event(done_in[k])
                if k >= 2:
                    stream.wait_event(done_out[k - 2])      # set k%2's outputs were copied out
                rv.relay_allreduce(bx + [None] * (R - A), by + [None] * (R - A), scratch, count,
                                   rv.BF16, A, R, SCALE, stream=stream)
                done_comp[k].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done_comp[k])
                    for a in range(A):
                        if mode in ("library", "library-out"):
                            rv.relay_copy(hy[a], by[a], max_ctas=link_ctas, stream=s_out)
                        else:
                            hy[a].copy_(by[a], non_blocking=True)
                    done_out[k].record(s_out)
            stream.wait_event(done_out[steps - 1])
            e1.record(stream)
            barrier()
            return e0.elapsed_time(e1)

        if args.e2e_copy == "auto":
            # the pipeline itself, 3 steps per way of copying, twice in turn, outside the
            # timed region; each way is scored by its slower trial. On some boxes the copy
            # engines slow down several-fold inside the pipeline, and not steadily, which the
            # single- and paired-copy rates alone do not predict.
            modes = ("torch", "library-in", "library-out", "library")
            trials = {m: [] for m in modes}
            for _ in range(2):
                for m in modes:
                    trials[m].append(pipeline(m, 3))
            calib["pipeline_3_steps_ms"] = {m: [round(t, 2) for t in ts] for m, ts in trials.items()}
            e2e_mode = min(modes, key=lambda m: max(trials[m]))
        e2e_ms = pipeline(e2e_mode, e2e_steps)
        del sets

    ms, e2e_ms, default_ms = slowest_rank([ms, e2e_ms if e2e_ms is not None else 0.0, default_ms],
                                          world)

    if rank == 0:
        peak, peak_kind = _peaks()
        theo = _theoretical_hbm_gbs(dev)
        # end-to-end ceiling: each direction's bytes at the faster calibrated single-direction
        # rate, both directions at once (full duplex, no interference: an upper bound)
        link_ceiling = link_pair = None
        if calib:
            t_in = A * count * 2 / (max(calib["h2d_engine_gbs"], calib["h2d_kernel_gbs"]) * 1e9)
            t_out = A * count * 2 / (max(calib["d2h_engine_gbs"], calib["d2h_kernel_gbs"]) * 1e9)
            link_ceiling = round(nbytes / max(t_in, t_out) / 1e9, 1)
            # the same with both directions at the rate the chosen pairing reached together
            pair_rate = calib[f"both_{e2e_mode}_gbs_each"] * 1e9
            link_pair = round(nbytes / (A * count * 2 / pair_rate) / 1e9, 1)
        value = whole_job_gbs(nbytes, args.steps, world, ms)
        e2e = whole_job_gbs(nbytes, e2e_steps, world, e2e_ms) if e2e_ms else None
        top = max(range(npass), key=lambda i: per_pass[i])
        top_bytes = passes[top]["bytes_read"] + passes[top]["bytes_written"]
        achieved = top_bytes / (per_pass[top] / 1e3) / 1e9
        traffic, _sha = _profiled_traffic()
        tr = traffic.get(passes[top]["name"]) if traffic else None
        sample = min(CPU_BASELINE_SAMPLE, count)
        cpu_t = None if args.kernel_only else _cpu_oracle(sample, inputs=hx)
        cpu_all = None if args.kernel_only else _cpu_oracle_all_cores(sample, inputs=hx)
        cpu_bytes, _ = _bytes_per_step(plan, rv, sample)
        cpu_val = cpu_bytes / cpu_t / 1e9 if cpu_t else None
        line = {
            "metric": "relay-pass HBM GB/s (allreduce A=2 of R=8, bf16)",
            "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16, generated on the device)",
            "config": {"workload": WORKLOAD if count == COUNT else
                       f"allreduce A=2 of R=8, bf16, {count} elements per rank (profiling case)",
                       "count": count, "A": A, "R": R,
                       "schedule": ["relay", "zero_chunk", "direct", "legacy"][plan.kind],
                       "numChunks": plan.H + 2, "chunk": plan.chunk,
                       "l2": "inputs larger than L2 (1 GiB per rank); no flush",
                       "bytes_per_step": nbytes, "parallelism": f"replicas x{world}"},
            "passes": {p["name"]: {"ms": round(t, 4), "bytes": p["bytes_read"] + p["bytes_written"],
                                   "gbs": round((p["bytes_read"] + p["bytes_written"]) / t / 1e6, 1),
                                   "frac": round((p["bytes_read"] + p["bytes_written"]) / t / 1e6
                                                 / peak, 4)}
                       for p, t in zip(passes, per_pass)},
            "roofline": {"kernel": f"relay_pass_kernel ({passes[top]['name']})", "bound": "hbm",
                         "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": tr,
                         "peak_source": f"{peak_kind} hbm_gbs (copy, burst)",
                         "hbm_theoretical_gbs": theo,
                         "frac_of_theoretical": None if not theo else round(achieved / theo, 4),
                         "algorithmic_bytes_per_launch": top_bytes},
            "cpu_baseline": None if cpu_t is None else {
                "value": round(cpu_val, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                "sample": f"oracle allreduce on the first {sample} elements of each rank's "
                          f"bench input ({cpu_t:.2f} s); GB/s counts the relay schedule's "
                          "algorithmic bytes for that count",
                "cpu_model": _cpu_model(),
                "all_cores": {"value": round(cpu_bytes / cpu_all[0] / 1e9, 3), "cores": cpu_all[1],
                              "seconds": round(cpu_all[0], 3),
                              "how": "the same sample split into one contiguous element range "
                                     "per host thread, each running the unchanged oracle"}},
            "e2e": None if e2e is None else {
                "value": round(e2e, 2), "unit": "GB/s", "h2d_bytes_per_step": A * count * 2,
                "d2h_bytes_per_step": A * count * 2, "steps": e2e_steps,
                "note": "pinned host inputs copied in and results copied out every step; "
                        "two device buffer sets overlap the copies with the passes",
                "link_ceiling_gbs": link_ceiling,
                "frac_of_link_ceiling": None if not link_ceiling else round(e2e / link_ceiling, 3),
                "link_pair_bound_gbs": link_pair,
                "host_placement": host_numa,
                "frac_of_link_pair_bound": None if not link_pair else round(e2e / link_pair, 3),
                "copies": {"library": "relay_copy both ways",
                           "library-in": "relay_copy in, copy engine out",
                           "library-out": "copy engine in, relay_copy out",
                           "torch": "copy engines both ways"}[e2e_mode]
                          + ("" if e2e_mode == "torch" else f" ({link_ctas} CTAs)")
                          + ("" if calib is None else
                             ", the fastest way in a 3-step trial of the pipeline on this GPU "
                             "(calibration outside the timed region: " + json.dumps(calib) + ")")},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "default_path": {
                "launch": default_form, "ms_per_step": round(default_ms / args.steps, 4),
                "value": round(whole_job_gbs(nbytes, args.steps, world, default_ms), 2),
                "unit": "GB/s",
                "frac": round(whole_job_gbs(nbytes, args.steps, world, default_ms) / world / peak, 4),
                "note": "the same steps without pass events, under the library's default launch "
                        "policy; the same algorithmic bytes per step. A chained launch runs each "
                        "tile's producer and consumer passes in one CTA, so the consumers' reads "
                        "of what their producers just wrote are served from L2, and the scratch "
                        "lines its last consumer has read are dropped from L2 unwritten: DRAM "
                        "traffic is below the algorithmic bytes and the fraction may exceed 1",
                "clocks": default_clocks,
                "keep_scratch": {
                    "launch": keep_form, "ms_per_step": round(keep_ms / args.steps, 4),
                    "value": round(whole_job_gbs(nbytes, args.steps, world, keep_ms), 2),
                    "frac": round(whole_job_gbs(nbytes, args.steps, world, keep_ms) / world / peak, 4),
                    "note": "the same chained steps with RELAY_FLAG_KEEP_SCRATCH: every scratch "
                            "line is written back to memory",
                    "clocks": keep_clocks}},
        }
        if per_wl is not None:
            head = {"workload": "2: allreduce A=2 of R=8, bf16, 1 GiB per rank (the headline above)",
                    "collective": "allreduce", "A": A, "R": R, "dtype": "bf16", "count": count,
                    "schedule": line["config"]["schedule"], "bytes_per_call": nbytes,
                    "calls_timed": args.steps, "ms": round(ms / args.steps, 5),
                    "gbs": round(nbytes / (ms / args.steps) / 1e6, 1),
                    "frac": round(nbytes / (ms / args.steps) / 1e6 / peak, 4),
                    "timing": "back-to-back calls, pass events, inputs larger than L2",
                    "clocks": clocks, "passes": line["passes"]}
            line["per_workload"] = [per_wl[0], head] + per_wl[1:]
        print(json.dumps(line))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


MB = 1 << 20


def per_workload_points():
    """One size of each workload the metric names, at the top of its range, plus the odd
    segmentCount the all-to-all workload asks for: (label, collective, A, dtype, count,
    schedule). count is the collective's own count (allreduce: elements per rank;
    reduce-scatter: recvCount; all-gather: sendCount; all-to-all: segmentCount)."""
    return [
        ("1: allreduce A=2 of R=8, fp32, 65536 elements, relay forced",
         "allreduce", 2, "f32", 65536, "relay"),
        ("3: reduce-scatter A=2 of R=8, fp32, 512 MB of input per rank",
         "reduce_scatter", 2, "f32", 512 * MB // 4 // 2, "auto"),
        ("3: reduce-scatter A=2 of R=8, int32, 512 MB of input per rank",
         "reduce_scatter", 2, "i32", 512 * MB // 4 // 2, "auto"),
        ("4: allreduce A=4 of R=8, bf16, 1 GiB per rank",
         "allreduce", 4, "bf16", 1024 * MB // 2, "auto"),
        ("4: reduce-scatter A=4 of R=8 (flat, fp32 partial), bf16, 1 GiB of input per rank",
         "reduce_scatter", 4, "bf16", 1024 * MB // 2 // 4, "auto"),
        ("5: all-gather A=4 of R=8, bf16, 1 GiB per rank",
         "all_gather", 4, "bf16", 1024 * MB // 2, "relay"),
        ("5: all-gather A=4 of R=8, int32, 1 GiB per rank",
         "all_gather", 4, "i32", 1024 * MB // 4, "relay"),
        ("5: all-to-all A=4 of R=8, bf16, 1 GiB workload count (segmentCount = count/12)",
         "all_to_all", 4, "bf16", 1024 * MB // 2 // 12, "relay"),
        ("5: all-to-all A=4 of R=8, bf16, 1 GiB workload count, odd segmentCount",
         "all_to_all", 4, "bf16", 1024 * MB // 2 // 12 + 1, "relay"),
        ("5: all-to-all A=4 of R=8, int32, 1 GiB workload count (odd segmentCount)",
         "all_to_all", 4, "i32", 1024 * MB // 4 // 12, "relay"),
    ]


def run_per_workload(rv, synth, dev, steps, warmup, peak, clk, min_window_s=0.3):
    """Each per_workload_points() entry timed on the device like the headline: warm-up
    calls, then rounds of `steps` calls, each call recording CUDA events before every pass
    and after the last, until at least `min_window_s` has passed so that the clock
    sampler sees the timed window. Calls whose buffers fit twice in L2 run one call per
    timed window after a flush (a buffer twice the L2 written, another read), timed around
    the call as a user makes it (the library's default launch policy, no pass events);
    larger ones run back to back (their inputs exceed L2)."""
    import torch
    colls = {"allreduce": rv.ALLREDUCE, "reduce_scatter": rv.REDUCE_SCATTER,
             "all_gather": rv.ALL_GATHER, "all_to_all": rv.ALL_TO_ALL}
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    flush_read = torch.ones(2 * l2 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    out = []
    for label, name, Ap, dt, count, sched in per_workload_points():
        coll, d = colls[name], rv.dtype_code(dt)
        opts0 = rv.make_opts(schedule=rv.SCHEDULE_RELAY if sched == "relay" else rv.SCHEDULE_AUTO)
        plan = rv.relay_plan(coll, count, d, Ap, R, opts0)
        passes = rv.relay_plan_passes(plan)
        nbytes = sum(q["bytes_read"] + q["bytes_written"] for q in passes)
        xs = [synth.rank_input(9, r, plan.input_elems, dt, device=dev) for r in range(Ap)]
        ys = [torch.empty(plan.output_elems, dtype=xs[0].dtype, device=dev) for _ in range(Ap)]
        scratch = rv.alloc_scratch(plan, dev)
        scale = 1.0 if (d == rv.I32 or coll in (rv.ALL_GATHER, rv.ALL_TO_ALL)) else 1.0 / Ap
        fn = rv.COLLECTIVES[coll]
        a0 = (xs + [None] * (R - Ap), ys + [None] * (R - Ap), scratch, count, d, Ap, R)

        def call(o):
            if coll in (rv.ALLREDUCE, rv.REDUCE_SCATTER):
                fn(*a0, scale, o)
            else:
                fn(*a0, o)
        working = sum(x.numel() * x.element_size() for x in xs + ys)
        small = working <= 2 * l2
        # warm-up: the call exactly as it is timed (pass events for the large ones)
        wev = [torch.cuda.Event(enable_timing=True) for _ in range(len(passes) + 1)]
        wopts = opts0 if small else rv.make_opts(schedule=opts0.schedule, pass_events=wev)
        for _ in range(warmup):
            call(wopts)
        torch.cuda.synchronize()
        per_call, per_pass, n_calls = [], [[] for _ in passes], 0
        t0 = time.time()
        total_ms, round_ms = 0.0, []
        while True:
            if small:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                for _ in range(steps):
                    flush.fill_(1.0)
                    flush_read.sum()
                    e0.record(stream)
                    call(opts0)
                    e1.record(stream)
                    torch.cuda.synchronize()
                    per_call.append(e0.elapsed_time(e1))
            else:
                ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(passes) + 1)]
                      for _ in range(steps)]
                ops = [rv.make_opts(schedule=opts0.schedule, pass_events=e) for e in ev]
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for k in range(steps):
                    call(ops[k])
                e1.record(stream)
                torch.cuda.synchronize()
                total_ms += e0.elapsed_time(e1)
                round_ms.append(e0.elapsed_time(e1) / steps)
                for k in range(steps):
                    for i in range(len(passes)):
                        per_pass[i].append(ev[k][i].elapsed_time(ev[k][i + 1]))
            n_calls += steps
            if time.time() - t0 >= min_window_s:
                break
        t1 = time.time()
        # large calls: the median over rounds of each round's time per call, so that a host
        # stall in one round (the GPU idles between calls) does not move the figure
        ms = statistics.median(per_call) if small else statistics.median(round_ms)
        gbs = nbytes / ms / 1e6
        row = {"workload": label, "collective": name, "A": Ap, "R": R, "dtype": dt, "count": count,
               "schedule": ["relay", "zero_chunk", "direct", "legacy"][plan.kind],
               "bytes_per_call": nbytes, "calls_timed": n_calls, "ms": round(ms, 5),
               "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
               "timing": ("median of single calls, each after an L2 flush, default launch "
                          "policy" if small else
                          "back-to-back calls, pass events, inputs larger than L2; median over "
                          "rounds of each round's time per call"),
               "clocks": clk.window(t0, t1) if clk is not None else None}
        if not small:
            row["rounds"] = len(round_ms)
            row["ms_mean_all_calls"] = round(total_ms / n_calls, 5)
        if small:
            # the same call captured in a CUDA graph: (a) one replay per timed window after
            # an L2 flush, timed around the replay (includes the graph launch); (b) 20 calls
            # in one graph replayed back to back, per call (warm L2, no host in the way)
            row["launch"] = rv.last_launch()
            s_g = torch.cuda.Stream()
            torch.cuda.synchronize()
            g1, g20 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            with torch.cuda.graph(g1, stream=s_g):
                call(opts0)
            with torch.cuda.graph(g20, stream=s_g):
                for _ in range(20):
                    call(opts0)
            g1.replay()
            g20.replay()
            torch.cuda.synchronize()
            rep = []
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            for _ in range(max(steps, 20)):
                flush.fill_(1.0)
                flush_read.sum()
                e0.record(stream)
                g1.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                rep.append(e0.elapsed_time(e1))
            e0.record(stream)
            for _ in range(5):
                g20.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            row["graph_replay_ms"] = round(statistics.median(rep), 5)
            row["graph_back_to_back_ms_per_call"] = round(e0.elapsed_time(e1) / 100, 5)
            del g1, g20
        if not small:
            # the same call under the library's default launch policy (no pass events:
            # one chained launch where the program allows it), back to back
            for _ in range(warmup):
                call(opts0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(steps):
                call(opts0)
            e1.record(stream)
            torch.cuda.synchronize()
            dms = e0.elapsed_time(e1) / steps
            row["default_path"] = {"launch": rv.last_launch(), "ms": round(dms, 5),
                                   "gbs": round(nbytes / dms / 1e6, 1),
                                   "frac": round(nbytes / dms / 1e6 / peak, 4)}
            row["passes"] = {}
            for q, ts in zip(passes, per_pass):
                b = q["bytes_read"] + q["bytes_written"]
                m = statistics.mean(ts)
                row["passes"][q["name"]] = {"ms": round(m, 5), "gbs": round(b / m / 1e6, 1),
                                            "frac": round(b / m / 1e6 / peak, 4)}
        out.append(row)
        del xs, ys, scratch, a0
        torch.cuda.empty_cache()
    del flush, flush_read
    torch.cuda.empty_cache()
    return out


def _sweep_points():
    """The five workloads of the metric at a spread of their sizes (bytes per rank)."""
    MB = 1 << 20
    pts = [("allreduce", 2, "f32", 65536 * 4, "relay")]
    pts += [("allreduce", 2, "bf16", b, "auto") for b in
            [64 * 1024, 256 * 1024, MB, 4 * MB, 16 * MB, 64 * MB, 256 * MB, 1024 * MB]]
    for dt in ("f32", "i32"):
        pts += [("reduce_scatter", 2, dt, b, "auto") for b in [2 * MB, 8 * MB, 32 * MB, 128 * MB, 512 * MB]]
    for coll in ("allreduce", "reduce_scatter"):
        pts += [(coll, 4, "bf16", b, "auto") for b in [MB, 4 * MB, 16 * MB, 64 * MB, 256 * MB, 1024 * MB]]
    for coll in ("all_gather", "all_to_all"):
        for dt in ("bf16", "i32"):
            pts += [(coll, 4, dt, b, "relay") for b in
                    [int(13.5 * MB), 54 * MB, 135 * MB, 512 * MB, 1024 * MB]]
    # the schedules the page retuned, executed for comparison: the three-group
    # numChunks = H+1 schedule (item 1, before) and the 780-permille offload (item 4)
    pts += [("allreduce", 2, "bf16", b, "legacy") for b in [64 * MB, 1024 * MB]]
    pts += [("reduce_scatter", 2, "f32", b, "legacy") for b in [128 * MB, 512 * MB]]
    pts += [("allreduce", 4, "bf16", b, "permille780") for b in [64 * MB, 1024 * MB]]
    return pts


ORACLE_SWEEP_SAMPLE = 1 << 23  # input elements per active rank in the sweep's oracle timing


def _sweep_oracle(rv, coll, A, dt, opts0):
    """The oracle timed beside a sweep row: the collective's results for a bounded sample
    (ORACLE_SWEEP_SAMPLE input elements per active rank) computed by the unchanged oracle
    on one host core -- one call for allreduce and all-gather (every active gets the same
    result), one per owner or destination for reduce-scatter and all-to-all. GB/s counts the
    relay schedule's algorithmic bytes for the sample's count, as the bench's CPU leg does."""
    import oracle as orc
    import synth
    d = rv.dtype_code(dt)
    S = ORACLE_SWEEP_SAMPLE
    count = {rv.ALLREDUCE: S, rv.REDUCE_SCATTER: S // A, rv.ALL_GATHER: S,
             rv.ALL_TO_ALL: S // (A * (A - 1))}[coll]
    plan = rv.relay_plan(coll, count, d, A, R, opts0)
    xs = [synth.to_numpy(synth.rank_input(9, r, plan.input_elems, dt)) for r in range(A)]
    od = {rv.F32: orc.F32, rv.BF16: orc.BF16, rv.I32: orc.I32}[d]
    scale = 1.0 if (d == rv.I32 or coll in (rv.ALL_GATHER, rv.ALL_TO_ALL)) else 1.0 / A
    orc.lib()
    t0 = time.perf_counter()
    if coll == rv.ALLREDUCE:
        orc.allreduce(od, xs, scale)
    elif coll == rv.REDUCE_SCATTER:
        rs = orc.reduce_scatter_wide if plan.wide_partial else orc.reduce_scatter
        for o in range(A):
            rs(od, xs, count, o, scale, plan.relay_total)
    elif coll == rv.ALL_GATHER:
        orc.all_gather(xs, count)
    else:
        for dst in range(A):
            orc.all_to_all(xs, count, dst)
    sec = time.perf_counter() - t0
    nbytes = sum(p["bytes_read"] + p["bytes_written"] for p in rv.relay_plan_passes(plan))
    return {"gbs": round(nbytes / sec / 1e9, 3), "seconds": round(sec, 3), "cores": 1,
            "sample_count": count, "kind": "oracle"}


def run_sweep(args):
    """Per collective and count: each pass's time (CUDA events; before every repetition
    a buffer twice the L2 is written and another read, so L2 holds no dirty lines),
    algorithmic bytes, GB/s and fraction of the measured HBM peak."""
    import torch
    import pack_virtual_rank_gb300.build as b
    b.build()
    import pack_virtual_rank_gb300 as rv
    import synth
    dev = torch.device("cuda", 0)
    peak, _ = _peaks()
    colls = {"allreduce": rv.ALLREDUCE, "reduce_scatter": rv.REDUCE_SCATTER,
             "all_gather": rv.ALL_GATHER, "all_to_all": rv.ALL_TO_ALL}
    dts = {"f32": rv.F32, "bf16": rv.BF16, "i32": rv.I32}
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    flush_read = torch.ones(2 * l2 // 4, dtype=torch.float32, device=dev)
    # the achievable copy rate on this device in this run, for reference: a 1 GiB bf16
    # device-to-device copy, best of 5, read + written bytes
    src = torch.ones(1 << 29, dtype=torch.bfloat16, device=dev)
    dst = torch.empty_like(src)
    best = None
    for _ in range(6):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        dst.copy_(src)
        a1.record()
        torch.cuda.synchronize()
        t = a0.elapsed_time(a1)
        best = t if best is None else min(best, t)
    copy_gbs = 2 * src.numel() * 2 / best / 1e6
    del src, dst
    print(json.dumps({"device_copy_gbs_this_run": round(copy_gbs, 1), "measured_peak_gbs": peak}),
          flush=True)
    rows = []
    clk = Clocks(0, period_ms=25).__enter__()   # one sampler for the sweep; each row its window
    for name, A, dt, nbytes, sched in _sweep_points():
        coll, d = colls[name], dts[dt]
        E = rv.ESIZE[d]
        elems = nbytes // E
        count = {rv.ALLREDUCE: elems, rv.REDUCE_SCATTER: elems // A, rv.ALL_GATHER: elems,
                 rv.ALL_TO_ALL: elems // (A * (A - 1))}[coll]
        opts0 = rv.make_opts(
            schedule={"relay": rv.SCHEDULE_RELAY, "legacy": rv.SCHEDULE_LEGACY}.get(sched, rv.SCHEDULE_AUTO),
            offload_permille=780 if sched == "permille780" else -1)
        plan = rv.relay_plan(coll, count, d, A, R, opts0)
        passes = rv.relay_plan_passes(plan)
        xs = [synth.rank_input(9, r, plan.input_elems, dt, device=dev) for r in range(A)]
        ys = [torch.empty(plan.output_elems, dtype=xs[0].dtype, device=dev) for _ in range(A)]
        scratch = rv.alloc_scratch(plan, dev)
        scale = 1.0 if (d == rv.I32 or coll in (rv.ALL_GATHER, rv.ALL_TO_ALL)) else 1.0 / A
        fn = rv.COLLECTIVES[coll]

        def call(opts):
            a = (xs + [None] * (R - A), ys + [None] * (R - A), scratch, count, d, A, R)
            if coll in (rv.ALLREDUCE, rv.REDUCE_SCATTER):
                fn(*a, scale, opts)
            else:
                fn(*a, opts)
        for _ in range(3):
            call(opts0)
        torch.cuda.synchronize()
        t_row0 = time.time()
        reps = args.steps
        times = [[] for _ in passes]
        totals = []
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(passes) + 1)]
        o = rv.make_opts(schedule=opts0.schedule, offload_permille=opts0.offload_permille,
                         pass_events=ev)
        graph = None
        if args.graph:
            # the whole call, pass events included, replayed from a CUDA graph: no host
            # launch gaps between the passes
            s = torch.cuda.Stream()
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=s):
                call(o)
        for _ in range(reps):
            flush.fill_(1.0)
            flush_read.sum()        # leaves clean lines in L2: no write-back inside the call
            if graph is not None:
                graph.replay()
            else:
                call(o)
            torch.cuda.synchronize()
            for i in range(len(passes)):
                times[i].append(ev[i].elapsed_time(ev[i + 1]))
            totals.append(ev[0].elapsed_time(ev[-1]))
        # the whole call under the library's default launch policy (one cooperative
        # launch for small calls), timed around the call
        whole = []
        default_form = None
        if not args.graph:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            for _ in range(reps):
                flush.fill_(1.0)
                flush_read.sum()
                e0.record()
                call(opts0)
                e1.record()
                torch.cuda.synchronize()
                whole.append(e0.elapsed_time(e1))
            default_form = rv.last_launch()
        # the same call replayed from a CUDA graph: device time only, without the host's
        # planning and launch work that the timing around a direct call includes
        whole_graph = []
        if not args.graph:
            s_g = torch.cuda.Stream()
            torch.cuda.synchronize()
            g_call = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_call, stream=s_g):
                call(opts0)
            g_call.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            for _ in range(reps):
                flush.fill_(1.0)
                flush_read.sum()
                e0.record()
                g_call.replay()
                e1.record()
                torch.cuda.synchronize()
                whole_graph.append(e0.elapsed_time(e1))
            del g_call
        # the same with the one-launch path forced at every size
        fused = []
        if not args.graph:
            of = rv.make_opts(schedule=opts0.schedule, offload_permille=opts0.offload_permille,
                              flags=rv.FLAG_FUSED_PASSES)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            for _ in range(reps):
                flush.fill_(1.0)
                flush_read.sum()
                e0.record()
                call(of)
                e1.record()
                torch.cuda.synchronize()
                fused.append(e0.elapsed_time(e1))
        prow = []
        for p, t in zip(passes, times):
            by = p["bytes_read"] + p["bytes_written"]
            med = statistics.median(t)
            prow.append({"pass": p["name"], "bytes": by, "ms_min": round(min(t), 4),
                         "ms_median": round(med, 4), "gbs": round(by / med / 1e6, 1),
                         "frac": round(by / med / 1e6 / peak, 3)})
        tot_b = sum(p["bytes_read"] + p["bytes_written"] for p in passes)
        med = statistics.median(totals)
        row = {"collective": name, "A": A, "dtype": dt, "bytes_per_rank": nbytes, "count": count,
               "timing": "cuda graph replay" if graph is not None else "direct calls",
               "schedule": ["relay", "zero_chunk", "direct", "legacy"][plan.kind] +
                           (" 780 permille" if sched == "permille780" else ""),
               "link_cost_bytes": rv.relay_plan_cost_bytes(plan),
               "ms_median": round(med, 4), "gbs": round(tot_b / med / 1e6, 1),
               "frac": round(tot_b / med / 1e6 / peak, 3), "passes": prow}
        if fused:
            fm = statistics.median(fused)
            row.update({"ms_call_fused_forced": round(fm, 4),
                        "frac_call_fused_forced": round(tot_b / fm / 1e6 / peak, 3)})
        if whole_graph:
            gm = statistics.median(whole_graph)
            row.update({"ms_call_default_policy_graph": round(gm, 4),
                        "frac_call_default_policy_graph": round(tot_b / gm / 1e6 / peak, 3)})
        if whole:
            wm = statistics.median(whole)
            row.update({"launch_default_policy": default_form,
                        "ms_call_default_policy": round(wm, 4),
                        "gbs_call_default_policy": round(tot_b / wm / 1e6, 1),
                        "frac_call_default_policy": round(tot_b / wm / 1e6 / peak, 3)})
        # a row whose timed calls took less than 0.15 s repeats the same call (L2 flushed
        # before each, as timed) until they have, so that the sampler sees it running
        while time.time() - t_row0 < 0.15:
            flush.fill_(1.0)
            flush_read.sum()
            call(opts0)
            torch.cuda.synchronize()
        row["clocks"] = clk.window(t_row0, time.time())
        key = (name, A, dt, sched)
        if sched in ("auto", "relay") and nbytes == max(b for n2, a2, d2, b, s2 in _sweep_points()
                                                        if (n2, a2, d2, s2) == key):
            row["oracle"] = _sweep_oracle(rv, coll, A, dt, opts0)
        rows.append(row)
        print(json.dumps(row), flush=True)
        del xs, ys, scratch, graph
        torch.cuda.empty_cache()
    t_rest = time.time()
    rows += _sweep_fused_groups(rv, synth, dev, peak, flush, flush_read, args.steps)
    rows += _sweep_flat_pack(rv, dev, peak, flush, flush_read, args.steps)
    rest_clocks = clk.window(t_rest, time.time())
    for row in rows:
        row.setdefault("clocks", rest_clocks)
    clk.__exit__(None, None, None)
    sweep_clocks = clk.summary()
    if args.sweep_out:
        with open(args.sweep_out, "w") as f:
            json.dump({"peak_gbs": peak, "device_copy_gbs_this_run": round(copy_gbs, 1),
                       "hbm_theoretical_gbs": _theoretical_hbm_gbs(dev),
                       "clocks": sweep_clocks, "rows": rows}, f, indent=1)
    return 0


def _timed(fn, reps, flush, flush_read):
    import torch
    ts = []
    for _ in range(reps):
        flush.fill_(1.0)
        flush_read.sum()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def _sweep_fused_groups(rv, synth, dev, peak, flush, flush_read, reps):
    """The fused multi-group call: every rank active in its own group and a helper in
    the others, all groups' passes merged phase by phase (commits D115998367, D115998376)."""
    import torch
    rows = []
    for name, coll, A, dt, per_rank in (("allreduce", rv.ALLREDUCE, 2, "bf16", 256 << 20),
                                        ("allreduce", rv.ALLREDUCE, 4, "bf16", 512 << 20),
                                        ("reduce_scatter", rv.REDUCE_SCATTER, 2, "bf16", 256 << 20)):
        G = R // A
        d = rv.dtype_code(dt)
        elems = per_rank // rv.ESIZE[d]
        count = elems if coll == rv.ALLREDUCE else elems // A
        counts = [count] * G
        plans = [rv.relay_plan(coll, c, d, A, R) for c in counts]
        xs = [synth.rank_input(9, r, plans[r // A].input_elems, dt, device=dev) for r in range(R)]
        ys = [torch.empty(plans[r // A].output_elems, dtype=xs[0].dtype, device=dev) for r in range(R)]
        scratch = rv.alloc_multi_scratch(coll, counts, d, A, dev)
        scale = 1.0 / A
        call = lambda: rv.relay_multi_group(coll, counts, xs, ys, scratch, d, A, scale)
        for _ in range(3):
            call()
        ms = _timed(call, reps, flush, flush_read)
        # bytes: every group's passes (the fused call runs them all)
        nbytes = sum(p["bytes_read"] + p["bytes_written"] for pl in plans for p in rv.relay_plan_passes(pl))
        link = rv.relay_multi_group_link_bytes(coll, counts, d, A)
        row = {"collective": f"{name} fused {G} groups", "A": A, "dtype": dt,
               "bytes_per_rank": per_rank, "count": count, "schedule": "relay",
               "link_cost_bytes": int(sum(t.max() for t in link)), "ms_median": round(ms, 4),
               "gbs": round(nbytes / ms / 1e6, 1), "frac": round(nbytes / ms / 1e6 / peak, 3),
               "passes": []}
        rows.append(row)
        print(json.dumps(row), flush=True)
        del xs, ys, scratch
        torch.cuda.empty_cache()
    return rows


def _sweep_flat_pack(rv, dev, peak, flush, flush_read, reps):
    """Packing 256 caller tensors of mixed sizes (1 GiB of bf16 in all) into one flat
    buffer and back, one launch each (the analogue of commit D115998366's pack/unpack);
    timed as graph replays."""
    import torch
    g = torch.Generator().manual_seed(3)
    sizes = torch.randint(1, 4 << 20, (256,), generator=g)
    sizes = (sizes * ((1 << 29) / sizes.sum())).long().clamp(min=1).tolist()
    ts = [torch.empty(n, dtype=torch.bfloat16, device=dev) for n in sizes]
    flat = torch.empty(sum(sizes), dtype=torch.bfloat16, device=dev)
    rows = []
    for name, fn in (("pack_flat", lambda: rv.relay_pack_flat(ts, flat)),
                     ("unpack_flat", lambda: rv.relay_unpack_flat(flat, ts))):
        for _ in range(3):
            fn()
        # replayed from a CUDA graph: the device time of the one launch, without the
        # host marshalling of 256 tensor pointers
        s = torch.cuda.Stream()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            fn()
        ms = _timed(graph.replay, reps, flush, flush_read)
        nbytes = 2 * flat.numel() * 2
        row = {"collective": name, "A": 0, "dtype": "bf16", "bytes_per_rank": flat.numel() * 2,
               "count": len(ts), "schedule": "-", "link_cost_bytes": 0, "ms_median": round(ms, 4),
               "gbs": round(nbytes / ms / 1e6, 1), "frac": round(nbytes / ms / 1e6 / peak, 3),
               "passes": []}
        rows.append(row)
        print(json.dumps(row), flush=True)
    return rows


def run_profile_case(args):
    """A named collective run W + K times under the library's default launch policy, for
    profiler captures of kernels the bench workload does not exercise (not a bench line).
    Case: COLLECTIVE:A:DTYPE:COUNT[:relay][:payload][:separate][:chained], COUNT in the
    collective's own count; "payload" carries 4-active reduce-scatter partials in the
    payload type; "separate" launches pass by pass, "chained" forces the chained launch."""
    import torch
    import pack_virtual_rank_gb300.build as b
    b.build()
    import pack_virtual_rank_gb300 as rv
    import synth
    name, a, dt, cnt, *rest = args.profile_case.split(":")
    Ap, count = int(a), int(cnt)
    coll = {"allreduce": rv.ALLREDUCE, "reduce_scatter": rv.REDUCE_SCATTER,
            "all_gather": rv.ALL_GATHER, "all_to_all": rv.ALL_TO_ALL}[name]
    d = {"f32": rv.F32, "bf16": rv.BF16, "i32": rv.I32}[dt]
    flags = ((rv.FLAG_PAYLOAD_PARTIAL if "payload" in rest else 0)
             | (rv.FLAG_SEPARATE_PASSES if "separate" in rest else 0)
             | (rv.FLAG_CHAINED if "chained" in rest else 0))
    opts = rv.make_opts(schedule=rv.SCHEDULE_RELAY if "relay" in rest else rv.SCHEDULE_AUTO,
                        flags=flags)
    dev = torch.device("cuda", 0)
    plan = rv.relay_plan(coll, count, d, Ap, R, opts)
    xs = [synth.rank_input(9, r, plan.input_elems, dt, device=dev) for r in range(Ap)]
    ys = [torch.empty(plan.output_elems, dtype=xs[0].dtype, device=dev) for _ in range(Ap)]
    scratch = rv.alloc_scratch(plan, dev)
    scale = 1.0 if (d == rv.I32 or coll in (rv.ALL_GATHER, rv.ALL_TO_ALL)) else 1.0 / Ap
    fn = rv.COLLECTIVES[coll]
    a0 = (xs + [None] * (R - Ap), ys + [None] * (R - Ap), scratch, count, d, Ap, R)
    call = (lambda: fn(*a0, scale, opts)) if coll in (rv.ALLREDUCE, rv.REDUCE_SCATTER) \
        else (lambda: fn(*a0, opts))
    for _ in range(args.warmup):
        call()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(args.steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    nbytes = sum(p["bytes_read"] + p["bytes_written"] for p in rv.relay_plan_passes(plan))
    print(json.dumps({"profile_case": args.profile_case, "passes": len(rv.relay_plan_passes(plan)),
                      "launch": rv.last_launch(), "ms_per_call": round(ms, 4),
                      "gbs": round(nbytes / ms / 1e6, 1)}))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--count", type=int, default=COUNT,
                    help="elements per rank (default 2^29 = 1 GiB of bf16); smaller counts are "
                         "for profiling captures, not bench lines")
    ap.add_argument("--profile-case", default=None,
                    help="COLLECTIVE:A:DTYPE:COUNT[:relay] run under the default launch policy "
                         "for profiler captures (not a bench line)")
    ap.add_argument("--sweep", action="store_true",
                    help="per-collective, per-count pass table of the five workloads "
                         "(not a bench line)")
    ap.add_argument("--sweep-out", default=None, help="write the sweep table as JSON here")
    ap.add_argument("--graph", action="store_true",
                    help="sweep: replay each call from a CUDA graph (device time without host gaps)")
    ap.add_argument("--e2e-copy", choices=["auto", "library", "library-in", "library-out", "torch"],
                    default="auto",
                    help="how the end-to-end leg moves inputs in and results out")
    ap.add_argument("--e2e-ctas", type=int, default=0,
                    help="CTA cap of the end-to-end leg's relay_copy launches (0: half the SMs)")
    ap.add_argument("--kernel-only", action="store_true",
                    help="time the device passes only (no end-to-end leg, no CPU baseline, "
                         "no per-workload table)")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the per-workload table (every other workload at one size)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)   # at least 3 untimed steps before timing
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.profile_case:
        return run_profile_case(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
