"""Benchmark: paged decode attention + paged cache write on GB300.

One step = one decode step of the 1.1B edge model shape over all 24 layers:
for every layer, write each sequence's new K/V row into its slot
(pa_cache_write) and run paged decode attention over the layer's cache
(pa_decode).  64 sequences, context lengths uniform in [16, 2048], 12 query /
2 kv heads, head dim 128, fp16, 16-token blocks, a randomly permuted pool of
1.2x the blocks needed, 24 distinct layer caches (about 1.6 GB, far above the
129 MB L2, so every step reads its K/V from HBM).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0.  ``value`` is achieved HBM GB/s over the
algorithmic bytes (K/V rows read, q read, out written, table and length reads,
the cache write's rows read and written), whole job.  ``--impl reference``
times the CPU oracle on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "paged decode attention: achieved HBM GB/s (% of GB300 peak) and KV tokens/s"
SPEC_PEAK_GBS = 8000.0


# ------------------------------------------------------------------------------------------
# byte ledger of one step
# ------------------------------------------------------------------------------------------

def decode_bytes(wl) -> int:
    """Algorithmic bytes of one pa_decode call: every context row of K and V, q read,
    out written, the table entries and lengths read.  Split partials are not counted."""
    e = 2
    D = wl.head_dim
    lens = wl.context_lens.to(torch.int64)
    kv = int(lens.sum()) * wl.num_kv_heads * D * e * 2
    qo = 2 * wl.num_seqs * wl.num_q_heads * D * e
    table = 4 * int(((lens + wl.block_size - 1) // wl.block_size).sum())
    return kv + qo + table + 4 * wl.num_seqs


def cache_write_bytes(wl) -> int:
    rows = wl.num_seqs * wl.num_kv_heads * wl.head_dim * 2 * 2   # K and V rows, 16-bit
    return 2 * rows + 8 * wl.num_seqs                             # read + written, slots read


# ------------------------------------------------------------------------------------------
# clocks sampled while the timed region runs
# ------------------------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = max(smax, float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def profiled_traffic(kernel_file: str, bench_op: str = "decode"):
    """DRAM bytes per launch from the committed ncu summary of the kernel on this bench line's
    workload (``bench_op``), if the kernel source still hashes to what was profiled (else None:
    the counters are stale)."""
    import glob
    import hashlib
    src = os.path.join(ROOT, kernel_file)
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        fields = {}
        for line in open(path, encoding="utf-8"):
            if ":" in line and not line.startswith((" ", "|", "#")):
                k, _, v = line.partition(":")
                fields[k.strip()] = v.strip()
        if (fields.get("kernel_source") == kernel_file and fields.get("source_sha256_16") == sha and
                fields.get("bench_op", "decode") == bench_op):
            try:
                return int(fields["traffic_bytes_per_launch"])
            except (KeyError, ValueError):
                return None
    return None


def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# ------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------

def _pack(tensors, device):
    """One contiguous device buffer holding copies of ``tensors`` (each at a 256-byte aligned
    offset) and views of it with their shapes and dtypes, so that a step's inputs (or outputs)
    cross the host link as one copy."""
    offs, n = [], 0
    for t in tensors:
        offs.append(n)
        n += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(n, dtype=torch.uint8, device=device)
    views = []
    for t, o in zip(tensors, offs):
        nb = t.numel() * t.element_size()
        v = buf[o:o + nb].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    return buf, views


class Step:
    """All device buffers of one bench step plus the captured CUDA graph.

    ``fused``: one pa_decode_append launch per layer (cache write of the new token + decode);
    otherwise pa_cache_write followed by pa_decode."""

    def __init__(self, wl, device, fused: bool = True, num_ctas: int = 0, planned: bool = True,
                 adaptive: bool = False):
        self.fused = fused
        self.num_ctas = num_ctas
        self.adaptive = adaptive
        self.planned = planned and fused
        import paged_kv_cache_08_gb300 as pa
        self.pa = pa
        self.wl = wl
        self.dev = device
        L = wl.layers
        slots = torch.from_numpy(pa.build_slot_mapping(wl.block_tables, wl.context_lens, wl.block_size))
        # every per-step input (queries, new K/V rows, tables, lengths, slots) in one buffer and
        # the outputs in another: the end-to-end pass moves each across the host link in one copy
        self.inbuf, views = _pack(list(wl.q) + list(wl.k_new) + list(wl.v_new) +
                                  [wl.block_tables, wl.context_lens, slots], device)
        wl.q = views[:L]
        wl.k_new = views[L:2 * L]
        wl.v_new = views[2 * L:3 * L]
        self.bt, self.lens, self.slots = views[3 * L:]
        self.outbuf, self.out = _pack([torch.zeros_like(wl.q[i]) for i in range(L)], device)
        S, Hq, D = wl.q[0].shape
        ws = pa.decode_workspace_size(S, Hq, wl.num_kv_heads, D, wl.block_size, wl.max_blocks_per_seq,
                                      num_ctas=num_ctas)
        self.ws = pa.new_workspace(ws, device)
        self.plan = None
        if self.planned:
            # the step's plan: built by the first launch of every step (inside the graph), read by
            # every layer's decode
            self.plan = pa.decode_plan(self.bt, self.lens, wl.num_q_heads, wl.num_kv_heads, wl.block_size,
                                       wl.num_blocks, num_ctas=num_ctas, adaptive=adaptive)
            self.ws = pa.new_planned_workspace(num_ctas, device)
        self.tps = pa.plan_tokens_per_split(S, Hq, wl.num_kv_heads, D, wl.block_size, wl.max_blocks_per_seq)
        self.graph = None
        self.ev = None

    def launch_layer(self, i, ev_pair=None):
        wl, pa = self.wl, self.pa
        if not self.fused:
            pa.cache_write(wl.k_new[i], wl.v_new[i], self.slots, wl.k_cache[i], wl.v_cache[i])
        if ev_pair is not None:
            ev_pair[0].record()
        if self.planned:
            # early reads from layer 1 on: the kernel before it is the previous layer's, which
            # writes other pools and never the plan (layer 0 follows the plan kernel)
            pa.decode_planned(wl.q[i], wl.k_cache[i], wl.v_cache[i], self.plan, wl.scale, k_new=wl.k_new[i],
                              v_new=wl.v_new[i], out=self.out[i], workspace=self.ws, early_reads=i > 0)
        elif self.fused:
            # early reads: the kernel before each launch is the previous layer's, which writes
            # other pools and never the tables or lengths
            pa.decode_append(wl.q[i], wl.k_new[i], wl.v_new[i], wl.k_cache[i], wl.v_cache[i], self.bt, self.lens,
                             wl.scale, wl.num_kv_heads, out=self.out[i], workspace=self.ws, num_ctas=self.num_ctas,
                             early_reads=True)
        else:
            pa.decode(wl.q[i], wl.k_cache[i], wl.v_cache[i], self.bt, self.lens, wl.scale, wl.num_kv_heads,
                      out=self.out[i], workspace=self.ws, num_ctas=self.num_ctas)
        if ev_pair is not None:
            ev_pair[1].record()

    def make_plan(self):
        wl = self.wl
        self.pa.decode_plan(self.bt, self.lens, wl.num_q_heads, wl.num_kv_heads, wl.block_size, wl.num_blocks,
                            plan=self.plan, num_ctas=self.num_ctas, adaptive=self.adaptive)

    def eager(self):
        if self.planned:
            self.make_plan()
        for i in range(self.wl.layers):
            self.launch_layer(i)

    def capture(self):
        self.eager()                       # warm every kernel / attribute outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.eager()
        self.graph = g

    def decode_launch_ms(self, rounds: int = 3):
        """Duration of every pa_decode call of the step, from CUDA events recorded on the
        launching stream around it.  The step is enqueued behind a spin kernel so that the
        GPU runs it back to back and host launch gaps stay outside the events."""
        times = []
        for _ in range(rounds):
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(self.wl.layers)]
            torch.cuda._sleep(50_000_000)
            if self.planned:
                self.make_plan()
            for i in range(self.wl.layers):
                self.launch_layer(i, evs[i])
            torch.cuda.synchronize()
            times += [a.elapsed_time(b) for a, b in evs]
        return times

    def replay(self):
        self.graph.replay()


def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's time (the job's time); identity on one process."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_shard(rank: int, world: int) -> dict:
    """Weak scaling: every rank runs the full step on its own replica of the workload (its own
    layer caches and queries, same shapes); sequences never exchange data, so no collective is
    on the data path."""
    return {"replica": rank, "of": world}


def _dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_ours(args):
    import torch.distributed as dist
    world, rank, local = _dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = workloads.config(2, device=dev, layers=args.layers)
    import paged_kv_cache_08_gb300 as pa
    kind = pa.kernel_kind(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads)
    fused = args.path in ("fused", "unplanned") and kind == 2
    planned = args.path == "fused" and fused
    st = Step(wl, dev, fused=fused, num_ctas=args.num_ctas, planned=planned, adaptive=args.adaptive)
    d_bytes = decode_bytes(wl)
    c_bytes = cache_write_bytes(wl)
    step_bytes = wl.layers * (d_bytes + c_bytes)
    kv_tokens = wl.layers * wl.total_context_tokens()

    st.capture()
    split_combine = kind != 2 and st.tps < wl.max_blocks_per_seq * wl.block_size
    # fused: one launch per layer; else cache write + decode (+ combine)
    launches_per_step = wl.layers * (1 if fused else 2 + (1 if split_combine else 0)) + (1 if planned else 0)

    for _ in range(args.warmup):
        st.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()

    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        st.pa.read_device_status(clear=True)
        start.record()
        for _ in range(args.steps):
            st.replay()
        stop.record()
        torch.cuda.synchronize()
        timed_status = st.pa.read_device_status(clear=True)
        decode_ms = st.decode_launch_ms()
    if timed_status:
        print(f"bench: the device status word read {timed_status:#x} after the timed region "
              "(a kernel skipped an index or gave up a wait): the number is not valid", file=sys.stderr)
    total_ms = max_over_ranks(start.elapsed_time(stop), dev)
    ms_per_step = total_ms / args.steps
    value = world * step_bytes / (ms_per_step * 1e-3) / 1e9

    # Roofline of the decode kernel.  Fused: the step is nothing but its back-to-back launches, so
    # the average launch duration is the timed region's event time over the launches in it (the
    # launches overlap one another's start and end).  Separate: events around each pa_decode call,
    # enqueued behind a spin kernel.  The isolated figure is reported beside it either way.
    peak, peak_kind = measured_peak_gbs()
    roof = None
    if decode_ms:
        iso_ms = statistics.mean(decode_ms)
        if fused:
            avg_ms = start.elapsed_time(stop) / (args.steps * wl.layers)
            how = ("timed-region events / decode launches in it (the step's plan launch included)" if planned
                   else "timed-region events / launches in it")
        else:
            avg_ms = iso_ms
            how = "events around each launch, enqueued behind a spin kernel"
        kernel_bytes = d_bytes + (c_bytes if fused else 0)   # the fused kernel also moves the new rows
        achieved = kernel_bytes / (avg_ms * 1e-3) / 1e9
        traffic = (profiled_traffic("paged_kv_cache_08_gb300/csrc/decode_planned.cu") if planned else
                   profiled_traffic("paged_kv_cache_08_gb300/csrc/decode_persist.cu") if kind == 2 else None)
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "algorithmic_bytes_per_launch": kernel_bytes,
                "kernel": "pa_decode_planned (append)" if planned else ("pa_decode_append" if fused else "pa_decode"),
                "avg_launch_us": round(avg_ms * 1e3, 2), "avg_launch_from": how,
                "isolated_launch_us": round(iso_ms * 1e3, 2),
                "isolated_achieved": round(kernel_bytes / (iso_ms * 1e-3) / 1e9, 1),
                "peak_source": f"{peak_kind} copy bandwidth",
                "frac_of_8TBs_spec": round(achieved / SPEC_PEAK_GBS, 4)}

    # e2e through the public API with host buffers: H2D of the step's inputs, D2H of its outputs
    e2e = run_e2e(st, wl, args, step_bytes) if rank == 0 else None

    # every configuration, one layer timed alone, with its raw error against the oracle
    per_config = None
    if rank == 0 and world == 1 and not args.no_per_config:
        del st
        torch.cuda.empty_cache()
        per_config = {}
        with ClockSampler(local) as clk_pc:
            for cfg, B in PER_CONFIG:
                key = f"config{cfg}" + (f"_B{B}" if B else "")
                per_config[key] = time_config(cfg, B, dev, 30, 3, args.num_ctas, errors=not args.no_cpu_baseline,
                                               adaptive=args.adaptive, with_adaptive=cfg != 1)
        per_config["clocks"] = clk_pc.summary()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, budget_s=args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": wl.name, "seqs": wl.num_seqs, "layers": wl.layers,
                       "context": "uniform [16, 2048]", "q_heads": wl.num_q_heads, "kv_heads": wl.num_kv_heads,
                       "head_dim": wl.head_dim, "block_size": wl.block_size, "pool_blocks": wl.num_blocks,
                       "decode_kernel": ("planned: one CTA per SM, two ranges streamed from both ends, "
                                         "mma.sync tensor cores" if planned else
                                         {1: "split grid, CUDA cores", 2: "persistent, tensor cores",
                                          3: "split grid, tensor cores"}[kind]),
                       "step": ("pa_decode_plan once, then pa_decode_planned with the cache write per layer"
                                if planned else "pa_decode_append per layer (cache write fused)" if fused
                                else "pa_cache_write + pa_decode per layer"),
                       "l2": "inputs larger than L2: %d distinct layer caches (%.2f GB) read once per step"
                             % (wl.layers, 2 * sum(t.numel() * 2 for t in wl.k_cache) / 1e9),
                       "parallelism": f"replicas x{world}", "cuda_graph": True},
            "pct_of_measured_peak": round(100 * value / world / peak, 2),
            "pct_of_8TBs_spec": round(100 * value / world / SPEC_PEAK_GBS, 2),
            "kv_tokens_per_s": round(world * kv_tokens / (ms_per_step * 1e-3), 1),
            "bytes_per_step": step_bytes,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "per_config": per_config,
            "gpu_launches": launches_per_step * args.steps,
            "device_status": timed_status,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_e2e(st, wl, args, step_bytes):
    """Same step through the public API with inputs in pinned host memory: every step copies
    q, the new K/V rows, the tables, lengths and slots to the device (one copy of the packed
    input buffer), runs the 24 layers and copies the outputs back (one copy).  Two buffer sets
    (and two captured graphs) let step k + 1's input copy and step k - 1's output copy run on
    copy streams while step k's kernels run; the timed region spans all copies of all steps."""
    st2 = Step(wl, st.dev, fused=st.fused, num_ctas=st.num_ctas, planned=st.planned, adaptive=st.adaptive)
    st2.capture()
    sets = [st, st2]
    host_in = st.inbuf.cpu().pin_memory()
    host_out = [torch.empty(x.outbuf.shape, dtype=x.outbuf.dtype).pin_memory() for x in sets]
    h2d = host_in.numel() * host_in.element_size()
    d2h = host_out[0].numel() * host_out[0].element_size()
    main = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    h2d_done, graph_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def h2d_copy(b):
        with torch.cuda.stream(up):
            up.wait_event(graph_done[b])          # the graph that last read this input set is done
            sets[b].inbuf.copy_(host_in, non_blocking=True)
            h2d_done[b].record(up)

    def run(steps):
        for b in range(2):                        # nothing in flight yet: every event completes at once
            graph_done[b].record(main)
            d2h_done[b].record(main)
        h2d_copy(0)
        for k in range(steps):
            b = k % 2
            if k + 1 < steps:
                h2d_copy(1 - b)
            main.wait_event(h2d_done[b])
            main.wait_event(d2h_done[b])          # the outputs this graph overwrites are on the host
            sets[b].replay()
            graph_done[b].record(main)
            with torch.cuda.stream(down):
                down.wait_event(graph_done[b])
                host_out[b].copy_(sets[b].outbuf, non_blocking=True)
                d2h_done[b].record(down)
        main.wait_stream(up)
        main.wait_stream(down)

    def serial(steps):
        for _ in range(steps):
            st.inbuf.copy_(host_in, non_blocking=True)
            st.replay()
            host_out[0].copy_(st.outbuf, non_blocking=True)

    def timed(fn):
        fn(max(3, args.warmup))
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b_ = torch.cuda.Event(enable_timing=True)
        a.record()
        fn(args.steps)
        b_.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b_) / args.steps

    ms = timed(run)
    ms_serial = timed(serial)
    return {"value": round(step_bytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "pipelined": "step k+1's input copy and step k-1's output copy overlap step k's kernels",
            "serial": {"value": round(step_bytes / (ms_serial * 1e-3) / 1e9, 1), "ms_per_step": round(ms_serial, 4),
                       "how": "input copy, the 24 layers, output copy, one stream"}}


# ------------------------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ------------------------------------------------------------------------------------------

def _oracle_layer(o, wl, i):
    import oracle as oracle_pkg
    kc = oracle_pkg.as_u16(wl.k_cache[i]).copy()
    vc = oracle_pkg.as_u16(wl.v_cache[i]).copy()
    t0 = time.perf_counter()
    slots = o.slot_mapping(wl.block_tables, wl.context_lens, wl.block_size)
    o.cache_write(wl.k_new[i], wl.v_new[i], slots, kc, vc)
    o.decode(wl.q[i], kc, vc, wl.block_tables, wl.context_lens, wl.scale, wl.num_kv_heads, wl.dtype == "bf16")
    return time.perf_counter() - t0


def _host_layer(wl, i):
    """A host copy of layer i (structure shared)."""
    sub = workloads.Workload(**{k: getattr(wl, k) for k in (
        "name", "dtype", "num_seqs", "num_q_heads", "num_kv_heads", "head_dim", "block_size", "num_blocks",
        "max_blocks_per_seq", "context_lens", "block_tables", "scale", "seed", "shared_prefix_blocks")})
    for key in ("q", "k_cache", "v_cache", "k_new", "v_new"):
        getattr(sub, key).append(getattr(wl, key)[i].cpu())
    return sub


def cpu_baseline(wl, budget_s=15.0):
    """The oracle, as it stands, on the host cores: whole layers of the same workload until
    about ``budget_s`` seconds of oracle time; GB/s over the same algorithmic bytes."""
    import oracle as oracle_pkg
    o = oracle_pkg.get()
    spent, layers = 0.0, 0
    for i in range(wl.layers):
        sub = _host_layer(wl, i)
        spent += _oracle_layer(o, sub, 0)
        layers += 1
        if spent >= budget_s:
            break
    byts = layers * (decode_bytes(wl) + cache_write_bytes(wl))
    return {"value": round(byts / spent / 1e9, 4), "unit": "GB/s", "cores": o.num_threads(), "kind": "oracle",
            "sample": f"{layers} of {wl.layers} layers of the same workload (cache write + decode, fp64)",
            "seconds": round(spent, 2)}


def run_reference(args):
    world, rank, _ = _dist_env()
    if rank != 0:
        return
    import oracle as oracle_pkg
    o = oracle_pkg.get()
    wl = workloads.config(2, layers=1)                     # one layer per step: a bounded sample
    step_bytes = decode_bytes(wl) + cache_write_bytes(wl)
    for _ in range(args.warmup):
        _oracle_layer(o, wl, 0)
    times = [_oracle_layer(o, wl, 0) for _ in range(args.steps)]
    ms = 1e3 * sum(times) / len(times)
    value = step_bytes / (ms * 1e-3) / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name + " (one layer of 24 per step)", "seqs": wl.num_seqs,
                       "block_size": wl.block_size, "parallelism": "host cores"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": o.num_threads(), "kind": "oracle",
                             "sample": "one layer of the 24-layer step per timed step"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# block copies: copy-on-write inside the cache, swap out to / in from pinned host memory
# ------------------------------------------------------------------------------------------

def _copy_pairs(num_blocks: int, n: int, seed: int):
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(num_blocks, generator=g)
    dst = perm[:n]
    src = perm[n:][torch.randint(0, num_blocks - n, (n,), generator=g)]
    return src.to(torch.int32), dst.to(torch.int32)


def _event_ms(fn, steps: int, warmup: int) -> float:
    for _ in range(warmup):
        fn(-1)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(steps):
        fn(i)
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def run_copy_blocks(args):
    """Copy-on-write at scale: 16384 random (src, dst) block pairs of a 1 GiB pool in the 1.1B
    shape (2 kv heads, 16-token blocks, fp16): 256 MiB read and 256 MiB written per call, four
    pair sets in rotation (each touches more than the L2).  Also the latency of one fork step's
    copies (64 pairs, one per sequence)."""
    import paged_kv_cache_08_gb300 as pa
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    NB, H, B, D = 65536, 2, 16, 128
    k = torch.empty((NB, H, B, D), dtype=torch.float16, device=dev).normal_()
    v = torch.empty_like(k).normal_()
    sets = [tuple(t.to(dev) for t in _copy_pairs(NB, 16384, seed=s)) for s in range(4)]
    small = [tuple(t.to(dev) for t in _copy_pairs(NB, 64, seed=100 + s)) for s in range(4)]
    blk_bytes = H * B * D * 2
    bytes_per_call = 16384 * 2 * blk_bytes * 2          # K and V blocks, read + written
    with ClockSampler(0) as clk:
        ms = _event_ms(lambda i: pa.copy_blocks(k, v, k, v, *sets[i % 4]), args.steps, args.warmup)
    small_ms = _event_ms(lambda i: pa.copy_blocks(k, v, k, v, *small[i % 4]), args.steps, args.warmup)
    peak, peak_kind = measured_peak_gbs()
    gbs = bytes_per_call / (ms * 1e-3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        o = oracle.get()
        nb = 8192
        hk = oracle.as_u16(k[:nb].cpu()).copy()
        hv = oracle.as_u16(v[:nb].cpu()).copy()
        src, dst = _copy_pairs(nb, 2048, seed=7)
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < min(args.cpu_seconds, 5.0):
            o.copy_blocks(hk, hv, hk, hv, src.numpy(), dst.numpy())
            reps += 1
        el = time.perf_counter() - t0
        cpu = {"value": round(reps * 2048 * 2 * blk_bytes * 2 / el / 1e9, 2), "unit": "GB/s", "cores": 1,
               "kind": "oracle", "sample": f"2048 pairs of an 8192-block pool, {reps} calls"}
    line = {"metric": "block copy (copy-on-write): achieved HBM GB/s", "value": round(gbs, 1), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic",
            "config": {"workload": "cow_copy_16384pairs_pool65536_kv2_B16_f16", "pool_gib": 1.0,
                       "l2": "four pair sets in rotation, 512 MiB moved per call"},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "traffic": None, "algorithmic_bytes_per_launch": bytes_per_call,
                         "kernel": "pa_copy_blocks", "avg_launch_us": round(ms * 1e3, 2),
                         "peak_source": f"{peak_kind} copy bandwidth"},
            "fork_step_64_pairs_us": round(small_ms * 1e3, 2),
            "cpu_baseline": cpu, "gpu_launches": args.steps, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def run_swap(args):
    """Swap out and in: the blocks of a 1 GiB device pool that fit a pinned host pool of 0.3 x its
    size (the tutorial's swap buffer) go to host memory and come back to other device blocks.
    The denominator is the same link measured by one large cudaMemcpyAsync each way."""
    import paged_kv_cache_08_gb300 as pa
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    NB, H, B, D = 65536, 2, 16, 128
    HB = int(0.3 * NB)
    k = torch.empty((NB, H, B, D), dtype=torch.float16, device=dev).normal_()
    v = torch.empty_like(k).normal_()
    hk = torch.empty((HB, H, B, D), dtype=torch.float16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    n = 16384
    g = torch.Generator().manual_seed(11)
    dev_ids = torch.randperm(NB, generator=g)[:n].to(torch.int32).to(dev)
    host_ids = torch.randperm(HB, generator=g)[:n].to(torch.int32).to(dev)
    back_ids = torch.randperm(NB, generator=g)[:n].to(torch.int32).to(dev)
    blk_bytes = H * B * D * 2
    moved = n * 2 * blk_bytes
    with ClockSampler(0) as clk:
        out_ms = _event_ms(lambda i: pa.copy_blocks(k, v, hk, hv, dev_ids, host_ids), args.steps, args.warmup)
        in_ms = _event_ms(lambda i: pa.copy_blocks(hk, hv, k, v, host_ids, back_ids), args.steps, args.warmup)
    flat_d = torch.empty(moved // 2, dtype=torch.uint8, device=dev)
    flat_h = torch.empty(moved // 2, dtype=torch.uint8).pin_memory()
    d2h_ms = _event_ms(lambda i: flat_h.copy_(flat_d, non_blocking=True), args.steps, args.warmup)
    h2d_ms = _event_ms(lambda i: flat_d.copy_(flat_h, non_blocking=True), args.steps, args.warmup)
    out_gbs = moved / (out_ms * 1e-3) / 1e9
    in_gbs = moved / (in_ms * 1e-3) / 1e9
    d2h = (moved // 2) / (d2h_ms * 1e-3) / 1e9
    h2d = (moved // 2) / (h2d_ms * 1e-3) / 1e9
    line = {"metric": "block swap out / in through pinned host memory: GB/s", "value": round(min(out_gbs, in_gbs), 1),
            "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(out_ms + in_ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": "swap_16384blocks_pool65536_host0.3_kv2_B16_f16",
                       "bytes_each_way": moved},
            "swap_out_gbs": round(out_gbs, 1), "swap_in_gbs": round(in_gbs, 1),
            "roofline": {"bound": "host link", "achieved": round(min(out_gbs, in_gbs), 1),
                         "peak": round(min(d2h, h2d), 1), "unit": "GB/s",
                         "frac": round(min(out_gbs / d2h, in_gbs / h2d), 4), "traffic": None,
                         "kernel": "pa_copy_blocks",
                         "peak_source": "one contiguous cudaMemcpyAsync of the same bytes each way, same run",
                         "d2h_copy_gbs": round(d2h, 1), "h2d_copy_gbs": round(h2d, 1)},
            "gpu_launches": 2 * args.steps, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def run_multi_query(args, new_tokens: int = 2):
    """Several new tokens per sequence (speculative-decoding verification of one draft token per
    sequence and its successor): the 1.1B edge shape of the decode bench, 24 layers, each layer
    writing the 2 newest tokens' K/V and attending over the cache (12 query rows per sequence
    and kv head) in one pa_multi_query_append launch with early reads (``--path separate``:
    pa_cache_write, then pa_multi_query), in a CUDA graph.  Bytes: the decode ledger with 2 query
    and output rows per sequence, plus the cache write of 2 rows per sequence."""
    import paged_kv_cache_08_gb300 as pa
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = workloads.config(2, device=dev, layers=args.layers)
    S, Hq, D, Hkv = wl.num_seqs, wl.num_q_heads, wl.head_dim, wl.num_kv_heads
    new = [new_tokens] * S
    q, qs, max_q = workloads.multi_query_inputs(wl, new, seed=777, device=dev)
    g = torch.Generator().manual_seed(778)
    k_new = [torch.randn((S * new_tokens, Hkv, D), generator=g).to(wl.torch_dtype).to(dev) for _ in range(wl.layers)]
    v_new = [torch.randn((S * new_tokens, Hkv, D), generator=g).to(wl.torch_dtype).to(dev) for _ in range(wl.layers)]
    bt, lens = wl.block_tables.to(dev), wl.context_lens.to(dev)
    # slots of each sequence's newest tokens: positions L - 2 and L - 1 (host bookkeeping)
    tables = wl.block_tables.numpy()
    slots = []
    for s_ in range(S):
        L = int(wl.context_lens[s_])
        for t in range(L - new_tokens, L):
            slots.append(int(tables[s_, t // wl.block_size]) * wl.block_size + t % wl.block_size)
    slots = torch.tensor(slots, dtype=torch.int64, device=dev)
    outs = [torch.empty_like(q) for _ in range(wl.layers)]
    ws = pa.new_workspace(pa.decode_workspace_size(S, Hq, Hkv, D, wl.block_size, wl.max_blocks_per_seq), dev)

    fused = args.path == "fused"

    def step():
        for i in range(wl.layers):
            if fused:
                pa.multi_query(q, wl.k_cache[i], wl.v_cache[i], bt, lens, qs, wl.scale, Hkv, max_q, out=outs[i],
                               workspace=ws, k_new=k_new[i], v_new=v_new[i], num_ctas=args.num_ctas,
                               early_reads=True)
                continue
            pa.cache_write(k_new[i], v_new[i], slots, wl.k_cache[i], wl.v_cache[i])
            pa.multi_query(q, wl.k_cache[i], wl.v_cache[i], bt, lens, qs, wl.scale, Hkv, max_q, out=outs[i],
                           workspace=ws, num_ctas=args.num_ctas)
    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        a.record()
        for _ in range(args.steps):
            graph.replay()
        b.record()
        torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    lens64 = wl.context_lens.to(torch.int64)
    kv = int(lens64.sum()) * Hkv * D * 2 * 2
    qo = 2 * S * new_tokens * Hq * D * 2
    table = 4 * int(((lens64 + wl.block_size - 1) // wl.block_size).sum())
    mq_bytes = kv + qo + table + 4 * (2 * S + 1)
    cw_bytes = 2 * (S * new_tokens * Hkv * D * 2 * 2) + 8 * S * new_tokens
    step_bytes = wl.layers * (mq_bytes + cw_bytes)
    gbs = step_bytes / (ms * 1e-3) / 1e9
    peak, peak_kind = measured_peak_gbs()
    per_layer_us = ms * 1e3 / wl.layers
    line = {"metric": "several-token paged attention (2 new tokens per sequence): achieved HBM GB/s",
            "value": round(gbs, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f16", "data": "synthetic",
            "config": {"workload": f"edge1p1b_64seq_ctx16-2048_gqa12x2_f16_B16_{new_tokens}new_x{wl.layers}layers",
                       "step": ("pa_multi_query_append (cache write + attention, early reads)" if fused
                                else "pa_cache_write + pa_multi_query") + " per layer", "cuda_graph": True,
                       "l2": "inputs larger than L2: distinct layer caches read once per step"},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "traffic": None,
                         "algorithmic_bytes_per_layer": mq_bytes + cw_bytes, "avg_layer_us": round(per_layer_us, 2),
                         "kernel": "pa_multi_query_append" if fused else "pa_multi_query (+ pa_cache_write)",
                         "peak_source": f"{peak_kind} copy bandwidth"},
            "gpu_launches": (1 if fused else 2) * wl.layers * args.steps, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def _half_ulp(t: torch.Tensor):
    """Half the spacing from |t| to the next representable magnitude of t's 16-bit dtype."""
    import numpy as np
    bits = t.detach().cpu().contiguous().view(torch.int16).numpy().astype(np.uint32) & 0x7FFF
    if t.dtype == torch.bfloat16:
        lo = (bits << 16).view(np.float32).astype(np.float64)
        hi = ((bits + 1) << 16).view(np.float32).astype(np.float64)
    else:
        lo = bits.astype(np.uint16).view(np.float16).astype(np.float64)
        hi = (bits + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    return (hi - lo) / 2


def time_config(cfg: int, block_size, dev, steps: int, warmup: int, num_ctas: int = 0, errors: bool = True,
                adaptive: bool = False, with_adaptive: bool = False):
    """One decode layer (the cache write of each sequence's new token plus attention) of a seeded
    configuration, timed alone: the step's plan built first (pa_decode_plan, timed separately),
    then ``steps`` pa_decode_planned launches, each after a 512 MB write that flushes the L2, by
    CUDA events (mean; one event pair resolves about 2 us, the mean of many finer).  The per-layer
    persistent launch (pa_decode_append) is timed the same way beside it.  With ``errors`` the
    output of one launch on fresh caches is compared with the fp64 oracle's on the host: the raw
    max-abs error, and the error beyond the output dtype's own rounding (bf16).  With ``adaptive``
    the plan is rebuilt after each warm-up launch, so that the CTAs' shares follow the rates the
    launches measured, and the timed launches use the last plan."""
    import numpy as np
    import paged_kv_cache_08_gb300 as pa
    wl = workloads.config(cfg, device=dev, layers=1, block_size=block_size)
    bt, lens = wl.block_tables.to(dev), wl.context_lens.to(dev)
    q, kn, vn = wl.q[0], wl.k_new[0], wl.v_new[0]
    kc0, vc0 = wl.k_cache[0], wl.v_cache[0]
    kc, vc = kc0.clone(), vc0.clone()
    out = torch.empty_like(q)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def timed(fn, n):
        ts = []
        for _ in range(n):
            flush.zero_()
            a, b = ev(), ev()
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.fmean(ts), statistics.median(ts)

    res = {}
    plan = pa.decode_plan(bt, lens, wl.num_q_heads, wl.num_kv_heads, wl.block_size, wl.num_blocks, num_ctas=num_ctas,
                          adaptive=adaptive)
    ws = pa.new_planned_workspace(num_ctas, dev)

    def planned():
        pa.decode_planned(q, kc, vc, plan, wl.scale, k_new=kn, v_new=vn, out=out, workspace=ws)

    def replan():
        pa.decode_plan(bt, lens, wl.num_q_heads, wl.num_kv_heads, wl.block_size, wl.num_blocks, plan=plan,
                       num_ctas=num_ctas, adaptive=adaptive)
    uws = pa.new_workspace(pa.decode_workspace_size(wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                                                    wl.block_size, wl.max_blocks_per_seq), dev)

    def unplanned():
        pa.decode_append(q, kn, vn, kc, vc, bt, lens, wl.scale, wl.num_kv_heads, out=out, workspace=uws)
    for fn in (planned, unplanned, replan):
        for _ in range(max(3, warmup)):
            fn()
    if adaptive:
        for _ in range(max(24, warmup)):
            flush.zero_()
            planned()
            replan()
    torch.cuda.synchronize()
    torch.cuda.synchronize()
    pa.read_device_status(clear=True)
    ms, med = timed(planned, steps)
    ms_u, _ = timed(unplanned, steps)
    status = pa.read_device_status(clear=True)
    if status:
        print(f"bench: device status {status:#x} after timing config {cfg}: not valid", file=sys.stderr)
    ms_p, _ = timed(replan, max(10, steps // 3))
    ms_a = None
    if with_adaptive and not adaptive:
        # the same launches through an adaptive plan, after rebuilds that let its shares settle
        aplan = pa.decode_plan(bt, lens, wl.num_q_heads, wl.num_kv_heads, wl.block_size, wl.num_blocks,
                               num_ctas=num_ctas, adaptive=True)

        def aplanned():
            pa.decode_planned(q, kc, vc, aplan, wl.scale, k_new=kn, v_new=vn, out=out, workspace=ws)
        for _ in range(max(24, warmup)):
            flush.zero_()
            aplanned()
            pa.decode_plan(bt, lens, wl.num_q_heads, wl.num_kv_heads, wl.block_size, wl.num_blocks, plan=aplan,
                           num_ctas=num_ctas, adaptive=True)
        torch.cuda.synchronize()
        pa.read_device_status(clear=True)
        ms_a, _ = timed(aplanned, steps)
        status |= pa.read_device_status(clear=True)
    nbytes = decode_bytes(wl) + cache_write_bytes(wl)
    peak, peak_kind = measured_peak_gbs()
    gbs = nbytes / (ms * 1e-3) / 1e9
    res.update({"workload": f"config{cfg}_{wl.num_seqs}seq_gqa{wl.num_q_heads}x{wl.num_kv_heads}_{wl.dtype}"
                            f"_B{wl.block_size}",
                "dtype": wl.dtype, "us": round(ms * 1e3, 2), "median_us": round(med * 1e3, 2),
                "value": round(gbs, 1), "unit": "GB/s", "frac": round(gbs / peak, 4),
                "frac_of_8TBs_spec": round(gbs / SPEC_PEAK_GBS, 4), "algorithmic_bytes": nbytes,
                "kv_tokens_per_s": round(float(wl.context_lens.sum()) / (ms * 1e-3), 1),
                "kernel": "pa_decode_planned (append)", "plan_us": round(ms_p * 1e3, 2),
                "per_layer_persistent_us": round(ms_u * 1e3, 2),
                "per_layer_persistent_gbs": round(nbytes / (ms_u * 1e-3) / 1e9, 1),
                "peak": peak, "peak_source": f"{peak_kind} copy bandwidth", "adaptive_plan": adaptive,
                "device_status": status, "l2": "flushed (512 MB write) before every timed launch"})
    if ms_a is not None:
        res.update({"adaptive_us": round(ms_a * 1e3, 2), "adaptive_gbs": round(nbytes / (ms_a * 1e-3) / 1e9, 1),
                    "adaptive_frac": round(nbytes / (ms_a * 1e-3) / 1e9 / peak, 4),
                    "adaptive_frac_of_8TBs_spec": round(nbytes / (ms_a * 1e-3) / 1e9 / SPEC_PEAK_GBS, 4)})
    if errors:
        import oracle as oracle_pkg
        o = oracle_pkg.get()
        kc.copy_(kc0)
        vc.copy_(vc0)
        planned()
        torch.cuda.synchronize()
        host = _host_layer(wl, 0)
        okc = oracle_pkg.as_u16(host.k_cache[0]).copy()
        ovc = oracle_pkg.as_u16(host.v_cache[0]).copy()
        t0 = time.perf_counter()
        slots = o.slot_mapping(host.block_tables, host.context_lens, host.block_size)
        o.cache_write(host.k_new[0], host.v_new[0], slots, okc, ovc)
        ref = o.decode(host.q[0], okc, ovc, host.block_tables, host.context_lens, host.scale, host.num_kv_heads,
                       host.dtype == "bf16")
        o_s = time.perf_counter() - t0
        got = out.float().cpu().numpy().astype(np.float64)
        d = np.abs(got - ref)
        allow = _half_ulp(out) if out.dtype == torch.bfloat16 else 0.0
        res.update({"max_abs_err_raw": float(d.max()) if d.size else 0.0,
                    "max_abs_err_beyond_rounding": float((d - allow).max()) if d.size else 0.0,
                    "cache_bit_exact": bool(np.array_equal(oracle_pkg.as_u16(kc.cpu()), okc) and
                                            np.array_equal(oracle_pkg.as_u16(vc.cpu()), ovc)),
                    "oracle_s": round(o_s, 3), "oracle_cores": o.num_threads()})
    del wl, kc, vc, flush
    torch.cuda.empty_cache()
    return res


PER_CONFIG = [(1, None), (2, None), (3, None), (4, None), (5, 16), (5, 32), (5, 64), (5, 128)]


def run_config(args):
    """``--op config``: one configuration through time_config, as one JSON line."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    with ClockSampler(0) as clk:
        r = time_config(args.config, args.block_size, dev, args.steps, args.warmup, args.num_ctas,
                        errors=not args.no_cpu_baseline, adaptive=args.adaptive, with_adaptive=args.config != 1)
    line = {"metric": METRIC, "value": r["value"], "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(r["us"] / 1e3, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": r["dtype"], "data": "synthetic",
            "config": {"workload": r["workload"], "step": "one pa_decode_planned launch (plan prebuilt), timed alone"},
            "roofline": {"bound": "hbm", "achieved": r["value"], "peak": r["peak"], "unit": "GB/s", "frac": r["frac"],
                         "traffic": None, "algorithmic_bytes_per_launch": r["algorithmic_bytes"],
                         "kernel": r["kernel"], "peak_source": r["peak_source"]},
            "detail": r, "gpu_launches": args.steps, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def run_prefill(args, seqs: int = 16, context: int = 4096, new_tokens: int = 512):
    """Chunked prefill: the last 512 tokens of 16 sequences of 4096 (their K/V already in the
    cache) attend causally over the paged cache, in the Llama-2-7B shape of the pages (32 query
    and 32 kv heads, head dim 128, fp16, 32-token blocks, randomly permuted pool, 1 GiB of K/V).
    Tensor-core bound: FLOPs = 4 * head_dim * (query row, visible token) pairs."""
    import paged_kv_cache_08_gb300 as pa
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = workloads.make_workload("prefill_llama7b", context_lens=[context] * seqs, num_q_heads=32, num_kv_heads=32,
                                 block_size=32, dtype="f16", seed=4242, device=dev, values=True)
    q, qs, max_q = workloads.multi_query_inputs(wl, [new_tokens] * seqs, seed=4243, device=dev)
    bt, lens = wl.block_tables.to(dev), wl.context_lens.to(dev)
    out = torch.empty_like(q)

    tiles = args.prefill_tiles

    def call(_):
        pa.multi_query(q, wl.k_cache[0], wl.v_cache[0], bt, lens, qs, wl.scale, wl.num_kv_heads, max_q, out=out,
                       tiles=tiles)
    with ClockSampler(0) as clk:
        ms = _event_ms(call, args.steps, args.warmup)
    pairs = seqs * wl.num_q_heads * sum(context - new_tokens + i + 1 for i in range(new_tokens))
    flops = 4 * wl.head_dim * pairs
    tflops = flops / (ms * 1e-3) / 1e12
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, kind = float(json.load(f)["bf16_tflops"]), "measured cuBLAS bf16 burst (fp16 has the same dense rate)"
    except (OSError, KeyError, ValueError):
        peak, kind = 1900.0, "fallback"
    line = {"metric": "chunked prefill paged attention: achieved TFLOP/s", "value": round(tflops, 1),
            "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": f"prefill_{seqs}seq_ctx{context}_new{new_tokens}_mha32_f16_B32",
                       "l2": "1 GiB of K/V, above L2", "tiles": tiles},
            "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(tflops / peak, 4),
                         "traffic": (profiled_traffic("paged_kv_cache_08_gb300/csrc/prefill_tc.cu", "prefill")
                                     if tiles == "tc" else None),
                         "flops_per_launch": flops,
                         "kernel": ("prefill_tc_kernel (tcgen05.mma, accumulators in tensor memory)" if tiles == "tc"
                                    else "prefill_mma_kernel (mma.sync m16n8k16)"), "peak_source": kind},
            "gpu_launches": args.steps, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def run_runs(args):
    """Slotted contexts: the decode bench's 24-layer 1.1B shape with every 16-token block of every
    context read as two runs cut at a seeded random offset (about 2 x 4300 runs per layer).  The
    step is one pa_decode_plan_runs (the token table and the cut, once for all layers) and one
    pa_decode_planned per layer (early reads from layer 1 on), in a CUDA graph; the one-call
    pa_decode_runs per layer (three launches each) is timed beside it, and the compaction of one
    layer's runs into fresh whole blocks (pa_gather_runs).  Bytes: the decode ledger with 12 bytes
    per run in place of 4 per table entry; the compaction moves every context row of K and V once
    (read + written)."""
    import paged_kv_cache_08_gb300 as pa
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl = workloads.config(2, device=dev, layers=args.layers)
    B = wl.block_size
    tables = wl.block_tables.numpy()
    g = torch.Generator().manual_seed(99)
    runs, seq_runs = [], [0]
    for s_, L in enumerate(wl.context_lens.tolist()):
        for t0 in range(0, L, B):
            n = min(B, L - t0)
            blk = int(tables[s_, t0 // B])
            cut = int(torch.randint(1, B, (1,), generator=g)) if n > 1 else n
            cut = min(cut, n)
            runs.append((blk, 0, cut))
            if n > cut:
                runs.append((blk, cut, n - cut))
        seq_runs.append(len(runs))
    runs_t = torch.tensor(runs, dtype=torch.int32, device=dev)
    seq_t = torch.tensor(seq_runs, dtype=torch.int32, device=dev)
    max_ctx = int(wl.context_lens.max())
    outs = [torch.empty_like(wl.q[i]) for i in range(wl.layers)]
    S, Hq, D, Hkv = wl.num_seqs, wl.num_q_heads, wl.head_dim, wl.num_kv_heads
    ws = pa.new_runs_workspace(wl.q[0], Hkv, B, max_ctx)
    plan = pa.decode_plan_runs(runs_t, seq_t, Hq, Hkv, B, wl.num_blocks, max_ctx)
    pws = pa.new_planned_workspace(0, dev)

    def step():
        pa.decode_plan_runs(runs_t, seq_t, Hq, Hkv, B, wl.num_blocks, max_ctx, plan=plan)
        for i in range(wl.layers):
            pa.decode_planned(wl.q[i], wl.k_cache[i], wl.v_cache[i], plan, wl.scale, out=outs[i], workspace=pws,
                              early_reads=i > 0)

    def step_one_call():
        for i in range(wl.layers):
            pa.decode_runs(wl.q[i], wl.k_cache[i], wl.v_cache[i], runs_t, seq_t, wl.scale, Hkv, max_ctx, out=outs[i],
                           workspace=ws)
    graphs = []
    for fn in (step, step_one_call):
        fn()
        torch.cuda.synchronize()
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_):
            fn()
        graphs.append(g_)
    pa.read_device_status(clear=True)
    with ClockSampler(0) as clk:
        ms = _event_ms(lambda _: graphs[0].replay(), args.steps, args.warmup)
    ms_one = _event_ms(lambda _: graphs[1].replay(), args.steps, args.warmup)
    status = pa.read_device_status(clear=True)
    lens64 = wl.context_lens.to(torch.int64)
    per_layer = int(lens64.sum()) * Hkv * D * 2 * 2 + 2 * S * Hq * D * 2 + 12 * len(runs) + 4 * (S + 1)
    gbs = wl.layers * per_layer / (ms * 1e-3) / 1e9
    # compaction of layer 0's runs into fresh whole blocks of a second pool
    moves, nxt = [], 0
    for s_ in range(S):
        t = 0
        for blk, off, ln in runs[seq_runs[s_]:seq_runs[s_ + 1]]:
            k = 0
            while k < ln:
                if t % B == 0:
                    nxt += 1
                take = min(ln - k, B - t % B)
                moves.append((blk, off + k, take, nxt - 1, t % B))
                t += take
                k += take
    moves_t = torch.tensor(moves, dtype=torch.int32, device=dev)
    dk = torch.empty((nxt,) + tuple(wl.k_cache[0].shape[1:]), dtype=wl.torch_dtype, device=dev)
    dv = torch.empty_like(dk)
    cms = _event_ms(lambda i: pa.gather_runs(wl.k_cache[i % wl.layers], wl.v_cache[i % wl.layers], dk, dv, moves_t),
                    args.steps, args.warmup)
    moved = 2 * 2 * int(lens64.sum()) * Hkv * D * 2
    peak, peak_kind = measured_peak_gbs()
    line = {"metric": "slotted-context paged decode (runs): achieved HBM GB/s", "value": round(gbs, 1), "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": f"edge1p1b_64seq_ctx16-2048_gqa12x2_f16_B16_2runs_per_block_x{wl.layers}layers",
                       "runs_per_layer": len(runs), "cuda_graph": True,
                       "l2": "inputs larger than L2: distinct layer caches read once per step"},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "traffic": None, "algorithmic_bytes_per_layer": per_layer,
                         "avg_layer_us": round(ms * 1e3 / wl.layers, 2),
                         "kernel": "decode_planned_kernel (runs: one bulk copy per K and V row)",
                         "peak_source": f"{peak_kind} copy bandwidth"},
            "one_call_per_layer": {"us_per_layer": round(ms_one * 1e3 / wl.layers, 2),
                                   "gbs": round(wl.layers * per_layer / (ms_one * 1e-3) / 1e9, 1),
                                   "how": "pa_decode_runs per layer: token table, plan and decode each time"},
            "device_status": status,
            "compaction": {"moves": len(moves), "us": round(cms * 1e3, 2),
                           "gbs": round(moved / (cms * 1e-3) / 1e9, 1), "frac": round(moved / (cms * 1e-3) / 1e9 / peak, 4)},
            "gpu_launches": (wl.layers + 2) * args.steps, "clocks": clk.summary()}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=24)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip timing every configuration's single layer (and its oracle error) after the step")
    ap.add_argument("--path", choices=["fused", "unplanned", "separate"], default="fused",
                    help="fused: one plan per step + pa_decode_planned (cache write fused) per layer; "
                         "unplanned: pa_decode_append per layer; separate: pa_cache_write + pa_decode")
    ap.add_argument("--num-ctas", type=int, default=0, help="persistent kernel grid (0 = library default)")
    ap.add_argument("--adaptive", action="store_true",
                    help="plans whose CTA shares follow the CTAs' measured streaming rates (PA_PLAN_ADAPTIVE)")
    ap.add_argument("--op", choices=["decode", "config", "copy_blocks", "swap", "multi_query", "prefill", "runs"],
                    default="decode",
                    help="decode step (default), one layer of another config (--config), or the block-copy, swap, "
                         "several-token, prefill and slotted benchmarks")
    ap.add_argument("--prefill-tiles", choices=["tc", "mma"], default="tc",
                    help="--op prefill: tcgen05 tiles of 128 rows or mma.sync tiles of 64 rows")
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5], help="--op config: which configuration")
    ap.add_argument("--block-size", type=int, default=None, help="--op config: block size (config 5 sweeps it)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.op == "copy_blocks" and args.impl == "ours":
        run_copy_blocks(args)
        return
    if args.op == "swap" and args.impl == "ours":
        run_swap(args)
        return
    if args.op == "multi_query" and args.impl == "ours":
        run_multi_query(args)
        return
    if args.op == "config" and args.impl == "ours":
        run_config(args)
        return
    if args.op == "prefill" and args.impl == "ours":
        run_prefill(args)
        return
    if args.op == "runs" and args.impl == "ours":
        run_runs(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
