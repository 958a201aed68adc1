"""Benchmark of the delta-rule fast-weight layer core on GB300.

One step = one fw_delta_forward call (DPFP of q and k fused, the chunked
delta rule, y and the final state written) over the B2 H8 L2048 d_key 64
nu 3 (d_dot 384) d_v 64 bf16 workload (chunk 64), with a non-zero initial
state W0 read and W_final written, inputs resident in HBM.  On this workload
the call is one cooperative launch (chunk_fused_kernel) in which the walk
over the chunks overlaps the preparation of the later chunks.  Every rank runs
its own replica of that workload (weak scaling, no data-path collective); the
timing is bracketed by a barrier and a device synchronisation on both sides
and the slowest rank's time is reported.

Between steps the inputs rotate over enough distinct sets that their total
exceeds 3x the 129 MB L2, so no step finds its inputs in L2.

The JSON line also carries the other rows of the hot path measured on their
own (the B4 H8 L512 nu 1 forward, the same nu = 3 forward with B = 16, the
standalone DPFP kernel, the decode step on its 512 MiB state, the sum rule,
the projected forward, the backward and the token-wise layer stack), the
roofline of the dominant kernel, an end-to-end number with host buffers,
clocks sampled over the whole run, and the CPU oracle's throughput on the
host cores (all threads, and one thread).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "delta-rule fast-weight forward tokens/s (1 GB300) + % tensor/HBM roofline"
WORKLOAD = "b2h8_l2048_nu3"
L2_BYTES = 129 * 1024 * 1024


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-rows", action="store_true", help="skip the per-row extra measurements")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    p.add_argument("--stack-steps", type=int, default=0,
                   help="only run this many token steps of the 6-layer stack workload (for profilers), then exit")
    p.add_argument("--backward-steps", type=int, default=0,
                   help="only run this many backward calls on the b4h8_l512 workload (for profilers), then exit")
    p.add_argument("--forward-steps", type=int, default=0,
                   help="only run this many forward calls on --forward-workload (for profilers), then exit")
    p.add_argument("--forward-workload", default="b4h8_l512", help="the workload of --forward-steps")
    p.add_argument("--projected-steps", type=int, default=0,
                   help="only run this many projected-forward calls on B1 H8 L1024 d_model 512 (for profilers), "
                        "then exit")
    return p.parse_args()


# ----------------------------------------------------------------- helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, source="fallback")


def forward_flops_per_head_token(C, d_dot, d_v):
    """Algorithmic FLOPs of the chunked form per (b,h,token): the chunk-local
    part plus the scan's state products, the C x C triangular products counted
    at half (only their lower triangle carries work)."""
    return prep_flops_per_head_token(C, d_dot, d_v) + scan_flops_per_head_token(d_dot, d_v)


def prep_flops_per_head_token(C, d_dot, d_v):
    """The chunk-local part: Gram, solve and the products with T and P."""
    return 2.0 * (1.5 * C * d_dot + C * d_v) + (2.0 / 3.0) * C * C


def scan_flops_per_head_token(d_dot, d_v):
    """The state part: W' S^T, Q' S^T and the update S += U^T K."""
    return 2.0 * 3.0 * d_dot * d_v


def forward_bytes(B, H, L, d_key, d_v, d_dot, io_bytes, w0=False, w_final=True):
    """Algorithmic HBM bytes of one forward: read q, k, v, beta, write y, and
    the fp32 state in / out when present."""
    return (B * H * L * io_bytes * (2 * d_key + 2 * d_v + 1)
            + (B * H * d_v * d_dot * 4) * (int(w0) + int(w_final)))


def roofline(name, flops, nbytes, ms, pk):
    """Achieved rate of one kernel against the resource that bounds it."""
    t_hbm = nbytes / (pk["hbm"] * 1e9)
    t_tc = flops / (pk["bf16"] * 1e12)
    secs = ms * 1e-3
    if t_hbm >= t_tc:
        a = nbytes / secs / 1e9
        r = {"bound": "hbm", "achieved": a, "peak": pk["hbm"], "unit": "GB/s", "frac": a / pk["hbm"]}
    else:
        a = flops / secs / 1e12
        r = {"bound": "tensor", "achieved": a, "peak": pk["bf16"], "unit": "TFLOP/s", "frac": a / pk["bf16"]}
    r.update({"kernel": name, "kernel_ms": ms, "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
              "hbm_frac": nbytes / secs / 1e9 / pk["hbm"],
              "tensor_frac": flops / secs / 1e12 / pk["bf16"], "peak_source": pk["source"]})
    return r


# fp32 FMA peak of the CUDA cores, from unit counts and clocks: 152 SMs x 128 fp32 lanes x 2 FLOP per FMA x
# the 2070 MHz maximum SM clock
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def alu_roofline(name, flops, ms):
    """Achieved fp32 rate of a path that runs on the CUDA cores' FMA units."""
    a = flops / (ms * 1e-3) / 1e12
    return {"bound": "alu", "achieved": a, "peak": FP32_ALU_TFLOPS, "unit": "TFLOP/s", "frac": a / FP32_ALU_TFLOPS,
            "kernel": name, "kernel_ms": ms, "algorithmic_flops": flops,
            "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 x 2.07 GHz"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs.

    One `nvidia-smi --query-gpu` call every `period` seconds from a thread:
    nvidia-smi's own loop mode buffers its output when writing to a pipe, so
    its samples only arrive when it exits (and are lost when it is stopped)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index, period=0.2):
        self.dev = device_index
        self.period = period
        self.lines = []
        self.failed = False
        self._stop = threading.Event()
        self._t = None

    def _query(self):
        r = subprocess.run(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                            "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=10)
        return r.stdout.strip().splitlines() if r.returncode == 0 else []

    def _loop(self):
        while not self._stop.is_set():
            try:
                self.lines.extend(self._query())
            except (OSError, subprocess.SubprocessError):
                self.failed = True
                return
            self._stop.wait(self.period)

    def start(self):
        self._t = threading.Thread(target=self._loop, daemon=True)
        self._t.start()

    def stop(self):
        self._stop.set()
        if self._t is not None:
            self._t.join(timeout=15)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons), "samples": len(sm)}


def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key, sources):
    """dram bytes per launch recorded from an ncu capture (profiles/traffic.json),
    or None when absent or when the kernel's source changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel_key)
    if not rec or rec.get("source_hash") != source_hash(sources):
        return None
    return rec.get("dram_bytes_per_launch")


def max_over_ranks(x, world, device):
    """The slowest rank's value (the job finishes when the last rank does)."""
    if world <= 1:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def replica_seed(rank, s):
    """Seed of input set s of rank `rank`: every rank runs its own replica
    (weak scaling), so the ranks' batches are independent draws."""
    return 1000 * rank + s


# ----------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    from delta_rule_linear_dpfp_gb300 import binding as fw
    from delta_rule_linear_dpfp_gb300 import build, inputs

    build.build()
    fw.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    cfg = inputs.FORWARD_CONFIGS[WORKLOAD]
    B, H, L, d_key, nu, d_v, C = (cfg[n] for n in ("B", "H", "L", "d_key", "nu", "d_v", "chunk"))
    d_dot = 2 * d_key * nu
    dt = inputs.torch_dtype(cfg["io"])
    io_bytes = 2 if dt == torch.bfloat16 else 4

    host = inputs.forward_inputs(WORKLOAD, seed=replica_seed(rank, 0))
    set_bytes = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    nsets = max(2, math.ceil(3 * L2_BYTES / set_bytes))
    sets = []
    for s in range(nsets):
        d = inputs.forward_inputs(WORKLOAD, seed=replica_seed(rank, s)) if s else host
        sets.append({k: (None if v is None else v.to(dev)) for k, v in d.items()})
    y = torch.empty(B, H, L, d_v, dtype=dt, device=dev)
    Wf = torch.empty(B, H, d_v, d_dot, dtype=torch.float32, device=dev)
    ws_bytes = fw.fw_delta_forward_workspace_size(B, H, L, d_key, nu, d_v, C, dt)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

    def step(i):
        d = sets[i % nsets]
        fw.fw_delta_forward(d["q"], d["k"], d["v"], d["beta"], W0=d.get("W0"), nu=nu, chunk=C,
                            y=y, W_final=Wf, workspace=ws, stream=stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # nvidia-smi samples from the warm-up to the end of the end-to-end loop
    clocks = ClockSampler(local_rank)
    clocks.start()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert fw.fw_device_status() == fw.FW_OK
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms_total = max_over_ranks(e0.elapsed_time(e1), world, dev)
    ms_step = ms_total / args.steps
    tokens_per_step = B * L
    value = tokens_per_step * world / (ms_step * 1e-3)

    # ---------------------------------------------------------------- e2e
    # A serving loop through the public API: every step copies its inputs
    # from pinned host memory (q, k, v, beta and W0 packed in one buffer: one
    # copy; the steps rotate over E2E_HOST_SETS distinct host buffers), runs
    # fw_delta_forward and reads y and W_final back (packed: one copy).
    # Two slots: the input copy of step i + 1 runs on a copy stream while the
    # forward of step i computes, and the read-back of step i on a third
    # stream; each step's own copies stay inside the timed region.
    names = tuple(n for n in ("q", "k", "v", "beta", "W0") if host.get(n) is not None)

    def packed(shapes_dtypes):
        offs, tot = [], 0
        for shape, dtype in shapes_dtypes:
            offs.append(tot)
            tot += (math.prod(shape) * torch.tensor([], dtype=dtype).element_size() + 255) // 256 * 256
        return offs, tot

    def views(buf, offs, shapes_dtypes):
        out = []
        for o, (shape, dtype) in zip(offs, shapes_dtypes):
            n = math.prod(shape) * torch.tensor([], dtype=dtype).element_size()
            out.append(buf[o:o + n].view(dtype).view(shape))
        return out

    in_sd = [(tuple(host[k].shape), host[k].dtype) for k in names]
    out_sd = [(tuple(y.shape), dt), (tuple(Wf.shape), torch.float32)]
    in_offs, in_tot = packed(in_sd)
    out_offs, out_tot = packed(out_sd)
    E2E_HOST_SETS = 4
    h_in = []
    for j in range(E2E_HOST_SETS):
        hb = torch.empty(in_tot, dtype=torch.uint8).pin_memory()
        src_set = host if j == 0 else inputs.forward_inputs(WORKLOAD, seed=replica_seed(rank, 1000 + j))
        for v_, src in zip(views(hb, in_offs, in_sd), (src_set[k] for k in names)):
            v_.copy_(src)
        h_in.append(hb)
    d_in = [torch.empty(in_tot, dtype=torch.uint8, device=dev) for _ in range(2)]
    d_out = [torch.empty(out_tot, dtype=torch.uint8, device=dev) for _ in range(2)]
    h_out = [torch.empty(out_tot, dtype=torch.uint8).pin_memory() for _ in range(2)]
    in_v = [views(d_in[i], in_offs, in_sd) for i in range(2)]
    out_v = [views(d_out[i], out_offs, out_sd) for i in range(2)]
    h2d = sum(math.prod(sh) * torch.tensor([], dtype=dty).element_size() for sh, dty in in_sd)
    d2h = sum(math.prod(sh) * torch.tensor([], dtype=dty).element_size() for sh, dty in out_sd)
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i, comp, reuse=True):
        sl = i & 1
        if reuse:                               # (in a graph, the first use of a slot has no predecessor)
            s_h2d.wait_event(ev_comp[sl])      # the forward that last read this slot is done
        with torch.cuda.stream(s_h2d):
            d_in[sl].copy_(h_in[i % E2E_HOST_SETS], non_blocking=True)
        ev_in[sl].record(s_h2d)
        comp.wait_event(ev_in[sl])
        if reuse:
            comp.wait_event(ev_out[sl])         # this slot's previous read-back is done
        ins = dict(zip(names, in_v[sl]))
        yo, Wo = out_v[sl]
        fw.fw_delta_forward(ins["q"], ins["k"], ins["v"], ins["beta"], W0=ins.get("W0"), nu=nu, chunk=C, y=yo,
                            W_final=Wo, workspace=ws, stream=comp)
        ev_comp[sl].record(comp)
        s_d2h.wait_event(ev_comp[sl])
        with torch.cuda.stream(s_d2h):
            h_out[sl].copy_(d_out[sl], non_blocking=True)
        ev_out[sl].record(s_d2h)

    # Measured twice over the same number of steps: eagerly (the C ABI
    # called for every step, its host-side checks inside the timed region:
    # the reported value), and with E2E_GRAPH steps captured once into a
    # CUDA graph that is then replayed (the copy streams fork from and join
    # the capture stream; every replay still copies in, computes and copies
    # out each of its steps), which takes the host's Python out of the loop.
    E2E_GRAPH = 32  # steps per replayed graph: the copy-in and copy-out at a replay boundary overlap nothing
    # as many end-to-end steps as timed steps; the graph form replays whole
    # graphs, so it covers that many rounded up to whole graphs
    e2e_steps = args.steps
    e2e_graph_steps = max(E2E_GRAPH, (args.steps + E2E_GRAPH - 1) // E2E_GRAPH * E2E_GRAPH)
    for i in range(4):                          # warm up
        e2e_step(i, stream)
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(e2e_steps):
        e2e_step(i, stream)
    stream.wait_stream(s_h2d)
    stream.wait_stream(s_d2h)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_eager_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, world, dev)

    graph = torch.cuda.CUDAGraph()
    for i in range(4):                          # warm up outside the capture
        e2e_step(i, stream)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        cap = torch.cuda.current_stream()
        fork = torch.cuda.Event()
        fork.record(cap)
        s_h2d.wait_event(fork)
        s_d2h.wait_event(fork)
        for i in range(E2E_GRAPH):
            e2e_step(i, cap, reuse=i >= 2)
        cap.wait_stream(s_h2d)
        cap.wait_stream(s_d2h)
    for _ in range(2):
        graph.replay()
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(e2e_graph_steps // E2E_GRAPH):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_graph_steps, world, dev)
    clk = clocks.stop()
    # the last step's results came back intact
    y_back = views(h_out[(E2E_GRAPH - 1) & 1], out_offs, out_sd)[0]
    assert torch.isfinite(y_back.float()).all()

    # ----------------------------------------------------------- roofline
    # fw_delta_forward runs either as one launch (chunk_fused_kernel: the
    # preparation and the walk overlapped) or as its two kernels; the two
    # kernels are also timed on their own (CUDA events on the launching
    # stream) to show the phases
    pk = peaks()
    has_w0 = host.get("W0") is not None
    launches_per_step = fw.fw_delta_forward_kernel_count(B, H, L, d_key, nu, d_v, C, torch.bfloat16)
    assert launches_per_step in (1, 2), launches_per_step
    kern = forward_kernels(fw, sets, y, Wf, ws, B, H, L, d_key, nu, d_v, C, io_bytes, stream, pk, WORKLOAD)
    fwd_name = "fw_delta_forward (one launch)" if launches_per_step == 1 else "fw_delta_forward (prepare + scan)"
    r_fwd = roofline(fwd_name, forward_flops_per_head_token(C, d_dot, d_v) * B * H * L,
                     forward_bytes(B, H, L, d_key, d_v, d_dot, io_bytes, w0=has_w0), ms_step, pk)
    r_prep, r_scan = kern["chunk_prep_kernel"], kern["chunk_scan_kernel"]
    if launches_per_step == 1:
        roof = dict(r_fwd, kernel="chunk_fused_kernel",
                    note="kernel_ms is the whole call: the one kernel plus the memset of its ready flags")
        roof["traffic"] = recorded_traffic(f"chunk_fused_kernel@{WORKLOAD}", FORWARD_SOURCES)
        kernels = {"chunk_fused_kernel": roof, "chunk_prep_kernel (two-kernel path, alone)": r_prep,
                   "chunk_scan_kernel (two-kernel path, alone)": r_scan, "forward": r_fwd}
    else:
        roof = dict(r_prep if r_prep["kernel_ms"] >= r_scan["kernel_ms"] else r_scan)
        kernels = {"chunk_prep_kernel": r_prep, "chunk_scan_kernel": r_scan, "forward": r_fwd}

    rows = None
    if rank == 0 and not args.no_rows:
        rows = measure_rows(fw, inputs, dev, stream, pk)
        for name in ROW_FORWARDS:
            rows[name] = forward_row(fw, inputs, name, dev, stream, pk)

    result = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_name(inputs.FORWARD_CONFIGS[WORKLOAD]),
                   "io": "bf16 in and out, fp32 state",
                   "global_batch": B * world, "seq_len": L,
                   "parallelism": "replicas" if world == 1 else f"replicas x{world}",
                   "l2": f"inputs rotate over {nsets} sets ({nsets * set_bytes / 2**20:.0f} MiB "
                         f"> 3x L2), no flush"},
        "clocks": clk,
        "e2e": {"value": tokens_per_step * world / (e2e_eager_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_eager_ms,
                "steps": e2e_steps, "graph_steps": e2e_graph_steps,
                "graph_value": tokens_per_step * world / (e2e_ms * 1e-3), "graph_ms_per_step": e2e_ms,
                "how": f"pinned host buffers (rotating over {E2E_HOST_SETS} distinct input sets); per step one "
                       f"packed copy in ({', '.join(names)}), fw_delta_forward through the C ABI, one packed "
                       f"copy out (y, W_final); two slots on three streams; value: the API called for every "
                       f"step; graph_value: the same steps, {E2E_GRAPH} per replayed CUDA graph"},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": roof,
        "kernels": kernels,
    }
    if rows is not None:
        result["rows"] = rows
    return result


# the sources the recorded DRAM traffic of the forward's kernels was captured from
FORWARD_SOURCES = ["delta_rule_linear_dpfp_gb300/csrc/fw_forward_tc.cu",
                   "delta_rule_linear_dpfp_gb300/csrc/fw_tc.cuh",
                   "delta_rule_linear_dpfp_gb300/csrc/fw_dpfp.cuh"]
# forward workloads measured as rows beside the headline: the nu = 1 workload, and the headline's
# shape with 8x the batch, where the serial chunk chain is not the only limit
ROW_FORWARDS = ["b4h8_l512", "b16h8_l2048_nu3"]


def phase_ms(fw, sets, y, Wf, ws, nu, C, stream, reps=200):
    """Average duration of the prepare and of the scan kernel, each timed over
    `reps` back-to-back launches with CUDA events on their stream."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(reps):
        d = sets[i % len(sets)]
        fw.fw_delta_forward_prepare(d["q"], d["k"], d["v"], d["beta"], ws, nu=nu, chunk=C, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_prep = e0.elapsed_time(e1) / reps
    e0.record(stream)
    for i in range(reps):
        fw.fw_delta_forward_scan(ws, y, W0=sets[0].get("W0"), W_final=Wf, nu=nu, chunk=C, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_scan = e0.elapsed_time(e1) / reps
    return ms_prep, ms_scan


def forward_kernels(fw, sets, y, Wf, ws, B, H, L, d_key, nu, d_v, C, io_bytes, stream, pk, workload):
    """Roofline entries of the forward's two kernels, each timed on its own."""
    d_dot = 2 * d_key * nu
    ms_prep, ms_scan = phase_ms(fw, sets, y, Wf, ws, nu, C, stream)
    BHL = B * H * L
    w0 = sets[0].get("W0") is not None
    r_prep = roofline("chunk_prep_kernel", prep_flops_per_head_token(C, d_dot, d_v) * BHL,
                      BHL * io_bytes * (2 * d_key + d_v + 1), ms_prep, pk)
    r_scan = roofline("chunk_scan_kernel", scan_flops_per_head_token(d_dot, d_v) * BHL,
                      BHL * io_bytes * d_v + B * H * d_v * d_dot * 4 * (1 + int(w0)), ms_scan, pk)
    for r in (r_prep, r_scan):
        r["traffic"] = recorded_traffic(f"{r['kernel']}@{workload}", FORWARD_SOURCES)
    return {"chunk_prep_kernel": r_prep, "chunk_scan_kernel": r_scan}


def forward_row(fw, inputs, name, dev, stream, pk, reps=50):
    """A whole forward call on one of inputs.FORWARD_CONFIGS, with its two kernels."""
    c = inputs.FORWARD_CONFIGS[name]
    B, H, L, d_key, nu, d_v, C = (c[n] for n in ("B", "H", "L", "d_key", "nu", "d_v", "chunk"))
    d_dot = 2 * d_key * nu
    one = inputs.forward_inputs(name)
    set_bytes = sum(t.numel() * t.element_size() for t in one.values() if t is not None)
    nsets = max(2, min(16, math.ceil(3 * L2_BYTES / set_bytes)))
    sets = [{k: (None if v is None else v.to(dev)) for k, v in (inputs.forward_inputs(name, seed=s) if s else one).items()}
            for s in range(nsets)]
    y = torch.empty(B, H, L, d_v, dtype=torch.bfloat16, device=dev)
    Wf = torch.empty(B, H, d_v, d_dot, dtype=torch.float32, device=dev)
    nws = fw.fw_delta_forward_workspace_size(B, H, L, d_key, nu, d_v, C, torch.bfloat16)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)

    def call(i):
        d = sets[i % nsets]
        fw.fw_delta_forward(d["q"], d["k"], d["v"], d["beta"], W0=d.get("W0"), nu=nu, chunk=C, y=y, W_final=Wf,
                            workspace=ws, stream=stream)
    ms = _time(call, reps, stream)
    w0 = sets[0].get("W0") is not None
    launches = fw.fw_delta_forward_kernel_count(B, H, L, d_key, nu, d_v, C, torch.bfloat16)
    r = roofline("fw_delta_forward (one launch)" if launches == 1 else "fw_delta_forward (prepare + scan)",
                 forward_flops_per_head_token(C, d_dot, d_v) * B * H * L,
                 forward_bytes(B, H, L, d_key, d_v, d_dot, 2, w0=w0), ms, pk)
    r["launches"] = launches
    r["tokens/s"] = B * L / (ms * 1e-3)
    r["kernels"] = forward_kernels(fw, sets, y, Wf, ws, B, H, L, d_key, nu, d_v, C, 2, stream, pk, name)
    r["workload"] = (f"B{B} H{H} L{L} d_key{d_key} nu{nu} (d_dot {d_dot}) d_v{d_v} bf16, chunk {C}, "
                     f"{'W0 in' if w0 else 'W0 = 0'}, y and W_final out, {nsets} rotating input sets")
    return r


def _time(fn, reps, stream):
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        fn(0)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(reps):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def measure_rows(fw, inputs, dev, stream, pk):
    rows = {}
    # a1 standalone: DPFP of the nu = 3 workload's q and k rows (65536 rows)
    g = torch.Generator().manual_seed(0)
    nrows = 2 * 8 * 2048 * 2
    xs = [torch.randn(nrows, 64, generator=g).to(torch.bfloat16).to(dev) for _ in range(4)]
    outs = [torch.empty(nrows, 384, dtype=torch.bfloat16, device=dev) for _ in range(4)]
    ms = _time(lambda i: fw.fw_dpfp(xs[i % 4], nu=3, out=outs[i % 4], stream=stream), 200, stream)
    nb = nrows * (64 + 384) * 2
    rows["dpfp_65536x64_nu3_bf16"] = roofline("dpfp_kernel", nrows * 384 * 4.0, nb, ms, pk)
    # a6: decode step, B256 H16 d_key64 nu2 d_v128, W 512 MiB fp32
    cfg = inputs.DECODE_CONFIGS["decode_b256"]
    B, H, d_key, nu, d_v = (cfg[n] for n in ("B", "H", "d_key", "nu", "d_v"))
    d = inputs.decode_inputs(B, H, d_key, nu, d_v, 8, "bf16", seed=0)
    dd = {k: v.to(dev) for k, v in d.items()}
    W = dd["W0"]
    yd = torch.empty(B, H, d_v, dtype=torch.bfloat16, device=dev)

    def dec(i):
        t = i % 8
        fw.fw_delta_decode_step(dd["q"][t], dd["k"][t], dd["v"][t], dd["beta"][t], W, nu=nu, y=yd,
                                stream=stream)
    ms = _time(dec, 100, stream)
    d_dot = 2 * d_key * nu
    nb = B * H * d_v * d_dot * 4 * 2 + B * H * (2 * d_key + 2 * d_v + 1) * 2
    r = roofline("decode_kernel", B * H * d_v * d_dot * 6.0, nb, ms, pk)
    r["tokens/s"] = B / (ms * 1e-3)
    # the same 128-step decode as one CUDA graph (each step its own launch inside the graph)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(128):
            t = i % 8
            fw.fw_delta_decode_step(dd["q"][t], dd["k"][t], dd["v"][t], dd["beta"][t], W, nu=nu, y=yd)
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(4):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    r["graph128_ms_per_step"] = e0.elapsed_time(e1) / (4 * 128)
    rows["decode_b256h16_nu2_dv128"] = r
    # the sum rule (linear attention, z-normalised) on the bench workload's shapes
    B, H, L, d_key, nu, d_v, C = 4, 8, 512, 64, 1, 64, 64
    d_dot = 2 * d_key * nu
    li = {k: (None if v is None else v.to(dev)) for k, v in inputs.linear_inputs(B, H, L, d_key, nu, d_v).items()}
    yl = torch.empty(B, H, L, d_v, dtype=torch.bfloat16, device=dev)
    Wl = torch.empty(B, H, d_v, d_dot, dtype=torch.float32, device=dev)
    zl = torch.empty(B, H, d_dot, dtype=torch.float32, device=dev)
    nws = fw.fw_linear_forward_workspace_size(B, H, L, d_key, nu, d_v, C, True)
    wsl = torch.empty(nws, dtype=torch.uint8, device=dev)
    ms = _time(lambda i: fw.fw_linear_forward(li["q"], li["k"], li["v"], nu=nu, normalize=True, chunk=C, y=yl,
                                              W_final=Wl, z_final=zl, workspace=wsl, stream=stream), 200, stream)
    flops = (C * d_dot + C * (d_v + 1) + 4.0 * d_dot * (d_v + 1)) * B * H * L
    nbytes = B * H * L * 2 * (2 * d_key + 2 * d_v) + B * H * (d_v + 1) * d_dot * 4
    r = roofline("fw_linear_forward (prepare + scan)", flops, nbytes, ms, pk)
    r["tokens/s"] = B * L / (ms * 1e-3)
    rows["linear_b4h8_l512_normalised"] = r
    # the projected workload from x: the projections folded into the prep, then the scan
    B, H, L, d_model, d_key, d_v, nu, C = 1, 8, 1024, 512, 64, 64, 1, 64
    d_dot = 2 * d_key * nu
    lx = inputs.layer_inputs(B, H, L, d_model, d_key, d_v)
    xp, Wp = lx["x"].to(dev), lx["W_all"].to(dev)
    yp = torch.empty(B, H, L, d_v, dtype=torch.bfloat16, device=dev)
    Wfp = torch.empty(B, H, d_v, d_dot, dtype=torch.float32, device=dev)
    nws = fw.fw_delta_forward_projected_workspace_size(B, L, d_model, H, d_key, nu, d_v, C)
    wsp = torch.empty(nws, dtype=torch.uint8, device=dev)
    ms = _time(lambda i: fw.fw_delta_forward_projected(xp, Wp, H, d_key, d_v, nu=nu, chunk=C, y=yp, W_final=Wfp,
                                                       workspace=wsp, stream=stream), 200, stream)
    N = H * (2 * d_key + d_v + 1)
    flops = 2.0 * B * L * d_model * N + forward_flops_per_head_token(C, d_dot, d_v) * B * H * L
    nbytes = B * L * d_model * 2 + d_model * N * 2 + B * H * L * d_v * 2 + B * H * d_v * d_dot * 4
    launches = fw.fw_delta_forward_kernel_count(B, H, L, d_key, nu, d_v, C, torch.bfloat16)
    r = roofline("fw_delta_forward_projected (prep from x + scan)" if launches == 2 and d_key <= 64 and d_v <= 64
                 else "fw_delta_forward_projected (projection GEMM + forward)", flops, nbytes, ms, pk)
    r["tokens/s"] = B * L / (ms * 1e-3)
    rows["projected_b1h8_l1024_dmodel512"] = r
    # the backward of the delta rule on the bench workload (dq, dk, dv, dbeta, dW0 from dy)
    c = inputs.FORWARD_CONFIGS["b4h8_l512"]
    B, H, L, d_key, nu, d_v = (c[n] for n in ("B", "H", "L", "d_key", "nu", "d_v"))
    d_dot = 2 * d_key * nu
    fi = {k: (None if v is None else v.to(dev)) for k, v in inputs.forward_inputs("b4h8_l512").items()}
    dyb = torch.randn(B, H, L, d_v, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).to(dev)
    nws = fw.fw_delta_backward_workspace_size(B, H, L, d_key, nu, d_v, torch.bfloat16)
    wsb = torch.empty(nws, dtype=torch.uint8, device=dev)
    ms = _time(lambda i: fw.fw_delta_backward(fi["q"], fi["k"], fi["v"], fi["beta"], dyb, nu=nu, workspace=wsb,
                                              stream=stream), 20, stream)
    # the recurrence's own work per head-token, whatever the method: the forward sweep (2 d_dot d_v) and
    # the reverse sweep (about 12 d_dot d_v), fp32
    flops = 14.0 * d_dot * d_v * B * H * L
    nbytes = B * H * L * 2 * (2 * 2 * d_key + 2 * 2 * d_v + 2) + B * H * d_v * d_dot * 4
    r = alu_roofline("fw_delta_backward (fp32, chunk-parallel)", flops, ms)
    r["algorithmic_bytes"] = nbytes
    r["tokens/s"] = B * L / (ms * 1e-3)
    rows["backward_b4h8_l512"] = r
    # the token-wise layer stack: one token of 256 sequences through 6 layers (d_model 512, 8 heads of 64,
    # d_ff 2048), each layer's 64 MiB of fast weights read and written once per token
    c = inputs.STACK_CONFIGS["stack_b256_l6"]
    B, H, d_key, nu, d_v, d_model, d_ff, nl = (c[n] for n in ("B", "H", "d_key", "nu", "d_v", "d_model", "d_ff",
                                                               "n_layers"))
    d_dot = 2 * d_key * nu
    si = inputs.stack_inputs(B, H, d_key, nu, d_v, d_model, d_ff, nl, 8, seed=0)
    sl = [{n: (None if t is None else t.to(dev)) for n, t in ly.items()} for ly in si["layers"]]
    sx = si["x"].to(dev)
    sg, sb = si["ln_gamma"].to(dev), si["ln_beta"].to(dev)
    so = torch.empty(B, d_model, dtype=torch.float32, device=dev)
    wss = torch.empty(fw.fw_decode_stack_workspace_size(B, H, d_key, d_v, d_model, d_ff), dtype=torch.uint8,
                      device=dev)

    def stack_step(i, st=stream):
        fw.fw_decode_stack_step(sx[i % 8], sl, H, d_key, d_v, nu=nu, ln_gamma=sg, ln_beta=sb, out=so, workspace=wss,
                                stream=st)
    ms = _time(stack_step, 50, stream)
    N = H * (2 * d_key + d_v + 1)
    wbytes = (d_model * sl[0]["W_in"].shape[1] + H * d_v * d_model + 2 * d_model * d_ff) * 2
    nbytes = nl * (2 * B * H * d_v * d_dot * 4 + wbytes) + 2 * B * d_model * 4
    flops = nl * (2.0 * B * (d_model * N + H * d_v * d_model + 2 * d_model * d_ff) + 6.0 * B * H * d_v * d_dot)
    r = roofline("fw_decode_stack_step (6 layers, 32 launches)", flops, nbytes, ms, pk)
    r["tokens/s"] = B / (ms * 1e-3)
    # the same token step captured once as a CUDA graph and replayed (8 tokens per timing)
    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(gs):
        stack_step(0, gs)
    gs.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        stack_step(0, gs)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(16):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    r["graph_ms_per_token"] = e0.elapsed_time(e1) / 16
    r["graph_tokens/s"] = B / (r["graph_ms_per_token"] * 1e-3)
    rows["stack_b256_l6_dmodel512"] = r
    return rows


def stack_only(steps):
    """`steps` token steps of the stack_b256_l6 workload through the public API
    (32 launches each), nothing else: the command the stack's launch list is
    captured from."""
    from delta_rule_linear_dpfp_gb300 import binding as fw, build, inputs
    build.build()
    fw.load()
    c = inputs.STACK_CONFIGS["stack_b256_l6"]
    B, H, d_key, nu, d_v, d_model, d_ff, nl = (c[n] for n in ("B", "H", "d_key", "nu", "d_v", "d_model", "d_ff",
                                                               "n_layers"))
    si = inputs.stack_inputs(B, H, d_key, nu, d_v, d_model, d_ff, nl, 4, seed=0)
    sl = [{n: (None if t is None else t.cuda()) for n, t in ly.items()} for ly in si["layers"]]
    sx, sg, sb = si["x"].cuda(), si["ln_gamma"].cuda(), si["ln_beta"].cuda()
    out = torch.empty(B, d_model, device="cuda")
    ws = torch.empty(fw.fw_decode_stack_workspace_size(B, H, d_key, d_v, d_model, d_ff), dtype=torch.uint8,
                     device="cuda")
    for i in range(steps):
        fw.fw_decode_stack_step(sx[i % 4], sl, H, d_key, d_v, nu=nu, ln_gamma=sg, ln_beta=sb, out=out, workspace=ws)
    torch.cuda.synchronize()
    print(json.dumps({"stack_steps": steps, "launches_per_step": 5 * nl + 2}))


def backward_only(steps):
    """`steps` fw_delta_backward calls on b4h8_l512 (bf16 I/O) through the public
    API (6 launches each), nothing else: the command the backward's profiles
    are captured from."""
    from delta_rule_linear_dpfp_gb300 import binding as fw, build, inputs
    build.build()
    fw.load()
    c = inputs.FORWARD_CONFIGS["b4h8_l512"]
    B, H, L, d_key, nu, d_v = (c[n] for n in ("B", "H", "L", "d_key", "nu", "d_v"))
    fi = {k: (None if v is None else v.cuda()) for k, v in inputs.forward_inputs("b4h8_l512").items()}
    dy = torch.randn(B, H, L, d_v, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).cuda()
    ws = torch.empty(fw.fw_delta_backward_workspace_size(B, H, L, d_key, nu, d_v, torch.bfloat16), dtype=torch.uint8,
                     device="cuda")
    for _ in range(steps):
        fw.fw_delta_backward(fi["q"], fi["k"], fi["v"], fi["beta"], dy, nu=nu, workspace=ws)
    torch.cuda.synchronize()
    print(json.dumps({"backward_steps": steps, "launches_per_step": 6}))


def forward_only(steps, name):
    """`steps` fw_delta_forward calls on one of inputs.FORWARD_CONFIGS through
    the public API, nothing else: the command the forward rows' profiles are
    captured from."""
    from delta_rule_linear_dpfp_gb300 import binding as fw, build, inputs
    build.build()
    fw.load()
    c = inputs.FORWARD_CONFIGS[name]
    B, H, L, d_key, nu, d_v, C = (c[n] for n in ("B", "H", "L", "d_key", "nu", "d_v", "chunk"))
    d = {k: (None if v is None else v.cuda()) for k, v in inputs.forward_inputs(name).items()}
    for _ in range(steps):
        fw.fw_delta_forward(d["q"], d["k"], d["v"], d["beta"], W0=d.get("W0"), nu=nu, chunk=C)
    torch.cuda.synchronize()
    print(json.dumps({"forward_steps": steps, "workload": name,
                      "launches_per_step": fw.fw_delta_forward_kernel_count(B, H, L, d_key, nu, d_v, C,
                                                                            torch.bfloat16)}))


def projected_only(steps):
    """`steps` fw_delta_forward_projected calls on B1 H8 L1024 d_model 512
    through the public API, nothing else (the projected row's profile)."""
    from delta_rule_linear_dpfp_gb300 import binding as fw, build, inputs
    build.build()
    fw.load()
    B, H, L, d_model, d_key, d_v = 1, 8, 1024, 512, 64, 64
    lx = inputs.layer_inputs(B, H, L, d_model, d_key, d_v)
    x, W = lx["x"].cuda(), lx["W_all"].cuda()
    for _ in range(steps):
        fw.fw_delta_forward_projected(x, W, H, d_key, d_v)
    torch.cuda.synchronize()
    print(json.dumps({"projected_steps": steps}))


def workload_name(cfg):
    """The bench workload as both arms name it in their config."""
    d_dot = 2 * cfg["d_key"] * cfg["nu"]
    w0 = f"W0 ~ N(0, {cfg['w0_var']}) in" if cfg.get("w0_var") else "W0 = 0"
    return (f"{WORKLOAD}: B{cfg['B']} H{cfg['H']} L{cfg['L']} d_key{cfg['d_key']} nu{cfg['nu']} "
            f"(d_dot {d_dot}) d_v{cfg['d_v']}, chunk {cfg['chunk']}, {w0}, y and W_final out")


# ------------------------------------------------------------ the oracle
class OracleSample:
    """The fp64 CPU oracle on the host cores over a bounded sample of the
    workload: whole (b,h) sequences when the time budget allows several, else
    the first tokens of one sequence.  Inputs are drawn and widened once."""

    def __init__(self, B, H, L, d_key, nu, d_v, io, w0_var=None, seed=0):
        import numpy as np

        import oracle
        from delta_rule_linear_dpfp_gb300 import inputs
        self.oracle, self.np = oracle, np
        d = inputs.random_forward_inputs(B, H, L, d_key, nu, d_v, io, w0_var, seed)
        flat = lambda t: np.ascontiguousarray(
            t.float().double().numpy().reshape((1, B * H) + tuple(t.shape[2:])))
        self.f = {k: flat(v) for k, v in d.items() if v is not None}
        self.B, self.H, self.L, self.nu = B, H, L, nu
        self.threads = oracle.default_threads()
        t0 = time.perf_counter()
        self._run(1, L, 1)
        self.t_pair = max(time.perf_counter() - t0, 1e-6)

    def _run(self, pairs, tokens, threads):
        f = self.f
        sl = lambda a: self.np.ascontiguousarray(a[:, :pairs, :tokens])
        W0 = self.np.ascontiguousarray(f["W0"][:, :pairs]) if "W0" in f else None
        self.oracle.delta_forward(sl(f["q"]), sl(f["k"]), sl(f["v"]), sl(f["beta"]), W0, self.nu,
                                  1e-6, threads)

    def plan(self, budget_s, threads):
        pairs = int(max(1, min(self.B * self.H, budget_s * threads / self.t_pair)))
        tokens = self.L
        if pairs == 1 and budget_s < self.t_pair:
            tokens = int(max(1, self.L * budget_s / self.t_pair))
        return pairs, tokens

    def measure(self, budget_s, max_threads=None):
        """Returns (tokens/s, threads used, sample description, seconds)."""
        cap = self.threads if max_threads is None else min(self.threads, max_threads)
        pairs, tokens = self.plan(budget_s, cap)
        threads = min(cap, pairs)
        t0 = time.perf_counter()
        self._run(pairs, tokens, threads)
        dt = time.perf_counter() - t0
        sample = (f"{pairs} of {self.B * self.H} (b,h) sequences x {tokens} of {self.L} tokens, "
                  f"fp64, {threads} threads")
        return pairs * tokens / self.H / dt, threads, sample, dt


def run_reference(args, rank, world):
    from delta_rule_linear_dpfp_gb300 import inputs
    cfg = inputs.FORWARD_CONFIGS[WORKLOAD]
    B, H, L, d_key, nu, d_v = (cfg[n] for n in ("B", "H", "L", "d_key", "nu", "d_v"))
    budget = max(0.002, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    orc = OracleSample(B, H, L, d_key, nu, d_v, cfg["io"], cfg.get("w0_var"))
    for _ in range(args.warmup):
        orc.measure(budget)
    tok, secs = 0.0, 0.0
    for _ in range(args.steps):
        v, cores, sample, dt = orc.measure(budget)
        tok += v * dt
        secs += dt
    value = tok / secs
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_name(cfg), "io": "fp64 throughout (the oracle)",
                   "global_batch": B, "seq_len": L, "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if args.stack_steps:
        stack_only(args.stack_steps)
        return
    if args.backward_steps:
        backward_only(args.backward_steps)
        return
    if args.forward_steps:
        forward_only(args.forward_steps, args.forward_workload)
        return
    if args.projected_steps:
        projected_only(args.projected_steps)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu:
            from delta_rule_linear_dpfp_gb300 import inputs
            cfg = inputs.FORWARD_CONFIGS[WORKLOAD]
            orc = OracleSample(cfg["B"], cfg["H"], cfg["L"], cfg["d_key"], cfg["nu"], cfg["d_v"],
                               cfg["io"], cfg.get("w0_var"))
            v, cores, sample, _ = orc.measure(12.0)
            v1, _, sample1, _ = orc.measure(6.0, max_threads=1)
            res["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                   "sample": sample,
                                   "single_thread": {"value": v1, "unit": "tokens/s", "cores": 1,
                                                     "sample": sample1}}
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
