#!/usr/bin/env python
"""Benchmark of the fused MLA decode query projection on one GB300.

Workload (one "step"): H = 16 heads, for each weight format / output dtype
pair (BF16 weights -> BF16 query, MXFP8 weights -> E4M3 query) and each
token count M in {1, 2, 4, 8, 16, 32}, one replay of a CUDA graph holding
one fused-query launch per layer over L distinct layers (L = 128 for BF16,
256 for MXFP8 so that the rotated weights, 256 / 264 MiB, are about twice
the 126 MiB L2), each launch reading its own weights, q_nope, q_pe and
writing its own [M,16,576] output.  Launches use programmatic dependent
launch (weights streamed before the dependency wait), the way consecutive
layers run in a decode step.

Metric: achieved HBM GB/s = algorithmic bytes (weights + scales + q_nope +
q_pe + output, per layer call) / time, and microseconds per layer call.

--op v_up measures the V up-projection after attention instead
(out[m,h,:128] = x[m,h,:512] @ W_UV[h], BF16 or MXFP8 W_UV, BF16 output),
same layer rotation, same metric on its own bytes (W_UV + scales + x + out).

--impl reference times the float64 CPU oracle on a bounded sample of the
same workload on the host cores (the only other code path this file runs).
"""

from __future__ import annotations

import os

# The CPU oracle leg runs on the host cores this process may use: numpy's
# BLAS gets that many threads (set before numpy loads it).  A one-core figure
# is taken in a child process with MLAQP_BENCH_BLAS_THREADS=1.
HOST_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
BLAS_THREADS = int(os.environ.get("MLAQP_BENCH_BLAS_THREADS", str(HOST_CORES)))
for _var in ("OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "OMP_NUM_THREADS"):
    os.environ[_var] = str(BLAS_THREADS)

import argparse
import json
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

H = 16
M_POINTS = (1, 2, 4, 8, 16, 32)
FORMATS = (("bf16", "bf16"), ("mxfp8", "e4m3"))
DEFAULT_LAYERS = {"bf16": 128, "mxfp8": 256}


def layers_for(fmt, h, v_up=False):
    """Rotated layers per graph: the H=16 defaults, raised for fewer heads so
    that the weights of one replay stay at least twice the L2 size."""
    per_layer = h * 512 * 128 * (2 if fmt == "bf16" else 1)
    need = -(-2 * L2_BYTES // per_layer)
    return max(DEFAULT_LAYERS[fmt], -(-need // 32) * 32)
CONFIG_INDEX = {"bf16": 1, "mxfp8": 3}  # seed family 1000*i + layer
V_CONFIG_INDEX = {"bf16": 6, "mxfp8": 7}
V_FORMATS = (("bf16", "bf16"), ("mxfp8", "bf16"))
Q_SCALE_SEED = 3
L2_BYTES = 126 * 2**20


def v_up_algorithmic_bytes(M, weight_format, h=H, latent=512, v_dim=128):
    wb = 2 if weight_format == "bf16" else 1
    scales = h * latent * (v_dim // 32) if weight_format == "mxfp8" else 0
    return h * latent * v_dim * wb + scales + 2 * M * h * latent + 2 * M * h * v_dim


def algorithmic_bytes(M, weight_format, out_dtype, h=H, nope=128):
    wb = 2 if weight_format == "bf16" else 1
    ob = 2 if out_dtype == "bf16" else 1
    scales = h * nope * 16 if weight_format == "mxfp8" else 0
    return h * nope * 512 * wb + scales + 2 * M * h * nope + 2 * M * h * 64 + M * h * 576 * ob


# --------------------------------------------------------------------------- device layer sets

class LayerSet:
    """L layers of one weight format resident on the GPU, plus per-M input
    and output buffers laid out [L, M, H, *] so each launch reads its own."""

    def __init__(self, weight_format, out_dtype, n_layers, h=H, m_points=M_POINTS, device="cuda",
                 config_index=None, nope=128, arm="auto", distinct=None, share=None):
        import torch
        from mla_decode_query_gb300 import inputs

        self.weight_format, self.out_dtype, self.L, self.H, self.K = weight_format, out_dtype, n_layers, h, nope
        self.arm = arm
        self.pdl_mode = 1
        self.shared_io = False  # True: every layer reads and writes the same q / out buffers
        self.m_points = tuple(m_points)
        ci = CONFIG_INDEX[weight_format] if config_index is None else config_index
        m_max = max(32, max(self.m_points))  # the first 32 token rows do not depend on m_max
        # `distinct` < n_layers: generate that many layers and repeat them at
        # distinct addresses (timing runs: the rotated bytes still stream from
        # DRAM); `share`: reuse another set's weights and inputs (same format
        # and head count, another output dtype).
        if share is not None:
            self.host, self.weight, self.scale = share.host, share.weight, share.scale
        else:
            nd = n_layers if not distinct else min(distinct, n_layers)
            gen = [inputs.make_layer(inputs.layer_seed(ci, l), h, weight_format, m_max=m_max, nope=nope)
                   for l in range(nd)]
            self.host = [gen[l % nd] for l in range(n_layers)]
            wdt = torch.int16 if weight_format == "bf16" else torch.uint8
            w = np.stack([d["weight"] for d in gen])
            w = torch.from_numpy(w.view(np.int16) if weight_format == "bf16" else w).to(device)
            reps = -(-n_layers // nd)
            self.weight = w.repeat((reps,) + (1,) * (w.dim() - 1))[:n_layers].contiguous()
            assert self.weight.dtype == wdt
            self.scale = None
            if weight_format == "mxfp8":
                sc = torch.from_numpy(np.stack([d["weight_scale"] for d in gen])).to(device)
                self.scale = sc.repeat((reps,) + (1,) * (sc.dim() - 1))[:n_layers].contiguous()
        self.q_scale_value = np.float32(inputs.make_q_scale(Q_SCALE_SEED)) if out_dtype == "e4m3" else None
        self.q_scale = (torch.tensor([self.q_scale_value], dtype=torch.float32, device=device)
                        if out_dtype == "e4m3" else None)
        odt = torch.int16 if out_dtype == "bf16" else torch.uint8
        self.q_nope_host, self.q_pe_host, self.q_nope, self.q_pe, self.out = {}, {}, {}, {}, {}
        for M in self.m_points:
            if share is not None:
                self.q_nope_host[M], self.q_pe_host[M] = share.q_nope_host[M], share.q_pe_host[M]
                self.q_nope[M], self.q_pe[M] = share.q_nope[M], share.q_pe[M]
            else:
                qn = np.stack([d["q_nope"][:M] for d in self.host]).view(np.int16)
                qp = np.stack([d["q_pe"][:M] for d in self.host]).view(np.int16)
                self.q_nope_host[M] = torch.from_numpy(qn).pin_memory()
                self.q_pe_host[M] = torch.from_numpy(qp).pin_memory()
                self.q_nope[M] = self.q_nope_host[M].to(device)
                self.q_pe[M] = self.q_pe_host[M].to(device)
            self.out[M] = torch.zeros((n_layers, M, h, 576), dtype=odt, device=device)

    def host_inputs(self, M):
        return [self.q_nope_host[M], self.q_pe_host[M]]

    def dev_inputs(self, M):
        return [self.q_nope[M], self.q_pe[M]]

    def kernel_name(self, M):
        """The kernel the library launches for M (its own plan, this device's SM count)."""
        import torch
        import mla_decode_query_gb300 as mq
        st, p = mq.mlaqp_debug_plan(M, self.H, self.weight_format, self.out_dtype, nope_dim=self.K,
                                    pdl=self.pdl_mode, arm=self.arm,
                                    sm_count=torch.cuda.get_device_properties(0).multi_processor_count)
        mq.check(st)
        return {"cta_mma": "mlaqp_fused_query_kernel", "tcgen05": "mlaqp_fused_query_large_kernel"}.get(
            p["arm"], "mlaqp_query_warp_kernel")

    def layer_args(self, M, l):
        io = 0 if self.shared_io else l
        return dict(q_nope=self.q_nope[M][io], q_pe=self.q_pe[M][io], weight=self.weight[l],
                    weight_scale=None if self.scale is None else self.scale[l], out=self.out[M][io],
                    out_row_stride=576 * self.H, q_scale=self.q_scale, M=M, H=self.H,
                    weight_format=self.weight_format, out_dtype=self.out_dtype)

    def launch_all(self, M, pdl=True, stream=None):
        import mla_decode_query_gb300 as mq
        if self.arm != "auto":  # a forced kernel form (measurement hook)
            for l in range(self.L):
                a = self.layer_args(M, l)
                mq.check(mq.mlaqp_debug_run_arm(a["q_nope"], self.H * self.K, self.K, a["q_pe"], self.H * 64, 64,
                                                a["weight"], a["weight_scale"], a["out"], a["out_row_stride"],
                                                a["q_scale"], M, self.H, self.K, self.weight_format, self.out_dtype,
                                                pdl=pdl, arm=self.arm, stream=stream))
            return
        if self.K != 128 or (pdl and self.pdl_mode == 2):  # the general entry point: nope dim, strides, pdl mode
            for l in range(self.L):
                a = self.layer_args(M, l)
                mq.check(mq.mlaqp_run_strided(a["q_nope"], self.H * self.K, self.K, a["q_pe"], self.H * 64, 64,
                                              a["weight"], a["weight_scale"], a["out"], a["out_row_stride"],
                                              a["q_scale"], M, self.H, self.K, self.weight_format, self.out_dtype,
                                              pdl=self.pdl_mode if pdl else 0, stream=stream))
            return
        run = mq.mlaqp_run_pdl if pdl else mq.mlaqp_run
        for l in range(self.L):
            mq.check(run(**self.layer_args(M, l), stream=stream))

    def capture(self, M, pdl=True):
        import torch
        import mla_decode_query_gb300 as mq
        mq.check(mq.mlaqp_prewarm(self.H, max(self.m_points), self.weight_format, self.out_dtype))
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.launch_all(M, pdl, stream=s)  # untimed eager warm-up
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.launch_all(M, pdl)
        return g

    def bytes_per_call(self, M):
        return algorithmic_bytes(M, self.weight_format, self.out_dtype, self.H, self.K)


class VLayerSet:
    """L layers of W_UV in one weight format, plus per-M attention outputs x
    and BF16 results laid out [L, M, H, *]; the V up-projection's LayerSet."""

    def __init__(self, weight_format, n_layers, h=H, m_points=M_POINTS, device="cuda"):
        import torch
        from mla_decode_query_gb300 import inputs

        self.weight_format, self.out_dtype, self.L, self.H = weight_format, "bf16", n_layers, h
        self.pdl_mode = 1
        self.m_points = tuple(m_points)
        ci = V_CONFIG_INDEX[weight_format]
        m_max = max(32, max(self.m_points))
        self.host = [inputs.make_v_layer(inputs.layer_seed(ci, l), h, weight_format, m_max=m_max)
                     for l in range(n_layers)]
        w = np.stack([d["weight"] for d in self.host])
        self.weight = torch.from_numpy(w.view(np.int16) if weight_format == "bf16" else w).to(device)
        self.scale = None
        if weight_format == "mxfp8":
            self.scale = torch.from_numpy(np.stack([d["weight_scale"] for d in self.host])).to(device)
        self.x_host, self.x, self.out = {}, {}, {}
        for M in self.m_points:
            self.x_host[M] = torch.from_numpy(np.stack([d["x"][:M] for d in self.host]).view(np.int16)).pin_memory()
            self.x[M] = self.x_host[M].to(device)
            self.out[M] = torch.zeros((n_layers, M, h, 128), dtype=torch.int16, device=device)

    def host_inputs(self, M):
        return [self.x_host[M]]

    def dev_inputs(self, M):
        return [self.x[M]]

    def kernel_name(self, M):
        """The kernel the library launches for M (its own plan, this device's SM count)."""
        import torch
        import mla_decode_query_gb300 as mq
        st, p = mq.mlaqp_debug_v_plan(M, self.H, self.weight_format, pdl=self.pdl_mode,
                                      sm_count=torch.cuda.get_device_properties(0).multi_processor_count)
        mq.check(st)
        return {"plain": "mlaqp_v_up_kernel", "multicast": "mlaqp_v_up_mc_kernel"}.get(
            p["form"], "mlaqp_v_up_large_kernel")

    def launch_all(self, M, pdl=True, stream=None):
        import mla_decode_query_gb300 as mq
        for l in range(self.L):
            mq.check(mq.mlaqp_v_up_run(self.x[M][l], self.H * 512, 512, self.weight[l],
                                       None if self.scale is None else self.scale[l], self.out[M][l],
                                       128 * self.H, M, self.H, self.weight_format,
                                       pdl=self.pdl_mode if pdl else 0, stream=stream))

    def capture(self, M, pdl=True):
        import torch
        import mla_decode_query_gb300 as mq
        mq.check(mq.mlaqp_v_up_prewarm(self.H, max(self.m_points), self.weight_format))
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.launch_all(M, pdl, stream=s)  # untimed eager warm-up
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.launch_all(M, pdl)
        return g

    def bytes_per_call(self, M):
        return v_up_algorithmic_bytes(M, self.weight_format, self.H)


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index, self.proc, self.lines = gpu_index, None, []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
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
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- distributed plumbing

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate_over_ranks(local_ms, local_bytes, world_size, backend_device=None):
    """Whole-job numbers: max time over ranks, sum of bytes over ranks."""
    if world_size == 1:
        return local_ms, local_bytes
    import torch
    import torch.distributed as dist
    dev = backend_device or "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    b = torch.tensor([float(local_bytes)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), float(b.item())


# --------------------------------------------------------------------------- CPU oracle timing

def oracle_samples(op="query"):
    """One layer of each format (layer 0 of its rotated set), host bits."""
    from mla_decode_query_gb300 import inputs
    samples = []
    if op == "v_up":
        for fmt, od in V_FORMATS:
            samples.append((fmt, od, inputs.make_v_layer(inputs.layer_seed(V_CONFIG_INDEX[fmt], 0), H, fmt), None))
        return samples
    for fmt, od in FORMATS:
        d = inputs.make_layer(inputs.layer_seed(CONFIG_INDEX[fmt], 0), H, fmt)
        qs = inputs.make_q_scale(Q_SCALE_SEED) if od == "e4m3" else None
        samples.append((fmt, od, d, qs))
    return samples


def time_oracle(budget_s, samples, m_points=M_POINTS, op="query"):
    """Time the oracle, as it stands, on a bounded sample: one layer call per
    (format, M) point, repeated until `budget_s` is spent (at least once).
    Returns (GB/s, calls, seconds)."""
    import oracle
    calls, nbytes, t0 = 0, 0, time.perf_counter()
    while True:
        for fmt, od, d, qs in samples:
            for M in m_points:
                if op == "v_up":
                    oracle.mla_v_up(d["x"][:M], d["weight"], d["weight_scale"], fmt)
                    nbytes += v_up_algorithmic_bytes(M, fmt)
                else:
                    oracle.mla_query(d["q_nope"][:M], d["q_pe"][:M], d["weight"], d["weight_scale"], fmt, od, qs)
                    nbytes += algorithmic_bytes(M, fmt, od)
                calls += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return nbytes / el / 1e9, calls, el


def oracle_threads():
    return BLAS_THREADS


def oracle_one_core(budget_s, op):
    """The same oracle timing in a child process whose BLAS has one thread."""
    env = dict(os.environ, MLAQP_BENCH_BLAS_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-only", "--cpu-budget", str(budget_s), "--op", op]
    try:
        out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=budget_s * 4 + 120)
        return json.loads(out.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError) as e:
        return {"error": str(e)[:200]}


# --------------------------------------------------------------------------- main arms

def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    samples = oracle_samples()
    for _ in range(args.warmup):
        time_oracle(0.0, samples)
    nbytes, total = 0.0, 0.0
    for _ in range(args.steps):
        gbs, calls, el = time_oracle(0.0, samples)
        total += el
        nbytes += gbs * el * 1e9
    value = nbytes / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "step": "one oracle layer call per (format, M) point: 12 calls"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle_threads(), "kind": "oracle",
                         "sample": "per step, one layer call of each of the 12 (format, M) points"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


METRIC_V = ("achieved HBM GB/s of the MLA V up-projection (W_UV+scales+x+out bytes per layer call / time), "
            "H=16, M in 1..32, BF16 and MXFP8 W_UV")
WORKLOAD_V = ("MLA V up-projection, H=16, latent 512 -> v 128; BF16 and MXFP8 W_UV, BF16 out; "
              "M in {1,2,4,8,16,32}; 128 (BF16) / 256 (MXFP8) rotated layers per CUDA-graph replay")
METRIC = ("achieved HBM GB/s of the fused MLA decode query projection (weights+scales+q_nope+q_pe+out "
          "bytes per layer call / time), H=16, M in 1..32, BF16 and MXFP8 weights")
WORKLOAD = ("fused MLA query projection, H=16, K=128, N=512, rope=64; BF16->BF16 and MXFP8->E4M3; "
            "M in {1,2,4,8,16,32}; 128 (BF16) / 256 (MXFP8) rotated layers per CUDA-graph replay")


def workload_name(nope, m_points, heads=(16,), formats=FORMATS, v_up=False):
    """The workload of a run, named by what it is; the default run's name is WORKLOAD."""
    w = WORKLOAD_V if v_up else WORKLOAD
    w = w.replace("M in {1,2,4,8,16,32}", "M in {" + ",".join(map(str, m_points)) + "}")
    if tuple(heads) != (16,):
        w = w.replace("H=16", "H in {" + ",".join(map(str, heads)) + "}")
    if not v_up and tuple(formats) != FORMATS:
        w = w.replace("BF16->BF16 and MXFP8->E4M3",
                      ", ".join(f"{a.upper()}->{b.upper()}" for a, b in formats))
    if not v_up and (tuple(heads) != (16,)):
        w = w.replace("128 (BF16) / 256 (MXFP8) rotated layers", "rotated layers (at least 2x L2 of weights)")
    return w if nope == 128 else w.replace("K=128", f"K={nope}")


def run_gpu(args):
    import torch
    import mla_decode_query_gb300 as mq

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    mq.load_library()
    if args.policy:
        trig, cap = (int(x) for x in args.policy.split(":"))
        mq.check(mq.mlaqp_debug_set_policy(trig, cap))

    m_points = tuple(int(x) for x in args.m.split(",")) if args.m else M_POINTS
    v_up = args.op == "v_up"
    formats = [f for f in (V_FORMATS if v_up else FORMATS) if not args.formats or f[0] in args.formats.split(",")]
    if args.pairs:  # explicit weight:output pairs, e.g. bf16:e4m3
        formats = [tuple(x.split(":")) for x in args.pairs.split(",")]
    heads = tuple(int(x) for x in args.heads.split(","))
    multi = len(heads) > 1
    sets = []
    for h in heads:
        for fmt, od in formats:
            L = args.layers or layers_for(fmt, h, v_up)
            sets.append(VLayerSet(fmt, L, h=h, m_points=m_points) if v_up else
                        LayerSet(fmt, od, L, h=h, m_points=m_points, nope=args.nope, arm=args.arm))

    for s in sets:
        s.pdl_mode = args.pdl_mode

    def key(s):
        return f"{s.weight_format}->{s.out_dtype}" + (f" H{s.H}" if multi else "")
    points = [(s, M) for s in sets for M in m_points]
    graphs = [s.capture(M, pdl=not args.no_pdl) for s, M in points]
    alt = None
    if not args.no_pdl and not args.pdl_only:
        alt = [s.capture(M, pdl=False) for s, M in points]
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    # untimed warm-up
    for _ in range(args.warmup):
        for g in graphs:
            g.replay()
    torch.cuda.synchronize()

    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in points]
          for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_start.record(stream)
    for k in range(args.steps):
        for i, g in enumerate(graphs):
            ev[k][i][0].record(stream)
            g.replay()
            ev[k][i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if ws > 1:
        torch.distributed.barrier()
    local_ms = t_start.elapsed_time(t_end)
    step_bytes = sum(s.bytes_per_call(M) * s.L for s, M in points)
    total_ms, total_bytes = aggregate_over_ranks(local_ms, step_bytes * args.steps, ws,
                                                 backend_device=f"cuda:{local}")
    value = total_bytes / (total_ms * 1e-3) / 1e9

    per_point = []
    kern_ms = {key(s): 0.0 for s in sets}
    kern_bytes = {key(s): 0 for s in sets}
    for i, (s, M) in enumerate(points):
        ms = [ev[k][i][0].elapsed_time(ev[k][i][1]) for k in range(args.steps)]
        med = statistics.median(ms)
        us = 1e3 * med / s.L
        p10, p90 = (1e3 * float(np.percentile(ms, q)) / s.L for q in (10, 90))
        per_point.append({"weights": s.weight_format, "out": s.out_dtype, "H": s.H, "M": M, "layers": s.L,
                          "us_per_layer": round(us, 4), "us_p10": round(p10, 4), "us_p90": round(p90, 4),
                          "gbs": round(s.bytes_per_call(M) / (us * 1e-6) / 1e9, 1)})
        kern_ms[key(s)] += sum(ms)
        kern_bytes[key(s)] += s.bytes_per_call(M) * s.L * args.steps

    if alt is not None:  # context: the same graphs launched without PDL (plain stream order)
        for i, (s, M) in enumerate(points):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            for _ in range(args.warmup):
                alt[i].replay()
            a.record(stream)
            for _ in range(args.steps):
                alt[i].replay()
            b.record(stream)
            torch.cuda.synchronize()
            per_point[i]["us_per_layer_no_pdl"] = round(1e3 * a.elapsed_time(b) / args.steps / s.L, 4)

    # end-to-end through the public API with host buffers
    e2e = None if args.no_e2e else run_e2e(sets, graphs, points, args)

    peaks = load_peaks()
    launches = args.steps * sum(s.L for s, _ in points)
    dominant = max(kern_ms, key=kern_ms.get)
    ach = kern_bytes[dominant] / (kern_ms[dominant] * 1e-3) / 1e9
    traffic_table = None if (v_up or args.nope != 128 or heads != (16,)) else measured_traffic()  # K=128, H=16
    traffic = None
    dom_points = [(s, M) for s, M in points if key(s) == dominant]
    if traffic_table and all((dominant, M) in traffic_table for _, M in dom_points):
        traffic = round(sum(traffic_table[(dominant, M)] * s.L for s, M in dom_points) /
                        sum(s.L for s, _ in dom_points))
    kernel_names = sorted({s.kernel_name(M) for s, M in dom_points})
    roof = {"bound": "hbm", "kernel": f"{' + '.join(kernel_names)} ({dominant})",
            "achieved": round(ach, 1), "peak": peaks[0], "unit": "GB/s",
            "frac": round(ach / peaks[0], 4), "peak_source": peaks[1], "traffic": traffic,
            "traffic_source": (TRAFFIC_FILE if traffic else
                               "no committed per-launch ncu table for this workload (the query op, K=128, H=16, "
                               "M in {1,2,4,8,16,32} has one)" if (v_up or args.nope != 128 or heads != (16,)
                                                                  or not all(M in M_POINTS for _, M in dom_points))
                               else "kernel changed since the last ncu capture"),
            "algorithmic_bytes_per_launch": round(kern_bytes[dominant] / (args.steps * sum(s.L for s, _ in dom_points))),
            "per_kernel_gbs": {f: round(kern_bytes[f] / (kern_ms[f] * 1e-3) / 1e9, 1) for f in kern_ms}}
    floor = launch_floor(args.steps, args.warmup)
    if rank == 0:
        line = {
            "metric": METRIC_V if v_up else METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_name(args.nope, m_points, heads, tuple(formats), v_up),
                       "heads": heads[0] if not multi else list(heads), "nope_dim": args.nope,
                       "m_points": list(m_points), "arm": args.arm,
                       **({"policy": args.policy} if args.policy else {}),
                       **({"pdl_mode": args.pdl_mode} if args.pdl_mode != 1 else {}),
                       "layers": {key(s): s.L for s in sets}, "pdl": not args.no_pdl,
                       "l2": f"rotated weights per replay {[s.L * s.bytes_per_call(1) >> 20 for s in sets]} MiB "
                             f"vs L2 {L2_BYTES >> 20} MiB (inputs larger than L2, no flush)",
                       "parallelism": f"replicas{ws}"},
            "us_per_layer_mean": round(1e3 * total_ms / args.steps / sum(s.L for s, _ in points), 4),
            "launch_floor_us": floor,
            "points": per_point,
            "roofline": roof,
            "gpu_launches": launches,
            "clocks": clk,
            "e2e": e2e,
        }
        if not args.no_extras and not v_up:
            line["config0_isolated_call"] = isolated_calls(max(20, args.steps))
            line["behind_producer"] = behind_producer(max(5, args.steps), args.warmup)
            line["workspace_reuse"] = workspace_reuse(args.sweep_steps, args.warmup)
            st = args.sweep_steps
            line["config4_sweep"] = {
                "columns": ["pair", "H", "M", "us_per_layer", "gbs"],
                "rows": sweep([("bf16", "bf16"), ("bf16", "e4m3"), ("mxfp8", "bf16"), ("mxfp8", "e4m3")],
                              (8, 11, 16), M_POINTS, st, args.warmup, 4)}
            all_m = tuple(range(1, 33))
            line["config2_points"] = {"columns": ["pair", "H", "M", "us_per_layer", "gbs"],
                                      "rows": sweep([("mxfp8", "bf16")], (8,), all_m, st, args.warmup, 2)}
            line["config3_points"] = {"columns": ["pair", "H", "M", "us_per_layer", "gbs"],
                                      "rows": sweep([("mxfp8", "e4m3")], (16,), all_m, st, args.warmup, 3)}
        if not args.no_cpu_baseline:
            gbs, calls, el = time_oracle(args.cpu_budget, oracle_samples(args.op), op=args.op)
            line["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": oracle_threads(),
                                    "host_cores": HOST_CORES, "kind": "oracle",
                                    "sample": f"{calls} oracle layer calls over 2 formats x M in "
                                              f"{{{','.join(map(str, M_POINTS))}}} (H={H}), {el:.1f} s, "
                                              f"layer 0 of each format; BLAS threads = usable host cores",
                                    "one_core": oracle_one_core(max(3.0, args.cpu_budget / 2), args.op)}
        print(json.dumps(line))
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def time_graph(g, layers, steps, warmup, stream=None):
    """Median over `steps` individually timed replays of graph `g`, in us per
    layer (the graph holds `layers` layer calls)."""
    import torch
    stream = stream or torch.cuda.current_stream()
    for _ in range(warmup):
        g.replay()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        a.record(stream)
        g.replay()
        b.record(stream)
    torch.cuda.synchronize()
    return 1e3 * statistics.median(a.elapsed_time(b) for a, b in ev) / layers


def sweep(pairs, heads, m_points, steps, warmup, config_index, distinct=32):
    """us per layer call and GB/s of every (pair, H, M): 128-512-layer PDL
    graph replays (at least twice the L2 of rotated weights), `distinct`
    generated layers repeated at distinct addresses."""
    import torch
    rows = []
    for h in heads:
        base = {}
        for fmt, od in pairs:
            ls = LayerSet(fmt, od, layers_for(fmt, h), h=h, m_points=m_points, config_index=config_index,
                          distinct=distinct, share=base.get(fmt))
            base.setdefault(fmt, ls)
            for M in m_points:
                g = ls.capture(M)
                us = time_graph(g, ls.L, steps, warmup)
                rows.append([f"{fmt}->{od}", h, M, round(us, 4), round(ls.bytes_per_call(M) / (us * 1e-6) / 1e9, 1)])
                del g
            del ls
        del base
        torch.cuda.empty_cache()
    return rows


def workspace_reuse(steps, warmup):
    """The headline chains (H = 16, rotated weights) with one q_nope / q_pe
    buffer and one output workspace shared by every layer, as in a decode
    step, where the producer has just written q and attention reads the
    output next.  The headline `points` rotate q and out with the weights."""
    rows = []
    for fmt, od in FORMATS:
        ls = LayerSet(fmt, od, layers_for(fmt, H), m_points=M_POINTS, distinct=32)
        ls.shared_io = True
        for M in M_POINTS:
            g = ls.capture(M)
            us = time_graph(g, ls.L, steps, warmup)
            rows.append([f"{fmt}->{od}", M, round(us, 4), round(ls.bytes_per_call(M) / (us * 1e-6) / 1e9, 1)])
            del g
        del ls
    return {"columns": ["pair", "M", "us_per_layer", "gbs"], "rows": rows,
            "note": "weights rotated as in the headline; q and out shared by all layers (a reused workspace)"}


def isolated_calls(steps):
    """One layer call on its own (no dependent chain): a CUDA graph of one
    plain launch, each replay timed alone.  warm: back to back (weights in
    L2 after the first); cold: a 256 MiB write before every replay evicts
    the weights and inputs from L2."""
    import torch
    out = {}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for fmt, od, ci in (("bf16", "bf16", 0), ("mxfp8", "e4m3", 3)):
        ls = LayerSet(fmt, od, 1, h=H, m_points=(1,), config_index=ci)
        g = ls.capture(1, pdl=False)
        warm = time_graph(g, 1, steps, 3)
        ms = []
        for _ in range(steps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            ms.append(a.elapsed_time(b))
        out[f"{fmt}->{od} H{H} M1"] = {"warm_us": round(warm, 4), "cold_us": round(1e3 * statistics.median(ms), 4)}
        del g, ls
    return out


def behind_producer(steps, warmup, m_points=(1, 8, 32)):
    """The op the way a decode step runs it: each layer call follows the
    kernels that produce its q_nope and q_pe (here two elementwise PyTorch
    kernels writing them, which, like most producers, do not trigger
    dependent launches early).  Graphs of 128 (BF16) / 256 (MXFP8) such
    layer steps, with the op launched with and without PDL, and with and
    without mlaqp_prefetch_weights on a parallel branch forked before the
    producers; op_us = layer step - the same graph without the op."""
    import torch
    import mla_decode_query_gb300 as mq
    res = []
    for fmt, od in FORMATS:
        ls = LayerSet(fmt, od, DEFAULT_LAYERS[fmt], h=H, m_points=m_points, distinct=32)
        for M in m_points:
            src_n, src_p = ls.q_nope[M].clone(), ls.q_pe[M].clone()

            def producers(l):
                torch.mul(src_n[l], 1, out=ls.q_nope[M][l])
                torch.mul(src_p[l], 1, out=ls.q_pe[M][l])

            side = torch.cuda.Stream()

            def layer_step(l, with_op, pdl, prefetch):
                main = torch.cuda.current_stream()
                if prefetch:  # a parallel branch that warms L2 with this layer's weights
                    side.wait_stream(main)
                    with torch.cuda.stream(side):
                        a = ls.layer_args(M, l)
                        mq.check(mq.mlaqp_prefetch_weights(a["weight"], a["weight_scale"], ls.H, ls.K,
                                                           ls.weight_format, stream=side))
                producers(l)
                if with_op:
                    run = mq.mlaqp_run_pdl if pdl else mq.mlaqp_run
                    mq.check(run(**ls.layer_args(M, l), stream=main))
                if prefetch:
                    main.wait_stream(side)

            def build(with_op, pdl, prefetch=False):
                s = torch.cuda.Stream()
                s.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(s):
                    for l in range(ls.L):
                        layer_step(l, with_op, pdl, prefetch)
                torch.cuda.current_stream().wait_stream(s)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for l in range(ls.L):
                        layer_step(l, with_op, pdl, prefetch)
                return g

            row = {"pair": f"{fmt}->{od}", "H": H, "M": M, "layers": ls.L}
            prod = time_graph(build(False, False), ls.L, steps, warmup)
            prod_pf = time_graph(build(False, False, True), ls.L, steps, warmup)
            row["producers_us"] = round(prod, 4)
            for name, pdl, pf in (("pdl", True, False), ("no_pdl", False, False),
                                  ("pdl_prefetch", True, True), ("no_pdl_prefetch", False, True)):
                step = time_graph(build(True, pdl, pf), ls.L, steps, warmup)
                row[f"step_us_{name}"] = round(step, 4)
                row[f"op_us_{name}"] = round(step - (prod_pf if pf else prod), 4)
            res.append(row)
        del ls
        torch.cuda.empty_cache()
    return res


def run_e2e(sets, graphs, points, args):
    """Same metric through the public API with host buffers.  Every step
    copies every point's q_nope / q_pe from pinned host memory, replays the
    point's graph and copies its outputs back to pinned host memory.  The
    copies run on their own streams, so point i+1's inputs travel while point
    i computes and point i's outputs travel while point i+1 computes; events
    keep each buffer's copy-in, use and copy-out in order, across steps too.
    The timed region runs from before the first copy to after the last
    copy-out of the last step."""
    import torch
    comp = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    n = len(points)
    host_out = [torch.empty(s.out[M].shape, dtype=s.out[M].dtype, pin_memory=True) for s, M in points]
    h2d = sum(t.numel() * t.element_size() for s, M in points for t in s.host_inputs(M))
    d2h = sum(s.out[M].numel() * s.out[M].element_size() for s, M in points)
    in_ready = [torch.cuda.Event() for _ in range(n)]  # point i's inputs are on the device
    computed = [torch.cuda.Event() for _ in range(n)]  # point i's graph has run (inputs read, outputs written)
    out_read = [torch.cuda.Event() for _ in range(n)]  # point i's outputs are on the host
    started = [False]

    def step():
        for i, ((s, M), g) in enumerate(zip(points, graphs)):
            if started[0]:
                h2d_s.wait_event(computed[i])  # the previous step's replay of i has read its inputs
            with torch.cuda.stream(h2d_s):
                for dst, src in zip(s.dev_inputs(M), s.host_inputs(M)):
                    dst.copy_(src, non_blocking=True)
            in_ready[i].record(h2d_s)
            comp.wait_event(in_ready[i])
            if started[0]:
                comp.wait_event(out_read[i])  # the previous step's outputs of i have left the device
            g.replay()
            computed[i].record(comp)
            d2h_s.wait_event(computed[i])
            with torch.cuda.stream(d2h_s):
                host_out[i].copy_(s.out[M], non_blocking=True)
            out_read[i].record(d2h_s)
        started[0] = True

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(comp)
    h2d_s.wait_event(a)
    d2h_s.wait_event(a)
    for _ in range(args.steps):
        step()
    comp.wait_stream(h2d_s)
    comp.wait_stream(d2h_s)
    b.record(comp)
    torch.cuda.synchronize()
    for i, (s, M) in enumerate(points):  # the host copies hold the last step's outputs
        if not torch.equal(host_out[i], s.out[M].cpu()):
            raise RuntimeError(f"e2e: host copy of point {i} differs from the device output")
    ms = a.elapsed_time(b)
    nbytes = sum(s.bytes_per_call(M) * s.L for s, M in points) * args.steps
    return {"value": round(nbytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(ms / args.steps, 4),
            "copies": "pinned host <-> device on two copy streams, overlapped with the previous / next point's replay"}


KERNEL_SOURCES = ("mla_decode_query_gb300/csrc/mlaqp_kernel.cuh", "mla_decode_query_gb300/csrc/mlaqp_kernels_bf16.cu",
                  "mla_decode_query_gb300/csrc/mlaqp_kernels_mxfp8.cu",
                  "mla_decode_query_gb300/csrc/mlaqp_kernel_warp.cuh",
                  "mla_decode_query_gb300/csrc/mlaqp_kernels_warp_bf16.cu",
                  "mla_decode_query_gb300/csrc/mlaqp_kernels_warp_mxfp8.cu")
TRAFFIC_FILE = "profiles/fused_query_dram_traffic_h16.txt"


def kernel_source_hash():
    import hashlib
    root = os.path.dirname(os.path.abspath(__file__))
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(root, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic():
    """Per-(pair, M) DRAM bytes per launch from the committed ncu summary, or
    None when the kernel sources changed since those counters were taken."""
    root = os.path.dirname(os.path.abspath(__file__))
    try:
        lines = open(os.path.join(root, TRAFFIC_FILE)).read().splitlines()
    except OSError:
        return None
    tag = [l for l in lines if l.startswith("# kernel-source-sha256-16")]
    if not tag or tag[0].split()[2] != kernel_source_hash():
        return None
    out = {}
    for l in lines:
        if l and not l.startswith("#"):
            pair, M, traffic, _ = l.split()
            out[(pair, int(M))] = int(traffic)
    return out


def launch_floor(steps, warmup):
    """us per launch of a CUDA graph of 128 dependent empty kernels (128 CTAs
    x 128 threads) with and without programmatic dependent launch: the floor
    of any one-launch-per-layer chain on this GPU."""
    import torch
    import mla_decode_query_gb300 as mq
    res = {}
    for pdl in (True, False):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            mq.check(mq.mlaqp_debug_launch_null(128, 128, pdl, stream=s))
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(128):
                mq.check(mq.mlaqp_debug_launch_null(128, 128, pdl))
        for _ in range(max(3, warmup)):
            g.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record()
        for _ in range(max(5, steps)):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        res["pdl" if pdl else "no_pdl"] = round(1e3 * a.elapsed_time(b) / max(5, steps) / 128, 4)
    return res


def load_peaks():
    p = os.path.join(os.path.dirname(os.path.abspath(__file__)), "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback 6.8 TB/s"


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=0, help="override layers per set")
    ap.add_argument("--m", type=str, default="", help="comma-separated token counts")
    ap.add_argument("--formats", type=str, default="", help="comma-separated subset of bf16,mxfp8")
    ap.add_argument("--pairs", type=str, default="", help="comma-separated weight:output pairs, e.g. bf16:e4m3")
    ap.add_argument("--nope", type=int, default=128, choices=(128, 192), help="nope dim (192: GLM shape)")
    ap.add_argument("--heads", type=str, default="16", help="comma-separated head counts (8, 11, 16)")
    ap.add_argument("--op", choices=["query", "v_up"], default="query",
                    help="query: the fused query projection (default); v_up: the V up-projection")
    ap.add_argument("--arm", choices=["auto", "warp_mma", "warp_fma", "cta_mma", "tcgen05"], default="auto",
                    help="force one kernel form (measurement; auto = the library's choice)")
    ap.add_argument("--policy", type=str, default="",
                    help="trig:cap override of the warp-tile kernel's launch policy (measurement)")
    ap.add_argument("--no-pdl", action="store_true")
    ap.add_argument("--compare-no-pdl", action="store_true", help="also time the graphs without PDL")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle timing")
    ap.add_argument("--pdl-only", action="store_true", help="skip the graphs without PDL")
    ap.add_argument("--pdl-mode", type=int, default=1, choices=(1, 2),
                    help="2: opt-in early trigger of the tcgen05 kernels (tensor-memory contract of pdl = 2)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the isolated-call, behind-producer and configuration sweeps")
    ap.add_argument("--sweep-steps", type=int, default=5, help="timed replays per point of the sweeps")
    ap.add_argument("--oracle-only", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.oracle_only:  # child process of the one-core oracle figure
        gbs, calls, el = time_oracle(args.cpu_budget, oracle_samples(args.op), op=args.op)
        print(json.dumps({"value": round(gbs, 4), "unit": "GB/s", "cores": oracle_threads(), "calls": calls,
                          "seconds": round(el, 2)}))
        return 0
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
