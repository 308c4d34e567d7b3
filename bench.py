"""Throughput benchmark of the fused AsymSpec verification step (CDA gate + delta-fusion).

One step = one asymspec_verify call over the whole batch of the B=64, K=2, V=151936 bf16
workload (64 requests x 3 rows of three logit tensors a, b, t = 175 MB), with inputs resident
in HBM.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

The K timed steps run back to back between two CUDA events on the launching stream; that region
is repeated (each repetition exactly K steps, bracketed by a barrier and a synchronize) until the
repetitions together last at least --min-region-s, so the clock sampler sees the kernel under
load, and the line reports the median repetition.  The `secondary` key carries device-timed
lines for the other workloads (the 1 x 3 x 32000 fp32 latency case, the 256 x 5 fp32 sweep, RAPID,
and the 1024 x 9 bf16 batch in AsymSpec, fused AsymSpec + E2-SCI and E2-SCI modes), each timed
the same way.

N > 1 runs under torchrun, one rank per GPU; requests are independent, so every rank verifies
its own batch (weak scaling, no collective on the data path).  `--impl reference` times the CPU
oracle (the double-precision restatement of the pages) on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gen  # noqa: E402

WORKLOAD = "asymspec_b64_k2_v151936_bf16"
METRIC = "verified logit rows/s and HBM GB/s vs ~8 TB/s, fused CDA+δ verify, V=151936"
BETA, GAMMA = 1.0, 0.5
N_SETS = 4  # rotating input copies: 4 x 175 MB, larger than the 129 MB L2
# The timed kernel's sources; its ncu summary under profiles/ records a hash of them (SHA-256 of the
# files' bytes concatenated in this order, first 16 hex digits).
KERNEL_SOURCES = ("asv_jsd.cu", "asv_jsd_common.cuh", "asv_device.cuh", "jsd_poly.inc", "asv_internal.h")
# The sources each profiled kernel is built from (the hash a committed ncu summary records).
KERNEL_SOURCES_OF = {"jsd_family": KERNEL_SOURCES,
                     "rapid_kernel": ("asv_rapid.cu", "asv_device.cuh", "asv_internal.h")}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def kernel_source_hash(kernel: str = "jsd_family") -> str:
    import hashlib
    csrc = os.path.join(ROOT, "speculative_decoding_logit_gb300", "csrc")
    h = hashlib.sha256()
    for name in KERNEL_SOURCES_OF[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _profiled_traffic(workload: str = WORKLOAD, kernel: str = "jsd_family"):
    """DRAM bytes per launch from the committed ncu summary of a kernel on a workload, or None when
    there is none or the kernel source has changed since that capture (the summary records a hash
    of the sources)."""
    prof = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(prof).read()
        h = kernel_source_hash(kernel)
    except (OSError, KeyError):
        return None
    m_sha = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not (m_sha and m_tr) or m_sha.group(1) != h:
        return None
    return float(m_tr.group(1))


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, period_ms: int = 50):
        self.cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    f"-lms={period_ms}", f"-i={gpu_index}"]
        self.lines = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=5)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def cpu_baseline_oracle(batch, budget_s: float = 20.0):
    """The oracle, as it stands, on the host: whole requests until ~budget_s of CPU work."""
    import oracle
    oracle.lib()
    rows = 0
    t0 = time.perf_counter()
    r = 0
    while r < batch.B and (time.perf_counter() - t0) < budget_s:
        oracle.asymspec_verify(batch.a[r:r + 1], batch.b[r:r + 1], batch.t[r:r + 1], batch.drafts[r:r + 1], BETA,
                               GAMMA)
        rows += batch.K + 1
        r += 1
    dt = time.perf_counter() - t0
    return {"value": rows / dt, "unit": "rows/s", "cores": 1, "kind": "oracle",
            "sample": f"{r} of {batch.B} requests ({rows} rows of V={batch.V}), one pass, single-threaded C, float64"}


def _oracle_requests(job):
    """Worker of the all-cores CPU baseline: generate this worker's requests (untimed), wait for the
    common start instant, then run the oracle, as it stands, over them.  Returns (rows, end time)."""
    requests, start_at = job
    import oracle
    w = gen.WORKLOADS[WORKLOAD]
    batch = gen.make_asymspec_batch(w.recipe, w.seed, w.B, w.K, w.V, w.dtype, requests=requests)
    oracle.lib()
    while time.time() < start_at:
        time.sleep(0.001)
    for r in range(batch.a.shape[0]):
        oracle.asymspec_verify(batch.a[r:r + 1], batch.b[r:r + 1], batch.t[r:r + 1], batch.drafts[r:r + 1], BETA,
                               GAMMA)
    return batch.a.shape[0] * (w.K + 1), time.time()


def cpu_baseline_oracle_parallel(per_worker: int = 4, lead_s: float = 8.0):
    """The same oracle code over requests on every host core: one process per core (spawn), each
    generating its own `per_worker` requests of the workload, all starting at one wall-clock instant;
    throughput = all rows / (last finish - start)."""
    import multiprocessing as mp
    w = gen.WORKLOADS[WORKLOAD]
    n = os.cpu_count() or 1
    reqs = min(w.B, n * per_worker)
    groups = [list(range(k, reqs, n)) for k in range(n)]
    groups = [g for g in groups if g]
    with mp.get_context("spawn").Pool(len(groups)) as pool:
        start_at = time.time() + lead_s
        res = pool.map(_oracle_requests, [(g, start_at) for g in groups])
    rows = sum(r for r, _ in res)
    dt = max(e for _, e in res) - start_at
    return {"value": rows / dt, "unit": "rows/s", "cores": len(groups), "kind": "oracle",
            "sample": f"{reqs} of {w.B} requests ({rows} rows of V={w.V}) over {len(groups)} processes started "
                      "together, single-threaded C, float64 each"}


def run_reference(args):
    """CPU oracle timed as the reference arm: each step verifies one request whose rows are
    cut to the first V' vocabulary entries (V' sized so the run ends within a few minutes);
    throughput counts each step as 3 * V'/V rows."""
    import oracle
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    w = gen.WORKLOADS[WORKLOAD]
    batch = gen.make_asymspec_batch(w.recipe, w.seed, 2, w.K, w.V, w.dtype)
    oracle.lib()
    t0 = time.perf_counter()
    oracle.asymspec_verify(batch.a[:1], batch.b[:1], batch.t[:1], batch.drafts[:1], BETA, GAMMA)
    per_req = time.perf_counter() - t0
    budget = 90.0 / max(1, args.steps + args.warmup)
    Vp = int(min(w.V, max(64, w.V * budget / per_req)))
    Vp -= Vp % 8
    cut = lambda x: np.ascontiguousarray(x[:1, :, :Vp])
    a, b, t = cut(batch.a), cut(batch.b), cut(batch.t)
    d = np.minimum(batch.drafts[:1], Vp - 1).astype(np.int32)
    for _ in range(args.warmup):
        oracle.asymspec_verify(a, b, t, d, BETA, GAMMA)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.asymspec_verify(a, b, t, d, BETA, GAMMA)
    dt = time.perf_counter() - t0
    rows = args.steps * (w.K + 1) * Vp / w.V
    val = rows / dt
    sample = f"per step: 1 request, rows cut to the first {Vp} of {w.V} entries (counted as {(w.K + 1) * Vp / w.V:.4f} rows)"
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "rows/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "B": w.B, "K": w.K, "V": w.V, "beta": BETA, "gamma": GAMMA},
            "cpu_baseline": {"value": val, "unit": "rows/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _timed_reps(step, steps, min_region_s, stream, dist=None):
    """Run `steps` calls of `step(i)` back to back between two CUDA events on `stream`, bracketed by a
    barrier and a synchronize; repeat until the repetitions together last at least `min_region_s`
    (the count is fixed from one calibration repetition, the largest over ranks, so every rank runs
    the same number).  Returns the per-repetition device times in ms."""
    import torch

    from speculative_decoding_logit_gb300.shard import max_over_ranks

    def rep():
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        return e0.elapsed_time(e1)

    first = rep()
    n = max(1, int(np.ceil(min_region_s * 1e3 / max(first, 1e-3))))
    n = int(max_over_ranks(n))
    return [first] + [rep() for _ in range(n - 1)]


def _graph_of(step, steps, warm=2):
    """The K-step loop captured once into a CUDA graph on a side stream (a few eager calls on that
    stream first, so per-stream state such as the binding's workspace exists before the capture)."""
    import torch

    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(gs):
        for i in range(warm):
            step(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=gs):
        for i in range(steps):
            step(i)
    torch.cuda.synchronize()
    g.replay()  # untimed
    torch.cuda.synchronize()
    return g


def _timed_graph_reps(g, min_region_s, dist=None):
    """Replays of a captured K-step graph between two CUDA events on the replaying stream, bracketed by
    a barrier and a synchronize, repeated as _timed_reps does.  Returns per-replay device times (ms)."""
    import torch

    from speculative_decoding_logit_gb300.shard import max_over_ranks

    stream = torch.cuda.current_stream()

    def rep():
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        return e0.elapsed_time(e1)

    first = rep()
    n = max(1, int(np.ceil(min_region_s * 1e3 / max(first, 1e-3))))
    n = int(max_over_ranks(n))
    return [first] + [rep() for _ in range(n - 1)]


def _gpu_id(dev):
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        return str(dev.index)


def run_ours(args):
    import torch

    import speculative_decoding_logit_gb300 as asv
    from speculative_decoding_logit_gb300.shard import max_over_ranks

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        dist = None
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    asv.build()
    lib = asv.library()

    w = gen.WORKLOADS[WORKLOAD]
    batch = gen.make_asymspec_batch(w.recipe, w.seed, w.B, w.K, w.V, w.dtype, processes=8)
    R = w.B * (w.K + 1)
    in_bytes = 3 * R * w.V * 2

    def todev(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)

    sets = [tuple(todev(x) for x in (batch.a, batch.b, batch.t)) for _ in range(N_SETS)]
    d = torch.from_numpy(batch.drafts).to(dev)
    out = asv.asymspec_verify(*sets[0], d, BETA, GAMMA)  # allocates outputs, loads the library
    wsbuf = torch.zeros(asv.workspace_bytes(asv.ASV_MODE_ASYMSPEC, w.B, w.K, w.V, asv.ASV_BF16), dtype=torch.uint8,
                        device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    fn = lib.asymspec_verify

    # Pre-marshalled argument lists (the stream handle included): one ctypes call per step.
    def marshalled(stream_handle):
        return [(a.data_ptr(), b.data_ptr(), t.data_ptr(), asv.ASV_BF16, d.data_ptr(), w.B, w.K, w.V,
                 BETA, GAMMA, out.accept_len.data_ptr(), out.tokens.data_ptr(), out.D.data_ptr(),
                 out.lse.data_ptr(), out.req_status.data_ptr(), wsbuf.data_ptr(), wsbuf.numel(), stream_handle)
                for (a, b, t) in sets]

    calls = marshalled(sh)

    def step(i):
        st = fn(*calls[i % N_SETS])
        if st != 0:
            raise RuntimeError(f"asymspec_verify failed: {st}")

    def step_on_current(i):
        st = fn(*marshalled(torch.cuda.current_stream(dev).cuda_stream)[i % N_SETS])
        if st != 0:
            raise RuntimeError(f"asymspec_verify failed: {st}")

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()

    # The timed region: the K calls captured once into a CUDA graph (as a serving loop issues them),
    # each repetition one replay between two events on the replaying stream; the kernel's average
    # launch duration is that region over K, the gaps between the graph's kernels included.  The
    # same K calls launched one by one from the host (eager) are timed too and reported beside it.
    clocks = ClockSampler(_gpu_id(dev))
    clocks.start()
    time.sleep(0.3)  # let the sampler start
    graph = _graph_of(step_on_current, args.steps)
    reps = _timed_graph_reps(graph, args.min_region_s, dist)
    eager_reps = _timed_reps(step, args.steps, min(0.25, args.min_region_s), stream, dist)
    clk = clocks.stop()
    del graph
    rep_ms = float(np.median(reps))
    elapsed_ms = max_over_ranks(rep_ms)
    launch_ms = rep_ms / args.steps
    rows_total = R * args.steps * ws
    value = rows_total / (elapsed_ms / 1e3)

    # End to end through the C ABI with host (pinned) buffers: H2D of the step's inputs,
    # the verification, D2H of the step's results, every step.
    e2e = None
    if not args.no_e2e:
        pin = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
        ha, hb, ht = (pin(x.view(np.int16)) for x in (batch.a, batch.b, batch.t))
        hd = pin(batch.drafts)
        o_acc = torch.empty(w.B, dtype=torch.int32).pin_memory()
        o_tok = torch.empty(w.B, w.K + 1, dtype=torch.int32).pin_memory()
        o_D = torch.empty(w.B, w.K + 1, dtype=torch.float32).pin_memory()
        o_st = torch.empty(w.B, dtype=torch.int32).pin_memory()
        arena = torch.zeros(asv.host_arena_bytes(w.B, w.K, w.V, asv.ASV_BF16), dtype=torch.uint8, device=dev)
        hcall = (ha.data_ptr(), hb.data_ptr(), ht.data_ptr(), asv.ASV_BF16, hd.data_ptr(), w.B, w.K, w.V, BETA, GAMMA,
                 o_acc.data_ptr(), o_tok.data_ptr(), o_D.data_ptr(), o_st.data_ptr(), arena.data_ptr(), arena.numel(),
                 sh)
        hfn = lib.asymspec_verify_host
        for _ in range(3):
            assert hfn(*hcall) == 0
        torch.cuda.synchronize()
        ne = max(10, min(200, args.steps // 50))
        h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h0.record(stream)
        for _ in range(ne):
            assert hfn(*hcall) == 0
        h1.record(stream)
        torch.cuda.synchronize()
        e_ms = max_over_ranks(h0.elapsed_time(h1))
        assert np.array_equal(o_tok.numpy(), out.tokens.cpu().numpy())
        h2d = 3 * R * w.V * 2 + w.B * w.K * 4
        d2h = w.B * 4 + R * 4 + R * 4 + w.B * 4
        e2e = {"value": R * ne * ws / (e_ms / 1e3), "unit": "rows/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": ne, "ms_per_step": e_ms / ne}

    peaks, peak_kind = _peaks()
    traffic = args.traffic if args.traffic is not None else _profiled_traffic()
    achieved = in_bytes / (launch_ms / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "traffic": traffic, "peak_kind": peak_kind,
            "frac_of_8tbs": achieved / 8000.0, "kernel_ms": launch_ms,
            "kernel_ms_from": "median replay of the K calls captured in one CUDA graph / K (CUDA events on the "
                              "replaying stream)",
            "algorithmic_bytes_per_launch": in_bytes}
    secondary = None
    if ws == 1 and not args.no_secondary:
        del sets, calls
        torch.cuda.empty_cache()
        secondary = {}
        for name in SECONDARY:
            secondary[name] = workload_line(name, args, dev, steps=None)
            torch.cuda.empty_cache()
    cpu = cpu_par = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_oracle(batch)
        cpu_par = cpu_baseline_oracle_parallel()
    plan = asv.query_plan(asv.ASV_MODE_ASYMSPEC, w.B, w.K, w.V, asv.ASV_BF16)
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": WORKLOAD, "B": w.B, "K": w.K, "V": w.V, "beta": BETA, "gamma": GAMMA,
                           "rows_per_step": R, "parallelism": f"replicas x{ws} (requests sharded, no collective)",
                           "l2": f"{N_SETS} rotating input sets of {in_bytes / 1e6:.0f} MB (> 129 MB L2)",
                           "timed_reps": len(reps), "rep_ms_min_median_max": [min(reps), rep_ms, max(reps)],
                           "launch": "the K calls captured once into a CUDA graph and replayed",
                           "eager_ms_per_step": float(np.median(eager_reps)) / args.steps,
                           "plan": plan},
                "roofline": roof, "cpu_baseline": cpu, "cpu_baseline_all_cores": cpu_par, "e2e": e2e,
                "gpu_launches": args.steps * len(reps), "clocks": clk, "secondary": secondary}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


# The other workloads, timed in the same run (device-timed lines under the `secondary` key).
SECONDARY = ("asymspec_b1_k2_v32000_f32", "asymspec_sweep_b256_k4_v151936_f32", "rapid_b32_g10_v128256_f32",
             "asymspec_b1024_k8_v151936_bf16", "sci_asymspec_b1024_k8_v151936_bf16", "sci_b1024_k8_v151936_bf16")

# Workload names that are modes of another workload's tensors: (source workload, mode).
_MODES = {"asymspec_b1024_k8_v151936_bf16": ("sci_asymspec_b1024_k8_v151936_bf16", "asymspec"),
          "sci_b1024_k8_v151936_bf16": ("sci_asymspec_b1024_k8_v151936_bf16", "sci"),
          "sci_asymspec_b1024_k8_v151936_bf16": ("sci_asymspec_b1024_k8_v151936_bf16", "fused")}


def workload_line(name, args, dev, steps=None):
    """Device-timed throughput of one workload: launches back to back between two CUDA events on the
    launching stream, repeated until the region lasts at least --min-region-s; inputs resident in
    HBM and larger than L2 (or rotating copies that together are).  Returns a dict in the shape of
    the headline line (no e2e or CPU leg)."""
    import dataclasses

    import torch

    import speculative_decoding_logit_gb300 as asv

    src, mode = _MODES.get(name, (name, None))
    w = gen.WORKLOADS[src]
    if mode is None:
        mode = {"asymspec": "asymspec", "rapid": "rapid", "sci": "fused"}[w.mode]
        if name == "asymspec_sweep_b256_k4_v151936_f32":
            mode = "sweep"
    if args.requests:
        # A smaller batch of the same workload (profiling captures must stay within a few GB).
        w = dataclasses.replace(w, B=min(w.B, args.requests))
    todev = lambda x, dt: (torch.from_numpy(np.ascontiguousarray(x)).to(dev) if dt == gen.F32 else
                           torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev))
    R = w.B * (w.K + 1)
    extra = {}
    per_step = 2 if mode == "rapid" else 1  # RAPID: verification launch + draw launch
    if mode == "rapid":
        b = gen.make_rapid_batch(w.seed, w.B, w.K, w.V)
        sets = [(todev(b.z, gen.F32), todev(b.q, gen.F32)) for _ in range(3)]
        d = torch.from_numpy(b.drafts).to(dev)
        eta = 10.0
        step_bytes = 2 * R * w.V * 4
        call = lambda i: asv.rapid_verify(*sets[i % 3], d, w.params["T"], eta, w.params["tail_frac"],
                                          w.params["philox_seed"])
        dtype, kernel = "f32", "rapid_kernel + rapid_draw_kernel"
        extra = {"eta": eta, "sets": 3}
    else:
        # Generated requests tiled along the batch when the workload is large (the kernel's work per
        # row does not depend on which request the row belongs to, and the rows are far apart).
        gen_B = min(w.B, 64)
        batch = gen.make_asymspec_batch(w.recipe, w.seed, gen_B, w.K, w.V, w.dtype,
                                        identical_frac=w.params.get("identical_frac", 0.0), processes=8)
        tile = (w.B + gen_B - 1) // gen_B
        rep = lambda x: np.concatenate([x] * tile, axis=0)[:w.B]
        a, b_, t = (todev(rep(x), w.dtype) for x in (batch.a, batch.b, batch.t))
        d = torch.from_numpy(rep(batch.drafts)).to(dev)
        s_el = 4 if w.dtype == gen.F32 else 2
        n_in = 2 if mode == "sci" else 3
        step_bytes = n_in * R * w.V * s_el
        nsets = max(1, min(4, int(np.ceil(4 * 129e6 / step_bytes))))
        sets = [(a, b_, t)] + [tuple(x.clone() for x in (a, b_, t)) for _ in range(nsets - 1)]
        dtype = "f32" if w.dtype == gen.F32 else "bf16"
        extra = {"requests_generated": gen_B, "tiled": tile, "sets": nsets}
        if mode == "sweep":
            betas, gammas = [0.0, 1.0, 1.5, 2.0], [0.4, 0.5, 0.7, 1.0]
            call = lambda i: asv.asymspec_verify_sweep(*sets[i % nsets], d, betas, gammas)
            kernel = "jsd_family_kernel (sweep: 4 betas x 4 gammas from one read)"
            extra["grid_points"] = 16
        elif mode == "fused":
            r_hat = torch.full((w.B,), w.params["r_hat0"], dtype=torch.float64, device=dev)
            call = lambda i: asv.asymspec_sci_verify(*sets[i % nsets], d, 1.0, 0.5, r_hat)
            kernel = "jsd_family_kernel (AsymSpec fused with E2-SCI, one read of a, b, t)"
        elif mode == "sci":
            r_hat = torch.full((w.B,), w.params["r_hat0"], dtype=torch.float64, device=dev)
            call = lambda i: asv.sci_verify(sets[i % nsets][0], sets[i % nsets][2], d, r_hat)
            kernel = "jsd_family_kernel (E2-SCI: draft a, target t)"
        else:
            call = lambda i: asv.asymspec_verify(*sets[i % nsets], d, 1.0, 0.5)
            kernel = "jsd_family_kernel"
    for i in range(max(3, args.warmup)):
        call(i)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    # enough launches per repetition that a repetition is at least ~2 ms
    t0 = time.perf_counter()
    call(0)
    torch.cuda.synchronize()
    est_ms = (time.perf_counter() - t0) * 1e3
    n_steps = steps or max(5, int(np.ceil(2.0 / max(est_ms, 1e-3))))
    clocks = ClockSampler(_gpu_id(dev))
    clocks.start()
    time.sleep(0.3)
    graph = _graph_of(call, n_steps)
    reps = _timed_graph_reps(graph, args.min_region_s)
    eager_reps = _timed_reps(call, n_steps, min(0.25, args.min_region_s), stream)
    clk = clocks.stop()
    del graph
    rep_ms = float(np.median(reps))
    launch_ms = rep_ms / n_steps
    peaks, peak_kind = _peaks()
    achieved = step_bytes / (launch_ms / 1e3) / 1e9
    kname = "rapid_kernel" if mode == "rapid" else "jsd_family"
    return {"metric": f"verified logit rows/s ({name})", "value": R * n_steps / (rep_ms / 1e3),
            "unit": "rows/s", "n_gpus": 1, "steps": n_steps, "ms_per_step": launch_ms, "higher_is_better": True,
            "dtype": dtype, "data": "synthetic",
            "config": dict({"workload": name, "B": w.B, "K": w.K, "V": w.V, "rows_per_step": R, "kernel": kernel,
                            "timed_reps": len(reps), "rep_ms_min_median_max": [min(reps), rep_ms, max(reps)],
                            "launch": "the calls captured once into a CUDA graph and replayed",
                            "eager_ms_per_step": float(np.median(eager_reps)) / n_steps},
                           **extra),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "frac_of_8tbs": achieved / 8000.0,
                         "traffic": _profiled_traffic(name, kname), "peak_kind": peak_kind, "kernel_ms": launch_ms,
                         "algorithmic_bytes_per_launch": step_bytes},
            "gpu_launches": per_step * n_steps * len(reps), "clocks": clk}


def run_workload(args):
    """One workload's device-timed line alone (the `--workload` flag)."""
    import torch
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    import speculative_decoding_logit_gb300 as asv
    asv.build()
    if args.cluster:
        asv.set_tuning(args.cluster)
    line = workload_line(args.workload, args, dev, steps=args.steps)
    if args.cluster:
        line["config"]["cluster_override"] = args.cluster
    line["warmup"] = args.warmup
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--min-region-s", type=float, default=1.0,
                    help="repeat the K-step timed region until the repetitions last this long in total")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch from an ncu capture of the current kernel (else null)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg (profiling runs)")
    ap.add_argument("--no-secondary", action="store_true", help="skip the other workloads' lines")
    ap.add_argument("--requests", type=int, default=0,
                    help="with --workload: verify only this many requests (small cases for ncu captures)")
    ap.add_argument("--cluster", type=int, default=0,
                    help="with --workload: CTAs per row (the library's tuning override; profiling captures of a "
                         "reduced batch in the full batch's plan)")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(set(gen.WORKLOADS) | set(_MODES)),
                    help="another workload (device-timed line only; the default is the headline workload)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.workload != WORKLOAD:
        return run_workload(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
