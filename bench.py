#!/usr/bin/env python
"""Benchmark of the attention-JVP hot path on GB300; prints ONE JSON line.

A step is one pass of the whole path over one batch of synthetic inputs:
the FP64 TrigFlow coefficients of the batch's times (host), the TrigFlow
tangent of the latent batch (GPU), and the fused attention forward + JVP
(GPU; split into key chunks + exact merge for the long-video workload).
The metric counts the attention's 12*B*H*N^2*d flops per step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the FP64 CPU oracle on host cores

Multi-GPU: launched by torchrun, each rank runs an independent replica of the
workload on its own GPU (the path shards into independent heads; no data
collective); timing is the max over ranks, value is the whole-job throughput.
"""
import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention-JVP TFLOPS (12·B·H·N²·d) and % of GB300 BF16 tensor peak"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "long_video"
# Other workloads timed in the same run, each as a device-timed sub-record.
DEFAULT_ALSO = "video_dit,stress,image_dit_1k"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Sources whose change invalidates a recorded DRAM-traffic capture of the fused kernel.
KERNEL_SOURCES = tuple(os.path.join(ROOT, "attention_jvp_gb300", "csrc", n) for n in ("attn_jvp_fwd.cu", "sm103_ptx.cuh"))
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    p.add_argument("--heads", type=int, default=None, help="override H (profiling on a smaller case)")
    p.add_argument("--skip-e2e", action="store_true")
    p.add_argument("--skip-cpu", action="store_true")
    p.add_argument("--skip-epilogue", action="store_true", help="skip the output-side kernels' bandwidth line")
    p.add_argument("--skip-backward", action="store_true", help="skip the primal-backward line")
    p.add_argument("--e2e-steps", type=int, default=5)
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    p.add_argument("--also", default=DEFAULT_ALSO,
                   help="comma-separated workloads timed after the main one as device-only sub-records ('' = none)")
    p.add_argument("--sub-steps", type=int, default=10, help="timed steps of each sub-record workload")
    p.add_argument("--sub-cpu-seconds", type=float, default=3.0,
                   help="target CPU time of each sub-record workload's oracle sample")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# host-side helpers (no GPU needed; covered by tests/test_bench_host.py)
# ---------------------------------------------------------------------------
def workload_spec(name, heads=None):
    from attention_jvp_gb300 import inputs
    spec = dict(inputs.WORKLOADS[name])
    if heads is not None:
        spec["H"] = int(heads)
    return spec


def attention_flops(spec, kv_len=None):
    """Algorithmic flops of one attention JVP pass: 12 d per (query, key) pair.

    2d for S, 4d for St (two d-deep products), 2d each for P~V, P~Vt and H~V.
    """
    kv = spec["N"] if kv_len is None else kv_len
    return 12.0 * spec["B"] * spec["H"] * spec["N"] * kv * spec["d"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return peaks, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def measure_epilogue(spec, dev, stream, peaks, reps=10, warmup=3):
    """Achieved bandwidth of the TrigFlow tangent and the two output-side kernels on a
    latent batch larger than L2.

    Algorithmic bytes per element: trigflow_tangent reads x0 and eps and writes the
    tangent (12 B); trigflow_output_jvp reads x, n and their tangents and
    writes F and its tangent (24 B); scm_tangent_loss reads F_theta, F_sg, F_teacher, x and
    F_t and writes g_n and df_dt (28 B); its in-place normalisation of g (one write and
    one re-read of the unnormalised g, 8 B more) is an implementation cost the figure
    does not credit."""
    import torch
    from attention_jvp_gb300 import binding, inputs

    batch = inputs.epilogue_batch(spec, device=dev)
    x, n, xt, nt, t, tt = (batch[k] for k in ("x", "n", "x_t", "n_t", "t", "t_t"))
    B, C, T, HW = x.shape
    shape = (B, C, T, HW)
    F, Ft = torch.empty_like(x), torch.empty_like(x)
    ws = binding.scm_workspace(shape, dev)
    elems = B * C * T * HW
    res = {"shape": [B, C, T, HW], "elements": elems}
    flat_x, flat_n = x.reshape(B, -1), n.reshape(B, -1)
    t_b = t[:, 0].contiguous()
    tangent_out = torch.empty_like(flat_x)
    ops = {
        "trigflow_tangent": (12, lambda: binding.trigflow_tangent(flat_x, flat_n, t_b, out=tangent_out,
                                                                  stream=stream)),
        "trigflow_output_jvp": (24, lambda: binding.trigflow_output_jvp(x, n, xt, nt, t, tt, out=F, out_t=Ft,
                                                                         stream=stream)),
        "scm_tangent_loss": (28, lambda: binding.scm_tangent_loss(F, x, n, xt, nt, t, 0.5, workspace=ws,
                                                                  stream=stream)),
    }
    peak = float(peaks["hbm_gbs"])
    for name, (bpe, fn) in ops.items():
        for _ in range(warmup):
            fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        gbs = bpe * elems / (ms * 1e-3) / 1e9
        res[name] = {"bound": "hbm", "algorithmic_bytes_per_elem": bpe, "ms": round(ms, 4),
                     "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4)}
    binding.attn_jvp_status()
    return res


def measure_qk_norm(x, dev, stream, peaks, reps=10, warmup=3):
    """Achieved bandwidth of qk_rmsnorm_jvp (the QK normalisation and its tangent) on the
    workload's Q, K and tangents, written to separate outputs.  Algorithmic bytes: 8 per
    element of Q and of K (read x and xt, write y and yt, bf16)."""
    import torch
    from attention_jvp_gb300 import binding
    q, qt, k, kt = x["q"], x["q_t"], x["k"], x["k_t"]
    d = q.shape[-1]
    w = torch.ones(d, dtype=torch.float32, device=dev)
    outs = tuple(torch.empty_like(t) for t in (q, qt, k, kt))

    def run():
        binding.qk_rmsnorm_jvp(q, qt, k, kt, w, w, eps=1e-6, out=outs, stream=stream)

    for _ in range(warmup):
        run()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    nb = 8 * (q.numel() + k.numel())
    peak = float(peaks["hbm_gbs"])
    gbs = nb / (ms * 1e-3) / 1e9
    del outs
    return {"bound": "hbm", "algorithmic_bytes": nb, "ms": round(ms, 4), "achieved": round(gbs, 1), "peak": peak,
            "unit": "GB/s", "frac": round(gbs / peak, 4),
            "note": "Q and K of the workload with their tangents: 8 B per element (bf16 x, xt in; y, yt out)"}


def measure_backward(x, spec, o, lse, dev, stream, peaks, reps=5, warmup=2):
    """Primal attention backward on the workload's Q, K, V with a random upstream gradient.

    ``tflops`` counts 10 d flops per (query, key) pair (S, dP, dV, dQ, dK), the usual
    figure for an attention backward; the two-pass kernels execute 14 d (they form S
    and dP in both passes), reported as ``tflops_executed``."""
    import torch
    from attention_jvp_gb300 import binding

    from attention_jvp_gb300 import inputs

    q, k, v = x["q"], x["k"], x["v"]
    dO = inputs.upstream_gradient(spec, q.shape, device=dev)
    dq, dk, dv = (torch.empty(t.shape, dtype=torch.float32, device=dev) for t in (q, k, v))
    n = binding.load().attn_bwd_workspace_bytes(q.shape[0], q.shape[1], q.shape[2])
    ws = torch.empty(n, dtype=torch.uint8, device=dev)

    def run():
        binding.attn_bwd(q, k, v, dO, o, lse, scale=x["scale"], dq=dq, dk=dk, dv=dv, workspace=ws, stream=stream)

    for _ in range(warmup):
        run()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    ms = e0.elapsed_time(e1) / reps
    B, H, N, d = q.shape
    pairs = B * H * float(N) * N
    executed = backward_executed_flops_per_pair(d)
    return {"ms": round(ms, 4), "tflops": round(10 * d * pairs / (ms * 1e-3) / 1e12, 2),
            "tflops_executed": round(executed * pairs / (ms * 1e-3) / 1e12, 2),
            "frac_of_sustained_peak": round(executed * pairs / (ms * 1e-3) / 1e12
                                            / float(peaks["bf16_tflops_sustained"]), 4),
            "flops_convention": "10 d per (query, key) pair; executed %d d (two passes%s)"
                                % (executed // d, ", two CTAs per row tile" if d > 128 else "")}


def backward_executed_flops_per_pair(d):
    """Tensor flops the two backward passes execute per (query, key) pair: each pass forms
    S and dP (2d + 2d), the dK/dV pass adds dV and dK (4d), the dQ pass dQ (2d): 14 d.
    At head dim 256 two CTAs share a row tile and each forms the full S and dP: 22 d."""
    return (22 if d > 128 else 14) * d


_COMMENT = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def kernel_source_sha():
    """Hash of the fused kernel's sources with comments removed and whitespace runs folded: a
    comment edit leaves the compiled kernel, and so its recorded traffic, unchanged; any code
    edit voids the record."""
    h = hashlib.sha256()
    for path in KERNEL_SOURCES:
        with open(path, encoding="utf-8") as f:
            h.update(" ".join(_COMMENT.sub(" ", f.read()).split()).encode())
    return h.hexdigest()[:16]


def traffic_per_launch(kernel, workload, heads):
    """DRAM bytes per launch from the committed ncu summary, or None if absent or stale."""
    try:
        with open(TRAFFIC_FILE) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    rec = table.get(kernel, {}).get(workload)
    if not rec or rec.get("source_sha") != kernel_source_sha():
        return None
    # counters scale with the number of heads processed (each head is independent)
    return float(rec["dram_bytes_per_launch"]) * heads / float(rec["heads"])


def aggregate(local_ms, local_units, world, reduce_max=None, reduce_sum=None):
    """Whole-job numbers from per-rank timings: max time over ranks, total units."""
    t = reduce_max(local_ms) if (world > 1 and reduce_max) else local_ms
    u = reduce_sum(local_units) if (world > 1 and reduce_sum) else local_units
    return t, u


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    @classmethod
    def summarize(cls, lines):
        sm, mx, reasons = [], [], set()
        for ln in lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(cls.REASONS, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}

    # Throttle reasons that void a timing; sw_power_cap is normal under a dense load and is kept.
    REJECT = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")

    @classmethod
    def rejection(cls, summary, locked_frac=0.75):
        """Why a timed region's clock record voids its number, or None.

        A slowdown or thermal reason seen at any sample voids it.  So does a median SM clock
        below ``locked_frac`` of the maximum with no reason active, the mark of a clock lock
        left behind by an earlier user.  No samples (no nvidia-smi) voids nothing.
        """
        bad = [r for r in summary.get("reasons", []) if r in cls.REJECT]
        if bad:
            return ",".join(bad)
        sm, mx = summary.get("sm_mhz"), summary.get("sm_max_mhz")
        if sm and mx and not summary.get("reasons") and sm < locked_frac * mx:
            return "sm clock %.0f of %.0f MHz with no reason active" % (sm, mx)
        return None


# ---------------------------------------------------------------------------
# CPU legs: the oracle on a bounded sample of the workload
# ---------------------------------------------------------------------------
def oracle_rows_for(spec, x_host_head, target_s, seed=0):
    """Number of query rows the FP64 oracle evaluates in about ``target_s`` seconds."""
    import oracle
    from attention_jvp_gb300 import inputs

    cores = oracle.default_threads()
    q, k, v, qt, kt, vt = x_host_head
    N = spec["N"]

    def per_row(n, s):
        rows = inputs.sample_rows(N, n, s).numpy()
        t0 = time.perf_counter()
        oracle.attn_jvp(q, k, v, qt, kt, vt, spec["scale"], rows=rows, nthreads=cores)
        return (time.perf_counter() - t0) / len(rows)

    # A row per thread is dominated by thread start-up and overstates the cost of a
    # row; a second run sized at a tenth of the target, with every thread busy, sets it.
    n0 = min(N, max(cores, 8))
    t_row = per_row(n0, seed)
    n1 = int(min(N, 0.1 * target_s / max(t_row, 1e-9)))
    if n1 > n0:
        t_row = per_row(n1, seed + 2)
    return int(max(n0, min(N, target_s / max(t_row, 1e-9))))


def oracle_sample(spec, x_host_head, n_rows, seed=0, with_outputs=False):
    """Time the FP64 oracle on ``n_rows`` query rows of one head against all N keys.

    Returns (tflops, cores, rows, seconds); flops are the same 12 d per
    (query, key) pair the GPU metric counts.  With ``with_outputs`` also the
    row indices and the oracle's (O, Ot, LSE, mu) at them.
    """
    import oracle
    from attention_jvp_gb300 import inputs

    cores = oracle.default_threads()
    q, k, v, qt, kt, vt = x_host_head
    N, d = spec["N"], spec["d"]
    rows = inputs.sample_rows(N, n_rows, seed + 1).numpy()
    t0 = time.perf_counter()
    ref = oracle.attn_jvp(q, k, v, qt, kt, vt, spec["scale"], rows=rows, nthreads=cores)
    dt = time.perf_counter() - t0
    res = (12.0 * len(rows) * N * d / dt / 1e12, cores, len(rows), dt)
    return res + (rows, ref) if with_outputs else res


def parity_on_rows(got, ref):
    """Errors of the GPU outputs (O, Ot, LSE, mu of one head, as host FP64 arrays at
    the sampled rows) against the oracle's: rel-L2 and max-abs / RMS(ref) for O, Ot and
    mu, max-abs for LSE."""
    import numpy as np
    out = {}
    for name, g, r in zip(("O", "Ot", "LSE", "mu"), got, ref):
        g, r = np.asarray(g, dtype=np.float64), np.asarray(r, dtype=np.float64)
        if name == "LSE":
            out[name] = {"max_abs": float(np.max(np.abs(g - r)))}
            continue
        rms = float(np.sqrt(np.mean(r * r)))
        out[name] = {"rel_l2": float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300)),
                     "max_abs_over_rms": float(np.max(np.abs(g - r)) / max(rms, 1e-300))}
    return out


def host_head(x, h=0):
    """FP64 host copies of one head's six inputs (the values the GPU sees)."""
    B, H, N, d = x["q"].shape
    return tuple(x[n].reshape(B * H, N, d)[h].to("cpu").double().numpy()
                 for n in ("q", "k", "v", "q_t", "k_t", "v_t"))


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import torch

    from attention_jvp_gb300 import inputs
    spec = workload_spec(args.workload, args.heads)
    spec["scale"] = inputs.default_scale(spec["d"])
    # one head's inputs, drawn on the CPU with the workload's recipe
    one = dict(spec, B=1, H=1)
    x = inputs.make_inputs(**one, device="cpu")
    xh = host_head(x)
    total = args.steps + args.warmup
    per_step = max(0.5, min(10.0, 150.0 / max(total, 1)))
    import oracle
    cores = oracle.default_threads()
    n_rows = oracle_rows_for(spec, xh, per_step)
    rates = []
    for s in range(total):
        tf, cores, rows_used, dt = oracle_sample(spec, xh, n_rows, seed=s)
        if s >= args.warmup:
            rates.append(tf)
    value = statistics.median(rates) if rates else None
    full = attention_flops(spec)
    rec = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": (full / (value * 1e12) * 1e3) if value else None,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "B": spec["B"], "H": spec["H"], "N": spec["N"], "d": spec["d"]},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "%d query rows of one head vs all %d keys per step; ms_per_step "
                                   "extrapolated to the full workload" % (rows_used, spec["N"])},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(rec))
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
# Dense bf16 tcgen05 rate of one SM per clock: a 128x128x16 MMA issues every 64
# clocks (2*128*128*16/64), measured on this GPU with one issuing thread.
TENSOR_FLOP_PER_CLK_SM = 8192.0


def merge_bytes(spec, n_chunks):
    """Algorithmic bytes of one merge: every chunk's O_c, Ot_c (d floats each) and
    LSE_c, mu_c are read once, O, Ot, LSE and mu written once."""
    rows = spec["B"] * spec["H"] * spec["N"]
    per_row = (2 * spec["d"] + 2) * 4
    return rows * per_row * (n_chunks + 1)


def tangent_bytes(elems):
    """Algorithmic bytes of trigflow_tangent: read x0 and eps, write the tangent (fp32)."""
    return 12 * elems


def clock_normalised_frac(tflops, sm_count, sm_mhz):
    """Achieved flops over the tensor pipe's own rate at the sampled SM clock."""
    if not sm_mhz:
        return None
    return tflops * 1e12 / (sm_count * TENSOR_FLOP_PER_CLK_SM * sm_mhz * 1e6)


class Path:
    """One workload's hot path on device-resident inputs: trigflow_coeffs (host,
    FP64) and trigflow_tangent of the latent batch, then the fused attention JVP
    (key chunks + exact merge where the workload is split).  ``step(record=True)``
    brackets every kernel launch with CUDA events on the launching stream."""

    def __init__(self, spec, dev, stream):
        import torch

        from attention_jvp_gb300 import binding, inputs
        self.spec, self.dev, self.stream = spec, dev, stream
        B, H, N, d = spec["B"], spec["H"], spec["N"], spec["d"]
        self.x = inputs.make_inputs(**spec, device=dev)
        self.scale = self.x["scale"]
        self.x0, self.eps, self.t = inputs.latent_for(spec, device=dev)
        self.t_host = self.t.cpu().tolist()
        self.dxdt = torch.empty_like(self.x0)
        self.out = torch.empty((B, H, N, d), dtype=torch.float32, device=dev)
        self.out_t = torch.empty_like(self.out)
        self.lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        self.mu = torch.empty_like(self.lse)
        self.n_chunks = spec.get("kv_chunks", 1)
        self.ws = binding.split_workspace((B, H, N, d), self.n_chunks, dev) if self.n_chunks > 1 else None
        self.bounds = binding.chunk_bounds(N, self.n_chunks)
        # attn_jvp_fwd cuts a short last wave into pieces and merges them in a second launch
        self.pieces = binding.attn_jvp_fwd_last_wave_split(B, H, N, N, d) if self.n_chunks == 1 else 1
        fwd_launches = 1 + (self.pieces > 1) if self.n_chunks == 1 else self.n_chunks + 1
        self.launches_per_step = 1 + fwd_launches
        self.events = {"attention": [], "merge": [], "tangent": []}  # (start, end, units)

    def _launch(self, kind, units, fn, record):
        import torch
        if not record:
            fn()
            return
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        fn()
        e1.record(self.stream)
        self.events[kind].append((e0, e1, units))

    def step(self, record=False):
        from attention_jvp_gb300 import binding
        x, st = self.x, self.stream
        coeffs = [binding.trigflow_coeffs(tt) for tt in self.t_host]  # FP64, host
        self._launch("tangent", self.x0.numel(),
                     lambda: binding.trigflow_tangent(self.x0, self.eps, self.t, out=self.dxdt, stream=st), record)
        args = (x["q"], x["k"], x["v"], x["q_t"], x["k_t"], x["v_t"])
        if self.n_chunks == 1:
            self._launch("attention", self.spec["N"],
                         lambda: binding.attn_jvp_fwd(*args, scale=self.scale, out=self.out, out_t=self.out_t,
                                                      lse=self.lse, mu=self.mu, stream=st), record)
        else:
            ws = self.ws
            for c, (a, n) in enumerate(self.bounds):
                self._launch("attention", n,
                             lambda c=c, a=a, n=n: binding.attn_jvp_fwd_chunk(
                                 *args, a, n, scale=self.scale, out=ws[0][c], out_t=ws[1][c], lse=ws[2][c],
                                 mu=ws[3][c], stream=st), record)
            self._launch("merge", self.n_chunks,
                         lambda: binding.attn_jvp_merge(*ws, out=self.out, out_t=self.out_t, lse=self.lse,
                                                        mu=self.mu, stream=st), record)
        return coeffs

    def clear_events(self):
        for v in self.events.values():
            v.clear()

    def mean_ms(self, kind):
        ev = self.events[kind]
        return sum(a.elapsed_time(b) for a, b, _ in ev) / len(ev) if ev else None


def timed_region(path, steps, sampler, world):
    """Times exactly ``steps`` steps between a barrier and a synchronize on each side,
    with the clocks sampled meanwhile; returns (ms, clock summary)."""
    import torch
    import torch.distributed as dist

    from attention_jvp_gb300 import binding
    path.clear_events()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)  # let the sampler take a first idle-to-load sample
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(path.stream)
    for _ in range(steps):
        path.step(record=True)
    ev1.record(path.stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    sampler.stop()
    binding.attn_jvp_status()
    return ev0.elapsed_time(ev1), ClockSampler.summarize(sampler.lines)


def measure_path(path, steps, warmup, sampler, world, dev):
    """Warm up, time, and retake once if the clock record voids the first region."""
    import torch
    import torch.distributed as dist

    from attention_jvp_gb300 import binding
    for _ in range(warmup):
        path.step()
    torch.cuda.synchronize()
    binding.attn_jvp_status()
    ms, clocks = timed_region(path, steps, sampler, world)
    why = ClockSampler.rejection(clocks)
    veto = float(why is not None)
    if world > 1:  # any rank's veto counts
        tv = torch.tensor([veto], dtype=torch.float64, device=dev)
        dist.all_reduce(tv, op=dist.ReduceOp.MAX)
        veto = float(tv.item())
    if veto:
        ms, clocks = timed_region(path, steps, sampler, world)
        clocks["remeasured"] = why or "another rank's clocks"
        clocks["rejected_again"] = ClockSampler.rejection(clocks)
    return ms, clocks


def kernel_report(path, workload, peaks, peak_src, clocks, sm_count):
    """Roofline of the fused attention kernel (tensor-bound) from its own launch events,
    plus the achieved bandwidth of the HBM-bound kernels of the step."""
    spec = path.spec
    B, H, d = spec["B"], spec["H"], spec["d"]
    ev = path.events["attention"]
    mean_launch_ms = path.mean_ms("attention")
    flops_launch = sum(attention_flops(spec, kv) for _, _, kv in ev) / len(ev)
    achieved = flops_launch / (mean_launch_ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops_sustained"])
    kname = "attn_jvp_fwd_kernel<%d, %d>" % (d, d)
    traffic = traffic_per_launch(kname, workload, H * B)
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": UNIT,
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": "%s bf16_tflops_sustained (kernel timed inside a long step)" % peak_src,
                "frac_of_burst_peak": round(achieved / float(peaks["bf16_tflops"]), 4),
                "kernel": kname, "launch_ms": round(mean_launch_ms, 4),
                "flops_per_launch": flops_launch}
    if path.pieces > 1:
        roofline["last_wave"] = ("cut into %d pieces per unit; launch_ms brackets the whole call, the fused "
                                 "kernel and the merge of the pieces" % path.pieces)
    cn = clock_normalised_frac(achieved, sm_count, clocks.get("sm_mhz"))
    if cn is not None:
        roofline["frac_of_tensor_pipe_at_sampled_clock"] = round(cn, 4)
        roofline["tensor_pipe_rate"] = ("%d SMs x %.0f flop/clk x %.0f MHz (median sampled) = %.1f TFLOP/s"
                                        % (sm_count, TENSOR_FLOP_PER_CLK_SM, clocks["sm_mhz"],
                                           sm_count * TENSOR_FLOP_PER_CLK_SM * clocks["sm_mhz"] * 1e-6))
    hbm = float(peaks["hbm_gbs"])
    others = {}
    t_ms = path.mean_ms("tangent")
    if t_ms:
        nb = tangent_bytes(path.x0.numel())
        others["trigflow_tangent_kernel"] = {
            "bound": "hbm", "algorithmic_bytes": nb, "launch_ms": round(t_ms, 5),
            "achieved": round(nb / (t_ms * 1e-3) / 1e9, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(nb / (t_ms * 1e-3) / 1e9 / hbm, 4),
            "note": "in the step: 12 B per element; %d elements, %.0f MB, a few microseconds of work, so "
                    "launch latency dominates; the epilogue object times it on a batch above L2"
                    % (path.x0.numel(), nb / 1e6)}
    m_ms = path.mean_ms("merge")
    if m_ms:
        nb = merge_bytes(spec, path.n_chunks)
        others["merge_kernel"] = {
            "bound": "hbm", "algorithmic_bytes": nb, "launch_ms": round(m_ms, 4),
            "achieved": round(nb / (m_ms * 1e-3) / 1e9, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(nb / (m_ms * 1e-3) / 1e9 / hbm, 4),
            "note": "%d chunk partials (O_c, Ot_c, LSE_c, mu_c) read, merged O, Ot, LSE, mu written"
                    % path.n_chunks}
    return roofline, others


def cpu_baseline_leg(path, seconds, dev):
    """The FP64 oracle on a bounded sample of ``path``'s workload (query rows of head 0
    against all keys, about ``seconds`` of host time), timed, and compared with the
    last timed step's outputs at the same rows."""
    import torch
    spec = dict(path.spec, scale=path.scale)
    B, H, N = spec["B"], spec["H"], spec["N"]
    xh = host_head(path.x)
    tf, cores, nrows, dt, rows, ref = oracle_sample(spec, xh, oracle_rows_for(spec, xh, seconds), with_outputs=True)
    ridx = torch.as_tensor(rows, device=dev)
    got = [t.reshape(B * H, N, *t.shape[3:])[0][ridx].to("cpu", torch.float64).numpy()
           for t in (path.out, path.out_t, path.lse, path.mu)]
    return {"value": tf, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "%d query rows of head 0 vs all %d keys (%.1f s FP64 on %d host threads)" % (nrows, N, dt, cores),
            "parity_of_the_timed_outputs": parity_on_rows(got, ref)}


def sub_record(name, args, dev, stream, peaks, peak_src, sampler, sm_count):
    """Device-timed line of another workload (same step, same timing rules), for the
    JSON line's ``workloads`` object."""
    import torch
    spec = workload_spec(name)
    path = Path(spec, dev, stream)
    ms, clocks = measure_path(path, args.sub_steps, max(3, args.warmup), sampler, 1, dev)
    flops = attention_flops(spec) * args.sub_steps
    value = flops / (ms * 1e-3) / 1e12
    roofline, others = kernel_report(path, name, peaks, peak_src, clocks, sm_count)
    rec = {"value": round(value, 3), "unit": UNIT, "steps": args.sub_steps, "warmup": max(3, args.warmup),
           "ms_per_step": round(ms / args.sub_steps, 4),
           "config": {"workload": name, "B": spec["B"], "H": spec["H"], "N": spec["N"], "d": spec["d"],
                      "kv_chunks": path.n_chunks},
           "roofline": roofline, "hbm_kernels": others, "clocks": clocks,
           "gpu_launches": path.launches_per_step * args.sub_steps}
    if not args.skip_cpu:
        rec["cpu_baseline"] = cpu_baseline_leg(path, args.sub_cpu_seconds, dev)
    del path
    torch.cuda.empty_cache()
    return rec


def run_gpu(args):
    import torch
    import torch.distributed as dist

    from attention_jvp_gb300 import _build, binding, inputs

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        _build.build()
    if world > 1:
        dist.barrier()
    binding.load()
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count

    spec = workload_spec(args.workload, args.heads)
    B, H, N, d = spec["B"], spec["H"], spec["N"], spec["d"]
    stream = torch.cuda.current_stream()
    path = Path(spec, dev, stream)
    x, scale, n_chunks = path.x, path.scale, path.n_chunks

    gpu_index = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local < len(ids) and ids[local].isdigit():
            gpu_index = int(ids[local])
    sampler = ClockSampler(gpu_index)

    local_ms, clocks = measure_path(path, args.steps, args.warmup, sampler, world, dev)
    flops_step = attention_flops(spec)

    def rmax(v):
        tt = torch.tensor([v], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        return float(tt.item())

    def rsum(v):
        tt = torch.tensor([v], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.SUM)
        return float(tt.item())

    job_ms, job_flops = aggregate(local_ms, flops_step * args.steps, world, rmax, rsum)
    value = job_flops / (job_ms * 1e-3) / 1e12

    peaks, peak_src = load_peaks()
    roofline, hbm_kernels = kernel_report(path, args.workload, peaks, peak_src, clocks, sm_count)
    out, lse = path.out, path.lse

    # ---- end to end through the C ABI with host buffers ----
    # Every step copies its inputs in from pinned host memory and its results
    # out: the latent batch around trigflow_tangent, and the six attention
    # inputs / four outputs through attn_jvp_fwd_host, which pipelines the
    # attention transfers against compute inside the library.
    e2e = None
    if not args.skip_e2e:
        x0, eps, t, dxdt, t_host = path.x0, path.eps, path.t, path.dxdt, path.t_host
        host_in = {n: torch.empty(x[n].shape, dtype=x[n].dtype, pin_memory=True) for n in inputs.NAMES}
        for n in inputs.NAMES:
            host_in[n].copy_(x[n])
        host_out = [torch.empty(tt.shape, dtype=tt.dtype, pin_memory=True)
                    for tt in (path.out, path.out_t, path.lse, path.mu)]
        lat_in = [torch.empty(tt.shape, dtype=tt.dtype, pin_memory=True) for tt in (x0, eps, t)]
        for hdst, src in zip(lat_in, (x0, eps, t)):
            hdst.copy_(src)
        lat_dev = [torch.empty_like(tt) for tt in (x0, eps, t)]
        lat_out = torch.empty(dxdt.shape, dtype=dxdt.dtype, pin_memory=True)
        ws_host = binding.host_workspace(tuple(x["q"].shape), n_chunks, device=dev)
        h2d = sum(tt.numel() * tt.element_size() for tt in list(host_in.values()) + lat_in)
        d2h = sum(tt.numel() * tt.element_size() for tt in host_out + [lat_out])

        # The latent batch's copies and tangent are independent of the attention, so
        # they run on a stream of their own beside the host path; the step ends when
        # both have (the caller's stream waits for the latent stream's last copy).
        lat_stream = torch.cuda.Stream(device=dev)

        def e2e_step():
            lat_stream.wait_stream(stream)
            with torch.cuda.stream(lat_stream):
                for hsrc, ddst in zip(lat_in, lat_dev):
                    ddst.copy_(hsrc, non_blocking=True)
                coeffs = [binding.trigflow_coeffs(tt) for tt in t_host]  # FP64, host
                binding.trigflow_tangent(lat_dev[0], lat_dev[1], lat_dev[2], out=dxdt, stream=lat_stream)
                lat_out.copy_(dxdt, non_blocking=True)
            binding.attn_jvp_fwd_host(*(host_in[n] for n in inputs.NAMES), *host_out, scale=scale,
                                      n_chunks=n_chunks, workspace=ws_host, stream=stream)
            stream.wait_stream(lat_stream)
            return coeffs

        e2e_step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e_ms, e_flops = aggregate(e0.elapsed_time(e1), flops_step * args.e2e_steps, world, rmax, rsum)
        e2e = {"value": round(e_flops / (e_ms * 1e-3) / 1e12, 3), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
               "ms_per_step": round(e_ms / args.e2e_steps, 3),
               "path": "attn_jvp_fwd_host (transfers pipelined against compute per head group)"}
        binding.attn_jvp_status()
        del host_in, host_out, lat_in, lat_dev, lat_out, ws_host

    # ---- output-side kernels (not part of the timed step): bandwidth on a batch above L2 ----
    epi = None
    if not args.skip_epilogue and rank == 0:
        epi = measure_epilogue(spec, dev, stream, peaks)

    # ---- QK normalisation JVP (the input side; not part of the timed step) ----
    qk_norm = None
    if not args.skip_epilogue and rank == 0:
        qk_norm = measure_qk_norm(x, dev, stream, peaks)

    # ---- primal attention backward (not part of the timed step) ----
    bwd = None
    if not args.skip_backward and rank == 0:  # on the (merged) forward's O and LSE
        bwd = measure_backward(x, spec, out, lse, dev, stream, peaks)

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1 only) ----
    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu:
        cpu = cpu_baseline_leg(path, args.cpu_seconds, dev)

    total_bytes = sum(x[n].numel() * x[n].element_size() for n in inputs.NAMES)
    launches = path.launches_per_step * args.steps
    del path, x, out, lse
    torch.cuda.empty_cache()

    # ---- the other workloads, device-timed under the same rules (rank 0, N = 1 only) ----
    subs = None
    if rank == 0 and world == 1 and args.also:
        subs = {}
        for name in [w for w in args.also.split(",") if w and w != args.workload]:
            subs[name] = sub_record(name, args, dev, stream, peaks, peak_src, sampler, sm_count)

    if rank == 0:
        rec = {
            "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(job_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": args.workload, "B": B, "H": H, "N": N, "d": d, "kv_chunks": n_chunks,
                       "parallelism": "replicas" if world > 1 else "single",
                       "l2": "inputs larger than L2 (%.2f GB of bf16 inputs per step vs 129 MB L2)"
                             % (total_bytes / 1e9)},
            "pct_of_peak": {"bf16_sustained_%.0f" % float(peaks["bf16_tflops_sustained"]):
                            round(100 * value / world / float(peaks["bf16_tflops_sustained"]), 2),
                            "bf16_burst_%.0f" % float(peaks["bf16_tflops"]):
                            round(100 * value / world / float(peaks["bf16_tflops"]), 2)},
            "roofline": roofline,
            "hbm_kernels": hbm_kernels,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "epilogue": epi,
            "qk_norm": qk_norm,
            "backward": bwd,
            "clocks": clocks,
            "workloads": subs,
        }
        print(json.dumps(rec))
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
