"""Throughput benchmark: context-parallel causal attention, forward + backward.

Workload (default): bf16, one 65536-token sequence, 32 query / 8 key-value
heads (GQA), head dim 128, cut into 8 context-parallel shards in the zigzag
layout; q, k, v, dout iid N(0, 1) (synthetic, seeded).

One step = the whole hot path on one batch: shard permutation of q, k, v,
dout (global -> sharded order), the fused forward (o, lse), the backward
(dq, dk, dv), and the permutation of o, dq, dk, dv back to global order.
``value`` counts attention FLOPs only over visible (query, key) pairs:
fwd = pairs * hq * (2 d_qk + 2 d_v), bwd = pairs * hq * (6 d_qk + 4 d_v).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N > 1 runs under torchrun, one process per GPU, each GPU an independent
replica of the workload (the path needs no exchange on one node: the KV ring
is a visiting order over shards already in device memory).
``--impl reference`` times the float64 CPU oracle on a bounded sample of the
same workload instead.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# Thread counts of the CPU oracle's BLAS and OpenMP pools, set before numpy
# and torch load them (an explicit setting from the environment wins).
for _var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
    os.environ.setdefault(_var, str(_host_cores()))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "CP causal attn TFLOP/s fwd & fwd+bwd (bf16, S=64K) and % of GB300 BF16 peak"
DEFAULT_WORKLOAD = "bf16_gqa_s64k_h32kv8_d128_c8_zigzag"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK), "fallback"


# ----------------------------------------------------------------------------- oracle (CPU baseline)

def oracle_sample(w: workloads.Workload, budget_tokens: int = 8192):
    """Times the float64 oracle's forward + backward on a bounded sample of the
    workload: the first `budget_tokens` tokens of the stream and the query
    heads of the first key/value head.  Returns (tflops, seconds, desc)."""
    import oracle

    lengths = w.lengths()
    Ts = min(budget_tokens, w.total_tokens)
    # the sample keeps the workload's sequence boundaries inside its prefix
    cu = [0]
    for L in lengths:
        if cu[-1] >= Ts:
            break
        cu.append(min(Ts, cu[-1] + L))
    G = w.hq // w.hkv
    sub = w.replace(total_tokens=Ts, hq=G, hkv=1, seqlens=tuple(np.diff(cu).tolist()), varlen_range=None)
    inp = workloads.make_inputs(sub, with_dout=True)
    t0 = time.perf_counter()
    oracle.attn_backward(inp["q"], inp["k"], inp["v"], inp["dout"], cu, w.scale, w.causal)
    dt = time.perf_counter() - t0
    flops = sub.flops_fwd() + sub.flops_bwd()
    desc = (f"float64 oracle fwd+bwd on the first {Ts} tokens, {G} query heads / 1 kv head "
            f"of the workload ({len(cu) - 1} sequence(s))")
    return flops / dt / 1e12, dt, desc


def kernel_source_digest(src: str) -> str:
    """First 16 hex digits of the sha256 over a kernel's .cu file followed by
    the two headers every kernel includes (internal.h, sm103_ptx.cuh)."""
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "context_long_sequence_zigzag_gb300", "csrc")
    for name in (src, "internal.h", "sm103_ptx.cuh"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/dram_traffic.txt), or None when none was recorded for this
    kernel and workload or the kernel's source changed since the capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    src = {"attn_fwd_tc_kernel": "attn_fwd_sm103.cu", "attn_bwd_dkdv_kernel": "attn_bwd_sm103.cu",
           "attn_bwd_dq_kernel": "attn_bwd_sm103.cu"}.get(kernel)
    if src is None:
        return None
    digest = kernel_source_digest(src)
    with open(path) as f:
        for line in f:
            fields = dict(tok.split("=", 1) for tok in line.split() if "=" in tok)
            if fields.get("kernel") == kernel and fields.get("workload") == workload and \
                    fields.get("source_sha256_16") == digest:
                return int(float(fields["bytes_per_launch"]))
    return None


def l2_note(w: workloads.Workload) -> str:
    """How the timed steps stand to the 129 MB L2: the inputs are not flushed
    between steps, so they have to be larger than L2."""
    q_bytes = w.total_tokens * w.hq * w.d_qk * (4 if w.dtype == "f32" else 2)
    mib = q_bytes / 2**20
    if q_bytes > 129e6:
        return f"inputs larger than L2 (q alone is {mib:.0f} MiB), not flushed between steps"
    return f"q is {mib:.1f} MiB, smaller than L2, not flushed between steps"


def chosen_workload(args) -> workloads.Workload:
    """The --workload preset with the command line's overrides applied; an
    overridden workload's name lists them."""
    w = workloads.get(args.workload)
    kw = {}
    if args.layout:
        kw["layout"] = args.layout
    if args.cp_size:
        kw["cp_size"] = args.cp_size
    if args.seed is not None:
        kw["seed"] = args.seed
    if args.heads:
        hq, hkv = (int(x) for x in args.heads.split(":"))
        if hq < 1 or hkv < 1 or hq % hkv:
            raise SystemExit("--heads wants HQ:HKV with HKV dividing HQ")
        kw["hq"], kw["hkv"] = hq, hkv
    if args.seq_len is not None:
        if args.seq_len < 1:
            raise SystemExit("--seq-len wants a positive token count")
        if w.seqlens is not None:
            raise SystemExit("--seq-len does not apply to a workload with fixed sequence lengths")
        kw["total_tokens"] = args.seq_len  # a varlen pack is drawn to this many tokens
    if not kw:
        return w
    tag = ",".join(f"{k}={v}" for k, v in kw.items())
    return w.replace(name=f"{w.name}[{tag}]", **kw)


def cpu_cores() -> int:
    return _host_cores()


def cpu_baseline_entry(w: workloads.Workload, tf: float, secs: float, desc: str) -> dict:
    """The oracle's measured rate on its sample, the thread counts it ran
    with, and a labelled extrapolation of that rate to the whole workload
    (the oracle's cost grows with the visible pairs, as the FLOP count does)."""
    full = w.flops_fwd() + w.flops_bwd()
    return {"value": round(tf, 6), "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle", "sample": desc,
            "seconds": round(secs, 2),
            "threads": {"OPENBLAS_NUM_THREADS": os.environ.get("OPENBLAS_NUM_THREADS"),
                        "OMP_NUM_THREADS": os.environ.get("OMP_NUM_THREADS"),
                        "torch_intraop": torch.get_num_threads()},
            "extrapolated_full_problem": {"seconds": round(full / (tf * 1e12), 1),
                                          "note": "estimate: the whole workload's fwd+bwd FLOPs at the sample's "
                                                  "measured rate; not measured"}}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- GPU arm

class Runner:
    """Holds device buffers and runs one step of the hot path through the C ABI."""

    def __init__(self, w: workloads.Workload, device: torch.device):
        import context_long_sequence_zigzag_gb300 as cpa

        self.cpa = cpa
        self.w = w
        self.dev = device
        inp = workloads.make_inputs(w, device=device, with_dout=True)
        self.cu = inp["cu_seqlens"].tolist()
        self.prob = cpa.Problem(w.total_tokens, w.hq, w.hkv, w.d_qk, w.d_v, w.cp_size, w.layout, self.cu,
                                w.causal, w.scale, "blocked", torch.bfloat16)
        self.g = {n: inp[n] for n in ("q", "k", "v", "dout")}  # global order (inputs)
        self.s = {n: torch.empty_like(t) for n, t in self.g.items()}  # sharded copies
        T = w.total_tokens
        bf = torch.bfloat16
        self.o = torch.empty(T, w.hq, w.d_v, dtype=bf, device=device)
        self.lse = torch.empty(w.hq, T, dtype=torch.float32, device=device)
        self.dq = torch.empty(T, w.hq, w.d_qk, dtype=bf, device=device)
        self.dk = torch.empty(T, w.hkv, w.d_qk, dtype=bf, device=device)
        self.dv = torch.empty(T, w.hkv, w.d_v, dtype=bf, device=device)
        self.out = {n: torch.empty_like(t) for n, t in
                    (("o", self.o), ("dq", self.dq), ("dk", self.dk), ("dv", self.dv))}
        self.ws_perm = cpa.workspace(self.prob, cpa.CP_OP_PERMUTE, device)
        self.ws_fwd = cpa.workspace(self.prob, cpa.CP_OP_FWD, device)
        self.ws_bwd = cpa.workspace(self.prob, cpa.CP_OP_BWD, device)
        self.ws_dkdv = cpa.workspace(self.prob, cpa.CP_OP_BWD_DKDV, device)
        self.ws_dq = cpa.workspace(self.prob, cpa.CP_OP_BWD_DQ, device)
        self.dpsum = torch.empty(w.hq, T, dtype=torch.float32, device=device)
        self.ev = []  # (fwd_start, fwd_end, bwd_start, bwd_end) per timed step
        self.launches_per_step = 4 + 1 + 3 + 4  # permute x4, fwd, D pre-pass, dK/dV, dQ, permute x4

    def step(self, record: bool = False, combined_bwd: bool = False):
        self.permute_in()
        self.attend(record, combined_bwd)
        self.permute_out()

    def permute_in(self):
        """Global-order inputs -> sharded order (what the C ranks would hold)."""
        for n in ("q", "k", "v", "dout"):
            self.cpa.cp_shard_permute(self.prob, self.g[n], out=self.s[n], ws=self.ws_perm)

    def permute_out(self):
        """Sharded o, dq, dk, dv -> global order."""
        for n, t in (("o", self.o), ("dq", self.dq), ("dk", self.dk), ("dv", self.dv)):
            self.cpa.cp_shard_permute(self.prob, t, inverse=True, out=self.out[n], ws=self.ws_perm)

    def attend(self, record: bool = False, combined_bwd: bool = False):
        """Forward, then backward, on the sharded buffers."""
        cpa = self.cpa
        e = [torch.cuda.Event(enable_timing=True) for _ in range(5)] if record else None
        if record:
            e[0].record()
        cpa.cp_attn_fwd(self.prob, self.s["q"], self.s["k"], self.s["v"], self.o, self.lse, self.ws_fwd)
        if record:
            e[1].record()
        if combined_bwd:
            cpa.cp_attn_bwd(self.prob, self.s["q"], self.s["k"], self.s["v"], self.o, self.lse, self.s["dout"],
                            self.dq, self.dk, self.dv, self.ws_bwd)
        else:
            # the same kernels as cp_attn_bwd, called one by one so that each
            # is timed on its own
            cpa.cp_attn_bwd_prep(self.prob, self.o, self.s["dout"], self.dpsum)
            if record:
                e[2].record()
            cpa.cp_attn_bwd_dkdv(self.prob, self.s["q"], self.s["k"], self.s["v"], self.lse, self.dpsum,
                                 self.s["dout"], self.dk, self.dv, self.ws_dkdv)
            if record:
                e[3].record()
            cpa.cp_attn_bwd_dq(self.prob, self.s["q"], self.s["k"], self.s["v"], self.lse, self.dpsum,
                               self.s["dout"], self.dq, self.ws_dq)
        if record:
            e[4].record()
            self.ev.append(e)

    def kernel_times_ms(self):
        """Mean device time of (fwd, whole bwd, dK/dV kernel, dQ kernel)."""
        fwd = [e[0].elapsed_time(e[1]) for e in self.ev]
        bwd = [e[1].elapsed_time(e[4]) for e in self.ev]
        dkdv = [e[2].elapsed_time(e[3]) for e in self.ev]
        dq = [e[3].elapsed_time(e[4]) for e in self.ev]
        return statistics.mean(fwd), statistics.mean(bwd), statistics.mean(dkdv), statistics.mean(dq)


def ulysses_measure(r: Runner, steps: int = 3, warmup: int = 2) -> dict:
    """The step's attention computed the Ulysses way on the same sharded
    inputs (all-to-all, full-sequence attention of every rank's heads,
    all-to-all back: cp_ulysses_attn_fwd / _bwd), device time per step, and
    the bandwidth of one all-to-all re-layout of q (read + write)."""
    cpa, w = r.cpa, r.w
    try:
        ws_f = cpa.workspace(r.prob, cpa.CP_OP_ULYSSES_FWD, r.dev)
        ws_b = cpa.workspace(r.prob, cpa.CP_OP_ULYSSES_BWD, r.dev)
    except cpa.CpError as e:
        return {"unavailable": str(e)}
    s = r.s
    times = []
    for i in range(warmup + steps):
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        cpa.cp_ulysses_attn_fwd(r.prob, s["q"], s["k"], s["v"], r.o, r.lse, ws_f)
        e[1].record()
        cpa.cp_ulysses_attn_bwd(r.prob, s["q"], s["k"], s["v"], r.o, r.lse, s["dout"], r.dq, r.dk, r.dv, ws_b)
        e[2].record()
        if i >= warmup:
            times.append(e)
    torch.cuda.synchronize()
    if cpa.cp_device_status() != 0:
        raise RuntimeError("device wait timeout in the Ulysses path")
    fwd = statistics.mean(a.elapsed_time(b) for a, b, _ in times)
    bwd = statistics.mean(b.elapsed_time(c) for _, b, c in times)
    del ws_f, ws_b
    # one re-layout of q: T*hq*d_qk bf16 read and written
    u = torch.empty(w.cp_size, w.total_tokens, w.hq // w.cp_size, w.d_qk, dtype=torch.bfloat16, device=r.dev)
    ws_a = cpa.workspace(r.prob, cpa.CP_OP_ULYSSES_A2A, r.dev)
    best = float("inf")
    for _ in range(6):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        cpa.cp_ulysses_a2a(r.prob, s["q"], out=u, ws=ws_a)
        b.record()
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b))
    nbytes = 2 * s["q"].numel() * 2
    return {"fwd_ms": round(fwd, 3), "bwd_ms": round(bwd, 3), "ms_per_step": round(fwd + bwd, 3),
            "a2a_q": {"bytes": nbytes, "ms": round(best, 4), "gbs": round(nbytes / (best * 1e-3) / 1e9, 1)}}


def linear_measure(dev, steps: int = 5, warmup: int = 3) -> dict:
    """Decayed linear attention with AllGather CP (cp_lin_attn_fwd) on a
    long-sequence configuration: S = 64K tokens, 16 heads of 128, C = 8
    contiguous pieces, bf16, decays alpha = exp(g) in (0.39, 0.95).  Its three
    passes run on the tensor cores (block states, output) and as a plain scan
    (the decayed prefix over the gathered states); what bounds them is HBM,
    so the roofline counts the bytes the method moves: the state pass reads
    k and v and writes one D x D state per (block, head); the prefix reads the
    states and writes the initial states; the output pass reads q, k, v and
    the initial states and writes o.  Tensor FLOPs of the chunked form are
    reported beside it."""
    import context_long_sequence_zigzag_gb300 as cpa

    T, H, D, C = 65536, 16, 128, 8
    BLOCK, CHUNK = 512, 128  # tokens per parallel block, tokens per chunk
    gen = torch.Generator(device=dev).manual_seed(7)
    q = (torch.randn(T, H, D, device=dev, generator=gen) * 0.5).to(torch.bfloat16)
    k = (torch.randn(T, H, D, device=dev, generator=gen) * 0.5).to(torch.bfloat16)
    v = torch.randn(T, H, D, device=dev, generator=gen).to(torch.bfloat16)
    g = -torch.rand(H, device=dev, generator=gen) * 0.9 - 0.05
    prob = cpa.Problem(T, H, H, D, D, C, "contiguous", None, True, D ** -0.5, "blocked", torch.bfloat16)
    ws = cpa.workspace(prob, cpa.CP_OP_LIN_FWD, dev)
    o = torch.empty_like(v)
    times = []
    for i in range(warmup + steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        cpa.cp_lin_attn_fwd(prob, q, k, v, g, o, ws)
        b.record()
        if i >= warmup:
            times.append((a, b))
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in times)
    nblocks = C * -(-(T // C) // BLOCK)
    state_bytes = nblocks * H * D * D * 4
    nbytes = T * H * D * 2 * (2 + 3 + 1) + 4 * state_bytes
    gbs = nbytes / (ms * 1e-3) / 1e9
    peaks, _ = load_peaks()
    peak_gbs = float(peaks.get("hbm_gbs", FALLBACK["hbm_gbs"]))
    # per 128-token chunk and head: Q K^T, A' V, Q H and the state update in
    # the output pass, the state update again in the state pass (2*C*D*D each)
    flops = float(T // CHUNK) * H * 5 * 2 * CHUNK * D * D
    return {"config": {"total_tokens": T, "heads": H, "head_dim": D, "cp_size": C, "layout": "contiguous",
                       "dtype": "bf16"},
            "ms": round(ms, 3), "tensor_tflops": round(flops / (ms * 1e-3) / 1e12, 2),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": round(peak_gbs, 1), "unit": "GB/s",
                         "frac": round(gbs / peak_gbs, 4), "traffic": None, "algorithmic_bytes": nbytes}}


def other_configs_measure(dev, main_name: str, steps: int = 2, warmup: int = 1) -> dict:
    """Device throughput of the other standard bf16 problems (S = 16K GQA, the
    128K-token varlen pack, the S = 256K MLA shape): the same step as the
    headline (permutes, forward, D pre-pass, dK/dV, dQ, permutes back), the
    same FLOP rule, and the forward / backward fractions of the bf16 peak.
    The fp32 S = 256 problem is a correctness case of the CUDA-core path
    and gets no throughput line."""
    peaks, _ = load_peaks()
    burst = float(peaks.get("bf16_tflops", FALLBACK["bf16_tflops"]))
    out = {}
    for name in workloads.ORDER:
        w = workloads.get(name)
        if name == main_name or w.dtype != "bf16":
            continue
        r = Runner(w, dev)
        for _ in range(warmup):
            r.step()
        torch.cuda.synchronize()
        r.ev.clear()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(steps):
            r.step(record=True)
        t1.record()
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / steps
        fwd_ms, bwd_ms, _, _ = r.kernel_times_ms()
        f_fwd, f_bwd = w.flops_fwd(), w.flops_bwd()
        fwd_tf, bwd_tf = f_fwd / (fwd_ms * 1e-3) / 1e12, f_bwd / (bwd_ms * 1e-3) / 1e12
        out[name] = {"ms_per_step": round(ms, 3), "tflops": round((f_fwd + f_bwd) / (ms * 1e-3) / 1e12, 2),
                     "fwd_tflops": round(fwd_tf, 2), "bwd_tflops": round(bwd_tf, 2),
                     "fwd_frac_of_burst": round(fwd_tf / burst, 4), "bwd_frac_of_burst": round(bwd_tf / burst, 4)}
        status = r.cpa.cp_device_status()
        if status != 0:
            raise RuntimeError(f"device wait timeout code {status:#x} ({name})")
        del r
        torch.cuda.empty_cache()
    return out


def e2e_measure(r: Runner, steps: int, warmup: int):
    """Same metric through the ABI with host buffers: every step copies its
    inputs (q, k, v, dout) in from pinned host memory and its results (o,
    dq, dk, dv) back out, all inside the timed region.  The copies are
    pipelined against the kernels the way a training loop prefetches: on
    two copy streams, step i+1's inputs go in once step i has permuted its
    own into sharded order, and step i's results come out while step i+1
    computes.  Events order every reuse of a buffer."""
    host_in = {n: t.cpu().pin_memory() for n, t in r.g.items()}
    host_out = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in r.out.items()}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def pipeline(n: int):
        h2d_done = [torch.cuda.Event() for _ in range(n)]
        perm_done = [torch.cuda.Event() for _ in range(n)]
        out_ready = [torch.cuda.Event() for _ in range(n)]
        d2h_done = [torch.cuda.Event() for _ in range(n)]
        s_in.wait_stream(comp)
        s_out.wait_stream(comp)

        def copy_in(i):
            with torch.cuda.stream(s_in):
                if i > 0:
                    s_in.wait_event(perm_done[i - 1])  # step i-1 no longer needs the global-order inputs
                for n_, t in host_in.items():
                    r.g[n_].copy_(t, non_blocking=True)
                h2d_done[i].record(s_in)

        copy_in(0)
        for i in range(n):
            comp.wait_event(h2d_done[i])
            r.permute_in()
            perm_done[i].record(comp)
            if i + 1 < n:
                copy_in(i + 1)
            r.attend(combined_bwd=True)
            if i > 0:
                comp.wait_event(d2h_done[i - 1])  # step i-1's results are out of the output buffers
            r.permute_out()
            out_ready[i].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(out_ready[i])
                for n_, t in host_out.items():
                    t.copy_(r.out[n_], non_blocking=True)
                d2h_done[i].record(s_out)
        comp.wait_stream(s_out)

    def serial(n: int):
        # every copy on the compute stream, in order: nothing overlaps
        for _ in range(n):
            for n_, t in host_in.items():
                r.g[n_].copy_(t, non_blocking=True)
            r.step(combined_bwd=True)
            for n_, t in host_out.items():
                t.copy_(r.out[n_], non_blocking=True)

    def timed(fn, n):
        fn(warmup)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(comp)
        fn(n)
        e1.record(comp)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    # the host link is shared with the node's other GPUs: the median of three
    # timed runs of each form
    ms_pipe = statistics.median(timed(pipeline, steps) for _ in range(3))
    ms_serial = statistics.median(timed(serial, max(2, steps // 4)) for _ in range(3))
    return ms_pipe, ms_serial, h2d, d2h


def ring_measure(r: Runner, steps: int = 3, warmup: int = 2) -> dict:
    """The forward as a ring with explicit KV transport (cp_ring_attn_fwd):
    C steps of block attention merged into an fp32 accumulator, while every
    rank's KV shard moves one rank on by device-to-device copies on a second
    stream.  Device time with the copies on their own stream (overlapped) and
    serialised on the compute stream, the same set of copies alone, and the
    share of the copy time the overlap hides."""
    cpa, w = r.cpa, r.w
    ws = cpa.workspace(r.prob, cpa.CP_OP_RING_FWD, r.dev)
    comm = torch.cuda.Stream(priority=-1)  # copies ahead of the attention kernel's waiting CTAs
    s = r.s

    def timed(overlap: bool) -> float:
        ev = []
        for i in range(warmup + steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            cpa.cp_ring_attn_fwd(r.prob, s["q"], s["k"], s["v"], r.o, r.lse, ws, comm_stream=comm, overlap=overlap)
            b.record()
            if i >= warmup:
                ev.append((a, b))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    ms_ovl, ms_ser = timed(True), timed(False)
    status = cpa.cp_device_status()
    if status != 0:
        raise RuntimeError(f"device wait timeout code {status:#x} (ring)")
    # the transfers alone: C - 1 steps, every rank's shard of K and of V
    off = cpa.cp_shard_offsets(r.prob)
    C = w.cp_size
    rows = max(off[i + 1] - off[i] for i in range(C))
    slot_k = torch.empty(2, C, rows, w.hkv, w.d_qk, dtype=torch.bfloat16, device=r.dev)
    slot_v = torch.empty(2, C, rows, w.hkv, w.d_v, dtype=torch.bfloat16, device=r.dev)
    nbytes = 0
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for rep in range(2):
        a.record()
        for st in range(C - 1):
            for rk in range(C):
                n = off[(rk - st) % C + 1] - off[(rk - st) % C]
                dst = (st + 1) % 2
                slot_k[dst, (rk + 1) % C, :n].copy_(slot_k[st % 2, rk, :n])
                slot_v[dst, (rk + 1) % C, :n].copy_(slot_v[st % 2, rk, :n])
                if rep == 0:
                    nbytes += n * w.hkv * (w.d_qk + w.d_v) * 2
        b.record()
        torch.cuda.synchronize()
    ms_copy = a.elapsed_time(b)
    del ws, slot_k, slot_v
    return {"ms_overlapped": round(ms_ovl, 3), "ms_serialised": round(ms_ser, 3),
            "ms_saved_by_overlap": round(ms_ser - ms_ovl, 3),
            "ms_copies_alone": round(ms_copy, 3), "copies_alone": "the same bytes by cudaMemcpyAsync with the GPU "
                                                                  "to itself (context for the transfer volume)",
            "copy_bytes": nbytes, "tflops_overlapped": round(w.flops_fwd() / (ms_ovl * 1e-3) / 1e12, 2),
            "transport": "per step, one copy kernel per tensor (one CTA per SM, beside the attention CTAs) on a "
                         "high-priority stream; unmeasured across GPUs"}


def aux_bandwidth(r: "Runner", reps: int = 5) -> dict:
    """HBM throughput of the bandwidth-bound kernels on buffers larger than L2:
    the shard permutation of q (one launch), one LSE merge of fp32 partials
    over all rows and heads (the stepwise ring's update) and the backward's
    pre-pass D = rowsum(dout * o)."""
    cpa, w, dev = r.cpa, r.w, r.dev
    out = {}
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    x = r.g["q"]
    y = torch.empty_like(x)
    nbytes = 2 * x.numel() * x.element_size()
    times = []
    for i in range(reps + 1):
        ev[0].record()
        cpa.cp_shard_permute(r.prob, x, out=y, ws=r.ws_perm)
        ev[1].record()
        torch.cuda.synchronize()
        if i:
            times.append(ev[0].elapsed_time(ev[1]))
    out["shard_permute"] = {"bytes": nbytes, "ms": round(min(times), 4),
                            "gbs": round(nbytes / (min(times) * 1e-3) / 1e9, 1)}
    rows = w.total_tokens
    o_acc = torch.randn(rows, w.hq, w.d_v, device=dev)
    o_part = torch.randn(rows, w.hq, w.d_v, device=dev)
    l_acc = torch.randn(w.hq, rows, device=dev)
    l_part = torch.randn(w.hq, rows, device=dev)
    nbytes = rows * w.hq * (3 * w.d_v * 4 + 12)
    times = []
    for i in range(reps + 1):
        ev[0].record()
        cpa.cp_lse_merge(r.prob, o_acc, l_acc, o_part, l_part)
        ev[1].record()
        torch.cuda.synchronize()
        if i:
            times.append(ev[0].elapsed_time(ev[1]))
    out["lse_merge"] = {"bytes": nbytes, "ms": round(min(times), 4),
                        "gbs": round(nbytes / (min(times) * 1e-3) / 1e9, 1)}
    del o_acc, o_part, l_acc, l_part, y
    # the backward's pre-pass D = rowsum(dout * o): reads o and dout, writes D
    dp = torch.empty(w.hq, w.total_tokens, dtype=torch.float32, device=dev)
    nbytes = 2 * r.o.numel() * r.o.element_size() + dp.numel() * 4
    times = []
    for i in range(reps + 1):
        ev[0].record()
        cpa.cp_attn_bwd_prep(r.prob, r.o, r.s["dout"], dp)
        ev[1].record()
        torch.cuda.synchronize()
        if i:
            times.append(ev[0].elapsed_time(ev[1]))
    out["bwd_preprocess"] = {"bytes": nbytes, "ms": round(min(times), 4),
                             "gbs": round(nbytes / (min(times) * 1e-3) / 1e9, 1)}
    return out


def slowest_rank_ms(ms: float, device) -> float:
    """The timed region of a multi-rank run lasts as long as its slowest
    rank: the maximum of every rank's time (any backend; on one rank, ms)."""
    dist = torch.distributed
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_gpu(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = chosen_workload(args)
    r = Runner(w, dev)
    cpa = r.cpa

    for _ in range(args.warmup):
        r.step()
    torch.cuda.synchronize()
    if cpa.cp_device_status() != 0:
        raise RuntimeError("device wait timeout during warm-up")

    clocks = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        r.step(record=True)
    t1.record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ms = slowest_rank_ms(t0.elapsed_time(t1) / args.steps, dev)
    status = cpa.cp_device_status()
    if status != 0:
        raise RuntimeError(f"device wait timeout code {status:#x}")
    fwd_ms, bwd_ms, dkdv_ms, dq_ms = r.kernel_times_ms()

    # at least 8 steps: one step's H2D before the first and one D2H after the last are
    # not overlapped, and the per-step number should be the steady state
    e2e_ms, e2e_serial_ms, h2d, d2h = e2e_measure(r, min(max(args.steps, 8), 16), 1)
    ring = ring_measure(r) if not args.no_ring else {"skipped": "--no-ring"}
    aux = aux_bandwidth(r)
    uly = ulysses_measure(r) if not args.no_ulysses else {"skipped": "--no-ulysses"}
    lin = linear_measure(dev) if not args.no_linear else {"skipped": "--no-linear"}
    others = (other_configs_measure(dev, args.workload) if world == 1 and not args.no_other_configs
              else {"skipped": "--no-other-configs" if args.no_other_configs else "N > 1"})

    peaks, peak_kind = load_peaks()
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK["bf16_tflops_sustained"]))
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK["bf16_tflops"]))
    f_fwd, f_bwd = w.flops_fwd(), w.flops_bwd()
    value = (f_fwd + f_bwd) * world / (ms * 1e-3) / 1e12
    fwd_tf = f_fwd / (fwd_ms * 1e-3) / 1e12
    bwd_tf = f_bwd / (bwd_ms * 1e-3) / 1e12
    # Each kernel is credited only the method's own GEMMs it performs over the
    # visible pairs: the forward its two (Q K^T, P V); dK/dV four of the
    # backward's five (Q K^T recomputed, dO V^T, P^T dO, dS^T Q); dQ the fifth
    # (dS K).  The dQ kernel also recomputes Q K^T and dO V^T, which the
    # dK/dV kernel already counts: that repeated work is not credited.
    pairs_h = float(w.visible_pairs()) * w.hq
    kernels = {
        "attn_fwd_tc_kernel": (fwd_ms, pairs_h * (2 * w.d_qk + 2 * w.d_v)),
        "attn_bwd_dkdv_kernel": (dkdv_ms, pairs_h * (4 * w.d_qk + 4 * w.d_v)),
        "attn_bwd_dq_kernel": (dq_ms, pairs_h * (2 * w.d_qk)),
    }
    executed_dq = pairs_h * (4 * w.d_qk + 2 * w.d_v)  # what the dQ kernel runs, recomputation included
    dom = max(kernels, key=lambda k: kernels[k][0])
    dom_ms, dom_flops = kernels[dom]
    dom_tf = dom_flops / (dom_ms * 1e-3) / 1e12

    result = None
    if rank == 0:
        traffic = recorded_traffic(dom, w.name)
        result = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms, 3),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded iid N(0,1) q, k, v, dout)",
            "config": {"workload": w.name, "total_tokens": w.total_tokens, "hq": w.hq, "hkv": w.hkv,
                       "d_qk": w.d_qk, "d_v": w.d_v, "cp_size": w.cp_size, "layout": w.layout, "causal": w.causal,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU, C virtual ranks",
                       "l2": l2_note(w)},
            "fwd_tflops": round(fwd_tf, 2),
            "bwd_tflops": round(bwd_tf, 2),
            "fwd_bwd_pct_of_peak": round(100 * value / world / peak_sus, 2),
            "roofline": {"bound": "tensor", "kernel": dom, "achieved": round(dom_tf, 2), "peak": peak_sus,
                         "unit": "TFLOP/s", "frac": round(dom_tf / peak_sus, 4),
                         "peak_kind": f"bf16 sustained, {peak_kind}", "traffic": traffic,
                         "ms_per_launch": round(dom_ms, 3),
                         "kernels": {k: {"ms": round(t, 3), "tflops": round(fl / (t * 1e-3) / 1e12, 2),
                                         "frac": round(fl / (t * 1e-3) / 1e12 / peak_sus, 4),
                                         "frac_of_burst": round(fl / (t * 1e-3) / 1e12 / peak_burst, 4)}
                                     for k, (t, fl) in kernels.items()},
                         "credit": "method GEMMs only: fwd 2d_qk+2d_v, dK/dV 4d_qk+4d_v, dQ 2d_qk (dS K) per "
                                   "pair and head",
                         "dq_kernel_executed_tflops": round(executed_dq / (dq_ms * 1e-3) / 1e12, 2),
                         "bwd_whole": {"ms": round(bwd_ms, 3), "tflops": round(bwd_tf, 2),
                                       "frac": round(bwd_tf / peak_sus, 4),
                                       "frac_of_burst": round(bwd_tf / peak_burst, 4)}},
            "hbm_kernels": {k: dict(v, frac=round(v["gbs"] / float(peaks.get("hbm_gbs", FALLBACK["hbm_gbs"])), 4),
                                    peak_gbs=float(peaks.get("hbm_gbs", FALLBACK["hbm_gbs"])))
                            for k, v in aux.items()},
            "fwd_frac_of_burst": round(fwd_tf / peak_burst, 4),
            "bwd_frac_of_burst": round(bwd_tf / peak_burst, 4),
            "e2e": {"value": round((f_fwd + f_bwd) * world / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 3),
                    "copies": "pinned host buffers; step i+1's H2D and step i's D2H on two copy streams, "
                              "overlapping the kernels; median of 3 timed runs (the host link is shared)",
                    "serialised": {"value": round((f_fwd + f_bwd) * world / (e2e_serial_ms * 1e-3) / 1e12, 2),
                                   "ms_per_step": round(e2e_serial_ms, 3),
                                   "copies": "the same copies in order on the compute stream, nothing overlapped"}},
            "clocks": clk,
            "gpu_launches": r.launches_per_step * args.steps,
            "rank_block_counts": cpa.cp_rank_block_counts(r.prob),
            "rank_balance": balance_report(cpa, w),
            "ulysses": uly,
            "ring_transport": ring,
            "other_configs": others,
            "linear_attention_cp": lin,
        }
        if "ms_per_step" in uly:
            hbm = float(peaks.get("hbm_gbs", FALLBACK["hbm_gbs"]))
            uly["tflops"] = round((f_fwd + f_bwd) / (uly["ms_per_step"] * 1e-3) / 1e12, 2)
            uly["ring_attention_ms_per_step"] = round(fwd_ms + bwd_ms, 3)
            uly["a2a_q"]["frac"] = round(uly["a2a_q"]["gbs"] / hbm, 4)
        if not args.no_cpu_baseline:
            tf, secs, desc = oracle_sample(w, args.cpu_tokens)
            result["cpu_baseline"] = cpu_baseline_entry(w, tf, secs, desc)
    if world > 1:
        torch.distributed.destroy_process_group()
    return result


def balance_report(cpa, w) -> dict:
    """Per-rank effective attention work of the workload under each shard
    layout: visible 128x128 tiles per rank (cp_rank_block_counts) and the
    slowest rank's share over the mean.  With one GPU per rank, the slowest
    rank would set the step time."""
    out = {}
    cu = workloads.make_cu_seqlens(w.lengths()).tolist()
    for layout in ("contiguous", "zigzag", "striped"):
        p = cpa.Problem(w.total_tokens, w.hq, w.hkv, w.d_qk, w.d_v, w.cp_size, layout, cu, w.causal, w.scale)
        c = cpa.cp_rank_block_counts(p)
        out[layout] = {"max_over_mean": round(max(c) / (sum(c) / len(c)), 4), "min": min(c), "max": max(c)}
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    w = chosen_workload(args)
    vals = []
    for _ in range(args.warmup):
        oracle_sample(w, args.cpu_tokens // 2)
    secs = []
    desc = ""
    for _ in range(args.steps):
        tf, s, desc = oracle_sample(w, args.cpu_tokens // 2)
        vals.append(tf)
        secs.append(s)
    v = statistics.mean(vals)
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "TFLOP/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1000 * statistics.mean(secs), 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded iid N(0,1) q, k, v, dout)",
        "config": {"workload": w.name, "total_tokens": w.total_tokens, "hq": w.hq, "hkv": w.hkv, "d_qk": w.d_qk,
                   "d_v": w.d_v, "cp_size": w.cp_size, "layout": w.layout},
        "cpu_baseline": cpu_baseline_entry(w, v, statistics.mean(secs), desc),
        "e2e": {"value": round(v, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(workloads.WORKLOADS))
    ap.add_argument("--cpu-tokens", type=int, default=8192)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-ulysses", action="store_true", help="skip the Ulysses comparison")
    ap.add_argument("--no-linear", action="store_true", help="skip the linear-attention CP measurement")
    ap.add_argument("--no-ring", action="store_true", help="skip the ring-with-transport measurement")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the throughput lines of the other standard problems")
    ap.add_argument("--layout", default=None, choices=["contiguous", "zigzag", "striped"],
                    help="shard layout instead of the workload's own (zigzag for the standard ones)")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="sequence length (single-sequence workloads) or total tokens of a varlen pack")
    ap.add_argument("--heads", default=None, help="query:key-value head counts, e.g. 32:8")
    ap.add_argument("--cp-size", type=int, default=None, help="number of context-parallel shards C")
    ap.add_argument("--seed", type=int, default=None, help="input generator seed")
    args = ap.parse_args()
    if args.impl == "reference":
        res = run_reference(args)
    else:
        res = run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
