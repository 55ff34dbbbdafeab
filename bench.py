"""Benchmark: fused Q+K RoPE forward/backward, achieved HBM GB/s and us/call.

One step = the forward rotation of (Q, K) followed by the backward rotation
of the incoming gradients (dQ, dK) of the same shapes -- one training step of
RoPE in one attention layer.  Default workload: the Llama-3-8B-shaped GQA
layer (bf16, split-half, Q [4,32,4096,128], K [4,8,4096,128], theta 5e5).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Throughput counts algorithmic bytes: the rotary span of every rotated Q/K
row read and written once, plus each distinct cos/sin row and the position
vector read once, per call.  The cos/sin table is built once before the timed
region (it depends only on theta, rotary_dim, the number of positions and the
interpolation factor) and its build time is reported separately.

With N > 1 (torchrun) every rank runs the same workload on its own GPU: the
method has no exchange step, so ranks are independent replicas.  ``value``
is the bytes all ranks moved divided by the slowest rank's time.

``--impl reference`` times the plain CPU oracle on this host's cores (the
pages publish no runnable implementation), on a bounded sample of the same
workload per step.

Two more operations have their own lines (not the contract line):
``--op attention`` times the attention with fused rotation (TFLOP/s on the
visible causal pairs of a Llama-3-8B-shaped prefill), ``--op xpos`` the
rotation with XPOS tables (one launch per tensor).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "fused Q+K RoPE fwd/bwd achieved HBM GB/s (% of GB300 peak) and µs/call"
DEFAULT_WORKLOAD = "llama3_8b_gqa_bf16"
PRE_ROLL_CYCLES = 1_000_000          # GPU clock cycles slept before a timed region (~0.5 ms)
FALLBACK_HBM_GBS = 6800.0
PROFILE_DIR = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = [os.path.join(ROOT, "rotary_position_embedding_rope_gb300", "csrc", f)
                  for f in ("rope_kernels.cuh", "rope_internal.cuh", "rope_api.cu")]
ATTN_SOURCES = [os.path.join(ROOT, "rotary_position_embedding_rope_gb300", "csrc", f)
                for f in ("rope_attention.cuh", "rope_attention.cu", "rope_kernels.cuh", "rope_internal.cuh",
                          "rope_api.cu")]


def kernel_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES if sources is None else sources:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# --------------------------------------------------------------------------
# distributed plumbing
# --------------------------------------------------------------------------
def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def aggregate(dist, device, local_ms: float, local_bytes: float):
    """Max time over ranks, total bytes over ranks (replicas: no data exchange)."""
    if dist is None:
        return local_ms, local_bytes
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    b = torch.tensor([local_bytes], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), float(b.item())


# --------------------------------------------------------------------------
# clocks during the timed region (NVML through ctypes; nvidia-smi fallback)
# --------------------------------------------------------------------------
REASON_BITS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}


class ClockSampler:
    def __init__(self, device_index: int):
        self.samples = []          # (sm_mhz, reasons_mask)
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._handle = None
        self._smi = None
        self.source = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            handle = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(device_index)
            uuid = str(getattr(props, "uuid", ""))
            ok = False
            for cand in (uuid, "GPU-" + uuid):
                if cand and nv.nvmlDeviceGetHandleByUUID(cand.encode(), ctypes.byref(handle)) == 0:
                    ok = True
                    break
            if not ok:
                vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
                idx = int(vis.split(",")[device_index]) if vis and vis.split(",")[0].isdigit() \
                    else device_index
                ok = nv.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(handle)) == 0
            if not ok:
                raise OSError("no NVML handle")
            self._nvml, self._handle = nv, handle
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self._reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.source = "nvml"
        except (OSError, AttributeError, ValueError, IndexError):
            self.source = "nvidia-smi"

    def _sample_nvml(self):
        mhz = ctypes.c_uint()
        mask = ctypes.c_ulonglong()
        if self._nvml.nvmlDeviceGetClockInfo(self._handle, 1, ctypes.byref(mhz)) == 0:
            self._reasons_fn(self._handle, ctypes.byref(mask))
            self.samples.append((float(mhz.value), int(mask.value)))

    def _run(self):
        while not self._stop.is_set():
            self._sample_nvml()
            time.sleep(0.002)

    def start(self):
        if self.source == "nvml":
            self._sample_nvml()
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        else:
            try:
                self._smi = subprocess.Popen(
                    ["nvidia-smi", "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-i", str(torch.cuda.current_device()),
                     "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self._smi = None

    def stop(self):
        if self.source == "nvml":
            self._sample_nvml()
            self._stop.set()
            if self._thread:
                self._thread.join()
        elif self._smi is not None:
            self._smi.terminate()
            out, _ = self._smi.communicate(timeout=10)
            for line in out.splitlines():
                parts = [p.strip() for p in line.split(",")]
                try:
                    self.samples.append((float(parts[0]), int(parts[2], 16)))
                    self.max_mhz = float(parts[1])
                except (ValueError, IndexError):
                    pass

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": self.source}
        mhz = [s[0] for s in self.samples]
        mask = 0
        for _, m in self.samples:
            mask |= m
        reasons = [name for bit, name in REASON_BITS.items() if mask & bit and bit != 0x1]
        return {"sm_mhz": float(np.median(mhz)), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(self.samples), "source": self.source}


# --------------------------------------------------------------------------
# roofline inputs
# --------------------------------------------------------------------------
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_NAMES = {2: "rope_scalar_kernel", 3: "rope_vec_kernel"}


def profiled_traffic(kernel: str, workload: str, sources=None):
    """DRAM bytes per launch of a kernel from a committed ncu summary, or None
    when there is none, the kernel sources changed since, or the library
    loaded is another build (ROPE_LIBRARY: a compile-time variant)."""
    if os.environ.get("ROPE_LIBRARY"):
        return None
    path = os.path.join(PROFILE_DIR, "%s_%s.md" % (kernel, workload))
    try:
        text = open(path).read()
    except OSError:
        return None
    src = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    val = re.search(r"dram_bytes_per_launch:\s*([0-9,]+)", text)
    if not src or not val or src.group(1) != kernel_source_hash(sources):
        return None
    return int(val.group(1).replace(",", ""))


# --------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and --impl reference)
# --------------------------------------------------------------------------
def oracle_sample_step(o, w, xs, pos, cos32, sin32, n_tok: int):
    """Oracle forward on Q, K and backward on dQ, dK restricted to batch 0 and
    the first n_tok tokens (all heads).  Returns the algorithmic bytes of that
    sample."""
    import oracle as O

    code = {"f32": O.F32, "bf16": O.BF16, "f16": O.F16}[w.dtype]
    sub = w.with_sizes(B=1, S=n_tok)
    p = None if pos is None else pos[:n_tok]
    for (x, H), backward in zip(xs, (False, False, True, True)):
        xb = W.bits(x[:1, :, :n_tok] if not w.seq_before_head else x[:1, :n_tok])
        rc, _, _ = o.apply(xb, code, 1, H, n_tok, w.D, w.rotary_dim, W.LAYOUTS[w.layout],
                           w.seq_before_head, backward, p, cos32, sin32, want_f64=False)
        assert rc == 0
    return 2 * W.algorithmic_bytes(sub)


def time_oracle(w, budget_s: float, xs, pos, cos32, sin32):
    """Run oracle steps on growing token samples until budget_s is spent."""
    import oracle as O

    o = O.load()
    n_tok = 16
    done_bytes = 0
    t0 = time.perf_counter()
    tokens = 0
    while True:
        n = min(n_tok, w.S)
        done_bytes += oracle_sample_step(o, w, xs, pos, cos32, sin32, n)
        tokens += n
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
        n_tok = min(n_tok * 2, w.S)
    return done_bytes, el, tokens


def reference_arm(args, w):
    world, rank, _ = dist_info()
    if rank != 0:
        return 0                               # rank 0 alone times the CPU oracle
    import oracle as O

    o = O.load()
    q, k, pos = W.make_inputs(w)
    dq, dk, _ = W.make_inputs(w, seed_offset=100)
    xs = [(q, w.Hq), (k, w.Hk), (dq, w.Hq), (dk, w.Hk)]
    cos32, sin32 = o.tables(w.theta, w.rotary_dim, w.table_rows, w.interpolate_factor, "f32")
    # the oracle is single-threaded; so is the slicing around it from here on
    torch.set_num_threads(1)
    # size one step so the whole run stays near two minutes of CPU work
    budget = reference_step_seconds(args)
    # a step costs about c0 + c1 * tokens: fit both from two sizes
    times = []
    for n in (8, 64):
        t0 = time.perf_counter()
        oracle_sample_step(o, w, xs, pos, cos32, sin32, min(n, w.S))
        times.append(time.perf_counter() - t0)
    c1 = max((times[1] - times[0]) / 56, 1e-9)
    c0 = max(times[0] - 8 * c1, 0.0)
    n_tok = int(max(1, min(w.S, (budget - c0) / c1)))
    for _ in range(args.warmup):
        oracle_sample_step(o, w, xs, pos, cos32, sin32, n_tok)
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        nbytes += oracle_sample_step(o, w, xs, pos, cos32, sin32, n_tok)
    el = time.perf_counter() - t0
    gbs = nbytes / el / 1e9
    sample = ("batch 0, first %d of %d tokens, all %d Q + %d K heads, forward on Q,K and "
              "backward on dQ,dK per step" % (n_tok, w.S, w.Hq, w.Hk))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "note": "the pages publish no runnable implementation; the reference arm is the "
                "single-threaded fp64 CPU oracle on this host",
    }
    print(json.dumps(line), flush=True)
    return 0


def reference_step_seconds(args) -> float:
    """CPU seconds of one reference-arm step: at most 0.25 s, and about two
    minutes for all warm-up and timed steps together."""
    return min(0.25, 120.0 / max(1, args.steps + args.warmup))


# --------------------------------------------------------------------------
# every workload, forward and backward timed apart (the per_workload block)
# --------------------------------------------------------------------------
def rotating_sets(w, device, min_bytes: float, max_sets: int = 256):
    """Device copies of the workload's Q, K: enough sets that one pass over
    them moves at least min_bytes (so each call reads memory the previous
    ones evicted from L2), two at least."""
    q, k, pos = W.make_inputs(w)
    per = sum(t.numel() * t.element_size() for t in (q, k) if t is not None)
    n = int(min(max_sets, max(2, -(-min_bytes // per))))
    sets = [(q.to(device), None if k is None else k.to(device)) for _ in range(n)]
    return sets, (None if pos is None else torch.from_numpy(pos).to(device)), per, (q, k, pos)


def time_direction(R, w, sets, cos, sin, pos_g, stream, backward: int, device, min_ms: float,
                   min_calls: int, graph_calls: int):
    """Back-to-back calls of one direction over the rotating sets, events at
    the two ends only (programmatic dependent launch stays on): eager through
    the binding, eager through a prepared call, and the replay of a CUDA
    graph of the same calls.  Returns a dict of µs per call, GB/s, fractions
    and the clock record of the eager region."""
    layout, sbh, dt = W.LAYOUTS[w.layout], int(w.seq_before_head), W.DTYPES[w.dtype]
    nsets = len(sets)

    def call(i):
        qx, kx = sets[i % nsets]
        R.rope_apply_qk(qx, kx, cos, sin, pos_g, w.B, w.Hq, w.Hk, w.S, w.D, w.rotary_dim, layout,
                        sbh, backward, dt, w.table_rows, stream)

    sampler = ClockSampler(device.index or 0)
    sampler.start()
    for i in range(10):
        call(i)
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for i in range(10):
        call(i)
    torch.cuda.synchronize(device)
    est = max((time.perf_counter() - t0) / 10, 1e-7)
    n = int(max(min_calls, min_ms * 1e-3 / est))

    def region(fn, count):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(count):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize(device)
        return e0.elapsed_time(e1) * 1e3 / count

    us = region(call, n)
    sampler.stop()
    prep = R.PreparedApply(sets[0][0], sets[0][1], cos, sin, pos_g, w.rotary_dim, w.layout,
                           w.seq_before_head, stream)
    pcall = (lambda i: prep(sets[i % nsets][0], sets[i % nsets][1], backward=bool(backward)))
    for i in range(10):
        pcall(i)
    us_prep = region(pcall, n)
    # the same calls captured once in a graph and replayed: device time
    # without the host's launch cost
    gcount = min(n, graph_calls)
    gs = torch.cuda.Stream(device)
    gs.wait_stream(torch.cuda.current_stream(device))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(gs):
        with torch.cuda.graph(g, stream=gs):
            for i in range(gcount):
                qx, kx = sets[i % nsets]
                R.rope_apply_qk(qx, kx, cos, sin, pos_g, w.B, w.Hq, w.Hk, w.S, w.D, w.rotary_dim,
                                layout, sbh, backward, dt, w.table_rows, gs)
    torch.cuda.synchronize(device)
    g.replay()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize(device)
    us_graph = e0.elapsed_time(e1) * 1e3 / gcount
    del g
    peak, _ = hbm_peak()
    nbytes = W.algorithmic_bytes(w)
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"us_per_call": round(us, 3), "gbs": round(gbs, 1),
            "frac_of_hbm_measured": round(gbs / peak, 4), "frac_of_nominal_8tbs": round(gbs / 8000.0, 4),
            "calls": n, "us_per_call_prepared": round(us_prep, 3),
            "us_per_call_graph_replay": round(us_graph, 3), "graph_calls": gcount,
            "gbs_graph_replay": round(nbytes / (us_graph * 1e-6) / 1e9, 1),
            "clocks": sampler.summary()}


def per_workload_block(R, device, stream, min_ms: float, min_calls: int, l2_bytes: int,
                       names=None, cpu_seconds: float = 0.0):
    """Every workload (the five and two launch-bound single calls), forward
    and backward apart; with cpu_seconds > 0 also the single-threaded oracle
    on growing prefixes of batch 0 for about that long per workload."""
    out = {}
    for name in names or list(W.ALL_BY_NAME):
        w = W.ALL_BY_NAME[name]
        sets, pos_g, per, host = rotating_sets(w, device, 2.2 * l2_bytes)
        cos = torch.empty((w.table_rows, w.rotary_dim // 2), dtype=torch.float32, device=device)
        sin = torch.empty_like(cos)
        R.rope_tables_build(w.theta, w.rotary_dim, w.table_rows, w.interpolate_factor, cos, sin,
                            stream)
        entry = {"bytes_per_call": W.algorithmic_bytes(w),
                 "config": {k: v for k, v in config_of(w).items() if k != "step"},
                 "rotating_sets": len(sets),
                 "l2": "%d sets of %.1f MB = %.0f MB per pass vs %.0f MB L2" % (
                     len(sets), per / 1e6, len(sets) * per / 1e6, l2_bytes / 1e6)}
        for backward, key in ((0, "forward"), (1, "backward")):
            entry[key] = time_direction(R, w, sets, cos, sin, pos_g, stream, backward, device,
                                        min_ms, min_calls, 400)
        assert R.rope_check_errors(stream) == R.ROPE_OK
        if cpu_seconds > 0:
            import oracle as O

            q, k, pos = host
            cos32, sin32 = O.load().tables(w.theta, w.rotary_dim, w.table_rows,
                                           w.interpolate_factor, "f32")
            threads = torch.get_num_threads()
            torch.set_num_threads(1)
            nb, el, toks = time_oracle(w, cpu_seconds, [(q, w.Hq), (k, w.Hk), (q, w.Hq),
                                                        (k, w.Hk)], pos, cos32, sin32)
            torch.set_num_threads(threads)
            entry["cpu_oracle"] = {"gbs": round(nb / el / 1e9, 4), "cores": 1,
                                   "sample": "batch 0, growing token prefixes (%d token-steps in "
                                             "%.1f s), forward and backward" % (toks, el)}
        out[name] = entry
        del sets
        torch.cuda.empty_cache()
    return out


def link_context(device, stream, nbytes: int = 256 << 20, reps: int = 3):
    """GB/s of pinned-host <-> device copies: host to device, device to host,
    and both at once on two streams (best of reps)."""
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_a = torch.empty(nbytes, dtype=torch.uint8, device=device)
    d_b = torch.empty(nbytes, dtype=torch.uint8, device=device)
    s2 = torch.cuda.Stream(device)

    def timed(fn):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize(device)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(device)
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        return best

    def both():
        s2.wait_stream(stream)
        d_a.copy_(h_in, non_blocking=True)
        with torch.cuda.stream(s2):
            h_out.copy_(d_b, non_blocking=True)
        stream.wait_stream(s2)

    h2d = timed(lambda: d_a.copy_(h_in, non_blocking=True))
    d2h = timed(lambda: h_out.copy_(d_b, non_blocking=True))
    bi = timed(both)
    gbs = lambda n, ms: round(n / (ms * 1e-3) / 1e9, 1)
    return {"h2d_gbs": gbs(nbytes, h2d), "d2h_gbs": gbs(nbytes, d2h),
            "both_directions_gbs": gbs(2 * nbytes, bi),
            "what": "256 MiB pinned-host copies, best of %d" % reps}


def config_of(w):
    return {"workload": w.name, "q_shape": list(w.q_shape), "k_shape": list(w.k_shape),
            "dtype": w.dtype, "layout": w.layout,
            "tensor_layout": "BSHD" if w.seq_before_head else "BHSD",
            "rotary_dim": w.rotary_dim, "theta": w.theta, "table_rows": w.table_rows,
            "positions": w.positions, "step": "forward(Q,K) + backward(dQ,dK), in place",
            "bytes_per_call": W.algorithmic_bytes(w)}


# --------------------------------------------------------------------------
# attention with fused rotation (--op attention)
# --------------------------------------------------------------------------
ATTN_WORKLOAD = dict(name="llama3_8b_prefill_attention_bf16", B=4, Hq=32, Hk=8, S=4096, D=128,
                     rotary_dim=128, theta=5e5, causal=True, dtype="bf16")


def attention_flops(B, Hq, Sq, Sk, D, causal):
    """Multiply-adds of S = Q K^T and O = P V over the visible (query, key)
    pairs, times 2: the work a causal kernel must do."""
    if causal:
        shift = Sk - Sq
        pairs = sum(max(0, min(Sk, i + shift + 1)) for i in range(Sq))
    else:
        pairs = Sq * Sk
    return 4.0 * B * Hq * D * pairs


def attention_inputs(a):
    """Seeded Q, K, V of the attention workload, on the CPU."""
    g = torch.Generator().manual_seed(6)
    q = W.draw((a["B"], a["Hq"], a["S"], a["D"]), a["dtype"], g)
    k = W.draw((a["B"], a["Hk"], a["S"], a["D"]), a["dtype"], g)
    v = W.draw((a["B"], a["Hk"], a["S"], a["D"]), a["dtype"], g)
    return q, k, v


def oracle_attention_rows(a, q, k, v, head, nq, c32, s32):
    """The oracle on the last nq query rows of (batch 0, head), at their own
    positions, against every key of its key/value head.  q, k, v may live on
    any device; only those rows and heads are copied.  Returns the flops of
    the visible pairs."""
    import oracle as O
    from oracle import attention as OA

    S = a["S"]
    hk = head // (a["Hq"] // a["Hk"])
    pos_q = np.arange(S - nq, S, dtype=np.int32)
    OA.attention(W.bits(q[:1, head:head + 1, S - nq:].cpu()), W.bits(k[:1, hk:hk + 1].cpu()),
                 W.bits(v[:1, hk:hk + 1].cpu()), O.BF16, a["rotary_dim"], O.SPLIT_HALF, c32, s32,
                 pos_q=pos_q, causal=True)
    return attention_flops(1, 1, nq, S, a["D"], True)


def attention_config(a, flops):
    return {"workload": a["name"], "q_shape": [a["B"], a["Hq"], a["S"], a["D"]],
            "kv_shape": [a["B"], a["Hk"], a["S"], a["D"]], "causal": a["causal"],
            "rotary_dim": a["rotary_dim"], "flops_per_call": flops}


def attention_reference_arm(args):
    """The oracle on a bounded sample of the attention workload: per step the
    last rows of one query head (heads taken in turn) against all keys."""
    world, rank, _ = dist_info()
    if rank != 0:
        return 0                               # rank 0 alone times the CPU oracle
    import oracle as O

    a = ATTN_WORKLOAD
    q, k, v = attention_inputs(a)
    c32, s32 = O.load().tables(a["theta"], a["rotary_dim"], a["S"], 1.0, "f32")
    budget = reference_step_seconds(args)
    # a step costs about c0 + c1 * rows: fit both from two sizes
    times = []
    for n in (16, 128):
        t0 = time.perf_counter()
        oracle_attention_rows(a, q, k, v, 0, n, c32, s32)
        times.append(time.perf_counter() - t0)
    c1 = max((times[1] - times[0]) / 112, 1e-9)
    c0 = max(times[0] - 16 * c1, 0.0)
    nq = int(max(1, min(a["S"], (budget - c0) / c1)))
    for i in range(args.warmup):
        oracle_attention_rows(a, q, k, v, i % a["Hq"], nq, c32, s32)
    flops = 0.0
    t0 = time.perf_counter()
    for i in range(args.steps):
        flops += oracle_attention_rows(a, q, k, v, i % a["Hq"], nq, c32, s32)
    el = time.perf_counter() - t0
    tflops = flops / el / 1e12
    sample = ("batch 0, one query head per step (heads in turn), its last %d of %d query rows "
              "against all keys (numpy fp64; threads as numpy uses them)" % (nq, a["S"]))
    line = {
        "impl": "reference", "metric": "fused rotary attention forward TFLOP/s", "op": "attention",
        "value": round(tflops, 6), "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(el / max(1, args.steps) * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": a["dtype"],
        "data": "synthetic", "config": attention_config(a, flops_of(a)),
        "cpu_baseline": {"value": round(tflops, 6), "unit": "TFLOP/s", "cores": os.cpu_count() or 0,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(tflops, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "note": "the pages publish no runnable implementation; the reference arm is the fp64 "
                "CPU oracle on this host",
    }
    print(json.dumps(line), flush=True)
    return 0


def tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def flops_of(a):
    return attention_flops(a["B"], a["Hq"], a["S"], a["S"], a["D"], a["causal"])


def attention_arm(args):
    world, rank, local = dist_info()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    from rotary_position_embedding_rope_gb300 import _build
    if local == 0:
        _build.build()
    if dist is not None:
        dist.barrier()
    import rotary_position_embedding_rope_gb300 as R

    a = ATTN_WORKLOAD
    q, k, v = (t.to(device) for t in attention_inputs(a))
    cos, sin = R.build_tables(a["theta"], a["rotary_dim"], a["S"], device=device)
    stream = torch.cuda.current_stream(device)
    o = torch.empty_like(q)
    kws = torch.empty_like(k)          # receives rot(K) once per call
    warmup = max(3, args.warmup)
    steps = max(1, min(args.steps, 200))

    def step(ws=kws):
        R.attention(q, k, v, cos, sin, rotary_dim=a["rotary_dim"], causal=a["causal"], out=o,
                    k_workspace=ws, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(device)
    assert R.rope_check_errors(stream) == R.ROPE_OK
    sampler = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(device)
    sampler.stop()
    ms = e0.elapsed_time(e1) / steps
    flops = flops_of(a)
    max_ms, all_flops = aggregate(dist, device, ms * steps, flops * steps)
    tflops = all_flops / (max_ms * 1e-3) / 1e12

    # context: the same call with the key tiles rotated inside the attention
    # kernel (no workspace: one launch per call)
    for _ in range(warmup):
        step(None)
    torch.cuda.synchronize(device)
    i0, i1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    i0.record(stream)
    for _ in range(steps):
        step(None)
    i1.record(stream)
    torch.cuda.synchronize(device)
    ims = i0.elapsed_time(i1) / steps
    inkernel = {"ms": round(ims, 4), "tflops": round(flops_of(a) / (ims * 1e-3) / 1e12, 1),
                "what": "k_workspace=None: each CTA rotates its key tiles (rope_attn_kernel)"}

    # context: the same call with an attn_mask -- all keys visible and key
    # padding (batch entry b keeps its first S - 512 b keys), both prefixes of
    # the keys, and a mask that hides a seeded ~10 % of the keys everywhere
    # (not a prefix: the kernel reads its bytes)
    masked = {}
    gm = torch.Generator(device=device).manual_seed(12)
    for label, m in (("all_visible", torch.ones((a["B"], a["S"]), dtype=torch.bool,
                                                device=device)),
                     ("key_padding", torch.arange(a["S"], device=device)[None, :] <
                      (a["S"] - 512 * torch.arange(a["B"], device=device))[:, None]),
                     ("scattered", torch.rand((a["B"], a["S"]), generator=gm, device=device) > 0.1)):
        mws = R.attention_workspace(k, m)   # rot(K), the key-tile counts, the prefix lengths

        def mstep(m=m, mws=mws):
            R.attention(q, k, v, cos, sin, rotary_dim=a["rotary_dim"], causal=a["causal"], out=o,
                        k_workspace=mws, attn_mask=m, stream=stream)
        for _ in range(warmup):
            mstep()
        torch.cuda.synchronize(device)
        m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        m0.record(stream)
        for _ in range(steps):
            mstep()
        m1.record(stream)
        torch.cuda.synchronize(device)
        mms = m0.elapsed_time(m1) / steps
        masked[label] = {"ms": round(mms, 4), "tflops_of_unmasked_flops":
                         round(flops_of(a) / (mms * 1e-3) / 1e12, 1)}
    masked["what"] = ("rope_attention_fwd_masked, workspace path with the mask's key-tile "
                      "counts and prefix lengths, [B, Sk] mask: all keys visible, or batch entry b "
                      "keeping its first S - 512 b keys (the key tiles past them skipped; both "
                      "prefixes, computed without reading the mask), or ~10 % of the keys hidden "
                      "at random (mask bytes read per key tile)")

    # context: the same result from the unfused path (rotation kernel, then
    # torch's scaled_dot_product_attention on the rotated tensors)
    unfused = None
    try:
        import torch.nn.functional as F

        qr, kr = q.clone(), k.clone()

        def unfused_step():
            qr.copy_(q)
            kr.copy_(k)
            R.apply_qk(qr, kr, cos, sin, stream=stream)
            return F.scaled_dot_product_attention(qr, kr, v, is_causal=True, enable_gqa=True)

        for _ in range(warmup):
            unfused_step()
        torch.cuda.synchronize(device)
        u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        u0.record(stream)
        for _ in range(steps):
            unfused_step()
        u1.record(stream)
        torch.cuda.synchronize(device)
        ums = u0.elapsed_time(u1) / steps
        unfused = {"ms": round(ums, 4), "tflops": round(flops / (ums * 1e-3) / 1e12, 1),
                   "what": "copy Q,K; rope_apply_qk; torch scaled_dot_product_attention"}
    except Exception as exc:  # noqa: BLE001 - context only
        unfused = {"unavailable": str(exc)[:200]}

    # end to end through the public API with host buffers: every step copies
    # Q, K, V from pinned host memory and O back to pinned host memory, one
    # batch chunk at a time, with the copies overlapping the calls
    from rotary_position_embedding_rope_gb300.host import HostAttention

    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    ho = torch.empty_like(hq).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size()
    pieces = a["B"]                    # one batch entry per call (more pieces measured slower)
    hat = HostAttention(device, chunks=pieces)

    def e2e_step(after):
        return hat.forward(hq, hk, hv, ho, cos, sin, rotary_dim=a["rotary_dim"],
                           causal=a["causal"], after=after)

    for _ in range(2):
        stream.wait_event(e2e_step(None))
    torch.cuda.synchronize(device)
    if dist is not None:
        dist.barrier()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    last = x0
    for i in range(args.e2e_steps):
        last = e2e_step(x0 if i == 0 else None)
    stream.wait_event(last)
    x1.record(stream)
    torch.cuda.synchronize(device)
    assert R.rope_check_errors(stream) == R.ROPE_OK
    e2e_ms, e2e_flops = aggregate(dist, device, x0.elapsed_time(x1), flops * args.e2e_steps)
    e2e = {"value": round(e2e_flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
           "ms_per_step": round(e2e_ms / args.e2e_steps, 4),
           "what": "pinned host Q, K, V in and O out; %d pieces (batch entry x group of "
                   "key/value heads), copies overlapping the calls" % pieces}

    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        import oracle as O

        c32, s32 = O.load().tables(a["theta"], a["rotary_dim"], a["S"], 1.0, "f32")
        # the last nq query rows of heads 0, 1, ... of batch 0 until cpu_seconds are spent
        nq, heads, sf = 64, 0, 0.0
        t0 = time.perf_counter()
        while heads < a["Hq"] and (heads == 0 or time.perf_counter() - t0 < args.cpu_seconds):
            sf += oracle_attention_rows(a, q, k, v, heads, nq, c32, s32)
            heads += 1
        el = time.perf_counter() - t0
        cpu = {"value": round(sf / el / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count() or 0,
               "kind": "oracle", "sample": "batch 0, query heads 0-%d, the last %d of %d query rows "
               "of each against all keys (numpy fp64; threads as numpy uses them)"
               % (heads - 1, nq, a["S"])}

    peak, peak_kind = tensor_peak()
    if rank == 0:
        line = {
            "metric": "fused rotary attention forward TFLOP/s", "op": "attention",
            "value": round(tflops, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": steps,
            "warmup": warmup, "ms_per_step": round(max_ms / steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": a["dtype"], "data": "synthetic",
            "config": attention_config(a, flops),
            "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(tflops / peak, 4),
                         "peak_source": "%s bf16 (MEASURED_PEAKS.json bf16_tflops)" % peak_kind,
                         "traffic": profiled_traffic("rope_attn_2sm_kernel", a["name"],
                                                     ATTN_SOURCES),
                         "kernel": "rope_attn_2sm_kernel",
                         "note": "achieved = flops per call / the call's time, which also holds "
                                 "the launch that rotates K into the workspace"},
            "e2e": e2e,
            "inkernel_keys_context": inkernel,
            "masked_context": masked,
            "unfused_context": unfused,
            "gpu_launches": 2 * steps,
            "clocks": sampler.summary(),
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


# --------------------------------------------------------------------------
# grid sizings of the rotation kernel side by side (--op sweep)
# --------------------------------------------------------------------------
def sweep_tunings(P: int, per_sm: int):
    """(label, ctas_per_sm, min_units, prefetch_next) of rope_tune_rotation_launch."""
    return [("rule", 0, 0, 0),
            ("persistent_balanced", per_sm, 1, 0),
            ("one_tile_per_lane_group", 64, P, 0),
            ("half_tile_per_lane_group", 64, max(1, P // 2), 0),
            ("quarter_tile_per_lane_group", 64, max(1, P // 4), 0),
            ("rule_no_next_tile_prefetch", 0, 0, -1)]


def sweep_arm(args):
    """Every workload under each grid sizing of sweep_tunings: forward calls
    back to back (as in per_workload), one JSON line per (workload, sizing).
    The results do not depend on the sizing; only the time does."""
    world, rank, local = dist_info()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from rotary_position_embedding_rope_gb300 import _build
    if local == 0:
        _build.build()
    import rotary_position_embedding_rope_gb300 as R

    R.load_library()
    stream = torch.cuda.current_stream(device)
    l2_bytes = torch.cuda.get_device_properties(device).L2_cache_size
    per_sm = 4                                # resident CTAs of 128 threads (its launch bounds)
    try:
        for name in W.ALL_BY_NAME:
            w = W.ALL_BY_NAME[name]
            sets, pos_g, _, _ = rotating_sets(w, device, 2.2 * l2_bytes)
            cos = torch.empty((w.table_rows, w.rotary_dim // 2), dtype=torch.float32,
                              device=device)
            sin = torch.empty_like(cos)
            R.rope_tables_build(w.theta, w.rotary_dim, w.table_rows, w.interpolate_factor, cos,
                                sin, stream)
            for label, cps, mu, pf in sweep_tunings(w.Hq + w.Hk, per_sm):
                R.rope_tune_rotation_launch(cps, mu, pf)
                r = time_direction(R, w, sets, cos, sin, pos_g, stream, 0, device,
                                   args.per_workload_ms or 20.0, 200, 400)
                if rank == 0:
                    print(json.dumps({"op": "sweep", "workload": name, "grid": label,
                                      "tuning": [cps, mu, pf], "us_per_call": r["us_per_call"],
                                      "gbs": r["gbs"], "us_per_call_graph_replay":
                                      r["us_per_call_graph_replay"],
                                      "clocks": r["clocks"]}), flush=True)
            assert R.rope_check_errors(stream) == R.ROPE_OK
            del sets
            torch.cuda.empty_cache()
    finally:
        R.rope_tune_rotation_launch(0, 0, 0)
    return 0


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------
# --------------------------------------------------------------------------
# XPOS rotation (--op xpos): frequency tables with the query/key scale folded in
# --------------------------------------------------------------------------
XPOS_SCALE_BASE = 512.0


def xpos_arm(args):
    """Llama-shaped layer with XPOS: Q rotated with the +1 table and K with the
    -1 table (one launch each), forward and backward, in place."""
    world, rank, local = dist_info()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    from rotary_position_embedding_rope_gb300 import _build
    if local == 0:
        _build.build()
    if dist is not None:
        dist.barrier()
    import rotary_position_embedding_rope_gb300 as R

    w = W.BY_NAME[DEFAULT_WORKLOAD]
    stream = torch.cuda.current_stream(device)
    kw = dict(theta=w.theta, xpos_scale_base=XPOS_SCALE_BASE, xpos_center=w.table_rows / 2,
              device=device, stream=stream)
    tq = R.build_tables_ex("lang", w.rotary_dim, w.table_rows, xpos_sign=1, **kw)
    tk = R.build_tables_ex("lang", w.rotary_dim, w.table_rows, xpos_sign=-1, **kw)
    g = torch.Generator().manual_seed(w.seed)
    nsets = 2
    sets = []
    for _ in range(nsets):
        q = W.draw((w.B, w.Hq, w.S, w.D), w.dtype, g).to(device)
        k = W.draw((w.B, w.Hk, w.S, w.D), w.dtype, g).to(device)
        sets.append((q, k, q.clone(), k.clone()))

    def step(i):
        q, k, dq, dk = sets[i % nsets]
        R.apply_qk_xpos(q, k, tq, tk, stream=stream)
        R.apply_qk_xpos(dq, dk, tq, tk, backward=True, stream=stream)

    warmup = max(3, args.warmup)
    steps = max(1, min(args.steps, 1000))
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(device)
    assert R.rope_check_errors(stream) == R.ROPE_OK
    sampler = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(device)
    sampler.stop()
    assert R.rope_check_errors(stream) == R.ROPE_OK
    ms = e0.elapsed_time(e1)
    # per direction: the fused call's bytes plus one more table (Q and K each
    # read their own)
    table = w.S * (w.rotary_dim // 2) * 4 * 2
    bytes_step = 2 * (W.algorithmic_bytes(w) + table)
    max_ms, all_bytes = aggregate(dist, device, ms, bytes_step * steps)
    value = all_bytes / (max_ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    if rank == 0:
        line = {
            "metric": "XPOS rotation of Q and K, fwd/bwd achieved HBM GB/s", "op": "xpos",
            "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": steps,
            "warmup": warmup, "ms_per_step": round(max_ms / steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "q_shape": [w.B, w.Hq, w.S, w.D],
                       "k_shape": [w.B, w.Hk, w.S, w.D], "tables": "lang theta=%g, XPOS base %g "
                       "centre %g, +1 for Q, -1 for K" % (w.theta, XPOS_SCALE_BASE, w.table_rows / 2),
                       "step": "Q and K forward, dQ and dK backward: 4 launches",
                       "bytes_per_step": bytes_step,
                       "l2": "inputs larger than L2: %d rotating sets of Q,K,dQ,dK" % nsets},
            "roofline": {"bound": "hbm", "achieved": round(value / world, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(value / world / peak, 4),
                         "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_kind,
                         "traffic": None, "kernel": "rope_vec_kernel"},
            "gpu_launches": 4 * steps,
            "clocks": sampler.summary(),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.ALL_BY_NAME))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--per-workload-ms", type=float, default=20.0,
                    help="rope: time every workload forward and backward apart, each region "
                         "at least this long (and 200 calls) before the headline; 0 skips it")
    ap.add_argument("--sets", type=int, default=0,
                    help="rope: rotating sets of Q, K, dQ, dK for the headline (0: enough that one "
                         "pass moves at least 2.2 x the L2 size, at least one)")
    ap.add_argument("--seq", type=int, default=0,
                    help="rope: run the workload with this sequence length instead (smaller "
                         "cases for profiling runs)")
    ap.add_argument("--op", choices=["rope", "attention", "xpos", "sweep"], default="rope",
                    help="rope: the fused Q+K rotation (default); attention: attention with the "
                         "rotation fused into the Q/K tile loads; xpos: the rotation with XPOS "
                         "tables, one launch per tensor; sweep: the rotation kernel's grid "
                         "sizings side by side")
    args = ap.parse_args()
    args.e2e_steps = max(1, args.e2e_steps)
    if args.op == "sweep":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "op": "sweep",
                              "unavailable": "the sweep compares grid sizings of the CUDA kernel"}))
            return 0
        return sweep_arm(args)
    if args.op == "xpos":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "op": "xpos",
                              "unavailable": "the reference arm times the rotation only"}))
            return 0
        return xpos_arm(args)
    if args.op == "attention":
        if args.impl == "reference":
            return attention_reference_arm(args)
        return attention_arm(args)
    w = W.ALL_BY_NAME[args.workload]
    if args.seq > 0:
        w = w.with_sizes(name="%s_S%d" % (w.name, args.seq), S=args.seq,
                         table_rows=max(w.table_rows, args.seq) if w.positions == "none"
                         else w.table_rows)
    if args.impl == "reference":
        return reference_arm(args, w)

    world, rank, local = dist_info()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")

    from rotary_position_embedding_rope_gb300 import _build
    if local == 0:
        _build.build()
    if dist is not None:
        dist.barrier()
    import rotary_position_embedding_rope_gb300 as R

    R.load_library()
    warmup = max(3, args.warmup)
    stream = torch.cuda.current_stream(device)
    l2_bytes = torch.cuda.get_device_properties(device).L2_cache_size

    # every workload, forward and backward timed apart, before the headline
    # (it also brings the GPU to its working clocks)
    per_workload = None
    if args.per_workload_ms > 0:
        per_workload = per_workload_block(
            R, device, stream, args.per_workload_ms, 200, l2_bytes,
            cpu_seconds=min(1.5, args.cpu_seconds / 5) if rank == 0 and world == 1 else 0.0)

    # inputs: seeded on the CPU, copied to rotating device sets so every call
    # reads memory last touched 3 steps (~1 GB of traffic) earlier: larger than L2
    q, k, pos = W.make_inputs(w)
    dq, dk, _ = W.make_inputs(w, seed_offset=100)
    set_bytes = sum(t.numel() * t.element_size() for t in (q, k, dq, dk) if t is not None)
    nsets = args.sets if args.sets > 0 else max(1, -(-int(2.2 * l2_bytes) // set_bytes))
    sets = [(q.to(device), k.to(device), dq.to(device), dk.to(device)) for _ in range(nsets)]
    pos_g = None if pos is None else torch.from_numpy(pos).to(device)

    cos = torch.empty((w.table_rows, w.rotary_dim // 2), dtype=torch.float32, device=device)
    sin = torch.empty_like(cos)
    ev_t0, ev_t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    R.rope_tables_build(w.theta, w.rotary_dim, w.table_rows, w.interpolate_factor, cos, sin, stream)
    ev_t0.record(stream)
    R.rope_tables_build(w.theta, w.rotary_dim, w.table_rows, w.interpolate_factor, cos, sin, stream)
    ev_t1.record(stream)
    torch.cuda.synchronize(device)
    table_ms = ev_t0.elapsed_time(ev_t1)

    layout, sbh, dt = W.LAYOUTS[w.layout], int(w.seq_before_head), W.DTYPES[w.dtype]

    def call(qx, kx, backward):
        R.rope_apply_qk(qx, kx, cos, sin, pos_g, w.B, w.Hq, w.Hk, w.S, w.D, w.rotary_dim, layout,
                        sbh, backward, dt, w.table_rows, stream)

    def step(i, events=None):
        qx, kx, dqx, dkx = sets[i % nsets]
        if events is not None:
            events[0].record(stream)
        call(qx, kx, 0)
        if events is not None:
            events[1].record(stream)
        call(dqx, dkx, 1)
        if events is not None:
            events[2].record(stream)

    # the clock sampler is set up and running before the warm-up, so nothing
    # slow (NVML's set-up) leaves the GPU idle between warm-up and timed region
    sampler = ClockSampler(local)
    sampler.start()
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(device)
    assert R.rope_check_errors(stream) == R.ROPE_OK

    # timed region: K steps and nothing else on the stream, bracketed by two
    # events.  No event sits between launches inside it: an event there would
    # stop the next launch from becoming resident early (programmatic
    # dependent launch), which a user's stream does not do.
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(device)
    # A GPU-side pause of ~0.5 ms before the start event (outside the timed
    # region): while the GPU sleeps, the host enqueues the region's first
    # launches, so a host-side delay at the start of a short region (thread
    # scheduling, a driver query) cannot appear as idle GPU time inside it.
    torch.cuda._sleep(PRE_ROLL_CYCLES)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(i)
    t_end.record(stream)
    torch.cuda.synchronize(device)
    sampler.stop()
    if dist is not None:
        dist.barrier()
    local_ms = t_start.elapsed_time(t_end)
    launches = 2 * args.steps
    assert R.rope_check_errors(stream) == R.ROPE_OK

    # per-call durations in isolation (an event on each side of every launch),
    # after the timed region
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(64)]
    for i, e in enumerate(evs):
        step(i, e)
    torch.cuda.synchronize(device)
    fwd_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    bwd_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in evs]))
    bytes_call = W.algorithmic_bytes(w)
    bytes_step = 2 * bytes_call
    max_ms, all_bytes = aggregate(dist, device, local_ms, bytes_step * args.steps)
    ms_per_step = max_ms / args.steps
    value = all_bytes / (max_ms * 1e-3) / 1e9

    # end to end through the public API with host buffers: every step copies
    # Q, K, dQ, dK from pinned host memory, rotates them, and copies the
    # results back to pinned host memory.  The host pipeline splits each call
    # along the batch so both copy directions and the kernels overlap.
    from rotary_position_embedding_rope_gb300.host import HostRotator

    hq, hk, hdq, hdk = (t.pin_memory() for t in (q, k, dq, dk))
    oq, ok_, odq, odk = (torch.empty_like(t).pin_memory() for t in (q, k, dq, dk))
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hdq, hdk))
    rot = HostRotator(device, chunks=4)

    def e2e_step(after):
        rot.apply_qk(hq, hk, cos, sin, oq, ok_, pos_g, w.rotary_dim, w.layout, w.seq_before_head,
                     False, after)
        return rot.apply_qk(hdq, hdk, cos, sin, odq, odk, pos_g, w.rotary_dim, w.layout,
                            w.seq_before_head, True)

    for _ in range(2):
        stream.wait_event(e2e_step(None))
    torch.cuda.synchronize(device)
    if dist is not None:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    last = e0
    for i in range(args.e2e_steps):
        # the pipeline orders every reuse of its staging buffers itself
        last = e2e_step(e0 if i == 0 else None)
    stream.wait_event(last)
    e1.record(stream)
    torch.cuda.synchronize(device)
    e2e_ms, e2e_bytes = aggregate(dist, device, e0.elapsed_time(e1), bytes_step * args.e2e_steps)
    e2e_value = e2e_bytes / (e2e_ms * 1e-3) / 1e9
    assert R.rope_check_errors(stream) == R.ROPE_OK

    # the host link the e2e leg is bound by: 256 MiB copies between pinned
    # host memory and the device, each direction alone and both at once on
    # two streams (plain runtime copies, context for the e2e figure)
    link = link_context(device, stream)

    # roofline of the dominant kernel.  The timed region holds only its
    # launches (2 per step), so its average launch duration is the region's
    # event time over the launch count.
    peak, peak_kind = hbm_peak()
    kernel_ms = local_ms / launches
    achieved = bytes_call / (kernel_ms * 1e-3) / 1e9
    qx0, kx0 = sets[0][0], sets[0][1]
    variant = R.rope_qk_kernel_variant(qx0, kx0, cos, sin, pos_g, w.B, w.Hq, w.Hk, w.S, w.D,
                                       w.rotary_dim, layout, sbh, 0, dt, w.table_rows)
    kernel_name = KERNEL_NAMES.get(variant, "unknown")
    traffic = profiled_traffic(kernel_name, w.name)

    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        import oracle as O

        o = O.load()
        cos32, sin32 = o.tables(w.theta, w.rotary_dim, w.table_rows, w.interpolate_factor, "f32")
        # the oracle is single-threaded; so is the slicing around it while it is timed
        threads = torch.get_num_threads()
        torch.set_num_threads(1)
        nb, el, toks = time_oracle(w, args.cpu_seconds, [(q, w.Hq), (k, w.Hk), (dq, w.Hq),
                                                         (dk, w.Hk)], pos, cos32, sin32)
        torch.set_num_threads(threads)
        cpu = {"value": round(nb / el / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": "batch 0, growing prefixes of the %d tokens (%d token-steps in %.1f s), "
                         "all heads, forward on Q,K + backward on dQ,dK; host has %d cores, "
                         "oracle is single-threaded" % (w.S, toks, el, os.cpu_count() or 0)}

    if rank == 0:
        clocks = sampler.summary()
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic", "config": dict(
                config_of(w),
                timed_region=("exactly %d steps between two events, after a synchronize and a "
                              "%d-cycle GPU-side sleep outside the region (the host enqueues the "
                              "first launches meanwhile)" % (args.steps, PRE_ROLL_CYCLES)),
                l2=("inputs larger than L2: %d rotating set(s) of Q,K,dQ,dK, %.0f MB each, "
                    "%.0f MB in all vs %.0f MB L2; each call's pair (%.0f MB) was last touched "
                    "%.0f MB of traffic earlier" % (
                        nsets, set_bytes / 1e6, nsets * set_bytes / 1e6, l2_bytes / 1e6,
                        set_bytes / 2e6, (2 * nsets - 1) * set_bytes / 2e6)),
                parallelism="replicas" if world > 1 else "single GPU"),
            "us_per_call": round(kernel_ms * 1e3, 3),
            "us_per_call_isolated": {"forward": round(fwd_ms * 1e3, 3),
                                     "backward": round(bwd_ms * 1e3, 3),
                                     "note": "an event on each side of every launch"},
            "table_build_us": round(table_ms * 1e3, 2),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_kind
                         if peak_kind == "measured" else "fallback 6.8 TB/s",
                         "traffic": traffic, "kernel": kernel_name,
                         "frac_of_nominal_8tbs": round(achieved / 8000.0, 4)},
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": h2d, "steps": args.e2e_steps,
                    "ms_per_step": round(e2e_ms / args.e2e_steps, 4),
                    "link_context": link},
            "gpu_launches": launches,
            "kernel_variant": variant,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        if per_workload is not None:
            line["per_workload"] = per_workload
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
