#!/usr/bin/env python
"""Benchmark of the KDA serving hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  state gather (16 rows of an fp32 cache [1024,32,128,128], 20% flags false)
  -> chunked prefill of the varlen batch (16 sequences, lengths U[512,8192],
     H=32, K=V=128, bf16 q/k/v, fp32 g/beta, chunk 64)
  -> state scatter of the 16 final states back to their rows
  -> one decode step (512 requests, bf16 cache [2048,32,128,128], 5% invalid).
value = prefill tokens per second of the whole step (decode time included).
The state-copy bandwidth of the copy workload (fp32 cache [4096,32,128,128]
with 64 KiB page gaps, 256 rows) is measured in the same run and reported
next to it, as the metric names both.  Further legs, each timed on its own:
the fused cache-indexed prefill with checkpoints, INT8 checkpoints, the short
convolution, target verification and the long single-sequence prefill
(131,072 tokens, the few-chain state pass).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

With --gpus N > 1 the script runs under torchrun, one replica per GPU (the
path has no exchange step), and reports the aggregate.  --impl reference runs
the fp64 CPU oracle on the host cores, a bounded sample of the workload per
step.  Prints ONE JSON line (rank 0).
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "KDA prefill tokens/s (H=32,K=V=128) + state gather/scatter GB/s vs HBM peak"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- ranks --

class Ranks:
    def __init__(self, want: int):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = False
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if torch.cuda.is_available():
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.pg = True
        self.want = want

    def barrier(self):
        if self.pg:
            import torch.distributed as dist
            dist.barrier()

    def max(self, x: float) -> float:
        return self._reduce(x, "max")

    def sum(self, x: float) -> float:
        return self._reduce(x, "sum")

    def _reduce(self, x: float, op: str) -> float:
        if not self.pg:
            return x
        import torch.distributed as dist
        dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            import torch.distributed as dist
            dist.destroy_process_group()


def aggregate(units_per_rank: float, seconds_per_rank: float, ranks: Ranks) -> tuple:
    """Whole-job throughput: units all ranks processed / the slowest rank's time."""
    total_units = ranks.sum(units_per_rank)
    slowest = ranks.max(seconds_per_rank)
    return total_units / slowest, slowest


# ---------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi samples (every 100 ms) during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = [r for r in csv.reader(io.StringIO(self.tmp.read())) if len(r) >= 9]
        os.unlink(self.tmp.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "", 1).isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------- peaks --

def peaks() -> tuple:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def traffic_record(kernel: str, units: int):
    """DRAM bytes per launch from a committed ncu capture (bytes per unit x the
    units this launch processes; the capture ran a smaller case of the same
    kernel, whose traffic grows in proportion to its chunk-heads), only while
    the kernel source it was taken from is unchanged (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src):
        return None
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return rec["bytes_per_unit"] * units if h == rec["source_sha256_16"] else None


# ------------------------------------------------------------- workloads --

def build_inputs(dev, seed=0, small=False):
    import kimi_delta_attention_varlen_gb300 as kda
    from kimi_delta_attention_varlen_gb300 import workloads as wl
    w = wl.varlen(seed, B=4) if small else wl.varlen(seed)
    H, D = w.H, w.K
    cu = [0]
    for n in w.lengths:
        cu.append(cu[-1] + n)
    T = cu[-1]
    P = {}
    P["w"] = w
    P["cu_list"] = cu
    P["cache3"] = wl.paged_cache(w.cache_rows, H, D, D, w.cache_dtype, w.cache_stride, seed=seed + 1, device=dev)
    P["inp"] = wl.token_inputs(T, H, D, D, w.io_dtype, seed=seed, device=dev)
    P["cu"] = torch.tensor(cu, dtype=torch.int32, device=dev)
    P["gidx"] = w.gather_idx.to(dev)
    P["gflags"] = w.gather_flags.to(dev)
    P["sidx"] = w.scatter_idx.to(dev)
    P["packed"] = torch.empty(w.B, H, D, D, dtype=torch.float32, device=dev)
    P["final"] = torch.empty(w.B, H, D, D, dtype=torch.float32, device=dev)
    P["out"] = torch.empty(T, H, D, dtype=w.io_dtype, device=dev)
    P["ws"] = torch.empty(kda.kda_prefill_workspace_size(T, w.B, H, D, D), dtype=torch.uint8, device=dev)
    dw = wl.decode(seed)
    P["dw"] = dw
    P["cache5"] = wl.paged_cache(dw.cache_rows, dw.H, dw.V, dw.K, dw.cache_dtype, None, seed=seed + 2, device=dev)
    P["dinp"] = wl.token_inputs(dw.R, dw.H, dw.K, dw.V, dw.io_dtype, seed=seed + 3, device=dev)
    P["didx"] = dw.idx.to(dev)
    P["dout"] = torch.empty(dw.R, dw.H, dw.V, dtype=dw.io_dtype, device=dev)
    return P


def run_step(P, ev=None, prep_only=False):
    """gather -> prefill -> scatter -> decode on the current stream.  `ev`: dict of
    events recorded at the boundaries (for the per-kernel breakdown); with prep_only
    just the two around the chunk-preparation kernel (each record costs stream time)."""
    import kimi_delta_attention_varlen_gb300 as kda
    inp, d = P["inp"], P["dinp"]
    full = ev is not None and not prep_only
    if full:
        ev["g0"].record()
    kda.kda_state_gather(P["cache3"].view, P["gidx"], P["packed"], P["gflags"])
    pev = None
    if ev is not None:
        pev = [None, ev["p1"], ev["p2"], None] if prep_only else [ev["p0"], ev["p1"], ev["p2"], ev["p3"]]
    kda.kda_prefill_varlen(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], P["cu"], P["out"], P["ws"],
                           init_state=P["packed"], final_state=P["final"], events=pev)
    kda.kda_state_scatter(P["cache3"].view, P["sidx"], P["final"])
    if full:
        ev["s1"].record()
    kda.kda_decode_step(d["q"], d["k"], d["v"], d["g"], d["beta"], P["cache5"].view, P["didx"], P["dout"])
    if full:
        ev["d1"].record()


LAUNCHES_PER_STEP = 7  # gather, chunk table, chunk prep, exact chunk prep (fix-up list), state pass, scatter, decode


def prefill_bytes(P) -> dict:
    """Algorithmic bytes of the step's kernels (each kernel's compulsory reads and writes)."""
    w, T, H, D = P["w"], P["cu_list"][-1], P["w"].H, P["w"].K
    io = 2  # bf16
    B = w.B
    n_chunks = sum((n + 63) // 64 for n in w.lengths)
    rec = (3 * 64 * D * 2) + 64 * 64 * 2 + D * 4 + D * 64 * 2
    token_in = T * H * (3 * D * io + D * 4 + 4)
    state = B * H * D * D * 4
    method = token_in + T * H * D * io + 2 * state  # q,k,v,g,beta in; o out; init in, final out
    return {"method": method, "prep": token_in + n_chunks * H * rec, "pass": n_chunks * H * rec + T * H * D * io
            + 2 * state, "n_chunks": n_chunks}


def prefill_flops(P) -> float:
    """Dense 64-tile FLOPs of the chunked form: per chunk and head, the two gated
    Gram products, W and U (2 * 64*64*D each), and the state pass (W S, Q S,
    K^T V_new: 2 * 64*D*D each, plus A_qk V_new: 2 * 64*64*D)."""
    w, D, H = P["w"], P["w"].K, P["w"].H
    n_chunks = sum((n + 63) // 64 for n in w.lengths)
    per = 4 * (2 * 64 * 64 * D) + 3 * (2 * 64 * D * D) + 2 * 64 * 64 * D
    return float(n_chunks * H * per)


def cached_measure(P, steps: int, warmup: int, ckpt_every: int = 1024) -> dict:
    """The fused cache-indexed prefill on the step's inputs (initial states read from
    cache rows, final states written back), without and with checkpoints every
    `ckpt_every` tokens (fp32); median device time of `steps` calls each."""
    import kimi_delta_attention_varlen_gb300 as kda
    inp, T = P["inp"], P["cu_list"][-1]
    n_ck = kda.kda_prefill_checkpoint_count(P["cu_list"], ckpt_every)
    w = P["w"]
    ck = torch.empty(n_ck, w.H, w.V, w.K, dtype=torch.float32, device=P["out"].device)
    res = {}
    for name, kw in (("no_checkpoints", {}), ("checkpoints", {"checkpoints": ck, "ckpt_every": ckpt_every})):
        def call():
            kda.kda_prefill_varlen_cached(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], P["cu"], P["out"],
                                          P["ws"], P["cache3"].view, P["gidx"], flags=P["gflags"],
                                          idx_out=P["sidx"], **kw)
        for _ in range(warmup):
            call()
        times = []
        for _ in range(steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            call()
            b.record()
            b.synchronize()
            times.append(a.elapsed_time(b))
        ms = statistics.median(times)
        res[name] = {"ms": ms, "tokens_per_s": T / (ms * 1e-3)}
    res["checkpoints"].update({"every_tokens": ckpt_every, "slots": n_ck, "dtype": "f32",
                               "bytes": n_ck * w.H * w.V * w.K * 4})
    return res


def ckpt_int8_measure(P, steps: int, warmup: int, pairs: int = 256) -> dict:
    """INT8 checkpoint store (active fp32 rows -> int8 slots) and load (slots -> rows)
    of `pairs` states of the step's cache [1024, 32, 128, 128]; median device time and
    GB/s of the compulsory bytes (state rows, codes, scales)."""
    import kimi_delta_attention_varlen_gb300 as kda
    pc = P["cache3"]
    N, H, V, K = pc.view.shape
    dev = pc.view.device
    rows = torch.randperm(N, generator=torch.Generator().manual_seed(21))[:pairs].to(torch.int32).to(dev)
    slots = torch.arange(pairs, dtype=torch.int32, device=dev)
    q = torch.empty(pairs, H, V, K, dtype=torch.int8, device=dev)
    sc = torch.empty(pairs, H, K, dtype=torch.float32, device=dev)
    state_b = pairs * H * V * K * pc.view.element_size()
    code_b = pairs * H * V * K + pairs * H * K * 4
    res = {"pairs": pairs, "cache": f"fp32 [{N},{H},{V},{K}]"}
    for name, fn in (("store", lambda: kda.kda_ckpt_store_int8(pc.view, rows, slots, q, sc)),
                     ("load", lambda: kda.kda_ckpt_load_int8(q, sc, slots, pc.view, rows))):
        for _ in range(warmup):
            fn()
        times = []
        for _ in range(steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            times.append(a.elapsed_time(b))
        ms = statistics.median(times)
        res[name] = {"ms": ms, "gbs": (state_b + code_b) / (ms * 1e-3) / 1e9, "bytes": state_b + code_b}
    return res


def conv1d_measure(P, steps: int, warmup: int, W: int = 4) -> dict:
    """The short causal convolution (width 4, SiLU, bf16 states) over the step's tokens
    for q, k and v as one [T, 3 H D] bf16 buffer, with initial and final states; median
    device time and GB/s of the compulsory bytes (x in, y out, states in and out)."""
    import kimi_delta_attention_varlen_gb300 as kda
    w = P["w"]
    T, B = P["cu_list"][-1], w.B
    C = 3 * w.H * w.K
    dev = P["out"].device
    g = torch.Generator(device=dev).manual_seed(31)
    x = torch.randn(T, C, generator=g, device=dev).to(torch.bfloat16)
    y = torch.empty_like(x)
    wt = torch.randn(C, W, generator=g, device=dev) * 0.5
    bias = torch.randn(C, generator=g, device=dev) * 0.1
    init = torch.randn(B, W - 1, C, generator=g, device=dev).to(torch.bfloat16)
    fin = torch.empty_like(init)

    def call():
        kda.kda_conv1d_varlen(x, P["cu"], wt, y, bias=bias, activation="silu", init_state=init, final_state=fin)
    for _ in range(warmup):
        call()
    times = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    nbytes = 2 * T * C * 2 + 2 * B * (W - 1) * C * 2 + C * (W + 1) * 4
    return {"ms": ms, "gbs": nbytes / (ms * 1e-3) / 1e9, "bytes": nbytes, "tokens_per_s": T / (ms * 1e-3),
            "shape": f"x [{T}, {C}] bf16, width {W}, SiLU, bf16 states"}


def long_prefill_measure(dev, steps: int, warmup: int, tokens: int | None = None) -> dict:
    """The long single-sequence prefill (131,072 tokens unless `tokens` says otherwise; 32 heads,
    head size 128, bf16, zero initial state, final state out).  Its state pass is one serial chain of
    T / 64 chunks per head over only 32 (sequence, head) pairs, the few-chain shape.  From 512
    chunks on, the prefill runs segmented (the state pass of each 256-chunk segment overlapping the
    next segment's preparation): prep_ms is then the time until the last segment is prepared and
    pass_ms the rest; unsegmented they are the two kernels' times."""
    import kimi_delta_attention_varlen_gb300 as kda
    from kimi_delta_attention_varlen_gb300 import workloads as wl
    w = wl.long_seq(0, T=tokens) if tokens else wl.long_seq(0)
    T, H, D = w.lengths[0], w.H, w.K
    inp = wl.token_inputs(T, H, D, D, w.io_dtype, seed=7, device=dev)
    out = torch.empty(T, H, D, dtype=w.io_dtype, device=dev)
    fin = torch.empty(1, H, D, D, dtype=torch.float32, device=dev)
    ws = torch.empty(kda.kda_prefill_workspace_size(T, 1, H, D, D), dtype=torch.uint8, device=dev)
    cu = torch.tensor([0, T], dtype=torch.int32, device=dev)

    def call(ev=None):
        kda.kda_prefill_varlen(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu, out, ws,
                               final_state=fin, events=ev)

    for _ in range(warmup):
        call()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for e in evs:
        call(e)
    torch.cuda.synchronize()
    med = statistics.median
    prep = med(e[1].elapsed_time(e[2]) for e in evs)
    pas = med(e[2].elapsed_time(e[3]) for e in evs)
    tot = med(e[0].elapsed_time(e[3]) for e in evs)
    del inp, out, fin, ws
    torch.cuda.empty_cache()
    form = "segmented (256-chunk segments, passes overlapping preparation)" if T >= 512 * 64 else "two kernels"
    return {"workload": w.name, "form": form, "prep_ms": prep, "pass_ms": pas, "ms": tot,
            "tokens_per_s": T / (tot * 1e-3)}


def compact_measure(P, dev, steps: int, warmup: int, long_tokens: int | None = None) -> dict:
    """The prefill's compact form (bf16, head size 128, a workspace of only the chunk table):
    the fused kernel on the step's varlen batch and on the long single sequence; median device
    time and the workspace bytes against the two-kernel form's."""
    import kimi_delta_attention_varlen_gb300 as kda
    from kimi_delta_attention_varlen_gb300 import workloads as wl
    res = {}
    w = P["w"]
    T, B, H, D = P["cu_list"][-1], w.B, w.H, w.K
    inp = P["inp"]
    ws = torch.empty(kda.kda_prefill_workspace_size_compact(T, B, H, D, D), dtype=torch.uint8, device=dev)
    ms = _time_calls(lambda: kda.kda_prefill_varlen(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], P["cu"],
                                                    P["out"], ws, init_state=P["packed"], final_state=P["final"]),
                     steps, warmup)
    res["varlen"] = {"ms": ms, "tokens_per_s": T / (ms * 1e-3), "workspace_bytes": ws.numel(),
                     "two_kernel_workspace_bytes": kda.kda_prefill_workspace_size(T, B, H, D, D)}
    lw = wl.long_seq(0, T=long_tokens) if long_tokens else wl.long_seq(0)
    TL = lw.lengths[0]
    li = wl.token_inputs(TL, H, D, D, lw.io_dtype, seed=7, device=dev)
    lo = torch.empty(TL, H, D, dtype=lw.io_dtype, device=dev)
    lf = torch.empty(1, H, D, D, dtype=torch.float32, device=dev)
    lcu = torch.tensor([0, TL], dtype=torch.int32, device=dev)
    lws = torch.empty(kda.kda_prefill_workspace_size_compact(TL, 1, H, D, D), dtype=torch.uint8, device=dev)
    ms = _time_calls(lambda: kda.kda_prefill_varlen(li["q"], li["k"], li["v"], li["g"], li["beta"], lcu, lo, lws,
                                                    final_state=lf), max(2, min(steps, 5)), 1)
    res["long"] = {"workload": lw.name, "ms": ms, "tokens_per_s": TL / (ms * 1e-3), "workspace_bytes": lws.numel(),
                   "two_kernel_workspace_bytes": kda.kda_prefill_workspace_size(TL, 1, H, D, D)}
    del li, lo, lf, lws, ws
    torch.cuda.empty_cache()
    return res


def verify_measure(P, steps: int, warmup: int, L: int = 4, requests: int | None = None) -> dict:
    """Speculative target verification of L draft tokens for the decode workload's
    requests (bf16 cache [2048, 32, 128, 128], R = 512): every token's state to its own
    bf16 pool slot.  Median device time; GB/s of the compulsory bytes (states read once,
    L intermediate states written, token inputs and outputs)."""
    import kimi_delta_attention_varlen_gb300 as kda
    from kimi_delta_attention_varlen_gb300 import workloads as wl
    dw, pc = P["dw"], P["cache5"]
    R, H, K, V = (requests or dw.R), dw.H, dw.K, dw.V
    didx = P["didx"][:R]
    dev = P["out"].device
    t = wl.token_inputs(R * L, H, K, V, dw.io_dtype, seed=41, device=dev)
    inp = {n: x.view(R, L, *x.shape[1:]) for n, x in t.items()}
    pool = torch.empty(R * L, H, V, K, dtype=pc.view.dtype, device=dev)
    inter = torch.arange(R * L, dtype=torch.int32, device=dev).view(R, L)
    out = torch.empty(R, L, H, V, dtype=dw.io_dtype, device=dev)

    def call():
        kda.kda_target_verify(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], pc.view, didx, pool, inter, out)
    for _ in range(warmup):
        call()
    times = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        call()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    valid = int((dw.idx[:R] >= 0).sum())
    st = H * V * K * pc.view.element_size()
    io = R * L * H * (3 * K * 2 + K * 4 + 4 + V * 2)
    nbytes = valid * st + R * L * st + io
    return {"ms": ms, "gbs": nbytes / (ms * 1e-3) / 1e9, "bytes": nbytes, "draft_tokens": L, "requests": R,
            "tokens_per_s": R * L / (ms * 1e-3)}


def _time_calls(fn, steps: int, warmup: int) -> float:
    """Median device time (ms) of `steps` calls, events on the current stream."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


def copy_measure(dev, steps: int, warmup: int, hbm_gbs: float, rows: int = 4096) -> dict:
    """The state-copy workload ([4096, 32, 128, 128] cache, 64 KiB page gaps, 256 selected
    rows, 10% invalid, flags p = 0.8) in every variant it names: fp32 cache with int32 and
    int64 indices, bf16 cache with int32 indices, and the scatter of fp32 packed states into
    the bf16 cache (RNE cast).  Algorithmic bytes: gather reads the valid flagged rows and
    writes every packed row; scatter reads and writes each valid row (4 B read + 2 B written
    per element when casting)."""
    import kimi_delta_attention_varlen_gb300 as kda
    from kimi_delta_attention_varlen_gb300 import workloads as wl
    res = {}
    for w in (wl.copy_fp32(N=rows), wl.copy_bf16(N=rows)):
        pc = wl.paged_cache(w.N, w.H, w.V, w.K, w.dtype, w.row_stride, seed=w.seed, device=dev)
        es = pc.view.element_size()
        P = w.H * w.V * w.K
        flags = wl.bernoulli_flags(w.S, w.p_flag, seed=w.seed + 2).to(dev)
        packed = torch.empty(w.S, w.H, w.V, w.K, dtype=w.dtype, device=dev)
        tag = "fp32" if w.dtype == torch.float32 else "bf16"
        itypes = (torch.int32, torch.int64) if w.dtype == torch.float32 else (torch.int32,)
        for it in itypes:
            gidx = wl.gather_indices(w.S, w.N, w.p_invalid, seed=w.seed + 1, dtype=it).to(dev)
            sidx = wl.scatter_indices(w.S, w.N, w.p_invalid, seed=w.seed + 3, dtype=it).to(dev)
            g_cpu, s_cpu = gidx.cpu(), sidx.cpu()
            n_g = int(((g_cpu >= 0) & (g_cpu < w.N) & flags.cpu()).sum())
            n_s = int(((s_cpu >= 0) & (s_cpu < w.N)).sum())
            name = f"{tag}_{'int32' if it == torch.int32 else 'int64'}"
            for op, fn, nbytes in (
                    ("gather", lambda: kda.kda_state_gather(pc.view, gidx, packed, flags), (n_g + w.S) * P * es),
                    ("scatter", lambda: kda.kda_state_scatter(pc.view, sidx, packed), 2 * n_s * P * es)):
                ms = _time_calls(fn, steps, warmup)
                gbs = nbytes / (ms * 1e-3) / 1e9
                res[f"{op}_{name}"] = {"ms": ms, "gbs": gbs, "frac": gbs / hbm_gbs, "bytes": nbytes}
            if w.dtype == torch.bfloat16:  # fp32 packed states cast into the bf16 cache
                src = torch.randn(w.S, w.H, w.V, w.K, device=dev)
                nbytes = n_s * P * (4 + 2)
                ms = _time_calls(lambda: kda.kda_state_scatter(pc.view, sidx, src), steps, warmup)
                gbs = nbytes / (ms * 1e-3) / 1e9
                res["scatter_fp32_to_bf16_int32"] = {"ms": ms, "gbs": gbs, "frac": gbs / hbm_gbs, "bytes": nbytes}
                del src
        del pc, packed
        torch.cuda.empty_cache()
    return {"workload": f"copy: cache [{rows},32,128,128] stride payload+64KiB, S=256, 10% invalid, flags p=0.8",
            "variants": res, "hbm_peak_gbs": hbm_gbs}


# ------------------------------------------------------------ CPU oracle --

def cpu_baseline(P, target_s: float = 12.0, steps: int | None = None) -> dict:
    """The oracle as it stands, timed on the host cores on a bounded sample of the
    prefill workload: the shortest sequences, all heads, from their gathered
    initial states."""
    import numpy as np

    import oracle
    w, cu = P["w"], P["cu_list"]
    order = sorted(range(w.B), key=lambda b: w.lengths[b])
    nthreads = os.cpu_count() or 1

    def host(b):
        t0, t1 = cu[b], cu[b + 1]
        inp = P["inp"]
        sl = [inp[k][t0:t1].detach().cpu().double().numpy() for k in ("q", "k", "v", "g", "beta")]
        return sl, P["packed"][b:b + 1].cpu().double().numpy()

    # calibrate on the shortest sequence, then size the sample to ~target_s
    sl, ini = host(order[0])
    t = time.perf_counter()
    oracle.prefill(*sl, [0, sl[0].shape[0]], init=ini, scale=w.K ** -0.5, nthreads=nthreads)
    dt = time.perf_counter() - t
    rate = sl[0].shape[0] / max(dt, 1e-9)
    budget = rate * target_s
    chosen, tok = [], 0
    for b in order:
        if tok + w.lengths[b] > budget and chosen:
            break
        chosen.append(b)
        tok += w.lengths[b]
    parts = [host(b) for b in chosen]
    q, k, v, g, beta = (np.concatenate([p[0][i] for p in parts]) for i in range(5))
    ini = np.concatenate([p[1] for p in parts])
    cu_s = [0]
    for b in chosen:
        cu_s.append(cu_s[-1] + w.lengths[b])
    t = time.perf_counter()
    oracle.prefill(q, k, v, g, beta, cu_s, init=ini, scale=w.K ** -0.5, nthreads=nthreads)
    dt = time.perf_counter() - t
    return {"value": tok / dt, "unit": UNIT, "cores": min(nthreads, len(chosen) * w.H), "kind": "oracle",
            "sample": f"{len(chosen)} shortest sequences ({tok} tokens) x {w.H} heads of the varlen workload, "
                      f"fp64 token-by-token recurrence, {dt:.1f} s"}


# ------------------------------------------------------------------ main --

def native(args, ranks: Ranks) -> dict | None:
    import kimi_delta_attention_varlen_gb300 as kda  # noqa: F401  (fails loudly if libkda.so is missing)
    dev = torch.device("cuda", ranks.local)
    torch.cuda.set_device(dev)
    if args.workload == "copy":  # the state-copy legs alone (profiler captures on a smaller cache)
        pk, pk_kind = peaks()
        res = copy_measure(dev, args.steps, args.warmup, pk["hbm_gbs"], rows=args.copy_rows)
        return {"metric": METRIC, "unit": "GB/s", "state_copy": res, "peak_source": pk_kind} if ranks.rank == 0 \
            else None
    P = build_inputs(dev, small=args.workload == "small")
    T = P["cu_list"][-1]
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        run_step(P)
    torch.cuda.synchronize()

    names = ["g0", "p0", "p1", "p2", "p3", "s1", "d1"]
    # evs: the timed steps (events around the chunk preparation only); evb: as many instrumented
    # steps after the timed region for the rest of the per-kernel breakdown
    evs = [{n: torch.cuda.Event(enable_timing=True) for n in names} for _ in range(args.steps)]
    evb = [{n: torch.cuda.Event(enable_timing=True) for n in names} for _ in range(args.steps)]
    for e in evs + evb:  # create the events outside the timed region
        for x in e.values():
            x.record()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(ranks.local)
    torch.cuda.synchronize()
    ranks.barrier()
    torch.cuda.synchronize()
    clocks.start()
    start.record(stream)
    for i in range(args.steps):
        run_step(P, evs[i], prep_only=True)
    stop.record(stream)
    torch.cuda.synchronize()
    ranks.barrier()
    torch.cuda.synchronize()
    clk = clocks.stop()
    sec = start.elapsed_time(stop) * 1e-3
    value, slowest = aggregate(T * args.steps, sec, ranks)
    for i in range(args.steps):
        run_step(P, evb[i])
    torch.cuda.synchronize()

    def med(a, b, src=evb):
        return statistics.median(e[a].elapsed_time(e[b]) for e in src)

    br = {"gather": med("g0", "p0"), "chunk_table": med("p0", "p1"), "chunk_prep": med("p1", "p2", evs),
          "state_pass": med("p2", "p3"), "scatter": med("p3", "s1"), "decode": med("s1", "d1")}
    if args.workload == "small":  # reduced sizes for profiler captures: the step, then one call of each next-row leg
        legs = {"cached_prefill": cached_measure(P, 1, 1),
                "ckpt_int8": ckpt_int8_measure(P, 1, 1, pairs=64),
                "conv1d": conv1d_measure(P, 1, 1),
                "target_verify": verify_measure(P, 1, 1, requests=128),
                "compact_prefill": compact_measure(P, dev, 1, 1, long_tokens=16384),
                "long_prefill": long_prefill_measure(dev, 1, 3, tokens=16384)}
        return {"metric": METRIC, "value": value, "unit": UNIT, "workload": P["w"].name, "tokens": T,
                "breakdown_ms": br, "legs": legs} if ranks.rank == 0 else None

    # end to end through the public API: every step copies its inputs from pinned host
    # memory to the device, runs, and reads its results back.  As a serving loop would,
    # the upload of step i + 1 (copy stream) overlaps step i's kernels, and the download
    # of step i (a second copy stream) overlaps step i + 1; two device sets of inputs and
    # outputs alternate, each reused only once its previous download has finished.
    in_keys = ("q", "k", "v", "g", "beta")
    small_keys = ("cu", "gidx", "gflags", "sidx", "didx")
    Q = dict(P)
    Q["inp"] = {k: torch.empty_like(P["inp"][k]) for k in P["inp"]}
    Q["dinp"] = {k: torch.empty_like(P["dinp"][k]) for k in P["dinp"]}
    for k in small_keys:
        Q[k] = torch.empty_like(P[k])
    Q["out"], Q["dout"] = torch.empty_like(P["out"]), torch.empty_like(P["dout"])
    sets = (P, Q)
    host_in = {k: P["inp"][k].cpu().pin_memory() for k in in_keys}
    host_d = {k: P["dinp"][k].cpu().pin_memory() for k in in_keys}
    small = {k: P[k].cpu().pin_memory() for k in small_keys}
    host_out = torch.empty(P["out"].shape, dtype=P["out"].dtype).pin_memory()
    host_dout = torch.empty(P["dout"].shape, dtype=P["dout"].dtype).pin_memory()
    bi = sum(t.numel() * t.element_size() for t in (*host_in.values(), *host_d.values(), *small.values()))
    bo = host_out.numel() * host_out.element_size() + host_dout.numel() * host_dout.element_size()
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_steps_run(n):
        free = [None, None]  # per set: the download that last read it
        s_up.wait_stream(stream)
        for i in range(n):
            S = sets[i % 2]
            if free[i % 2] is not None:
                s_up.wait_event(free[i % 2])
            with torch.cuda.stream(s_up):
                for k2, t in host_in.items():
                    S["inp"][k2].copy_(t, non_blocking=True)
                for k2, t in host_d.items():
                    S["dinp"][k2].copy_(t, non_blocking=True)
                for k2, t in small.items():
                    S[k2].copy_(t, non_blocking=True)
            stream.wait_stream(s_up)
            run_step(S)
            s_down.wait_stream(stream)
            with torch.cuda.stream(s_down):
                host_out.copy_(S["out"], non_blocking=True)
                host_dout.copy_(S["dout"], non_blocking=True)
                free[i % 2] = s_down.record_event()
        stream.wait_stream(s_down)

    e2e_steps = max(1, args.steps)  # the same K steps as the device-resident measurement
    e2e_steps_run(min(args.warmup, 3))
    torch.cuda.synchronize()
    ranks.barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    e2e_steps_run(e2e_steps)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_value, _ = aggregate(T * e2e_steps, a.elapsed_time(b) * 1e-3, ranks)
    del Q, sets

    pk, pk_kind = peaks()
    leg_steps = max(5, min(args.steps, 50))  # the secondary legs report medians of up to 50 calls
    copy = copy_measure(dev, max(5, min(args.steps, 20)), max(3, args.warmup), pk["hbm_gbs"])
    fused = cached_measure(P, leg_steps, max(3, args.warmup))
    ck8 = ckpt_int8_measure(P, leg_steps, max(3, args.warmup))
    conv = conv1d_measure(P, leg_steps, max(3, args.warmup))
    ver = verify_measure(P, leg_steps, max(3, args.warmup))
    long_pf = long_prefill_measure(dev, 5, 3)
    compact = compact_measure(P, dev, leg_steps, max(3, args.warmup))
    nb = prefill_bytes(P)
    flops = prefill_flops(P)
    prefill_ms = br["chunk_table"] + br["chunk_prep"] + br["state_pass"]
    # dominant kernel of the step, by measured time.  Its roofline uses the method's algorithmic
    # bytes for the units the launch processes: a prefill kernel processes the whole batch
    # (49,280 B per token at H = 32, K = V = 128 bf16, plus 2 H D^2 4 B of initial and final
    # state per sequence); the kernel's own compulsory bytes (its inputs plus the per-(chunk,
    # head) records it writes or reads) are reported beside them.
    kern = {"chunk_prep": (br["chunk_prep"], nb["method"], nb["prep"]),
            "state_pass": (br["state_pass"], nb["method"], nb["pass"]),
            "state_gather": (br["gather"], None, None), "decode_step": (br["decode"], None, None)}
    dom = max(kern, key=lambda k2: kern[k2][0])
    dom_ms, dom_bytes, dom_compulsory = kern[dom]
    if dom_bytes is None:
        dw = P["dw"]
        dom_bytes = dom_compulsory = 2 * int((dw.idx >= 0).sum()) * dw.H * dw.K * dw.V * 2
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    traffic = traffic_record(dom, nb["n_chunks"] * P["w"].H)

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ranks.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": slowest * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": P["w"].name + " + gather/scatter fp32 cache [1024,32,128,128] + decode R=512",
                   "tokens_per_step": T, "lengths": P["w"].lengths, "heads": 32, "head_dim": 128, "chunk": 64,
                   "step": "state gather -> chunked prefill -> state scatter -> decode step",
                   "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{ranks.world}"},
        "breakdown_ms": br,
        "breakdown_source": "chunk_prep: events around it in every timed step; the other kernels: the same "
                            "number of fully instrumented steps right after the timed region",
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
                     "peak_source": pk_kind, "bytes_per_launch": dom_bytes,
                     "bytes_convention": "algorithmic: 49,280 B per token + 2 H D^2 4 B per sequence",
                     "compulsory_bytes_per_launch": dom_compulsory,
                     "compulsory_frac": dom_compulsory / (dom_ms * 1e-3) / 1e9 / pk["hbm_gbs"]},
        "prefill_roofline": {
            "ms": prefill_ms, "algorithmic_bytes": nb["method"],
            "achieved_gbs": nb["method"] / (prefill_ms * 1e-3) / 1e9,
            "frac_hbm": nb["method"] / (prefill_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
            "dense_tile_tflops": flops / (prefill_ms * 1e-3) / 1e12,
            "frac_bf16": flops / (prefill_ms * 1e-3) / 1e12 / pk["bf16_tflops"],
            "attainable_frac": (nb["method"] / (prefill_ms * 1e-3)) /
                               min(pk["bf16_tflops"] * 1e12 * nb["method"] / flops, pk["hbm_gbs"] * 1e9),
            "flop_convention": "dense 64x64 tiles", "peak_source": pk_kind},
        "state_copy": copy,
        "decode": {"ms": br["decode"], "requests_per_s": P["dw"].R / (br["decode"] * 1e-3)},
        "cached_prefill": {**fused, "unfused_ms": br["gather"] + prefill_ms + br["scatter"]},
        "conv1d": {**conv, "frac": conv["gbs"] / pk["hbm_gbs"]},
        "target_verify": {**ver, "frac": ver["gbs"] / pk["hbm_gbs"]},
        "long_prefill": long_pf,
        "compact_prefill": compact,
        "ckpt_int8": {**ck8, "store_frac": ck8["store"]["gbs"] / pk["hbm_gbs"],
                      "load_frac": ck8["load"]["gbs"] / pk["hbm_gbs"]},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo},
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "clocks": clk,
    }
    if ranks.rank == 0 and ranks.world == 1:
        result["cpu_baseline"] = cpu_baseline(P)
    return result if ranks.rank == 0 else None


def reference(args, ranks: Ranks) -> dict | None:
    """The oracle arm: each step runs the fp64 CPU oracle on a bounded sample of
    the same workload (rank 0 only)."""
    if ranks.rank != 0:
        return None
    import numpy as np

    import oracle
    from kimi_delta_attention_varlen_gb300 import workloads as wl
    w = wl.varlen()
    cu = [0]
    for n in w.lengths:
        cu.append(cu[-1] + n)
    b = min(range(w.B), key=lambda i: w.lengths[i])  # the shortest sequence, all heads
    L = w.lengths[b]
    inp = wl.token_inputs(L, w.H, w.K, w.V, w.io_dtype, seed=0, device="cpu")  # same shapes and draws
    sl = [inp[k].double().numpy() for k in ("q", "k", "v", "g", "beta")]
    init = np.zeros((1, w.H, w.V, w.K))
    nthreads = os.cpu_count() or 1
    for _ in range(args.warmup):
        oracle.prefill(*sl, [0, L], init=init, scale=w.K ** -0.5, nthreads=nthreads)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.prefill(*sl, [0, L], init=init, scale=w.K ** -0.5, nthreads=nthreads)
    sec = time.perf_counter() - t
    value = L * args.steps / sec
    sample = (f"1 sequence of {L} tokens (the workload's shortest length) x {w.H} heads per step, same "
              f"distributions, fp64 oracle")
    return {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ranks.world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": sec * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": w.name, "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": min(nthreads, w.H), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=["full", "small", "copy"], default="full",
                    help="small: 4-sequence varlen batch, step timing plus one call of each next-row leg "
                         "at reduced sizes (for profiler captures); copy: the state-copy variants alone")
    ap.add_argument("--copy-rows", type=int, default=4096,
                    help="cache rows of the state-copy workload (--workload copy; 4096 is the full size)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    ranks = Ranks(args.gpus)
    try:
        res = reference(args, ranks) if args.impl == "reference" else native(args, ranks)
    finally:
        ranks.close()
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
