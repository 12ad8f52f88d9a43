"""Layer-step benchmark of the GB300 Flash-dLLM hot path.

Workload (the LLaDA-8B-shaped single layer, bf16, batch 1, prompt 512 + gen
256): one step = fused QKV + RoPE + KV scatter for 64 refresh rows (32
masked-window + 32 tracked), scheduled attention over the 768 cached keys
with the Eq. (2) tracker, tracker top-32, and eps unmasking of the 32 window
rows over vocab 126464. Metric: query rows per second of whole layer-steps.

Timing: W warm-up steps, then exactly K timed steps between CUDA events on
the launching stream, bracketed by a barrier and torch.cuda.synchronize().
Weights, caches, hidden rows and logits rotate over enough copies that the
step's working set is several times the L2 size, so no step reads a
previous step's data out of L2. The dominant kernel (the QKV projection,
which streams the 100.7 MB weight) is timed for the roofline figure by CUDA
events around back-to-back graph launches of it alone, right after the
timed steps (events inside the step graph would slow the step itself). SM
clocks and throttle reasons are sampled with nvidia-smi during the timed
region.

--impl reference times the float64 CPU oracle (the reference arm of this
build; there is no upstream implementation to install) on bounded samples
of the same workload on the host cores.

Multi-GPU (torchrun): every rank runs an independent replica of the
workload (the path shards by sequence with no exchange); value is the total
rows of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "layer-step query-tokens/s at LLaDA-8B shapes; % of bf16 TC peak / HBM GB/s"
WORKLOAD = "llada8b_layer_bf16_b1_p512_g256_w32_t32"


# DRAM traffic of one projection call on this workload (its two kernels,
# the weight stream and the merge: dram__bytes_read.sum +
# dram__bytes_write.sum with the caches left alone), from the ncu capture
# summarised in profiles/gemm_stream_kernel_llada8b_layer.txt. It is reported
# only while the sources it was taken from hash to the recorded value; after
# any change to them the figure is stale and the line carries null.
QKV_TRAFFIC = {"sources_sha256": "cf3bad7dad7c9043b34f7298f0bbe083a682322157db4c31d44a1b42fd64df9d",
               "bytes": 102338304 + 3235584 + 256 + 562176}
QKV_SOURCES = ("kv_cache_attention_gb300/csrc/fdl_qkv_tc.cu", "kv_cache_attention_gb300/csrc/fdl_gemm_tc.cu", "kv_cache_attention_gb300/csrc/fdl_gemm_stream.cu", "kv_cache_attention_gb300/csrc/fdl_qkv.cu",
               "kv_cache_attention_gb300/csrc/tc_ptx.cuh", "kv_cache_attention_gb300/csrc/fdl_internal.cuh")


def sources_sha256(paths) -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def qkv_traffic():
    if QKV_TRAFFIC["sources_sha256"] and QKV_TRAFFIC["sources_sha256"] == sources_sha256(QKV_SOURCES):
        return QKV_TRAFFIC["bytes"]
    return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class Clocks:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.reader = None

    def __enter__(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        if self.proc:
            def read():
                for line in self.proc.stdout:
                    self.lines.append(line)
            self.reader = threading.Thread(target=read, daemon=True)
            self.reader.start()
        return self

    def wait_live(self, timeout_s: float):
        """Waits (up to timeout_s) until the sampler has printed a sample."""
        end = time.perf_counter() + timeout_s
        while self.proc and not self.lines and time.perf_counter() < end and self.proc.poll() is None:
            time.sleep(0.01)

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.reader:
                self.reader.join(timeout=5)
        self.out = "".join(self.lines)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


class Nvml:
    """SM clock and throttle reasons read straight from the driver's NVML
    library (libnvidia-ml, part of the driver) through ctypes: one read takes
    microseconds, so it can bracket a timed region closely. Only queries;
    nothing is set."""
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap"}

    def __init__(self, index: int):
        import ctypes
        self.ok = False
        try:
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
            if self.lib.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
                return
            self.ok = True
        except OSError:
            pass

    def read(self):
        import ctypes
        if not self.ok:
            return None
        mhz, mx, why = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) != 0:   # NVML_CLOCK_SM
            return None
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
        reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        reasons(self.h, ctypes.byref(why))
        return {"sm_mhz": int(mhz.value), "sm_max_mhz": int(mx.value),
                "reasons": sorted(n for bit, n in self.REASONS.items() if why.value & bit)}


def clock_record(clk, before, after):
    """The line's clocks: the sampler's median SM clock and reasons over the
    loaded window, plus the NVML reads that bracket the timed steps."""
    rec = clk.summary()
    rec["nvml_before_timed"] = before
    rec["nvml_after_timed"] = after
    reasons = set(rec["reasons"])
    for r in (before, after):
        if r:
            reasons.update(r["reasons"])
    rec["reasons"] = sorted(reasons)
    if rec["sm_mhz"] is None and before and after:
        rec["sm_mhz"] = (before["sm_mhz"] + after["sm_mhz"]) / 2
        rec["sm_max_mhz"] = max(before["sm_max_mhz"], after["sm_max_mhz"])
    rec["how"] = ("nvidia-smi every 50 ms from an untimed 0.3 s pre-roll under load through the warm-ups, the "
                  "timed steps and the roofline replays (sm_mhz = median of those samples); NVML SM clock and "
                  "reasons read immediately before and after the timed steps")
    return rec


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if os.environ.get("FDL_BENCH_BACKEND", "nccl") == "nccl" else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest of the ranks' x (every rank gets it): the job's time is
    the slowest replica's."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(rows_per_rank_step: int, steps: int, ms_max: float, world: int) -> float:
    """Rows of all ranks' steps over the slowest rank's time (rows/s); every
    rank runs the same replica workload."""
    return world * rows_per_rank_step * steps / (ms_max * 1e-3)


# ---------------------------------------------------------------------------
# CPU oracle leg
# ---------------------------------------------------------------------------
def oracle_step(wl, n_rows: int):
    """One oracle layer-step of the workload restricted to its first n_rows
    query rows (the bounded sample); returns the rows processed."""
    import oracle
    e, s, g = wl.extra, wl.shape, wl.geom
    rows = e["rows"]
    sel = slice(0, n_rows)
    x = e["x"].values()[sel]
    q, kc, vc = oracle.qkv_rope_cache_write(
        x, e["w_vals"], s.n_heads, s.head_dim, s.rope_theta, rows.row_rope_pos[sel], rows.row_seq[sel],
        rows.row_cache_pos[sel], g.block_table, g.page_size, e["kc_vals"], e["vc_vals"], s.dtype)
    cu = np.array([0, n_rows], np.int32)
    _, _, tr = oracle.sched_attn(q, kc, vc, g.block_table, g.page_size, cu, wl.seq_len, rows.row_kind[sel],
                                 max_seq=wl.max_seq, dtype=s.dtype)
    oracle.track_topk(tr.astype(np.float32), e["eligible"], wl.seq_len, e["topk"])
    n_logit_rows = min(n_rows, 32)
    oracle.unmask(e["logit_vals"][:n_logit_rows], np.zeros(n_logit_rows, np.int32),
                  e["window_pos"][:n_logit_rows], 1, e["eps"], False, e["max_search"])
    return n_rows


def cpu_leg(wl, budget_s: float):
    """Times the oracle as it stands on the host cores for about budget_s."""
    e = wl.extra
    e.setdefault("w_vals", e["w"].values())
    e.setdefault("kc_vals", e["k_cache"].values())
    e.setdefault("vc_vals", e["v_cache"].values())
    e.setdefault("logit_vals", e["logits"].values())
    n_rows = e["rows"].n_rows
    done, t0 = 0, time.perf_counter()
    steps = 0
    while True:
        done += oracle_step(wl, n_rows)
        steps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return done / dt, steps, dt


def flash_verify_oracle_sample(fv, budget_s: float):
    """Times the oracle on a bounded sample of the Flash-Verify stress
    layer-step: the draft forward's layer for its first sequence (32 window +
    32 tracked rows against that sequence's 1536 cached keys), that
    sequence's top-32 and the eps unmasking of its 32 window rows over the
    126464-entry vocabulary, repeated for about budget_s."""
    import oracle
    e, s, g = fv.extra, fv.shape, fv.geom
    rows = e["rows"]
    n = int(rows.cu_seqlens[1])
    slots = g.page_size
    w = e.setdefault("w_vals", e["w"].values())
    kc = e["k_cache"].values()[:slots]
    vc = e["v_cache"].values()[:slots]
    x = e["x"].values()[:n]
    logits = e["logits"].values()[:32]
    bt = np.zeros((1, 1), np.int32)
    done, steps, t0 = 0, 0, time.perf_counter()
    while True:
        q, kc2, vc2 = oracle.qkv_rope_cache_write(
            x, w, s.n_heads, s.head_dim, s.rope_theta, rows.row_rope_pos[:n], np.zeros(n, np.int32),
            rows.row_cache_pos[:n], bt, slots, kc, vc, s.dtype)
        _, _, tr = oracle.sched_attn(q, kc2, vc2, bt, slots, np.array([0, n], np.int32), fv.seq_len[:1],
                                     rows.row_kind[:n], max_seq=fv.max_seq, dtype=s.dtype)
        oracle.track_topk(tr.astype(np.float32), e["eligible"][:1], fv.seq_len[:1], e["topk"])
        oracle.unmask(logits, np.zeros(32, np.int32), e["window_pos"], 1, e["eps"], False, e["max_search"])
        done += n
        steps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return done / (time.perf_counter() - t0), steps, time.perf_counter() - t0


def cpu_leg_subprocess(budget_s: float, threads: int):
    """cpu_leg in a fresh interpreter whose BLAS and OpenMP pools are held to
    `threads` threads (set before numpy loads)."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = str(threads)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-leg", "--cpu-seconds", str(budget_s)],
                       env=env, capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return None
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_reference(args, world, rank):
    """The oracle as the reference arm: W untimed steps, then exactly K timed
    steps, each a bounded sample of the layer-step (its first r of the 64
    query rows, r sized from one calibration step so that the K steps take
    about a minute)."""
    if rank != 0:
        return
    import synth
    wl = synth.llada_layer()
    e = wl.extra
    e.setdefault("w_vals", e["w"].values())
    e.setdefault("kc_vals", e["k_cache"].values())
    e.setdefault("vc_vals", e["v_cache"].values())
    e.setdefault("logit_vals", e["logits"].values())
    R = e["rows"].n_rows
    t0 = time.perf_counter()
    oracle_step(wl, R)                                  # calibration, untimed
    full_step_s = time.perf_counter() - t0
    per_row = full_step_s / R
    K = args.steps
    r = int(max(1, min(R, 60.0 / (K * per_row))))
    for _ in range(args.warmup):
        oracle_step(wl, r)
    t0 = time.perf_counter()
    done = sum(oracle_step(wl, r) for _ in range(K))
    dt = time.perf_counter() - t0
    value = done / dt
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "query-rows/s", "n_gpus": args.gpus,
        "steps": K, "warmup": args.warmup, "ms_per_step": 1e3 * dt / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": 1, "seq_len": 768, "rows_per_step": 64,
                   "rows_per_timed_sample": r,
                   "ms_per_step_is": f"the time of one {r}-row sample of the 64-row layer-step",
                   "full_64_row_step_ms": 1e3 * full_step_s},
        "cpu_baseline": {"value": value, "unit": "query-rows/s", "cores": cores, "kind": "oracle",
                         "rows_per_sample": r,
                         "sample": f"{K} layer-steps of the float64 numpy oracle, each over the first {r} of "
                                   f"the 64 query rows (the whole K-step run {dt:.1f} s); one untimed full "
                                   f"64-row step took {1e3 * full_step_s:.0f} ms"},
        "e2e": {"value": value, "unit": "query-rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU leg
# ---------------------------------------------------------------------------
def run_gpu(args, world, rank, local):
    import torch

    import kv_cache_attention_gb300 as fdl
    import synth
    from kv_cache_attention_gb300 import build as fdl_build

    torch.cuda.set_device(local)
    fdl_build.build()
    wl = synth.llada_layer(seed=1002)
    e, s, g = wl.extra, wl.shape, wl.geom
    Hh, hd, N, d = s.n_heads, s.head_dim, wl.max_seq, s.d_model
    rows = e["rows"]
    R = rows.n_rows
    Rw, ms, k, V = 32, e["max_search"], e["topk"], e["vocab"]
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    ctx = fdl.fdl_create(d, Hh, hd, s.rope_theta, 1, N, wl.max_views, g.page_size, g.n_pages, R, V, "bf16",
                         stream=stream)
    # The top-k runs on a second stream with a context of its own (one
    # context per stream): it needs only the layer's tracker and the
    # unmasking only the step's logits, so once the layer is done the two run
    # concurrently. (Measured: 68.8 us per step, against 70.0 with the two in
    # sequence and 73.7 with the unmasking on the second stream instead.)
    side_stream = torch.cuda.Stream()
    ctx_side = fdl.fdl_create(d, Hh, hd, s.rope_theta, 1, N, wl.max_views, g.page_size, g.n_pages, R, V, "bf16",
                              stream=side_stream)
    layer_done, side_done = torch.cuda.Event(), torch.cuda.Event()

    def bf(t):
        return torch.from_numpy(np.ascontiguousarray(t.data).view(np.int16)).view(torch.bfloat16)

    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    w_host, x_host, l_host = bf(e["w"]), bf(e["x"]), bf(e["logits"])
    kc_host, vc_host = bf(e["k_cache"]), bf(e["v_cache"])
    per_copy = (w_host.numel() + x_host.numel() + l_host.numel() + 2 * kc_host.numel()) * 2
    n_copies = max(2, int(np.ceil(4 * l2 / per_copy)))
    Ws = [w_host.cuda() for _ in range(n_copies)]
    Xs = [x_host.cuda() for _ in range(n_copies)]
    Ls = [l_host.cuda() for _ in range(n_copies)]
    KC = [kc_host.cuda() for _ in range(n_copies)]
    VC = [vc_host.cuda() for _ in range(n_copies)]
    i32 = lambda a: torch.as_tensor(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    row_seq, row_rope, row_cache, row_kind = (i32(rows.row_seq), i32(rows.row_rope_pos),
                                              i32(rows.row_cache_pos), i32(rows.row_kind))
    cu, kv_len, bt = i32(rows.cu_seqlens), i32([N]), i32(g.block_table)
    elig = torch.as_tensor(e["eligible"]).cuda()
    seq_len = i32([N])
    win_seq, win_pos = i32(np.zeros(Rw)), i32(e["window_pos"])
    q = torch.empty((R, Hh, hd), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((R, Hh), dtype=torch.float32, device="cuda")
    track = torch.zeros((1, N), dtype=torch.float32, device="cuda")
    # The step's results (decisions and tracked set) are views of one device
    # buffer, so the end-to-end loop reads them back with one copy.
    res_layout = [("conf", torch.float32, (Rw,)), ("arg", torch.int32, (Rw,)), ("com", torch.uint8, (Rw,)),
                  ("srows", torch.int32, (1, ms)), ("nsr", torch.int32, (1,)), ("idx", torch.int32, (1, k)),
                  ("cnt", torch.int32, (1,))]
    res_off, off = {}, 0
    for name, dt, shp in res_layout:
        res_off[name] = off
        off += (int(np.prod(shp)) * torch.empty((), dtype=dt).element_size() + 15) // 16 * 16
    res_buf = torch.zeros(off, dtype=torch.uint8, device="cuda")
    res = {name: res_buf[res_off[name]:res_off[name] + int(np.prod(shp)) * torch.empty((), dtype=dt).element_size()]
           .view(dt).view(shp) for name, dt, shp in res_layout}
    conf, arg, com, srows, nsr, idx, cnt = (res[n] for n in ("conf", "arg", "com", "srows", "nsr", "idx", "cnt"))
    launches_per_step = 6  # projection (weight stream + merge), attention + tracker sums, top-k, unmask

    def qkv_part(c, X=None):
        X = Xs[c] if X is None else X
        ctx.qkv_rope_cache_write(X, Ws[c], row_seq, row_rope, row_cache, bt, KC[c], VC[c], q)

    def rest_part(c, L=None):
        L = Ls[c] if L is None else L
        ctx.sched_attn(q, KC[c], VC[c], bt, cu, kv_len, row_kind, o, lse_out=lse, track_scores=track)
        # fork: the unmasking stays on the layer's stream (after the layer,
        # as it would wait for the LM head's logits after the last layer), the
        # top-k goes to the side stream; join before the next step
        layer_done.record(stream)
        ctx.unmask_verify(1, ms, logits=L, row_seq=win_seq, row_pos=win_pos, eps=e["eps"], force_progress=False,
                          conf=conf, argmax=arg, commit=com, search_rows=srows, n_search=nsr)
        side_stream.wait_event(layer_done)
        ctx_side.track_topk(track, elig, seq_len, k, idx, cnt)
        # the top-k has consumed this step's scores: reset them for the next
        # step's first layer here, on the side stream, beside the unmasking
        with torch.cuda.stream(side_stream):
            track.zero_()
        side_done.record(side_stream)
        stream.wait_event(side_done)

    def step(c, X=None, L=None):
        # the tracker accumulates over a step's layers and is zero before a
        # step's first layer: zeroed once before the first step, then by each
        # step after its top-k has read it
        qkv_part(c, X)
        rest_part(c, L)

    track.zero_()
    for i in range(args.warmup):
        step(i % n_copies)
    ctx.sync_status()
    ctx_side.sync_status()
    # The device-resident step is replayed from CUDA graphs (one per rotating
    # input copy) so host launch cost does not stand in for GPU time; the
    # graphs hold exactly the kernels a direct call launches. Nothing else is
    # put inside the step graph: event-record nodes between its kernels were
    # measured to add about 9 us per step.
    step_graphs = []
    for c in range(n_copies):
        g_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step, stream=stream):
            step(c)
        step_graphs.append(g_step)
    # The dominant kernel's launch duration: one graph holding the projection
    # once per rotating copy, replayed back to back right after the timed
    # steps, between CUDA events on the same stream.
    qkv_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(qkv_graph, stream=stream):
        for c in range(n_copies):
            qkv_part(c)
    K = args.steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nvml = Nvml(local)
    n_qkv = max(20, K // n_copies)
    q0e, q1e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # The nvidia-smi sampler runs from before a short untimed pre-roll (so
    # that it is live and the clocks have settled under load) through the
    # warm-ups, the timed steps and the roofline replays; NVML reads taken
    # right before and right after the timed steps bracket them closely even
    # when they last only a millisecond.
    with Clocks(local) as clk:
        clk.wait_live(5.0)
        pre_end, i = time.perf_counter() + 0.3, 0
        while time.perf_counter() < pre_end:
            for _ in range(50):
                step_graphs[i % n_copies].replay()
                i += 1
            torch.cuda.synchronize()
        for i in range(args.warmup):
            step_graphs[i % n_copies].replay()
        qkv_graph.replay()
        ctx.sync_status()
        ctx_side.sync_status()
        barrier(world)
        torch.cuda.synchronize()
        nv_before = nvml.read()
        t0.record(stream)
        for i in range(K):
            step_graphs[i % n_copies].replay()
        t1.record(stream)
        torch.cuda.synchronize()
        nv_after = nvml.read()
        barrier(world)
        ctx.sync_status()
        ctx_side.sync_status()
        q0e.record(stream)
        for i in range(n_qkv):
            qkv_graph.replay()
        q1e.record(stream)
        torch.cuda.synchronize()
    ms_total = t0.elapsed_time(t1)
    ms_total = max_over_ranks(ms_total, world)
    ms_step = ms_total / K
    value = whole_job_rate(R, K, ms_total, world)
    qkv_ms = [q0e.elapsed_time(q1e) / (n_qkv * n_copies)]
    qkv_timing = (f"CUDA events over {n_qkv * n_copies} back-to-back graph launches of the projection "
                  f"(rotating copies), right after the timed steps")

    # end to end: pinned host inputs in, step results out, every step. The
    # step's inputs (hidden rows and logits) sit in one pinned host buffer and
    # one device buffer, and its results in one device buffer, so each
    # direction is one copy.
    nx, nl = x_host.numel(), l_host.numel()
    in_pin = torch.empty(nx + nl, dtype=torch.bfloat16).pin_memory()
    in_pin[:nx].copy_(x_host.reshape(-1))
    in_pin[nx:].copy_(l_host.reshape(-1))
    in_dev = torch.empty_like(in_pin, device="cuda")
    xd, ld_ = in_dev[:nx].view(x_host.shape), in_dev[nx:].view(l_host.shape)
    out_pin = torch.empty_like(res_buf, device="cpu").pin_memory()
    K_e2e = min(K, 1000)
    h2d = in_pin.numel() * 2
    d2h = out_pin.numel()

    def e2e_step(c):
        in_dev.copy_(in_pin, non_blocking=True)
        step(c, X=xd, L=ld_)
        out_pin.copy_(res_buf, non_blocking=True)

    for i in range(args.warmup):
        e2e_step(i % n_copies)
    barrier(world)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(K_e2e):
        e2e_step(i % n_copies)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b), world)
    e2e_value = whole_job_rate(R, K_e2e, e2e_ms, world)

    if rank != 0:
        return
    hbm, tc, src = peaks()
    qkv_bytes = 3 * d * d * 2 + R * d * 2 + R * d * 2 + 2 * R * d * 2
    qkv_avg = statistics.mean(qkv_ms)
    achieved = qkv_bytes / (qkv_avg * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "query-rows/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": world, "seq_len": N, "rows_per_step": R,
                   "parallelism": f"replicas{world}", "launch": "one CUDA graph replay per step; top-k and unmasking concurrent on two streams",
                   "l2_hygiene": f"{n_copies} rotating copies of W/X/cache/logits "
                   f"({per_copy * n_copies / 1e9:.2f} GB > 4x L2 {l2 / 1e6:.0f} MB)"},
        "e2e": {"value": e2e_value, "unit": "query-rows/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * K,
        "roofline": {"kernel": "qkv_rope_cache_write", "bound": "hbm", "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "traffic": qkv_traffic(), "peak_source": src,
                     "algorithmic_bytes": qkv_bytes, "avg_launch_us": qkv_avg * 1e3,
                     "timing": qkv_timing},
        "clocks": clock_record(clk, nv_before, nv_after),
    }
    if not args.no_configs:
        # kernel fractions on the other configurations (ragged batch, one
        # layer of the 32-layer chain, Flash-Verify stress), a few seconds of
        # GPU time, so that they are recorded with the headline
        fv = synth.flash_verify()
        cfgs = config_results(("ragged", "chain", "flash_verify"), reps_scale=0.5, workloads={"flash_verify": fv})
        line["configs"] = {r.pop("config"): {k: v for k, v in r.items() if k != "peaks"} for r in cfgs}
    else:
        fv = None
    if not args.no_cpu_baseline:
        cpu_value, cpu_steps, cpu_dt = cpu_leg(wl, args.cpu_seconds)
        line["cpu_baseline"] = {"value": cpu_value, "unit": "query-rows/s", "cores": os.cpu_count(),
                                "threads": "numpy default (all cores for BLAS)", "kind": "oracle",
                                "sample": f"{cpu_steps} full layer-steps (64 rows) of the float64 numpy oracle "
                                          f"in {cpu_dt:.1f} s"}
        one = cpu_leg_subprocess(args.cpu_seconds, 1)
        if one:
            line["cpu_baseline"]["one_thread"] = {
                "value": one["value"], "unit": "query-rows/s", "threads": 1,
                "sample": f"{one['steps']} full layer-steps (64 rows) in {one['dt']:.1f} s, BLAS and OpenMP "
                          f"pools held to one thread"}
        if fv is not None:
            v, n, dt = flash_verify_oracle_sample(fv, args.cpu_seconds / 2)
            line["cpu_baseline"]["flash_verify_sample"] = {
                "value": v, "unit": "query-rows/s", "cores": os.cpu_count(),
                "sample": f"{n} repetitions in {dt:.1f} s of one sequence of the Flash-Verify stress layer-step "
                          f"(64 draft rows: projection, attention over 1536 keys with the tracker, top-32, eps "
                          f"unmasking of 32 rows over 126464 logits); a sample, not the 32-sequence step"}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# Per-configuration kernel measurements (--configs)
# ---------------------------------------------------------------------------
CONFIG_SECTIONS = ("ragged", "chain", "flash_verify", "lm_head", "refresh", "flash_step")


def run_configs(args):
    """Prints one JSON line per configuration of config_results."""
    sections = CONFIG_SECTIONS if args.configs == "all" else (args.configs,)
    for r in config_results(sections):
        print(json.dumps(r), flush=True)


def config_results(sections, reps_scale: float = 1.0, workloads=None):
    """Times each kernel of the path on the ragged batch, one layer of the
    32-layer chain and the Flash-Verify stress workload, and the fused LM
    head + unmasking over the LLaDA vocabulary: CUDA-graph replays of one
    call, µs per call, and algorithmic TFLOP/s or GB/s against the measured
    peaks. Then one layer's projection + attention over a whole scripted
    decode under each KV-cache refresh policy, against the sum of the
    per-kernel roofline floors, and whole denoising steps of a 32-layer
    LLaDA-8B-shaped model. Returns one dict per configuration."""
    import torch

    import kv_cache_attention_gb300 as fdl
    import synth
    from kv_cache_attention_gb300 import build as fdl_build

    fdl_build.build()
    hbm, tc, src = peaks()
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)

    def bf(t):
        return torch.from_numpy(np.ascontiguousarray(t.data).view(np.int16)).view(torch.bfloat16).cuda()

    def i32(a):
        return torch.as_tensor(np.ascontiguousarray(a, dtype=np.int32)).cuda()

    def timed(fns, reps):
        """Average µs of one call; fns rotate over input copies, one per graph."""
        reps = max(len(fns), int(reps * reps_scale))
        graphs = []
        for fn in fns:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            graphs.append(g)
        for i in range(3 * len(graphs)):
            graphs[i % len(graphs)].replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(reps):
            graphs[i % len(graphs)].replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps * 1e3

    def entry(us, flops=None, nbytes=None):
        e = {"us": round(us, 2)}
        if flops:
            e["tflops"] = round(flops / us * 1e-6, 1)
            e["frac_bf16_peak"] = round(flops / us * 1e-6 / tc, 3)
        if nbytes:
            e["gbs"] = round(nbytes / us * 1e-3, 1)
            e["frac_hbm"] = round(nbytes / us * 1e-3 / hbm, 3)
        return e

    def layer_kernels(name, wl, rows, x, w_copies, kc, vc, ctx, track_rows=True, search=None, reps=50):
        s, g = wl.shape, wl.geom
        d, Hh, hd = s.d_model, s.n_heads, s.head_dim
        R = rows.n_rows
        q = torch.empty((R, Hh, hd), dtype=torch.bfloat16, device="cuda")
        o = torch.empty_like(q)
        lse = torch.empty((R, Hh), dtype=torch.float32, device="cuda")
        track = torch.zeros((wl.batch, wl.max_seq), dtype=torch.float32, device="cuda") if track_rows else None
        rs, rp, rc, rk, cu = (i32(rows.row_seq), i32(rows.row_rope_pos), i32(rows.row_cache_pos),
                              i32(rows.row_kind), i32(rows.cu_seqlens))
        bt, kvl = i32(g.block_table), i32(wl.seq_len)
        out = {"rows": R}
        qkv_fns = [lambda W=W: ctx.qkv_rope_cache_write(x, W, rs, rp, rc, bt, kc, vc, q) for W in w_copies]
        qkv_fl = 2.0 * R * 3 * d * d
        qkv_by = 2.0 * (3 * d * d + R * d + 3 * R * d)
        out["qkv_rope_cache_write"] = entry(timed(qkv_fns, reps), qkv_fl, qkv_by)
        kw = {}
        n_keys = wl.seq_len.astype(np.int64).copy()
        if search is not None:
            kw = {"search_pos": i32(search[0]), "n_search": i32(search[1])}
            n_keys = n_keys + 2 * np.asarray(search[1], np.int64)
        rows_b = np.diff(rows.cu_seqlens).astype(np.int64)
        att_fl = 4.0 * d * float((rows_b * n_keys).sum())
        att_by = 2.0 * (2 * d * float(wl.seq_len.astype(np.int64).sum()) + 2 * R * d)
        att_fn = lambda: ctx.sched_attn(q, kc, vc, bt, cu, kvl, rk, o, lse_out=lse, track_scores=track, **kw)
        out["sched_attn"] = entry(timed([att_fn], reps), att_fl, att_by)
        return out

    results = []

    def want(name):
        return name in sections

    if want("ragged"):
        # ragged batch of 16 (paged cache, half full refresh)
        wl = synth.ragged_batch()
        e, s, g = wl.extra, wl.shape, wl.geom
        rows = e["rows"]
        ctx = fdl.fdl_create(s.d_model, s.n_heads, s.head_dim, s.rope_theta, wl.batch, wl.max_seq, 0, g.page_size,
                             g.n_pages, rows.n_rows, 16, "bf16", stream=stream)
        Ws = [bf(e["w"]), bf(e["w"])]
        res = layer_kernels("ragged_batch", wl, rows, bf(e["x"]), Ws, bf(e["k_cache"]), bf(e["v_cache"]), ctx, reps=20)
        results.append({"config": "ragged_batch_b16_p64", **res})
        ctx.close()
        del Ws

    if want("chain"):
        # one layer of the 32-layer chain: 8 sequences x (32 window + 32 tracked)
        wl = synth.layer_chain()
        e, s, g = wl.extra, wl.shape, wl.geom
        d = s.d_model
        rng = np.random.default_rng(7)
        per_seq = [synth.draft_rows(e["window_pos"], np.sort(rng.choice(e["prompt"], 32, replace=False)))
                   for _ in range(wl.batch)]
        rows = synth.build_rows(per_seq)
        ctx = fdl.fdl_create(d, s.n_heads, s.head_dim, s.rope_theta, wl.batch, wl.max_seq, 0, g.page_size,
                             g.n_pages, rows.n_rows, 16, "bf16", stream=stream)
        n_slots = g.n_pages * g.page_size
        kc = torch.randn((n_slots, d), device="cuda").mul_(0.02 * d ** 0.5).bfloat16()
        vc = torch.randn((n_slots, d), device="cuda").mul_(0.02 * d ** 0.5).bfloat16()
        Ws = [bf(synth.chain_weight(e["seed"], l, d)) for l in range(2)]
        x = bf(synth.chain_hidden(e["seed"], 1, 0, rows.n_rows, d))
        res = layer_kernels("layer_chain", wl, rows, x, Ws, kc, vc, ctx)
        results.append({"config": "layer_chain_b8_one_layer", **res})
        ctx.close()
        del Ws, kc, vc

    if want("flash_verify"):
        # Flash-Verify stress: draft forward, eps unmasking, verify acceptance, top-k
        wl = (workloads or {}).get("flash_verify") or synth.flash_verify()
        e, s, g = wl.extra, wl.shape, wl.geom
        rows = e["rows"]
        B, ms, V = wl.batch, e["max_search"], e["vocab"]
        ctx = fdl.fdl_create(s.d_model, s.n_heads, s.head_dim, s.rope_theta, B, wl.max_seq, wl.max_views,
                             g.page_size, g.n_pages, rows.n_rows, V, "bf16", stream=stream)
        Ws = [bf(e["w"]), bf(e["w"])]
        res = layer_kernels("flash_verify", wl, rows, bf(e["x"]), Ws, bf(e["k_cache"]), bf(e["v_cache"]), ctx)
        del Ws
        logits = bf(e["logits"])
        Rw = logits.shape[0]
        wseq, wpos = i32(e["window_row_seq"]), i32(e["window_row_pos"])
        conf = torch.empty(Rw, dtype=torch.float32, device="cuda")
        arg = torch.empty(Rw, dtype=torch.int32, device="cuda")
        com = torch.empty(Rw, dtype=torch.uint8, device="cuda")
        srows = torch.empty((B, ms), dtype=torch.int32, device="cuda")
        nsr = torch.empty((B,), dtype=torch.int32, device="cuda")
        um = lambda: ctx.unmask_verify(B, ms, logits=logits, row_seq=wseq, row_pos=wpos, eps=e["eps"],
                                       force_progress=False, conf=conf, argmax=arg, commit=com, search_rows=srows,
                                       n_search=nsr)
        res["unmask (eps rule)"] = entry(timed([um], 50), None, 2.0 * Rw * V)
        um()
        torch.cuda.synchronize()
        ns_host = nsr.cpu().numpy()
        mask_logits = torch.empty((B * ms, V), dtype=torch.bfloat16, device="cuda")
        mask_logits.copy_(logits[: B * ms])
        draft = arg[: B * ms].clone()
        acc = torch.empty(B * ms, dtype=torch.uint8, device="cuda")
        nacc = torch.empty(B, dtype=torch.int32, device="cuda")
        mconf = torch.empty(B * ms, dtype=torch.float32, device="cuda")
        marg = torch.empty(B * ms, dtype=torch.int32, device="cuda")
        vf = lambda: ctx.unmask_verify(B, ms, mask_logits=mask_logits, draft_tok=draft, gamma=e["gamma"], n_search=nsr,
                                       accept=acc, n_accept=nacc, mask_conf=mconf, mask_argmax=marg)
        res["verify (acceptance)"] = entry(timed([vf], 50), None, 2.0 * float(ns_host.sum()) * V)
        res["verify (acceptance)"]["valid_rows"] = int(ns_host.sum())
        track = torch.rand((B, wl.max_seq), device="cuda")
        elig, sl = torch.as_tensor(e["eligible"]).cuda(), i32(wl.seq_len)
        idx = torch.empty((B, 32), dtype=torch.int32, device="cuda")
        cnt = torch.empty((B,), dtype=torch.int32, device="cuda")
        res["track_topk"] = entry(timed([lambda: ctx.track_topk(track, elig, sl, 32, idx, cnt)], 200))
        ctx.sync_status()
        results.append({"config": "flash_verify_b32", **res})
        ctx.close()

    if want("lm_head"):
        # fused LM head + eps unmasking (the step after the layers): the LLaDA
        # vocabulary and width against the 32 window rows; the weight (1.04 GB,
        # two seeded copies) is the algorithmic traffic
        d, V, Rw = 4096, 126464, 32
        ctx = fdl.fdl_create(d, 32, 128, 5e5, 1, 64, 0, 64, 1, 64, V, "bf16", stream=stream)
        gen = torch.Generator(device="cuda").manual_seed(1009)
        W_lm = [(torch.randn((V, d), device="cuda", generator=gen) * 0.02).bfloat16() for _ in range(2)]
        hid = torch.randn((Rw, d), device="cuda", generator=gen).bfloat16()
        rs, rp = i32(np.zeros(Rw)), i32(512 + np.arange(Rw))
        conf = torch.empty(Rw, dtype=torch.float32, device="cuda")
        arg = torch.empty(Rw, dtype=torch.int32, device="cuda")
        com = torch.empty(Rw, dtype=torch.uint8, device="cuda")
        srows = torch.empty((1, 16), dtype=torch.int32, device="cuda")
        nsr = torch.empty((1,), dtype=torch.int32, device="cuda")
        lm = [lambda W=W: ctx.lm_head_unmask(hid, W, 1, 16, row_seq=rs, row_pos=rp, eps=0.9, force_progress=True,
                                             conf=conf, argmax=arg, commit=com, search_rows=srows, n_search=nsr)
              for W in W_lm]
        res = {"lm_head_unmask": entry(timed(lm, 50), 2.0 * Rw * V * d, 2.0 * (V * d + Rw * d))}
        ctx.sync_status()
        results.append({"config": "lm_head_llada_vocab_w32", "rows": Rw, **res})
        ctx.close()
        # the Flash-Verify stress scale: 32 sequences x 32 window rows, and the
        # verify side's 32 x 16 mask views (tensor-bound: about R FLOP per byte)
        B5, W5, M5 = 32, 32, 16
        ctx = fdl.fdl_create(d, 32, 128, 5e5, B5, 64, 0, 64, 1, B5 * W5, V, "bf16", stream=stream)
        R5 = B5 * W5
        hid5 = torch.randn((R5, d), device="cuda", generator=gen).bfloat16()
        rs5, rp5 = i32(np.repeat(np.arange(B5), W5)), i32(np.tile(512 + np.arange(W5), B5))
        conf5 = torch.empty(R5, dtype=torch.float32, device="cuda")
        arg5 = torch.empty(R5, dtype=torch.int32, device="cuda")
        com5 = torch.empty(R5, dtype=torch.uint8, device="cuda")
        sr5 = torch.empty((B5, M5), dtype=torch.int32, device="cuda")
        ns5 = torch.empty((B5,), dtype=torch.int32, device="cuda")
        lm5 = [lambda W=W: ctx.lm_head_unmask(hid5, W, B5, M5, row_seq=rs5, row_pos=rp5, eps=0.9,
                                              force_progress=True, conf=conf5, argmax=arg5, commit=com5,
                                              search_rows=sr5, n_search=ns5) for W in W_lm]
        res5 = {"lm_head_unmask": entry(timed(lm5, 10), 2.0 * R5 * V * d, 2.0 * (V * d + R5 * d))}
        Rv = B5 * M5
        nsv = i32(np.full(B5, M5))
        drv = torch.zeros(Rv, dtype=torch.int32, device="cuda")
        accv = torch.empty(Rv, dtype=torch.uint8, device="cuda")
        nav = torch.empty(B5, dtype=torch.int32, device="cuda")
        mcv = torch.empty(Rv, dtype=torch.float32, device="cuda")
        mav = torch.empty(Rv, dtype=torch.int32, device="cuda")
        lmv = [lambda W=W: ctx.lm_head_verify(hid5[:Rv], W, B5, M5, n_search=nsv, draft_tok=drv, gamma=0.8,
                                              accept=accv, n_accept=nav, mask_conf=mcv, mask_argmax=mav)
               for W in W_lm]
        res5["lm_head_verify (512 mask views)"] = entry(timed(lmv, 10), 2.0 * Rv * V * d, 2.0 * (V * d + Rv * d))
        ctx.sync_status()
        results.append({"config": "lm_head_llada_vocab_b32_w32", "rows": R5, **res5})
        ctx.close()
        del W_lm

    if want("refresh"):
        # KV-cache refresh policies over one scripted decode of one layer: LLaDA
        # layer shape, batch 1, prompt 512 + gen 256, block (window) 32, two
        # positions unmasked per step (128 steps). Each step is the projection
        # and the attention of the rows the policy chooses, one graph per step,
        # replayed in order; the two weight copies alternate between steps
        # (200 MB > L2).
        d, Hh, hd, P, G, blk = 4096, 32, 128, 512, 256, 32
        N = P + G
        ctx = fdl.fdl_create(d, Hh, hd, 5e5, 1, N, 0, N, 1, N, 16, "bf16", stream=stream)
        gen = torch.Generator(device="cuda").manual_seed(1011)
        Ws = [(torch.randn((3 * d, d), device="cuda", generator=gen) * 0.02).bfloat16() for _ in range(2)]
        X = torch.randn((N, d), device="cuda", generator=gen).bfloat16()
        kc = torch.zeros((N, d), dtype=torch.bfloat16, device="cuda")
        vc = torch.zeros_like(kc)
        q = torch.empty((N, Hh, hd), dtype=torch.bfloat16, device="cuda")
        o = torch.empty_like(q)
        lse = torch.empty((N, Hh), dtype=torch.float32, device="cuda")
        track = torch.zeros((1, N), dtype=torch.float32, device="cuda")
        bt, kvl = i32([[0]]), i32([N])
        names = {fdl.FDL_REFRESH_FULL: "full_recompute", fdl.FDL_REFRESH_PREFIX: "fastdllm_prefix_cache",
                 fdl.FDL_REFRESH_DUAL: "fastdllm_dual_cache", fdl.FDL_REFRESH_FREECACHE: "freecache",
                 fdl.FDL_REFRESH_FLASH_DRAFT: "flash_dllm_draft_forward_only"}
        for policy, name in names.items():
            rng = np.random.default_rng([1011, policy])
            masked = np.zeros((1, N), np.uint8)
            masked[0, P:] = 1
            state = np.full(1, -1, np.int32)
            steps = []
            while masked.any():
                tracked = n_tracked = None
                if policy == fdl.FDL_REFRESH_FLASH_DRAFT:
                    tracked = rng.permutation(np.nonzero(masked[0] == 0)[0])[:32].astype(np.int32)[None]
                    n_tracked = np.array([tracked.shape[1]], np.int32)
                rows = fdl.fdl_refresh_rows(policy, [P], [N], masked, blk, state, tracked, n_tracked)
                steps.append(rows)
                masked[0, synth.trace_unmask(rng, rows.row_rope_pos[rows.row_kind == 1], 2, 2)] = 0
            graphs, keep, n_rows, floor_us = [], [], 0, 0.0
            for t, rows in enumerate(steps):
                R = rows.n_rows
                args_t = (i32(rows.row_seq), i32(rows.row_rope_pos), i32(rows.row_kind), i32(rows.cu_seqlens))
                keep.append(args_t)
                rs, rp, rk, cu = args_t
                tr = track if policy == fdl.FDL_REFRESH_FLASH_DRAFT else None
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    ctx.qkv_rope_cache_write(X[:R], Ws[t % 2], rs, rp, rp, bt, kc, vc, q[:R])
                    ctx.sched_attn(q[:R], kc, vc, bt, cu, kvl, rk, o[:R], lse_out=lse[:R], track_scores=tr)
                graphs.append(g)
                n_rows += R
                qkv_fl, qkv_by = 2.0 * R * 3 * d * d, 2.0 * (3 * d * d + 4 * R * d)
                att_fl, att_by = 4.0 * d * R * N, 2.0 * (2 * d * N + 2 * R * d)
                floor_us += max(qkv_by / hbm * 1e-3, qkv_fl / tc * 1e-6) + max(att_by / hbm * 1e-3, att_fl / tc * 1e-6)
            for _ in range(2):
                for g in graphs:
                    g.replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            passes = 5
            a.record(stream)
            for _ in range(passes):
                for g in graphs:
                    g.replay()
            b.record(stream)
            torch.cuda.synchronize()
            ctx.sync_status()
            us = a.elapsed_time(b) / passes * 1e3
            results.append({"config": f"refresh_{name}_llada_b1_p512_g256_blk32", "steps": len(steps),
                            "rows": n_rows, "us_per_decode_layer": round(us, 1),
                            "us_per_step": round(us / len(steps), 2),
                            "rows_per_s": round(n_rows / us * 1e6, 1),
                            "roofline_floor_us": round(floor_us, 1), "frac_roofline": round(floor_us / us, 3)})
            del graphs, keep
        ctx.close()
        del Ws

    if want("flash_step"):
        # Whole denoising steps of a LLaDA-8B-shaped model with random weights
        # (32 layers, d_model 4096, 32 heads, SwiGLU 12288, vocab 126464; 16 GB
        # of bf16 weights): batch 1, prompt 512 + gen 256, window 32, 32 tracked,
        # up to 16 search tokens. The first step is the full forward over all 768
        # positions; the steady steps run a draft forward over 64 rows, the LM
        # head, a verify forward and the acceptance. Wall time per call (the step
        # reads its decisions back three times). The floor counts the weights
        # read by both forwards and both LM-head passes, and each forward's cache
        # read, at the measured HBM rate.
        L, d, F, V, Hh, hd = 32, 4096, 12288, 126464, 32, 128
        P, G, Wn, BTk, MSk = 512, 256, 32, 32, 16
        N = P + G
        ctx = fdl.fdl_create(d, Hh, hd, 5e5, 1, N, 2 * MSk, N + 2 * MSk, 1, N, V, "bf16", stream=stream)
        gen = torch.Generator(device="cuda").manual_seed(1017)

        def rnd(*shape, std=0.02):
            return (torch.randn(shape, device="cuda", generator=gen, dtype=torch.bfloat16) * std)

        ones = torch.ones(d, dtype=torch.bfloat16, device="cuda")
        model = dict(ffn=F, eps=1e-5, embed=rnd(V, d, std=1.0), g_final=ones,
                     layers=[dict(g_attn=ones, w_qkv=rnd(3 * d, d), w_o=rnd(d, d), g_mlp=ones, w_gu=rnd(2 * F, d),
                                  w_down=rnd(d, F)) for _ in range(L)])
        w_lm = rnd(V, d)
        kcs = [torch.zeros((N + 2 * MSk, d), dtype=torch.bfloat16, device="cuda") for _ in range(L)]
        vcs = [torch.zeros_like(kcs[0]) for _ in range(L)]
        params = dict(window=Wn, track_budget=BTk, max_search=MSk, eps=0.9, gamma=0.8, force_progress=True,
                      mask_id=V - 1, max_views=2 * MSk)
        rng = np.random.default_rng(1017)
        toks = np.full((1, N), V - 1, np.int32)
        toks[0, :P] = rng.integers(0, V - 1, P)
        msk = np.zeros((1, N), np.uint8)
        msk[0, P:] = 1
        seqs = dict(prompt_len=np.array([P], np.int32), seq_len=np.array([N], np.int32), tokens=toks, masked=msk,
                    tracked=np.full((1, BTk), -1, np.int32), n_tracked=np.zeros(1, np.int32),
                    state=np.full(1, -1, np.int32))
        ws = torch.empty(ctx.flash_workspace_bytes(F, params, 1, N), dtype=torch.uint8, device="cuda")
        bt = i32([[0]])
        times, decoded, rows = [], [], []
        for t in range(10):
            before = int(seqs["masked"].sum())
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            rec = ctx.flash_step(model, w_lm, kcs, vcs, bt, params, seqs, ws, trace=False)
            torch.cuda.synchronize()
            times.append((time.perf_counter() - t0) * 1e3)
            decoded.append(before - int(seqs["masked"].sum()))
        ctx.sync_status()
        layer_w = 2.0 * (3 * d * d + d * d + 2 * F * d + F * d)
        fwd_bytes = L * layer_w + L * 2.0 * 2 * d * N            # weights + one K and V read of the cache
        floor_ms = (2 * fwd_bytes + 2 * 2.0 * V * d) / (hbm * 1e9) * 1e3
        steady = times[2:]
        results.append({"config": "flash_step_llada8b_shape_32_layers_b1_p512_g256", "first_step_ms": round(times[0], 2),
                        "steady_step_ms": round(statistics.median(steady), 2),
                        "steady_steps_timed": len(steady), "tokens_decoded_per_step": decoded,
                        "weights_gb": round((L * layer_w + 2 * 2.0 * V * d) / 1e9, 2),
                        "steady_floor_ms": round(floor_ms, 2),
                        "frac_hbm_floor": round(floor_ms / statistics.median(steady), 3),
                        "note": "random weights: confidences sit near 1/vocab, so each step commits its one forced "
                                "token and the verify forward runs on 16 search tokens",
                        "timing": "wall clock of each fdl_flash_step call (direct launches; the step reads its "
                                  "decisions back three times), median of the steady steps"})
        ctx.close()
        del model, w_lm, kcs, vcs
    for r in results:
        r.setdefault("timing", "CUDA-graph replays of one call on the dedicated stream; algorithmic work")
        r["peaks"] = {"hbm_gbs": hbm, "bf16_tflops": tc, "source": src}
    torch.cuda.synchronize()
    return results


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="fdl", choices=["fdl", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="leave the other configurations' kernel fractions out of the headline line")
    ap.add_argument("--cpu-leg", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--configs", nargs="?", const="all", default=None, metavar="SECTION",
                    help="time each kernel on the ragged-batch, 32-layer-chain and Flash-Verify workloads, "
                         "the fused LM head, one layer's decode under each KV-cache refresh policy and whole "
                         "denoising steps of a 32-layer model (all, or one of ragged, chain, flash_verify, "
                         "lm_head, refresh, flash_step)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.cpu_leg:
        # the oracle on the headline workload only (run in a subprocess with
        # limited threads by cpu_leg_subprocess)
        import synth
        v, n, dt = cpu_leg(synth.llada_layer(), args.cpu_seconds)
        print(json.dumps({"value": v, "steps": n, "dt": dt}), flush=True)
        return
    if args.configs:
        if args.configs != "all" and args.configs not in CONFIG_SECTIONS:
            raise SystemExit(f"unknown configuration {args.configs!r}; one of {', '.join(CONFIG_SECTIONS)}")
        run_configs(args)
        return
    world, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_gpu(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
