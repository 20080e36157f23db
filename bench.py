"""Benchmark: causal attention forward + backward at 32K tokens on GB300.

One step = the whole attention path on one batch: attn_fwd, then the three
stages of attn_bwd (D preprocess, dQ, dK/dV) -- exactly the work of
attn_fwd + attn_bwd -- on device-resident inputs, timed with CUDA events on
the launching stream (events between the stages give per-kernel times).
Inputs (Q 384 MiB, K 384 MiB, V/dO 256 MiB) exceed the 129 MB L2, so no flush
is needed between steps.

Reported: TFLOP/s of the algorithmic work (visible causal pairs only:
fwd 2*N*(dqk+dv), bwd 2*N*(3*dqk+2*dv)), ms per step, % of the dense BF16
tensor peak, an end-to-end figure through host buffers, the roofline of the
dominant kernel, and the FP64 oracle on a bounded sample as the CPU baseline.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
Multi-GPU (torchrun): every rank runs its own copy of the workload (weak
scaling, no collective in the data path); time = max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "b1_h32_s32768_d192_128"
METRIC = "causal attn fwd+bwd ms & TFLOP/s at 32K seq, % of GB300 BF16 tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = {"fwd": "fwd.cu", "dq": "bwd_dq.cu", "dkdv": "bwd_dkdv.cu", "pre": "small.cu"}


def visible_pairs(w, lengths=None):
    """Sum over sequences and query heads of visible (query, key) pairs."""
    lens = lengths if lengths is not None else w.lengths()
    n = 0
    for L in lens:
        if w.window[0] >= 0:
            W = w.window[0] + 1
            n += sum(min(i + 1, W) for i in range(L))
        else:
            n += L * (L + 1) // 2
    return n * w.heads_q


def score_blocks(w, lengths=None):
    """Visible 128-query x 128-key blocks over sequences and query heads
    (causal, with the workload's left window): one 32 KiB dS block each on
    the dS path of the backward."""
    lens = lengths if lengths is not None else w.lengths()
    n = 0
    for L in lens:
        for qt in range((L + 127) // 128):
            i0, i1 = 128 * qt, min(128 * qt + 127, L - 1)
            j0 = max(0, i0 - w.window[0]) if w.window[0] >= 0 else 0
            n += i1 // 128 - j0 // 128 + 1
    return n * w.heads_q


def flops(w, lengths=None):
    nv = visible_pairs(w, lengths)
    fwd = 2 * nv * (w.d_qk + w.d_v)
    bwd = 2 * nv * (3 * w.d_qk + 2 * w.d_v)
    # per-kernel attribution of the algorithmic work (sums to fwd + bwd):
    # head dims <= 256: dK/dV kernel S, dP, dV, dK; dQ kernel dQ (its S/dP
    # recompute is not credited).  On the materialising path (head dims 256
    # and 512 in these workloads) the dq stage runs the scores kernel (S, dP)
    # and the dQ GEMM, the dkdv stage the dV and dK GEMMs.
    if w.d_qk >= 256:
        kern = {"fwd": fwd, "dq": 2 * nv * (2 * w.d_qk + w.d_v), "dkdv": 2 * nv * (w.d_qk + w.d_v)}
    else:
        kern = {"fwd": fwd, "dkdv": 2 * nv * (2 * w.d_qk + 2 * w.d_v), "dq": 2 * nv * w.d_qk}
    return {"fwd": fwd, "bwd": bwd, "total": fwd + bwd, "n_visible": nv, "kernel": kern}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def file_hash(name):
    p = os.path.join(ROOT, "bwd_tcgen05_tmem_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def load_profile_value(fname, kernel):
    """A per-kernel figure from a committed ncu summary (`kernel value hash`
    lines; a stage may have one line per source file, e.g. the dq stage of each
    backward path), or None if there is none for the kernel's current source."""
    path = os.path.join(ROOT, "profiles", fname)
    if not os.path.exists(path):
        return None
    want = file_hash(KERNEL_SOURCES[kernel.split("+")[0]])
    with open(path) as f:
        for line in f:
            parts = line.split()
            if (len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel and
                    parts[2] == want):
                return float(parts[1])
    return None


def load_traffic(kernel):
    """DRAM bytes per full-size launch of `kernel` (ncu, scaled from the 8K case)."""
    return load_profile_value("dram_traffic.txt", kernel)


def load_tensor_pipe(kernel):
    """Tensor-pipe active % of `kernel` (ncu sm__pipe_tensor_cycles_active, 8K case)."""
    return load_profile_value("tensor_pipe.txt", kernel)


def cpu_model():
    """Host CPU model string (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def spread(xs):
    """Median and spread of a list of per-step times."""
    ys = sorted(xs)
    n = len(ys)
    q = lambda f: ys[min(n - 1, max(0, int(round(f * (n - 1)))))]  # noqa: E731
    return {"median": statistics.median(ys), "min": ys[0], "max": ys[-1],
            "p25": q(0.25), "p75": q(0.75), "n": n}


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.out.close()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    p = [x.strip() for x in line.split(",")]
                    if len(p) >= 9:
                        rows.append(p)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_median": statistics.median([num(r[3]) for r in rows
                                                     if num(r[3]) is not None] or [0])}


def cpu_baseline(w, seconds_target=15.0):
    """The FP64 oracle, as it stands, on a bounded sample of the workload: the
    last `rows` query rows of every head against every key (bottom-right
    causal), forward + backward.  Returns TFLOP/s of the sample's algorithmic
    work.  The oracle runs one thread per (sequence, head) work item."""
    import oracle
    from bwd_tcgen05_tmem_gb300 import synth
    S = w.seqlen
    ncpu = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    nthreads = min(ncpu, w.heads_q)
    q = synth.normal((1, S, w.heads_q, w.d_qk), synth.SEED_Q, w.torch_dtype)[0]
    k = synth.normal((1, S, w.heads_kv, w.d_qk), synth.SEED_K, w.torch_dtype)[0]
    v = synth.normal((1, S, w.heads_kv, w.d_v), synth.SEED_V, w.torch_dtype)[0]
    do = synth.normal((1, S, w.heads_q, w.d_v), synth.SEED_DO, w.torch_dtype)[0]
    k, v = (t.double().numpy() for t in (k, v))

    def run(rows):
        qs = q[S - rows:].double().numpy()
        dos = do[S - rows:].double().numpy()
        t0 = time.perf_counter()
        oracle.fwd(qs, k, v, [0, rows], [0, S], scale=w.scale, causal=True, bottom_right=True,
                   nthreads=nthreads)
        oracle.bwd(qs, k, v, dos, [0, rows], [0, S], scale=w.scale, causal=True,
                   bottom_right=True, nthreads=nthreads)
        dt = time.perf_counter() - t0
        nv = w.heads_q * sum(S - rows + i + 1 for i in range(rows))
        return dt, 2 * nv * (w.d_qk + w.d_v) + 2 * nv * (3 * w.d_qk + 2 * w.d_v)

    rows = 4
    dt, f = run(rows)
    while dt < 1.0 and rows < S:
        rows = min(S, rows * 4)
        dt, f = run(rows)
    if dt < seconds_target and rows < S:
        rows = min(S, max(rows, int(rows * seconds_target / dt)))
        dt, f = run(rows)
    return {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": nthreads,
            "kind": "oracle", "seconds": round(dt, 2), "cpu_model": cpu_model(),
            "host_cores": ncpu,
            "sample": f"FP64 oracle fwd+bwd of the last {rows} query rows of all "
                      f"{w.heads_q} heads (bottom-right causal against all {S} keys), "
                      f"{nthreads} threads of {ncpu} host cores"}


def max_over_ranks(value, device=None):
    """The slowest rank's value (the job's time); a no-op on one process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_rank, ms, world):
    """Whole-job throughput: every rank processed `flops_per_rank` in at most `ms`."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    samples = []
    for i in range(args.warmup + args.steps):
        cb = cpu_baseline(w, seconds_target=5.0)
        if i >= args.warmup:
            samples.append(cb)
    val = statistics.median(s["value"] for s in samples)
    fl = flops(w)
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": fl["total"] / (val * 1e12) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "seq_len": w.seqlen,
                   "heads": w.heads_q, "d_qk": w.d_qk, "d_v": w.d_v, "causal": True},
        "cpu_baseline": {**samples[-1], "value": val},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "note": "the reference arm is the FP64 CPU oracle timed on a bounded sample; "
                "ms_per_step is extrapolated to the whole workload",
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cp", action="store_true")
    ap.add_argument("--bwd-ds", default="auto", choices=["auto", "ds", "recompute"],
                    help="backward path at head dims 128/192 (attn_params_t.bwd_ds)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    from bwd_tcgen05_tmem_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
        return

    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    from bwd_tcgen05_tmem_gb300 import attn

    peaks0, peak_src0 = load_peaks()
    inp = synth.make_inputs(w)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "dout"))
    kw = dict(causal=True, scale=w.scale, window=w.window)
    if w.is_thd:  # packed documents: [tokens, heads, d], LSE [heads, tokens]
        cu = inp["cu_seqlens"].to(dev)
        kw.update(cu_seqlens_q=cu, cu_seqlens_k=cu, max_seqlen_q=inp["max_seqlen"],
                  max_seqlen_k=inp["max_seqlen"])
        fl = flops(w, (inp["cu_seqlens"][1:] - inp["cu_seqlens"][:-1]).tolist())
        lse = torch.empty((w.heads_q, q.shape[0]), dtype=torch.float32, device=dev)
    else:
        fl = flops(w)
        lse = torch.empty((q.shape[0], w.heads_q, q.shape[1]), dtype=torch.float32, device=dev)
    o = torch.empty((*q.shape[:-1], w.d_v), dtype=q.dtype, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fws = torch.empty(attn.workspace_size("fwd", q, k, v, **kw), dtype=torch.uint8, device=dev)
    bkw = dict(kw, bwd_ds={"auto": 0, "ds": 1, "recompute": -1}[args.bwd_ds])
    bws = torch.empty(attn.workspace_size("bwd", q, k, v, **bkw), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    # the stage order of attn_bwd: on the dS path the dK/dV kernel writes the
    # dS blocks that the dQ GEMM then reads
    bwd_path = attn.bwd_path(q, k, v, **bkw)
    if bwd_path == attn.BWD_DS:
        KERNEL_SOURCES["dq"] = "bwd_dq_ds.cu"
        stages = ("fwd", "pre", "dkdv", "dq")
    else:
        stages = ("fwd", "pre", "dq", "dkdv")
    api_stages = tuple({"pre": "preprocess"}.get(st, st) for st in stages[1:])

    def step(ev=None):
        n = 0
        if ev:
            ev[0].record(stream)
        attn.fwd(q, k, v, out=o, lse=lse, workspace=fws, **kw)
        n += attn.last_launch_count()
        for i, st in enumerate(api_stages):
            if ev:
                ev[i + 1].record(stream)
            attn.bwd(q, k, v, o, do, lse, dq=dq, dk=dk, dv=dv, workspace=bws, stage=st, **bkw)
            n += attn.last_launch_count()
        if ev:
            ev[4].record(stream)
        return n

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    attn.query_status(bws)
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    launches = 0
    with ClockSampler(local) as clk:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for s in range(args.steps):
            launches += step(events[s])
        t1.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    attn.query_status(bws)
    total_ms = t0.elapsed_time(t1)
    per_kernel = {st: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in events)
                  for i, st in enumerate(stages)}
    step_spread = spread([e[0].elapsed_time(e[4]) for e in events])
    kernel_spread = {st: spread([e[i].elapsed_time(e[i + 1]) for e in events])
                     for i, st in enumerate(stages)}
    ms = total_ms / args.steps
    ms = max_over_ranks(ms, dev)
    clocks = clk.summary()

    # ---- end to end through host buffers (pinned), copies inside the timed region.
    # Every step runs attn_fwd_bwd_host_stages of the C ABI in its three stages:
    # upload the step's inputs from pinned host memory into a device arena,
    # forward + backward there, download all outputs (O, LSE, dQ, dK, dV) into
    # host memory.  Uploads, compute and downloads have a stream each, ordered
    # by events, with two arenas: step s+1 uploads and step s-1 downloads while
    # step s computes, and the compute of consecutive steps stays in order.
    host_in = [t.cpu().pin_memory() for t in (q, k, v, do)]
    outs0 = (o, lse, dq, dk, dv)
    host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs0]
                for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    hkw = dict(bkw)
    if w.is_thd:  # host metadata for the host-buffer call, pinned like the tensors (a
        # copy from pageable memory would hold the host until its stream drains)
        cu_h = inp["cu_seqlens"].pin_memory()
        hkw.update(cu_seqlens_q=cu_h, cu_seqlens_k=cu_h)
    h_o, h_lse, h_dq, h_dk, h_dv = host_out[0]
    arena_bytes = attn.host_arena_size(*host_in, h_o, h_dq, h_dk, h_dv, **hkw)
    arenas = [torch.empty(arena_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    up_s, comp_s, down_s = (torch.cuda.Stream(device=dev) for _ in range(3))

    def e2e_run(n, spans=None):
        # spans: per step and stage (upload, compute, download) a pair of
        # timing events around the stage, to see where a step waits
        cur = torch.cuda.current_stream()
        for st_ in (up_s, comp_s, down_s):
            st_.wait_stream(cur)
        ev = [[torch.cuda.Event() for _ in range(3)] for _ in range(n)]  # up, compute, down
        for s_ in range(n):
            a_ = s_ % 2
            args = (*host_in, *host_out[a_], arenas[a_])
            for i_, (st_, stage) in enumerate(((up_s, attn.HOST_UPLOAD), (comp_s, attn.HOST_COMPUTE),
                                               (down_s, attn.HOST_DOWNLOAD))):
                if i_ == 0 and s_ >= 2:  # arena a_: step s_-2 has read its inputs
                    up_s.wait_event(ev[s_ - 2][1])
                if i_ == 1:
                    comp_s.wait_event(ev[s_][0])
                    if s_ >= 2:  # and its outputs are downloaded
                        comp_s.wait_event(ev[s_ - 2][2])
                if i_ == 2:
                    down_s.wait_event(ev[s_][1])
                if spans:
                    spans[s_][i_][0].record(st_)
                attn.fwd_bwd_host(*args, stream=st_, stages=stage, **hkw)
                if spans:
                    spans[s_][i_][1].record(st_)
                ev[s_][i_].record(st_)
        for st_ in (up_s, comp_s, down_s):
            cur.wait_stream(st_)

    # a fixed 16 steps (whatever --steps is), so that the unoverlapped first
    # upload and last download (about 7 ms each at the host link's rate) weigh
    # under 1 ms per step of a 32K step
    e2e_steps = 16
    e2e_run(2)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    spans = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(3)]
             for _ in range(e2e_steps)]
    e0.record(stream)
    e2e_run(e2e_steps, spans)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    # mean stage durations, and the mean gap between consecutive compute stages
    stage_ms = {name: statistics.mean(sp[i_][0].elapsed_time(sp[i_][1]) for sp in spans)
                for i_, name in enumerate(("upload", "compute", "download"))}
    stage_ms["compute_gap"] = (statistics.mean(spans[s_ - 1][1][1].elapsed_time(spans[s_][1][0])
                                               for s_ in range(1, e2e_steps)))
    # the timed region around the compute stages: before the first one starts
    # (its upload), from its start to the last one's end (per step), and after
    # that (the last download)
    stage_ms["lead"] = e0.elapsed_time(spans[0][1][0])
    stage_ms["compute_span_per_step"] = (spans[0][1][0].elapsed_time(spans[-1][1][1]) /
                                         e2e_steps)
    stage_ms["tail"] = spans[-1][1][1].elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, dev)
    for a_ in arenas:  # device-detected problems: forward, then backward status word
        attn.query_status(a_)
        attn.query_status(a_[256:])

    # the same host copies alone (no kernels): the host link's rate, each
    # direction on its own and both at once, to read the e2e figure against
    del arenas
    dev_in = [[torch.empty_like(t) for t in (q, k, v, do)]]
    dev_out = [[torch.empty_like(t) for t in outs0]]
    up_st, down_st = up_s, down_s

    def copy_run(up, down, n=3):
        cur = torch.cuda.current_stream()
        up_st.wait_stream(cur)
        down_st.wait_stream(cur)
        for _ in range(n):
            if up:
                with torch.cuda.stream(up_st):
                    for d_, h_ in zip(dev_in[0], host_in):
                        d_.copy_(h_, non_blocking=True)
            if down:
                with torch.cuda.stream(down_st):
                    for h_, d_ in zip(host_out[0], dev_out[0]):
                        h_.copy_(d_, non_blocking=True)
        cur.wait_stream(up_st)
        cur.wait_stream(down_st)

    copy_gbs = {}
    for name, up, down in (("h2d", True, False), ("d2h", False, True), ("both", True, True)):
        copy_run(up, down, 1)
        torch.cuda.synchronize()
        e0.record(stream)
        copy_run(up, down, 3)
        e1.record(stream)
        torch.cuda.synchronize()
        nbytes = 3 * ((h2d if up else 0) + (d2h if down else 0))
        copy_gbs[name] = nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9
    del dev_in, dev_out

    # ---- one-GPU context-parallel ring emulation (dual chunk swap, 8 ranks)
    cp_obj = None
    if not args.no_cp and not w.is_thd and w.batch == 1 and w.seqlen % 16 == 0:
        from bwd_tcgen05_tmem_gb300 import cp as cpmod
        ring = cpmod.CPRing(q, k, v, do, cp=8, scale=w.scale)
        for _ in range(2):
            ring.forward()
            ring.backward()
        torch.cuda.synchronize()
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c2 = torch.cuda.Event(enable_timing=True)
        n_cp = 3
        fwd_ms = bwd_ms = 0.0
        for _ in range(n_cp):
            c0.record(stream)
            ring.forward()
            c1.record(stream)
            ring.backward()
            c2.record(stream)
            torch.cuda.synchronize()
            fwd_ms += c0.elapsed_time(c1) / n_cp
            bwd_ms += c1.elapsed_time(c2) / n_cp
        # the LSE-merge kernel alone: every rank's merge, back to back on one
        # stream; algorithmic bytes = the parts' FP32 O and LSE read once plus
        # the merged O (bf16) and LSE written once
        n_m = 5
        m_bytes = 0
        for r_, pcs in enumerate(ring.pieces):
            for pc in pcs:
                m_bytes += pc.q_rows[1] * w.heads_q * (4 * w.d_v + 4)
            m_bytes += 2 * ring.chunk * w.heads_q * (2 * w.d_v + 4)
        # replayed from a CUDA graph, so that the host's per-call argument
        # marshalling (eight launches) does not sit between the kernels
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            ring.merge_all()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        merge_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(merge_graph):
            ring.merge_all()
        merge_graph.replay()
        c0.record(stream)
        for _ in range(n_m):
            merge_graph.replay()
        c1.record(stream)
        torch.cuda.synchronize()
        merge_ms = c0.elapsed_time(c1) / n_m
        del merge_graph
        cp_obj = {"cp": 8, "chunks": 16, "chunk_tokens": w.seqlen // 16,
                  "merge": {"ms": merge_ms, "bytes": m_bytes,
                            "gbs": m_bytes / (merge_ms * 1e-3) / 1e9,
                            "hbm_frac": m_bytes / (merge_ms * 1e-3) / 1e9 / peaks0["hbm_gbs"],
                            "launches": 8,
                            "note": "attn_lse_merge of all 8 ranks (FP32 partials of every "
                                    "ring step), timed alone on one stream, replayed "
                                    "from a CUDA graph"},
                  "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "ms": fwd_ms + bwd_ms,
                  "tflops": fl["total"] / ((fwd_ms + bwd_ms) * 1e-3) / 1e12,
                  "launches": ring.launches,
                  "note": "partials per ring step (FP32) + LSE merge per rank + per-step "
                          "backward with FP32 accumulation, all ranks on this GPU"}
        del ring
        # all-gather variant: one call per local query chunk on the trimmed keys
        ag = cpmod.CPAllGather(q, k, v, do, cp=8, scale=w.scale, window=(w.window[0], 0))
        for _ in range(2):
            ag.forward()
            ag.backward()
        torch.cuda.synchronize()
        fwd_ms = bwd_ms = 0.0
        for _ in range(n_cp):
            c0.record(stream)
            ag.forward()
            c1.record(stream)
            ag.backward()
            c2.record(stream)
            torch.cuda.synchronize()
            fwd_ms += c0.elapsed_time(c1) / n_cp
            bwd_ms += c1.elapsed_time(c2) / n_cp
        cp_obj["allgather"] = {
            "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "ms": fwd_ms + bwd_ms,
            "tflops": fl["total"] / ((fwd_ms + bwd_ms) * 1e-3) / 1e12, "launches": ag.launches,
            "note": "KV gathered and trimmed per query chunk, bottom-right causal, no LSE "
                    "merge; dK/dV partials summed in FP32 (the reduce-scatter), one GPU"}
        del ag
        # all-to-all variant: relayout to head shards, full-sequence attention per rank
        a2a = cpmod.CPA2A(q, k, v, do, cp=8, scale=w.scale, window=(w.window[0], 0))
        for _ in range(2):
            a2a.forward()
            a2a.backward()
        torch.cuda.synchronize()
        fwd_ms = bwd_ms = 0.0
        for _ in range(n_cp):
            c0.record(stream)
            a2a.forward()
            c1.record(stream)
            a2a.backward()
            c2.record(stream)
            torch.cuda.synchronize()
            fwd_ms += c0.elapsed_time(c1) / n_cp
            bwd_ms += c1.elapsed_time(c2) / n_cp
        # the relayout kernel alone: Q to head shards (read + write bytes)
        r0 = torch.cuda.Event(enable_timing=True)
        r1 = torch.cuda.Event(enable_timing=True)
        r0.record(stream)
        for _ in range(5):
            attn.cp_relayout(a2a.q_seq, a2a.q_h, to_heads=True, cp=8)
        r1.record(stream)
        torch.cuda.synchronize()
        rl_ms = r0.elapsed_time(r1) / 5
        cp_obj["a2a"] = {
            "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "ms": fwd_ms + bwd_ms,
            "tflops": fl["total"] / ((fwd_ms + bwd_ms) * 1e-3) / 1e12, "launches": a2a.launches,
            "relayout_q_ms": rl_ms,
            "relayout_q_gbs": 2 * q.numel() * q.element_size() / (rl_ms * 1e-3) / 1e9,
            "note": "sequence shards -> head shards (attn_cp_relayout), attention over the "
                    "whole sequence for H/cp heads per rank, outputs and gradients back"}
        del a2a

    peaks, peak_src = peaks0, peak_src0
    # the kernels run at close to the maximum SM clock (sampled below), so the
    # burst figure is the denominator; the sustained one (measured under the
    # power cap at a lower clock) is reported beside it
    peak_tf = peaks.get("bf16_tflops", peaks.get("bf16_tflops_sustained"))
    peak_sus = peaks.get("bf16_tflops_sustained", peak_tf)
    dom = max(("fwd", "dq", "dkdv"), key=lambda s: per_kernel[s])
    ach = fl["kernel"][dom] / (per_kernel[dom] * 1e-3) / 1e12

    def pkey(k_):  # the profile entry of a kernel: the dK/dV kernel that writes dS has its own
        return k_ + "+ds" if (k_ == "dkdv" and bwd_path == attn.BWD_DS) else k_

    # the committed ncu figures describe the 192/128 kernels on the 8K case
    # (traffic scaled to the 32K workload): reported for that workload only
    profiled = w.name == WORKLOAD
    traffic = load_traffic(pkey(dom)) if profiled else None
    value = job_tflops(fl["total"], ms, world)
    lens_b = ((inp["cu_seqlens"][1:] - inp["cu_seqlens"][:-1]).tolist() if w.is_thd else None)
    rows_q = q.shape[0] * (1 if w.is_thd else q.shape[1])
    rows_k = k.shape[0] * (1 if w.is_thd else k.shape[1])
    dq_bytes = (score_blocks(w, lens_b) * 32768 + rows_q * w.heads_q * w.d_qk * 2 +
                rows_k * w.heads_kv * w.d_qk * 2)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch * world, "seq_len": w.seqlen,
                   "heads": w.heads_q, "heads_kv": w.heads_kv, "d_qk": w.d_qk, "d_v": w.d_v,
                   "causal": True, "parallelism": f"replicas{world}",
                   "l2": "inputs larger than L2 (no flush)"},
        "pct_of_peak": 100.0 * (value / world) / peak_tf,
        "pct_of_peak_sustained": 100.0 * (value / world) / peak_sus,
        "peak_tflops": peak_tf,
        "peak_tflops_sustained": peak_sus,
        "peak_source": f"{peak_src} (bf16 burst; sustained beside it)",
        "step_ms": step_spread,
        "kernel_ms_spread": kernel_spread,
        "tflops_fwd": fl["fwd"] / (per_kernel["fwd"] * 1e-3) / 1e12,
        "tflops_bwd": fl["bwd"] / ((per_kernel["pre"] + per_kernel["dq"] + per_kernel["dkdv"])
                                   * 1e-3) / 1e12,
        "kernel_ms": {k_: round(v_, 4) for k_, v_ in per_kernel.items()},
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": ach, "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": ach / peak_tf, "traffic": traffic,
                     "peak_source": f"{peak_src} bf16_tflops (burst)",
                     "peak_sustained": peak_sus, "frac_sustained": ach / peak_sus,
                     "sm_mhz": clocks.get("sm_mhz"),
                     "work_per_launch": fl["kernel"][dom],
                     # on the dS path the dK/dV kernel also streams the dS blocks out
                     "ds_write_bytes": (score_blocks(w, lens_b) * 32768
                                        if bwd_path == attn.BWD_DS and dom == "dkdv" else None)},
        "bwd_path": {attn.BWD_RECOMPUTE: "recompute", attn.BWD_DS: "ds",
                     attn.BWD_PDS: "pds"}[bwd_path],
        "dq_gemm_hbm": None if bwd_path != attn.BWD_DS else {
            "bound": "hbm", "unit": "GB/s", "peak": peaks["hbm_gbs"],
            "bytes": dq_bytes, "achieved": dq_bytes / (per_kernel["dq"] * 1e-3) / 1e9,
            "frac": dq_bytes / (per_kernel["dq"] * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "note": "dQ GEMM of the dS path: dS blocks (32 KiB per visible 128 x 128 "
                    "tile and query head) read once, K read once, dQ written once"},
        "kernels": {k_: {"ms": per_kernel[k_],
                         "tflops": fl["kernel"][k_] / (per_kernel[k_] * 1e-3) / 1e12,
                         "frac": fl["kernel"][k_] / (per_kernel[k_] * 1e-3) / 1e12 / peak_tf,
                         "tensor_pipe_pct": load_tensor_pipe(pkey(k_)) if profiled else None}
                    for k_ in ("fwd", "dq", "dkdv")},
        # D preprocess: O and dO read, LSE read, {LSE log2 e, D} written, per row
        "pre_gbs": (q.shape[0] * (1 if w.is_thd else q.shape[1]) * w.heads_q * (2 * w.d_v * 2 + 12)) /
                   (per_kernel["pre"] * 1e-3) / 1e9,
        "pre_hbm_frac": (q.shape[0] * (1 if w.is_thd else q.shape[1]) * w.heads_q *
                         (2 * w.d_v * 2 + 12)) / (per_kernel["pre"] * 1e-3) / 1e9 / peaks["hbm_gbs"],
        "e2e": {"value": job_tflops(fl["total"], e2e_ms, world), "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "stage_ms": {k_: round(v_, 3) for k_, v_ in stage_ms.items()},
                "steps": e2e_steps, "copy_only_gbs": copy_gbs,
                "note": "C ABI attn_fwd_bwd_host_stages per step: inputs uploaded from "
                        "pinned host memory, forward + backward, all outputs downloaded; "
                        "upload, compute and download streams ordered by events over two "
                        "device arenas; copy_only_gbs: the same copies alone (h2d, d2h, "
                        "both at once)"},
        "gpu_launches": launches,
        "clocks": clocks,
        "cp_emulation": cp_obj,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
