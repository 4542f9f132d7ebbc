"""Benchmark: query-aware block selection + sparse decode attention on GB300.

Default workload: the Qwen3-4B-shaped GQA batch decode (batch 16, 32 q / 8 KV
heads, head_dim 128, 32768 cached tokens in blocks of 32, keep 12.5 % = 128
blocks, 36 layers with distinct buffers, about 74 GB of KV on the device).

One step = one decode step through all 36 layers; per layer it runs every
device step of the hot path through the C ABI: the append of the new token
with the open block's summary update, score + Top-k + spans, and the sparse
decode attention. The metric is layer-steps per second. The keep-ratio budget
(kvsel_budget, host arithmetic) is called once per step when the step is
enqueued; the timed steps are one CUDA-graph replay, so it ran at capture and
is not inside the timed region (it costs well under a microsecond).

Device timing: CUDA events on the bench stream around exactly --steps steps
after --warmup steps, with a device sync (and a barrier under torchrun) on
both sides; the max over ranks is reported. The 36 distinct layers (74 GB)
exceed the 129 MB L2, so no flush is needed between steps. Each decode and
score launch is also bracketed by events for the per-kernel roofline.

--impl reference times the fp64 CPU oracle on this machine's host cores on a
bounded sample (one layer, a few sequences) of the same workload.
"""
from __future__ import annotations

import argparse
import gc
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse decode-attn steps/s per layer; achieved HBM GB/s vs GB300 peak"
UNIT = "layer-steps/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kvsel", choices=["kvsel", "reference"])
    ap.add_argument("--layers", type=int, default=None, help="override the layer count (debug)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-offload", action="store_true", help="skip the C4 offload-tier measurement")
    ap.add_argument("--ref-seqs", type=int, default=4, help="sequences per oracle sample")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-layer step on the other workload shapes")
    ap.add_argument("--no-window", action="store_true",
                    help="skip the step with a forced sink block and recency window")
    return ap.parse_args()


def max_over_ranks(x: float, device) -> float:
    """The largest value of x over the ranks of the default process group
    (the slowest replica's time is the job's time)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, layers: int, steps: int, elapsed_ms: float) -> float:
    """Layer-steps per second of the whole job: every replica runs `steps`
    steps of `layers` layers on its own sequences (weak scaling), and the job
    takes as long as its slowest replica."""
    return world * layers * steps / (elapsed_ms / 1e3)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


DECODE_SOURCES = ("query_aware_sparse_block_gb300/csrc/sparse_decode.cu",
                  "query_aware_sparse_block_gb300/csrc/kvsel_common.cuh")


def decode_source_hash() -> str:
    """sha256 over the decode kernel's sources: ties an ncu capture to the code it measured."""
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def decode_traffic():
    """DRAM bytes (read + write) of one decode launch on this workload from the committed ncu
    capture, or None when there is none or the kernel changed since it was taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    if t.get("source_sha256") != decode_source_hash():
        return None
    return t.get("sparse_decode_bytes_per_launch")


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ------------------------------------------------------------------ clocks ---

class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ GPU workload ---

class Workbench:
    """All layers of the workload resident on the device, plus per-step inputs."""

    def __init__(self, w, layers, total_steps, device):
        import torch

        from query_aware_sparse_block_gb300.runtime import SparseDecoder
        from workloads.generate import generate_layer

        self.w, self.L, self.device = w, layers, device
        B = w.block_size
        # the last step ends with exactly seq_len cached tokens
        self.T0 = w.seq_len - total_steps
        self.max_blocks = (w.seq_len + B - 1) // B
        self.k = w.k_for(w.keep[0])
        self.dec = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, B, self.max_blocks,
                                 k_max=self.k, device=device)
        self.layers = []
        for l in range(layers):
            x = generate_layer(w, l, device=device, max_blocks=self.max_blocks, perm=False,
                               seq_lens=[self.T0] * w.batch)
            summ, acc = self.dec.new_summaries()
            self.dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
            g = torch.Generator(device=device)
            g.manual_seed(w.seed(l) + 104729)
            shape = (w.batch, w.n_kvheads, w.head_dim)
            new_k = torch.randn(shape, generator=g, device=device).to(torch.bfloat16)
            new_v = torch.randn(shape, generator=g, device=device).to(torch.bfloat16)
            out = torch.empty((w.batch, w.n_qheads, w.head_dim), dtype=torch.float32, device=device)
            lse = torch.empty((w.batch, w.n_qheads), dtype=torch.float32, device=device)
            self.layers.append(dict(x=x, summ=summ, acc=acc, new_k=new_k, new_v=new_v, out=out,
                                    lse=lse))
            torch.cuda.synchronize()
        # per-step positions: step s appends token T0 + s, then attends over T0 + s + 1 tokens
        s = torch.arange(total_steps, device=device, dtype=torch.int32).view(-1, 1)
        self.append_pos = (self.T0 + s).expand(total_steps, w.batch).contiguous()
        self.seq_lens = self.append_pos + 1
        self.dec.k_per_seq.fill_(self.k)
        self.step_i = 0
        from query_aware_sparse_block_gb300 import kvsel as K
        from query_aware_sparse_block_gb300.runtime import BoundLayer
        import ctypes
        self.K = K
        self.bound = [BoundLayer(self.dec, d["x"]["q"], d["x"]["kv_pages"],
                                 d["x"]["block_table"], d["summ"], d["acc"], d["out"], d["lse"],
                                 gamma=w.gamma, new_k=d["new_k"], new_v=d["new_v"])
                      for d in self.layers]
        self.pos_ptrs = [ctypes.c_void_p(self.append_pos[i].data_ptr()) for i in range(total_steps)]
        self.len_ptrs = [ctypes.c_void_p(self.seq_lens[i].data_ptr()) for i in range(total_steps)]
        # graph mode: one pair of device buffers advanced in place after every step
        self.pos_buf = torch.zeros((w.batch,), dtype=torch.int32, device=device)
        self.len_buf = torch.zeros((w.batch,), dtype=torch.int32, device=device)

    def budget_k(self):
        """kvsel_budget on the host: keep ratio (12.5 % override, no floor) -> k."""
        w = self.w
        N = (self.T0 + self.step_i + w.block_size) // w.block_size
        r = self.K.kvsel_budget(w.block_size, w.n_kvheads, w.head_dim, 2, 2560, N, 6.7e12, 1.7e15,
                                keep_override=w.keep[0], gamma=w.gamma)
        return r

    def step(self, stream, ev_score=None, ev_dec=None, q_ptrs=None, out_ptrs=None, nk_ptrs=None,
             nv_ptrs=None, graph=False, record=None):
        """One decode step through all layers (enqueue only): the host-side
        budget, then per layer the append + selection call and the decode
        call. With graph=True the step reads its positions from pos_buf /
        len_buf and advances them; a captured step replays only the device
        work, so the budget then runs once, at capture."""
        import ctypes
        i = self.step_i
        if graph:
            pos = ctypes.c_void_p(self.pos_buf.data_ptr())
            lens = ctypes.c_void_p(self.len_buf.data_ptr())
        else:
            pos, lens = self.pos_ptrs[i], self.len_ptrs[i]
        sp = ctypes.c_void_p(stream.cuda_stream)
        rec = record or (lambda ev: ev.record(stream))
        self.budget_k()
        for l, bl in enumerate(self.bound):
            if ev_score is not None and l == 0:
                rec(ev_score[0][0])             # later layers start at the previous merge's event
            # the token's summary update and the block selection, one call
            bl.append_select(pos, lens, sp, None if nk_ptrs is None else nk_ptrs[l],
                             None if nv_ptrs is None else nv_ptrs[l],
                             None if q_ptrs is None else q_ptrs[l])
            if ev_score is not None:
                rec(ev_score[1][l])
            bl.attend(lens, sp, None if q_ptrs is None else q_ptrs[l],
                      None if out_ptrs is None else out_ptrs[l])
            if ev_dec is not None:
                rec(ev_dec[1][l])
        if graph:
            self.pos_buf.add_(1)
            self.len_buf.add_(1)
        self.step_i += 1

    def decode_bytes(self):
        w = self.w
        sel = self.k * w.n_kvheads * 2 * w.block_size * w.head_dim * 2 * w.batch
        q = w.batch * w.n_qheads * w.head_dim * 2
        out = w.batch * w.n_qheads * (w.head_dim + 1) * 4
        return sel + q + out

    def score_bytes(self, N):
        w = self.w
        summ = w.batch * N * w.n_kvheads * w.head_dim * 2
        q = w.batch * w.n_qheads * w.head_dim * 2
        scores = w.batch * N * 4
        sel = w.batch * self.k * 4 * 3
        return summ + q + scores + sel


def load_cudart():
    """The CUDA runtime already loaded by torch (for external event records)."""
    import ctypes
    for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
        try:
            lib = ctypes.CDLL(name)
            lib.cudaEventRecordWithFlags.restype = ctypes.c_int
            return lib
        except OSError:
            pass
    with open("/proc/self/maps") as f:
        for ln in f:
            if "libcudart" in ln:
                lib = ctypes.CDLL(ln.split()[-1])
                lib.cudaEventRecordWithFlags.restype = ctypes.c_int
                return lib
    raise RuntimeError("libcudart not found in this process")


def run_gpu(args):
    import ctypes

    import torch
    import torch.distributed as dist

    from workloads import C3

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    w = C3
    layers = args.layers or w.layers
    n_e2e = 0 if args.no_e2e else max(3, args.steps // 2)
    n_win = 0 if args.no_window else max(3, args.steps // 2)
    total_steps = args.warmup + args.steps + 2 + n_e2e + 2 + n_win + 2
    wb = Workbench(w, layers, total_steps, device)
    K = wb.K
    stream = torch.cuda.Stream(device=device)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            wb.step(stream)
        stream.synchronize()
        err = K.kvsel_get_error(stream)
        if err:
            raise RuntimeError(f"device error {err} during warm-up")
        ev_s = [[torch.cuda.Event(enable_timing=True) for _ in range(layers * args.steps)] for _ in range(2)]
        ev_d = [[torch.cuda.Event(enable_timing=True) for _ in range(layers * args.steps)] for _ in range(2)]
        for e in ev_s[0] + ev_s[1] + ev_d[0] + ev_d[1]:
            e.record(stream)            # creates the events before capture
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        # The K timed steps are captured once into a CUDA graph, so the device
        # timing does not depend on how fast the host can enqueue. The kernels of
        # a layer are chained by programmatic dependent launch; an event node
        # between two of them would turn that edge into a full dependency, so the
        # timing events sit on a side branch: each one waits for everything
        # enqueued on the main stream so far and records when that completes.
        # A layer's score + Top-k call (summary append folded in) runs from the
        # end of the previous layer's merge grid (or the step's start) to the
        # end of its last kernel (the cluster launch, or the Top-k grid of the
        # two-grid form); its decode call from there to the end of its merge
        # grid.
        cudart = load_cudart()
        side = torch.cuda.Stream(device=device)
        ssp = side.cuda_stream
        forks = []

        def rec_ext(ev):
            fork = torch.cuda.Event()
            forks.append(fork)
            fork.record(stream)
            side.wait_event(fork)
            rc = cudart.cudaEventRecordWithFlags(ctypes.c_void_p(ev.cuda_event), ctypes.c_void_p(ssp), 1)
            if rc:
                raise RuntimeError(f"cudaEventRecordWithFlags failed: {rc}")

        first = wb.step_i
        acc_snap = [d["acc"].clone() for d in wb.layers]

        def reset_state():
            wb.pos_buf.copy_(wb.append_pos[first])
            wb.len_buf.copy_(wb.seq_lens[first])
            for d, a in zip(wb.layers, acc_snap):
                d["acc"].copy_(a)

        reset_state()
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        launches0 = K.kvsel_launch_count()
        h0 = time.perf_counter()
        with torch.cuda.graph(graph, stream=stream):
            for s in range(args.steps):
                sl = slice(s * layers, (s + 1) * layers)
                wb.step(stream, ev_score=(ev_s[0][sl], ev_s[1][sl]), ev_dec=(ev_s[1][sl], ev_d[1][sl]),
                        graph=True, record=rec_ext)
            join = torch.cuda.Event()
            join.record(side)
            stream.wait_event(join)
        host_ms = (time.perf_counter() - h0) * 1e3 / args.steps
        launches = K.kvsel_launch_count() - launches0
        graph.replay()                  # uploads the graph; untimed
        stream.synchronize()
        reset_state()
        clocks = ClockSampler(local)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        clocks.start()
        t0.record(stream)
        graph.replay()
        t1.record(stream)
        stream.synchronize()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        clk = clocks.stop()
        elapsed_ms = t0.elapsed_time(t1)
        err = K.kvsel_get_error(stream)
        if err:
            raise RuntimeError(f"device error {err} in the timed region")
        if world > 1:
            elapsed_ms = max_over_ranks(elapsed_ms, device)
        dec_ms = [a.elapsed_time(b) for a, b in zip(ev_s[1], ev_d[1])]
        # A layer's score call starts where the previous layer's decode call
        # ended, on that same event: consecutive event nodes of the side branch
        # fire about 2.5 us apart, so a second event at the same point would
        # shift the start.
        sc_start = [ev_s[0][i] if i % layers == 0 else ev_d[1][i - 1] for i in range(layers * args.steps)]
        sc_ms = [a.elapsed_time(b) for a, b in zip(sc_start, ev_s[1])]

        # ---- e2e: pinned host inputs in, results out, through the public API ----
        e2e = None
        if n_e2e:
            # Double-buffered: step s+1's inputs travel on one copy stream and
            # step s-1's outputs come back on another while step s computes,
            # as a serving loop would pipeline them. Every step's copies are in
            # the timed region; the last read-back ends it.
            q_host = torch.stack([d["x"]["q"] for d in wb.layers]).cpu().pin_memory()
            kv_host = torch.stack([torch.stack([d["new_k"], d["new_v"]]) for d in wb.layers]).cpu().pin_memory()
            q_dev = [torch.empty_like(q_host, device=device) for _ in range(2)]
            kv_dev = [torch.empty_like(kv_host, device=device) for _ in range(2)]
            out_shape = (layers, w.batch, w.n_qheads, w.head_dim)
            out_dev = [torch.empty(out_shape, dtype=torch.float32, device=device) for _ in range(2)]
            out_host = [torch.empty(out_shape, dtype=torch.float32).pin_memory() for _ in range(2)]
            import ctypes
            vp = ctypes.c_void_p
            bufs = [dict(q=[vp(q_dev[i][l].data_ptr()) for l in range(layers)],
                         nk=[vp(kv_dev[i][l, 0].data_ptr()) for l in range(layers)],
                         nv=[vp(kv_dev[i][l, 1].data_ptr()) for l in range(layers)],
                         out=[vp(out_dev[i][l].data_ptr()) for l in range(layers)]) for i in range(2)]
            h2d = torch.cuda.Stream(device=device)
            d2h = torch.cuda.Stream(device=device)
            ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of buffer i landed
            ev_used = [torch.cuda.Event() for _ in range(2)]   # the step on buffer i finished
            ev_out = [torch.cuda.Event() for _ in range(2)]    # outputs of buffer i read back
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)

            def load(s):
                i = s % 2
                if s >= 2:
                    h2d.wait_event(ev_used[i])      # step s-2 is done with buffer i
                with torch.cuda.stream(h2d):
                    q_dev[i].copy_(q_host, non_blocking=True)
                    kv_dev[i].copy_(kv_host, non_blocking=True)
                    ev_in[i].record(h2d)

            torch.cuda.synchronize()
            e0.record(stream)
            h2d.wait_stream(stream)
            d2h.wait_stream(stream)
            load(0)
            for s in range(n_e2e):
                i = s % 2
                if s + 1 < n_e2e:
                    load(s + 1)
                stream.wait_event(ev_in[i])
                if s >= 2:
                    stream.wait_event(ev_out[i])    # buffer i's last outputs were read back
                wb.step(stream, q_ptrs=bufs[i]["q"], out_ptrs=bufs[i]["out"], nk_ptrs=bufs[i]["nk"],
                        nv_ptrs=bufs[i]["nv"])
                ev_used[i].record(stream)
                d2h.wait_event(ev_used[i])
                with torch.cuda.stream(d2h):
                    out_host[i].copy_(out_dev[i], non_blocking=True)
                    ev_out[i].record(d2h)
            stream.wait_stream(d2h)
            e1.record(stream)
            stream.synchronize()
            e2e_ms = e0.elapsed_time(e1) / n_e2e
            e2e = {"value": layers / (e2e_ms / 1e3), "unit": UNIT,
                   "h2d_bytes_per_step": q_host.numel() * 2 + kv_host.numel() * 2,
                   "d2h_bytes_per_step": out_host[0].numel() * 4,
                   "ms_per_step": e2e_ms, "steps": n_e2e,
                   "copies": "pinned host buffers, double-buffered on two copy streams that overlap "
                             "the neighbouring steps' compute"}

        window = run_window(wb, stream, n_win, elapsed_ms / args.steps) if n_win else None
    configs = None
    if world == 1 and not args.no_configs:
        configs = run_configs(device)
        configs.append(run_summary_build(device))

    form, ctas = K.kvsel_score_path_for(wb.dec.p, True)
    score_form = {"form": "cluster" if form == K.KVSEL_SCORE_PATH_CLUSTER else "two_grid",
                  "cluster_ctas": ctas}
    ms_per_step = elapsed_ms / args.steps
    value = whole_job_rate(world, layers, args.steps, elapsed_ms)
    peak, peak_kind = peaks()
    N = (wb.T0 + args.warmup + w.block_size) // w.block_size   # blocks at the first timed step
    dec_bytes = wb.decode_bytes()
    dec_avg_ms = statistics.mean(dec_ms)
    sc_avg_ms = statistics.mean(sc_ms)
    dec_gbs = dec_bytes / (dec_avg_ms / 1e3) / 1e9
    sc_bytes = wb.score_bytes(N)
    sc_gbs = sc_bytes / (sc_avg_ms / 1e3) / 1e9
    traffic = decode_traffic()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "n_qheads": w.n_qheads,
                   "n_kvheads": w.n_kvheads, "head_dim": w.head_dim, "seq_len": w.seq_len,
                   "block_size": w.block_size, "keep": w.keep[0], "k": wb.k, "layers": layers,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (distinct buffers per layer, no flush)",
                   "score_form": score_form},
        "roofline": {"kernel": "sparse_decode", "bound": "hbm", "achieved": dec_gbs, "peak": peak,
                     "unit": "GB/s", "frac": dec_gbs / peak, "peak_kind": peak_kind,
                     "frac_of_nominal": dec_gbs / NOMINAL_HBM_GBS,
                     "traffic": traffic, "bytes_per_launch": dec_bytes,
                     "avg_launch_us": dec_avg_ms * 1e3},
        "kernels": {
            "score_topk": {"bytes_per_launch": sc_bytes, "avg_launch_us": sc_avg_ms * 1e3,
                           "achieved_gbs": sc_gbs, "frac": sc_gbs / peak,
                           "frac_of_nominal": sc_gbs / NOMINAL_HBM_GBS},
            "sparse_decode": {"bytes_per_launch": dec_bytes, "avg_launch_us": dec_avg_ms * 1e3,
                              "achieved_gbs": dec_gbs, "frac": dec_gbs / peak,
                              "frac_of_nominal": dec_gbs / NOMINAL_HBM_GBS},
        },
        "gpu_launches": int(launches),
        "host_capture_ms_per_step": host_ms,
        "timing": "one CUDA-graph replay of the timed steps (kernels launched through the C ABI "
                  "during capture, chained by programmatic dependent launch); per-call durations "
                  "from external event nodes on a side branch of the graph: score_topk (the "
                  "token's summary append folded in) from the end of the previous layer's merge "
                  "grid to the end of its last kernel (the cluster launch, or the Top-k grid of the "
                  "two-grid form), sparse_decode from there to the end of its merge grid",
        "clocks": clk,
        "e2e": e2e,
        "window": window,
        "configs": configs,
    }
    if world == 1 and not args.no_offload:
        line["offload"] = run_offload(device, K)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_subprocess(args.ref_seqs, reps=5)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


NOMINAL_HBM_GBS = 7900.0    # GB300 HBM3e, nominal


def run_summary_build(device, reps=3):
    """The FULL summary build (prefill; off the per-step path) on one layer of
    the Qwen3-4B-shaped batch (1 GiB of keys) and on the MiniCPM-shaped
    sequence (64 MiB): key bytes read per second and fp64 additions per second
    (one per key element; the sum is sequential in token order by definition)."""
    import torch

    from query_aware_sparse_block_gb300.runtime import SparseDecoder
    from workloads import C2, C3
    from workloads.generate import generate_layer

    peak, _ = peaks()
    res = {"kind": "summary_build_full"}
    for w in (C3, C2):
        x = generate_layer(w, 0, device=device, perm=False)
        dec = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, x["max_blocks"],
                            k_max=1, device=device)
        summ, acc = dec.new_summaries()
        dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(reps):
            dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
        t1.record()
        torch.cuda.synchronize()
        us = t0.elapsed_time(t1) * 1e3 / reps
        elems = w.batch * w.seq_len * w.n_kvheads * w.head_dim
        res[w.name] = {"us": us, "key_bytes": elems * 2, "key_gbs": elems * 2 / (us / 1e6) / 1e9,
                       "frac_of_hbm": elems * 2 / (us / 1e6) / 1e9 / peak,
                       "fp64_add_per_s": elems / (us / 1e6)}
        del x, dec, summ, acc
        torch.cuda.empty_cache()
    return res


def run_configs(device, passes=4, min_pass_bytes=400e6):
    """The decode step (score + Top-k, then sparse decode; no append) on the
    other workload shapes: tiny MHA (C0), OPT-6.7B-shaped MHA at keep 50 % and
    10 % (C1), MiniCPM4.1-8B-shaped GQA at 128K tokens (C2). Enough distinct
    layers are resident that one pass over them moves more than three times
    the L2; a CUDA graph of `passes` passes is timed with events. Reports
    layer-steps/s and the step's algorithmic bytes (summaries, q, selected K/V,
    outputs) per second against the measured and the nominal HBM bandwidth."""
    import ctypes

    import torch

    from query_aware_sparse_block_gb300.runtime import BoundLayer, SparseDecoder
    from workloads import C0, C1, C2
    from workloads.generate import generate_layer

    peak, _ = peaks()
    out = []
    for w in (C0, C1, C2):
        for k in w.ks:
            N = w.n_blocks
            per_layer = (w.batch * N * w.n_kvheads * w.head_dim * 2 + w.batch * w.n_qheads * w.head_dim * 2
                         + w.batch * k * w.n_kvheads * 2 * w.block_size * w.head_dim * 2
                         + w.batch * w.n_qheads * (w.head_dim + 1) * 4)
            nl = max(2, int(math.ceil(min_pass_bytes / per_layer)))
            dec = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, N, k_max=k,
                                device=device)
            dec.k_per_seq.fill_(k)
            layers, keep = [], []
            for l in range(nl):
                x = generate_layer(w, l, device=device, perm=False)
                summ, acc = dec.new_summaries()
                dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
                keep.append((x, summ, acc))
                layers.append(BoundLayer(dec, x["q"], x["kv_pages"], x["block_table"], summ, acc,
                                         dec.out, dec.lse, gamma=2.0))
            lens = ctypes.c_void_p(keep[0][0]["seq_lens"].data_ptr())
            s = torch.cuda.Stream(device=device)
            sp = ctypes.c_void_p(s.cuda_stream)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for _ in range(passes):
                    for bl in layers:
                        bl.select(lens, sp)
                        bl.attend(lens, sp)
            with torch.cuda.stream(s):
                g.replay()
                s.synchronize()
                t0 = torch.cuda.Event(enable_timing=True)
                t1 = torch.cuda.Event(enable_timing=True)
                t0.record(s)
                g.replay()
                t1.record(s)
                s.synchronize()
            us = t0.elapsed_time(t1) * 1e3 / (passes * nl)
            gbs = per_layer / (us / 1e6) / 1e9
            out.append({"workload": w.name, "k": k, "layers_resident": nl, "us_per_layer_step": us,
                        "layer_steps_per_s": 1e6 / us, "bytes_per_layer_step": per_layer,
                        "achieved_gbs": gbs, "frac": gbs / peak, "frac_of_nominal": gbs / NOMINAL_HBM_GBS})
            del g, layers, keep, dec
            torch.cuda.empty_cache()
    return out


def run_window(wb, stream, steps, plain_ms_per_step, n_sink=1, n_recent=4):
    """The same decode step with the first block and the last four blocks of
    every sequence forced into the selection (the recency window that the
    DKV abstract attends exactly beside the Top-k blocks, plus one leading
    block), Top-k over the blocks between: kvsel_score_topk_window with the
    token's append folded in, then kvsel_sparse_decode, captured into a CUDA
    graph and timed as a whole like the main step."""
    import torch

    from query_aware_sparse_block_gb300.runtime import BoundLayer, SparseDecoder

    w = wb.w
    dec = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, wb.max_blocks,
                        k_max=wb.k + n_sink + n_recent, device=wb.device)
    dec.k_per_seq.fill_(wb.k)
    bound = [BoundLayer(dec, d["x"]["q"], d["x"]["kv_pages"], d["x"]["block_table"], d["summ"],
                        d["acc"], d["out"], d["lse"], gamma=w.gamma, new_k=d["new_k"],
                        new_v=d["new_v"], window=(n_sink, n_recent)) for d in wb.layers]
    plain, wb.bound = wb.bound, bound
    try:
        first = wb.step_i
        acc_snap = [d["acc"].clone() for d in wb.layers]

        def reset_state():
            wb.pos_buf.copy_(wb.append_pos[first])
            wb.len_buf.copy_(wb.seq_lens[first])
            for d, a in zip(wb.layers, acc_snap):
                d["acc"].copy_(a)

        reset_state()
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        launches0 = wb.K.kvsel_launch_count()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(steps):
                wb.step(stream, graph=True)
        launches = wb.K.kvsel_launch_count() - launches0
        for _ in range(2):              # upload and warm up; untimed
            graph.replay()
            stream.synchronize()
            reset_state()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(stream)
        graph.replay()
        t1.record(stream)
        stream.synchronize()
        ms = t0.elapsed_time(t1) / steps
        err = wb.K.kvsel_get_error(stream)
        if err:
            raise RuntimeError(f"device error {err} in the window step")
        n_sel = dec.n_sel.cpu().tolist()
    finally:
        wb.bound = plain
    return {"n_sink": n_sink, "n_recent": n_recent, "k_topk": wb.k, "n_sel": n_sel[0],
            "value": len(wb.layers) / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "steps": steps,
            "gpu_launches": int(launches),
            "vs_plain_step": plain_ms_per_step / ms,
            "selected_kv_bytes_ratio": (wb.k + n_sink + n_recent) / wb.k}


# ------------------------------------------------------------ offload tier ---

def run_offload(device, K, reps=5, layer_prefetch=True):
    """C4 shape (64 sequences of 131072 tokens, 32 q / 2 KV heads, d 128, B 64):
    the full K/V in pinned host memory, summaries on the GPU. Reports the
    measured host-to-device copy rate of one large pinned copy, the budget
    model's keep ratio and dense decision for this link, and for the keep
    ratios 5 % (the floor) and 12.5 % the span gather (kvsel_fetch_spans) as
    link bytes per second and as a fraction of the measured copy rate, plus
    the whole offloaded decode (gather + attention); then the block cache
    (cross-step reuse) and, with `layer_prefetch`, the layer-ahead prefetch
    into per-layer caches."""
    import torch
    from query_aware_sparse_block_gb300.runtime import SparseDecoder
    from workloads import C4
    from workloads.generate import generate_layer, host_tier_layout

    w = C4
    N = w.n_blocks
    x = generate_layer(w, 0, device=device, perm=False)
    page = tuple(x["kv_pages"].shape[1:])
    page_bytes = int(np.prod(page)) * 2
    host = torch.empty((w.batch, N) + page, dtype=torch.bfloat16, pin_memory=True)
    host_tier_layout(x["kv_pages"], x["block_table"], N, out=host)
    dec = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, x["max_blocks"],
                        k_max=N, device=device)
    summ, acc = dec.new_summaries()
    dec.build_summaries(x["kv_pages"], x["block_table"], x["seq_lens"], summ, acc)
    torch.cuda.synchronize()
    del x["kv_pages"]
    torch.cuda.empty_cache()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def timed(fn, n):
        fn()
        torch.cuda.synchronize()
        ev[0].record()
        for _ in range(n):
            fn()
        ev[1].record()
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]) / n / 1e3    # seconds per call

    # The link's copy rate, three ways; the largest is the denominator of every
    # fraction below: (a) one large pinned host -> device copy (2 GiB), best of
    # 3; (b) four 512 MiB pinned copies on four streams at once, best of 3; (c)
    # the span gather itself (every 8th block of every sequence, 128 MiB) at 1
    # to 16 CTAs per SM, the best.
    src = host.view(-1)[: 1 << 30]
    dst = torch.empty(src.shape, dtype=src.dtype, device=device)
    copy_s = min(timed(lambda: dst.copy_(src, non_blocking=True), 1) for _ in range(3))
    copy_gbs = src.numel() * 2 / copy_s / 1e9
    streams = [torch.cuda.Stream(device=device) for _ in range(4)]
    quarter = src.numel() // 4

    def four_copies():
        cur = torch.cuda.current_stream()
        for i, st in enumerate(streams):
            st.wait_stream(cur)
            with torch.cuda.stream(st):
                dst[i * quarter:(i + 1) * quarter].copy_(src[i * quarter:(i + 1) * quarter], non_blocking=True)
        for st in streams:
            cur.wait_stream(st)

    conc_s = min(timed(four_copies, 1) for _ in range(3))
    conc_gbs = src.numel() * 2 / conc_s / 1e9
    del dst
    torch.cuda.empty_cache()
    k8 = N // 8
    sel8 = torch.arange(0, N, 8, dtype=torch.int32, device=device).repeat(w.batch, 1)
    dec8 = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, x["max_blocks"],
                         k_max=k8, device=device)
    dec8.sel_idx.copy_(sel8)
    dec8.n_sel.fill_(k8)
    K.kvsel_merge_spans(dec8.p, dec8.sel_idx, dec8.n_sel, dec8.span_start, dec8.span_len, dec8.n_spans)
    staging8 = torch.empty((w.batch, k8) + page, dtype=torch.bfloat16, device=device)
    gather_gbs = {}
    for per_sm in (1, 2, 4, 8, 16):
        kv8 = K.kv_host(host, N, staging8, k8, fetch_ctas=per_sm * torch.cuda.get_device_properties(device).multi_processor_count)
        t = timed(lambda: K.kvsel_fetch_spans(dec8.p, kv8, x["seq_lens"], dec8.span_start, dec8.span_len,
                                              dec8.n_spans, None), reps)
        gather_gbs[per_sm] = w.batch * k8 * page_bytes / t / 1e9
    del staging8, dec8
    torch.cuda.empty_cache()
    h2d_gbs = max(copy_gbs, conc_gbs, max(gather_gbs.values()))
    peak_f = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak_f = json.load(f).get("bf16_tflops_sustained")
    except (OSError, ValueError):
        pass
    flops = (peak_f or 1700.0) * 1e12
    bud = K.kvsel_budget(w.block_size, w.n_kvheads, w.head_dim, 2, w.hidden, N, h2d_gbs * 1e9, flops,
                         keep_floor=w.keep_floor, gamma=w.gamma)
    res = {"workload": w.name, "h2d_copy_gbs": h2d_gbs,
           "h2d_denominator": "max of one 2 GiB pinned copy, four concurrent 512 MiB copies and the "
                              "span gather at 1-16 CTAs per SM",
           "h2d_one_copy_gbs": copy_gbs, "h2d_four_streams_gbs": conc_gbs,
           "h2d_gather_gbs_by_ctas_per_sm": {str(k): v for k, v in gather_gbs.items()},
           "h2d_copy_bytes": src.numel() * 2,
           "budget_model": {"c_copy_s": bud.c_copy_s, "c_rec_s": bud.c_rec_s, "r_model": bud.r_model,
                            "r": bud.r, "k": int(bud.k), "dense": bool(bud.dense),
                            "recompute_flops_per_s": flops}}
    for keep in (w.keep_floor, 0.125):
        k = w.k_for(keep)
        dec.k_per_seq.fill_(k)
        dec.select(x["q"], summ, x["seq_lens"], gamma=w.gamma)
        torch.cuda.synchronize()
        n_dense = int(dec.dense_flag.sum())
        staging = torch.empty((w.batch, k) + page, dtype=torch.bfloat16, device=device)
        kv = K.kv_host(host, N, staging, k)
        fetch_s = timed(lambda: K.kvsel_fetch_spans(dec.p, kv, x["seq_lens"], dec.span_start,
                                                    dec.span_len, dec.n_spans, dec.dense_flag), reps)
        link_bytes = int(dec.n_sel.sum()) * page_bytes
        decode_s = timed(lambda: dec.attend(x["q"], kv, x["seq_lens"]), reps)
        # the attention kernel reading the host tier itself (no staging pass)
        kv_direct = K.kv_host_direct(host, N)
        direct_s = timed(lambda: dec.attend(x["q"], kv_direct, x["seq_lens"]), reps)
        err = K.kvsel_get_error()
        if err:
            raise RuntimeError(f"device error {err} in the offload measurement")
        res[f"keep_{keep:g}"] = {
            "k": k, "dense_sequences": n_dense, "link_bytes_per_step": link_bytes,
            "fetch_us": fetch_s * 1e6, "fetch_gbs": link_bytes / fetch_s / 1e9,
            "frac_of_h2d_copy": link_bytes / fetch_s / 1e9 / h2d_gbs,
            "fetch_plus_attend_us": decode_s * 1e6,
            "host_direct_attend_us": direct_s * 1e6,
            "host_direct_gbs": link_bytes / direct_s / 1e9,
            "host_direct_frac_of_h2d_copy": link_bytes / direct_s / 1e9 / h2d_gbs}
        del staging
    # the step the budget model decides for this link: r = 1, k = N, every
    # sequence dense, all of its K/V fetched over the link and attended
    k = int(bud.k)
    dec.k_per_seq.fill_(k)
    dec.select(x["q"], summ, x["seq_lens"], gamma=w.gamma)
    torch.cuda.synchronize()
    n_dense = int(dec.dense_flag.sum())
    staging = torch.empty((w.batch, N) + page, dtype=torch.bfloat16, device=device)
    kv = K.kv_host(host, N, staging, N)
    fetch_s = timed(lambda: K.kvsel_fetch_spans(dec.p, kv, x["seq_lens"], dec.span_start,
                                                dec.span_len, dec.n_spans, dec.dense_flag), 2)
    link_bytes = (n_dense * N + int(dec.n_sel[dec.dense_flag == 0].sum())) * page_bytes
    decode_s = timed(lambda: dec.attend(x["q"], kv, x["seq_lens"]), 2)
    err = K.kvsel_get_error()
    if err:
        raise RuntimeError(f"device error {err} in the dense offload measurement")
    res["model_decided"] = {
        "k": k, "dense_sequences": n_dense, "link_bytes_per_step": link_bytes,
        "fetch_us": fetch_s * 1e6, "fetch_gbs": link_bytes / fetch_s / 1e9,
        "frac_of_h2d_copy": link_bytes / fetch_s / 1e9 / h2d_gbs,
        "fetch_plus_attend_us": decode_s * 1e6}
    del staging
    torch.cuda.empty_cache()
    res["block_cache"] = run_block_cache(device, K, w, host, page, summ, x, timed, h2d_gbs,
                                         res[f"keep_{w.keep_floor:g}"]["fetch_plus_attend_us"])
    if layer_prefetch:
        res["layer_prefetch"] = run_layer_prefetch(device, K, w, host, page, summ, x, h2d_gbs)
    res["copy_unit_sweep"] = run_copy_unit_sweep(device, K, host, timed, h2d_gbs)
    del host
    torch.cuda.empty_cache()
    return res


def run_layer_prefetch(device, K, w, host, page, summ, x, h2d_gbs, layers=4, steps=8, rho=0.95,
                       rounds=3):
    """Layer-ahead prefetch into per-layer block caches, against the same
    caches without it, on the C4 shape at the keep floor (k = 102 of 2 048
    blocks, 64 sequences), for prediction widths m of 2 to 16 blocks. Each
    of `layers` layers has its own cache (2(k + 16) slots per sequence) and its own drifting queries (q_s = rho q_(s-1) +
    sqrt(1 - rho^2) e_s); they share the host tier and the summaries. Per
    step and layer the compute stream selects (keeping the score rows),
    fetches through the layer's cache and attends. With prefetch, once layer
    l's fetch is done a second stream takes the next layer's Top-(k + m) of
    its previous scores (kvsel_select_scores) and prefetches it into that
    layer's cache (kvsel_cache_prefetch); the next layer's fetch waits for
    it ("layer_ahead"). The other placement ("step_ahead") predicts on the
    compute stream right after a layer's select and prefetches that layer's
    next step on the second stream once its fetch is done, while the
    following layers run. Steps run back to back behind one bounded device-side delay; the
    figures are the steady-state time per layer-step (steps 1..), the
    blocks the compute stream's fetches copied (the critical path) and the
    blocks prefetched, medians over `rounds` rounds of every variant."""
    import torch
    from query_aware_sparse_block_gb300.runtime import BlockPredictor, HostBlockCache, SparseDecoder

    N = w.n_blocks
    k = w.k_for(w.keep_floor)
    ms = (2, 4, 8, 16)
    k_max = k + max(ms)
    slots = 2 * k_max
    page_bytes = int(np.prod(page)) * 2
    seq_lens = x["seq_lens"]
    decs, caches, preds, scores = [], [], [], []
    for _ in range(layers):
        dec = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size,
                            x["max_blocks"], k_max=k_max, device=device)
        dec.k_per_seq.fill_(k)
        decs.append(dec)
        caches.append(HostBlockCache(dec, slots, page))
        preds.append(BlockPredictor(dec, k_max))
        scores.append([torch.empty((w.batch, x["max_blocks"]), dtype=torch.float32, device=device)
                       for _ in range(2)])
    # every query of the run, made before it is timed
    qs = []
    for l in range(layers):
        g = torch.Generator(device=device).manual_seed(900 + l)
        q = x["q"].float() if l == 0 else torch.randn(x["q"].shape, generator=g, device=device)
        row = []
        for s in range(steps):
            if s:
                q = rho * q + math.sqrt(1 - rho * rho) * torch.randn(q.shape, generator=g, device=device)
            row.append(q.to(torch.bfloat16))
        qs.append(row)
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream(device=device)

    def run(m, mode="layer_ahead"):
        for c in caches:
            c.reset()
        for pr in preds:
            pr.k_pred.fill_(k + (m or 0))
        log_fetch = torch.zeros((steps, layers, w.batch), dtype=torch.int32, device=device)
        log_pref = torch.zeros((steps, layers, w.batch), dtype=torch.int32, device=device)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        pending = [None] * layers
        last_step = [-1] * layers
        torch.cuda.synchronize()
        # a bounded device-side delay (about 10 ms) while the host enqueues the run
        torch.cuda._sleep(20_000_000)
        for s in range(steps):
            ev[s].record(compute)
            for l in range(layers):
                dec = decs[l]
                dec.select(qs[l][s], summ, seq_lens, gamma=w.gamma, scores_out=scores[l][s % 2])
                if pending[l] is not None:
                    compute.wait_event(pending[l])
                    pending[l] = None
                if m and mode == "step_ahead":
                    preds[l].from_scores(scores[l][s % 2], seq_lens)
                caches[l].fetch(host, N, seq_lens, dec.sel_idx, dec.n_sel)
                log_fetch[s, l].copy_(caches[l].n_fetched)
                last_step[l] = s
                fetched = torch.cuda.Event()
                fetched.record(compute)
                if m and mode == "step_ahead" and s + 1 < steps:
                    # this layer's next step, prefetched while the following layers run
                    copy.wait_event(fetched)
                    with torch.cuda.stream(copy):
                        caches[l].prefetch(host, N, seq_lens, preds[l].pred_idx, preds[l].n_pred,
                                           stream=copy)
                        log_pref[s + 1, l].copy_(caches[l].n_prefetched)
                    done = torch.cuda.Event()
                    done.record(copy)
                    pending[l] = done
                dec.attend(qs[l][s], caches[l].kv, seq_lens, use_dense_flag=False)
                nl = (l + 1) % layers
                if m and mode == "layer_ahead" and last_step[nl] >= 0 and (nl > l or s + 1 < steps):
                    copy.wait_event(fetched)
                    with torch.cuda.stream(copy):
                        preds[nl].from_scores(scores[nl][last_step[nl] % 2], seq_lens, stream=copy)
                        caches[nl].prefetch(host, N, seq_lens, preds[nl].pred_idx, preds[nl].n_pred,
                                            stream=copy)
                        log_pref[s if nl > l else s + 1, nl].copy_(caches[nl].n_prefetched)
                    done = torch.cuda.Event()
                    done.record(copy)
                    pending[nl] = done
        ev[steps].record(compute)
        torch.cuda.synchronize()
        err = K.kvsel_get_error()
        if err:
            raise RuntimeError(f"device error {err} in the layer-prefetch measurement")
        warm = slice(1, steps)
        crit = log_fetch[warm].sum().item() / ((steps - 1) * layers)
        pref = log_pref[warm].sum().item() / ((steps - 1) * layers)
        return {"layer_us": ev[1].elapsed_time(ev[steps]) * 1e3 / ((steps - 1) * layers),
                "critical_blocks": crit, "prefetched_blocks": pref}

    variants = [(None, None)] + [(m, mode) for mode in ("layer_ahead", "step_ahead") for m in ms]
    gc_was_on = gc.isenabled()
    gc.disable()
    try:
        runs = {v: [] for v in variants}
        for _ in range(rounds):
            for v in variants:
                runs[v].append(run(*v))
    finally:
        if gc_was_on:
            gc.enable()
    out = {"layers": layers, "steps": steps, "rho": rho, "k": k, "slots": slots, "rounds": rounds,
           "predictor": "Top-(k + m) of the layer's previous-step scores",
           "layer_ahead": "prediction and prefetch of layer l+1 on the copy stream once layer l's fetch is done",
           "step_ahead": ("prediction on the compute stream after the layer's select; the prefetch of its "
                          "next step on the copy stream once its fetch is done")}
    base = None
    for v in variants:
        med = {key: statistics.median(r[key] for r in runs[v]) for key in runs[v][0]}
        row = {"layer_us": med["layer_us"],
               "layer_us_per_round": [round(r["layer_us"], 1) for r in runs[v]],
               "critical_link_bytes_per_layer_step": med["critical_blocks"] * page_bytes,
               "prefetch_link_bytes_per_layer_step": med["prefetched_blocks"] * page_bytes}
        if v[0] is None:
            base = row
            # the share of the layer-step in which the compute stream's fetch leaves the link idle
            row["link_idle_fraction"] = 1.0 - (row["critical_link_bytes_per_layer_step"]
                                               / (h2d_gbs * 1e9 * row["layer_us"] * 1e-6))
            out["without_prefetch"] = row
        else:
            row["speedup_vs_without"] = base["layer_us"] / row["layer_us"]
            row["critical_bytes_vs_without"] = (row["critical_link_bytes_per_layer_step"]
                                                / max(1.0, base["critical_link_bytes_per_layer_step"]))
            out[f"{v[1]}_m_{v[0]}"] = row
    del caches, decs
    torch.cuda.empty_cache()
    return out


def run_copy_unit_sweep(device, K, host, timed, h2d_gbs, reps=5):
    """Does the size of one copied unit matter on this link? The span gather
    on 64 sequences whose selection is every 16th block (spans of one block,
    so every unit is one page) for pages of 16, 32, 64 and 256 KiB (block
    sizes 16 / 32 / 64 with 2 KV heads, 64 with 8), d 128, over the first
    GiB of the pinned host tier viewed in each layout."""
    import torch
    from query_aware_sparse_block_gb300 import kvsel as KK

    out = []
    flat = host.view(-1)[: 1 << 29]                 # 1 GiB of bf16
    for B, Hkv in ((16, 2), (32, 2), (64, 2), (64, 8)):
        page = (Hkv, 2, 2, B, 64)
        page_elems = int(np.prod(page))
        batch = 64
        N = flat.numel() // (batch * page_elems)
        k = N // 16
        tier = flat[: batch * N * page_elems].view((batch, N) + page)
        p = KK.problem(batch, 4 * Hkv, Hkv, 128, B, N, k)
        i32 = dict(dtype=torch.int32, device=device)
        starts = (torch.arange(k, **i32) * 16).repeat(batch, 1).contiguous()
        lens = torch.ones((batch, k), **i32)
        n_spans = torch.full((batch,), k, **i32)
        seq_lens = torch.full((batch,), N * B, **i32)
        staging = torch.empty((batch, k) + page, dtype=torch.bfloat16, device=device)
        kv = KK.kv_host(tier, N, staging, k)
        t = timed(lambda: KK.kvsel_fetch_spans(p, kv, seq_lens, starts, lens, n_spans, None), reps)
        nbytes = batch * k * page_elems * 2
        out.append({"page_kib": page_elems * 2 // 1024, "units_per_step": batch * k,
                    "bytes_per_step": nbytes, "fetch_us": t * 1e6, "gbs": nbytes / t / 1e9,
                    "frac_of_h2d_copy": nbytes / t / 1e9 / h2d_gbs})
        del staging
    err = K.kvsel_get_error()
    if err:
        raise RuntimeError(f"device error {err} in the copy-unit sweep")
    return out


def run_block_cache(device, K, w, host, page, summ, x, timed, h2d_gbs, uncached_us, steps=8,
                    rho=0.95, repeats=5):
    """The floor selection (k = 102 of 2048 blocks) served through the GPU
    block cache (kvsel_cache_fetch, 2k slots per sequence) over consecutive
    steps whose queries drift, q_s = rho q_(s-1) + sqrt(1 - rho^2) e_s with
    e_s ~ N(0, 1): per warm step the blocks that crossed the link, the hit
    rate, the fetch time and rate against the measured copy rate, and select
    + fetch + attend against the uncached gather + attend. The eight-step leg
    runs `repeats` times from an empty cache with the same seeded drift (the
    same selections); the headline figures are medians over the repeats, and
    the SM clocks sampled during the repeats are reported beside them."""
    reps = []
    clocks = ClockSampler(torch_device_index(device))
    clocks.start()
    for _ in range(repeats):
        reps.append(_block_cache_leg(device, K, w, host, page, summ, x, h2d_gbs, uncached_us, steps, rho))
    clk = clocks.stop()
    out = dict(reps[0])
    for key in ("fetch_us", "fetch_gbs", "frac_of_h2d_copy", "select_fetch_attend_us", "fetch_gbs_median_step"):
        out[key] = statistics.median(r[key] for r in reps)
    out["repeats"] = repeats
    out["fetch_gbs_per_repeat"] = [round(r["fetch_gbs"], 1) for r in reps]
    out["clocks"] = clk
    return out


def torch_device_index(device):
    import torch
    return torch.device(device).index or 0


def _block_cache_leg(device, K, w, host, page, summ, x, h2d_gbs, uncached_us, steps, rho):
    import torch
    from query_aware_sparse_block_gb300.runtime import HostBlockCache, SparseDecoder

    N = w.n_blocks
    k = w.k_for(w.keep_floor)
    page_bytes = int(np.prod(page)) * 2
    dec = SparseDecoder(w.batch, w.n_qheads, w.n_kvheads, w.head_dim, w.block_size, x["max_blocks"],
                        k_max=k, device=device)
    dec.k_per_seq.fill_(k)
    cache = HostBlockCache(dec, 2 * k, page)
    g = torch.Generator(device=device).manual_seed(4242)
    q = x["q"].float()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    rows, host_us = [], []
    # no collector pause may fall between two of a step's calls (the events
    # would then time an idle GPU)
    gc_was_on = gc.isenabled()
    gc.disable()
    try:
        for step in range(steps):
            if step:
                q = rho * q + math.sqrt(1 - rho * rho) * torch.randn(q.shape, generator=g, device=device)
            qb = q.to(torch.bfloat16)
            torch.cuda.synchronize()
            # a bounded device-side delay (about 4 ms) while the host enqueues the
            # whole step, so that the events time the GPU and not the host calls
            torch.cuda._sleep(8_000_000)
            ev[0].record()
            dec.select(qb, summ, x["seq_lens"], gamma=w.gamma)
            ev[1].record()
            h0 = time.perf_counter()
            cache.fetch(host, N, x["seq_lens"], dec.sel_idx, dec.n_sel)
            host_us.append((time.perf_counter() - h0) * 1e6)
            ev[2].record()
            dec.attend(qb, cache.kv, x["seq_lens"], use_dense_flag=False)
            ev[3].record()
            torch.cuda.synchronize()
            if int(dec.dense_flag.sum()):
                raise RuntimeError("a sequence went dense at the keep floor")
            fetched = int(cache.n_fetched.sum())
            rows.append((fetched, ev[1].elapsed_time(ev[2]) * 1e3, ev[0].elapsed_time(ev[3]) * 1e3))
    finally:
        if gc_was_on:
            gc.enable()
    err = K.kvsel_get_error()
    if err:
        raise RuntimeError(f"device error {err} in the block-cache measurement")
    warm = rows[1:]
    blocks = statistics.mean(r[0] for r in warm)
    fetch_us = statistics.mean(r[1] for r in warm)
    step_us = statistics.mean(r[2] for r in warm)
    link = blocks * page_bytes
    del cache
    torch.cuda.empty_cache()
    return {"k": k, "slots": 2 * k, "rho": rho, "steps": steps,
            "cold_step_blocks": rows[0][0], "blocks_per_step": blocks,
            "hit_rate": 1.0 - blocks / (w.batch * k), "link_bytes_per_step": link,
            "fetch_us": fetch_us, "fetch_gbs": link / (fetch_us / 1e6) / 1e9,
            "frac_of_h2d_copy": link / (fetch_us / 1e6) / 1e9 / h2d_gbs,
            "fetch_gbs_median_step": statistics.median(r[0] * page_bytes / r[1] / 1e3 for r in warm),
            "select_fetch_attend_us": step_us, "uncached_fetch_plus_attend_us": uncached_us,
            "fetch_call_host_us": statistics.median(host_us),
            "per_step": [[r[0], round(r[1], 1)] for r in rows]}


# ------------------------------------------------------ oracle (reference) ---

def oracle_sample_inputs(n_seqs: int):
    """One layer of the workload on the CPU, restricted to the first sequences."""
    from workloads import C3
    from workloads.generate import bits, generate_layer, logical_kv

    w = C3.scaled(batch=n_seqs)
    x = generate_layer(w, 0, device="cpu", perm=False)
    seqs = []
    for b in range(n_seqs):
        seqs.append(dict(q=bits(x["q"][b]), k=bits(logical_kv(x["kv_pages"], x["block_table"], b, w.seq_len, 0)),
                         v=bits(logical_kv(x["kv_pages"], x["block_table"], b, w.seq_len, 1))))
    return w, seqs


def oracle_step(w, seqs, k, scale, state):
    """The decode step of one layer on the sampled sequences, in the oracle:
    append of the last token into the open block, score, Top-k, spans, gamma
    rule and attention over the selected blocks."""
    import oracle as o

    T = w.seq_len
    for s, st in zip(seqs, state):
        _, sb_open = o.append_token(st["acc"], s["k"][T - 1], T - 1, w.block_size)
        summ = st["bits"].copy()
        summ[(T - 1) // w.block_size] = sb_open
        scores = o.block_scores(s["q"], summ)
        sel = o.topk_blocks(scores, k)
        starts, _ = o.merge_spans(sel)
        dense = o.dense_fallback(len(starts), len(sel), len(scores), w.gamma, 0.0)
        blocks = np.arange(len(scores)) if dense else sel
        o.attend(s["q"], s["k"], s["v"], o.tokens_of_blocks(blocks, T, w.block_size), scale)


def oracle_state(w, seqs):
    """Summaries of the first T-1 tokens and the open block's accumulator."""
    import oracle as o

    state = []
    for s in seqs:
        bits_, _, acc = o.block_summaries(s["k"], w.seq_len - 1, w.block_size)
        full = np.zeros((w.n_blocks,) + bits_.shape[1:], dtype=np.uint16)
        full[: bits_.shape[0]] = bits_
        state.append(dict(bits=full, acc=acc))
    return state


def _oracle_worker(n_seqs, reps, out_path):
    w, seqs = oracle_sample_inputs(n_seqs)
    state = oracle_state(w, seqs)
    k = w.k_for(w.keep[0])
    scale = 1.0 / math.sqrt(w.head_dim)
    times = []
    t_start = time.perf_counter()
    while len(times) < reps or time.perf_counter() - t_start < 10.0:
        t = time.perf_counter()
        oracle_step(w, seqs, k, scale, state)
        times.append(time.perf_counter() - t)
    with open(out_path, "w") as f:
        json.dump({"times": times, "n_seqs": n_seqs, "batch": 16}, f)


def _oracle_timing(n_seqs: int, reps: int, threads: int):
    """Median seconds per sample step of the oracle in a fresh process whose
    BLAS / OpenMP thread count is `threads`, and the number of steps timed."""
    env = dict(os.environ)
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[v] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    with tempfile.TemporaryDirectory() as td:
        out = os.path.join(td, "o.json")
        code = (f"import sys; sys.path.insert(0, {ROOT!r}); import bench; "
                f"bench._oracle_worker({n_seqs}, {reps}, {out!r})")
        subprocess.run([sys.executable, "-c", code], env=env, check=True, timeout=900)
        with open(out) as f:
            r = json.load(f)
    return statistics.median(r["times"]), r["batch"] / r["n_seqs"], len(r["times"])


def cpu_baseline_subprocess(n_seqs: int, reps: int):
    """Times the oracle in fresh processes with the BLAS thread count pinned:
    once on every host core this process may use, once on one core."""
    cores = len(os.sched_getaffinity(0))
    t, scale, n = _oracle_timing(n_seqs, reps, cores)
    t1, _, n1 = _oracle_timing(n_seqs, reps, 1)
    return {"value": 1.0 / (t * scale), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"one layer, {n_seqs} of 16 sequences (append, score, Top-k, spans, "
                      f"attention over 128 blocks), repeated for >= 10 s ({n} reps on {cores} cores, "
                      f"{n1} on one); median rep scaled to a 16-sequence layer-step",
            "seconds_per_sample": t,
            "single_thread": {"value": 1.0 / (t1 * scale), "unit": UNIT, "cores": 1,
                              "seconds_per_sample": t1}}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from workloads import C3

    cores = len(os.sched_getaffinity(0))
    w, seqs = oracle_sample_inputs(args.ref_seqs)
    state = oracle_state(w, seqs)
    k = w.k_for(w.keep[0])
    scale = 1.0 / math.sqrt(w.head_dim)
    for _ in range(args.warmup):
        oracle_step(w, seqs, k, scale, state)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(w, seqs, k, scale, state)
    el = time.perf_counter() - t
    sample_step_s = el / args.steps
    per_layer_step = sample_step_s * (C3.batch / args.ref_seqs)
    value = 1.0 / per_layer_step
    sample = (f"each timed step: one layer, {args.ref_seqs} of {C3.batch} sequences of {C3.name} "
              f"(append, score, Top-k, spans, attention); value = that rate scaled to a "
              f"{C3.batch}-sequence layer-step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sample_step_s * 1e3,
            "step": f"one layer of {args.ref_seqs} sequences (the timed sample)",
            "scaled_to_workload": {"ms_per_layer_step": per_layer_step * 1e3,
                                   "ms_per_step_all_layers": per_layer_step * 1e3 * C3.layers,
                                   "sequences": C3.batch, "layers": C3.layers},
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": C3.name, "batch": C3.batch, "n_qheads": C3.n_qheads,
                       "n_kvheads": C3.n_kvheads, "head_dim": C3.head_dim, "seq_len": C3.seq_len,
                       "block_size": C3.block_size, "keep": C3.keep[0], "k": k, "layers": C3.layers,
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
