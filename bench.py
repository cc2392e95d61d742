#!/usr/bin/env python3
"""Benchmark of one decode step of GQA attention over a paged KV cache on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                    [--config NAME] [--per-call] [--no-extra-configs]

A step is one pass of the whole hot path (RoPE + append + split-KV attention
+ merge) over one batch.  The default workload is the largest configuration:
the Qwen3-8B-shaped continuous batch (32/8 heads, d 128, batch 64, cached
lengths log-uniform in [128, 8192], page 16) over its 36 independent layer
caches, decoded by one kvattn_decode_layers call per step (``--per-call``:
one kvattn_decode call per layer cache instead).  Inputs are seeded synthetic
N(0, 1) draws already resident in HBM; a step reads 18 GB of K/V, far above
the 129 MB L2 (single-layer configs rotate over independent caches whose
total is at least 4x L2).  The timed window is replayed from CUDA graphs that
each hold many consecutive steps, so no host launch gap falls inside it, and
is timed with CUDA events on the launching stream; rank 0 prints one JSON
line.  Every other configuration is timed in the same run under
``per_config``, each with its own roofline and end-to-end figure.

With N > 1 (torchrun) every rank decodes its own batch (weak scaling, no data
exchange); the timing is the max over ranks.  ``--impl reference`` times the
CPU oracle (the only reference this method has) on a bounded sample of the
same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from decode_phase_gqa_gb300 import workloads as W  # noqa: E402

METRIC = "decode-attn tokens/s and KV-read HBM GB/s (% of GB300 peak) per config"
PRIMARY = "qwen3"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
SRC_FILES = ["decode_common.cuh", "decode_mma.cuh", "kvattn_internal.cuh", "angle_table.inc",
             "storage.cuh", "kvattn_api.cu", "decode_bf16.cu", "decode_int8.cu",
             "decode_bf16_layers.cu", "decode_int8_layers.cu", "combine.cu"]


def workload_desc(wl: W.Workload) -> str:
    return {
        "tiny": "Tiny: 1 seq, 4/1 heads, d64, 256 cached + 1 new, page 16",
        "smollm3": "SmolLM3-3B-shaped layer: 16/4 heads, d128, batch 8, L~U[512,4096], page 16",
        "qwen3": "Qwen3-8B-shaped continuous batch: 32/8 heads, d128, batch 64, "
                 "L log-uniform [128,8192], page 16, 36 layer caches per step",
        "llama1b": "Llama-3.2-1B-shaped long context: 32/8 heads, d64, batch 32, "
                   "half L=32768, half L~U[1,2048], page 16",
        "int8": "Int8 KV cache, Qwen3-8B-shaped: 32/8 heads, d128, batch 128, "
                "L~U[1024,4096], page 16, per-token-per-head fp32 scales",
        "qwen3_b512": "Qwen3-8B-shaped large continuous batch: 32/8 heads, d128, batch 512, "
                      "L log-uniform [128,8192], page 16, one layer cache",
    }.get(wl.name, wl.name)


# --------------------------------------------------------------- dist ---

def dist_setup(use_gpu: bool = True):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (use_gpu and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (timing plumbing, not a data path)."""
    if world == 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------- clocks ---

class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self, t_start: float, t_end: float):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [r for r in rows if t_start <= r[0] <= t_end] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside)}


# ------------------------------------------------------------- native ---

def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in SRC_FILES:
        with open(os.path.join(ROOT, "decode_phase_gqa_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(config: str):
    """DRAM bytes per decode-kernel launch from the committed ncu summary, if it
    was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(config)
    if not entry or entry.get("source_hash") != kernel_source_hash():
        return None
    return entry.get("dram_bytes_per_launch")


class NativeCase:
    """Device-resident inputs of one config: `copies` independent caches (or the
    36 layer caches of the Qwen config), one workspace, one output buffer."""

    def __init__(self, name: str, seed: int, device, min_bytes: int = 4 * L2_BYTES,
                 layers=None, layered=False):
        from decode_phase_gqa_gb300 import kvattn as K
        self.K = K
        self.wl = W.make_workload(name, seed=seed)
        wl = self.wl
        if layers is not None:   # fewer layer caches per step (profiling runs only)
            wl.layers = max(1, min(wl.layers, layers))
        self.device = device
        # a step of a multi-layer config: one kvattn_decode call per layer cache,
        # or (layered) one kvattn_decode_layers call over all of them
        self.layered = bool(layered) and wl.layers > 1
        self.calls_per_step = 1 if self.layered else wl.layers
        per_cache = wl.kv_bytes
        if wl.layers > 1:
            self.copies = wl.layers           # a step reads every layer cache once
        else:
            # enough independent caches that a rotation reads min_bytes of KV;
            # capped for latency-bound toy shapes (their KV sits in L2 anyway)
            self.copies = min(64, max(2, math.ceil(min_bytes / max(per_cache, 1))))
        self.l2_resident = self.copies * per_cache * wl.layers < 2 * L2_BYTES
        if wl.layers > 1:
            # layer caches in layer-major arrays (what kvattn_decode_layers
            # takes); the per-layer calls use views of them
            self.stacked = {}
            for i in range(self.copies):
                t = W.make_tensors(wl, layer=i, device=device)
                for k, v in t.items():
                    if v is None:
                        self.stacked[k] = None
                        continue
                    if k not in self.stacked:
                        self.stacked[k] = torch.empty((self.copies,) + tuple(v.shape),
                                                      dtype=v.dtype, device=device)
                    self.stacked[k][i].copy_(v)
                del t
            self.caches = [{k: (None if v is None else v[i]) for k, v in self.stacked.items()}
                           for i in range(self.copies)]
        else:
            self.caches = [W.make_tensors(wl, layer=i, device=device) for i in range(self.copies)]
        self.bt = torch.from_numpy(wl.block_table).to(device)
        self.sl = torch.from_numpy(wl.seq_lens).to(device)
        self.pos = torch.from_numpy(wl.positions).to(device)
        lead = (wl.layers,) if self.layered else ()
        self.out = torch.empty(lead + (wl.n_seq, wl.n_qh, wl.head_dim), dtype=torch.bfloat16,
                               device=device)
        self.ws = K.alloc_workspace(wl.n_seq, wl.n_qh, wl.n_kvh, wl.head_dim, device=device,
                                    n_layers=wl.layers if self.layered else 1)
        self.graphs = []

    def call(self, i, stream=None, out=None):
        if self.layered:
            c = self.stacked
            self.K.kvattn_decode_layers(
                c["q"], c["k_new"], c["v_new"], c["k_pages"], c["v_pages"], self.bt, self.sl,
                self.pos, self.out if out is None else out, rope_theta=self.wl.rope_theta,
                scale=self.wl.scale, workspace=self.ws, k_scales=c["k_scales"],
                v_scales=c["v_scales"], stream=stream)
            return
        c = self.caches[i]
        self.K.kvattn_decode(c["q"], c["k_new"], c["v_new"], c["k_pages"], c["v_pages"],
                             self.bt, self.sl, self.pos, self.out if out is None else out,
                             rope_theta=self.wl.rope_theta, scale=self.wl.scale,
                             workspace=self.ws, k_scales=c["k_scales"], v_scales=c["v_scales"],
                             stream=stream)

    def step_groups(self):
        """Cache indices of each distinct step (a step = calls_per_step calls)."""
        if self.layered:
            return [[0]]
        if self.calls_per_step > 1:
            return [list(range(self.copies))]
        return [[i] for i in range(self.copies)]

    def capture(self, stream):
        """One graph per step (its calls), used for the warm-up steps."""
        for grp in self.step_groups():
            for i in grp:          # warm the library's per-device set-up first
                self.call(i, stream)
        torch.cuda.synchronize()
        for grp in self.step_groups():
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in grp:
                    self.call(i, stream)
            self.graphs.append(g)
        torch.cuda.synchronize()

    def replay(self, step):
        self.graphs[step % len(self.graphs)].replay()

    def capture_window(self, stream, first, n, max_calls=1024):
        """Graphs that replay steps first .. first + n - 1 (rotation order) with
        no host launch gap inside: a graph of C consecutive steps (C a multiple
        of the rotation's length, so every replay starts at the same cache),
        replayed n // C times, then a graph of the n % C steps left.  A graph
        holds at most max_calls library calls (two kernels each)."""
        groups = self.step_groups()
        r = len(groups)
        cap = max(1, max_calls // self.calls_per_step)
        assert r <= cap, "a rotation must fit one graph"
        chunk = n if n <= cap else r * (cap // r)

        def graph_of(k):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for s in range(first, first + k):
                    for i in groups[s % r]:
                        self.call(i, stream)
            return g

        self.window = [(graph_of(chunk), n // chunk)]
        if n % chunk:
            self.window.append((graph_of(n % chunk), 1))
        torch.cuda.synchronize()

    def replay_window(self):
        for g, reps in self.window:
            for _ in range(reps):
                g.replay()

    def check_status(self):
        return self.K.kvattn_read_device_status(self.ws)


def time_steps(case: NativeCase, steps: int, warmup: int, world: int, stream):
    case.capture_window(stream, warmup, steps)
    with torch.cuda.stream(stream):
        for s in range(warmup):
            case.replay(s)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.time()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        case.replay_window()
        end.record(stream)
        torch.cuda.synchronize()
        t1 = time.time()
        barrier(world)
    case.window = None
    return start.elapsed_time(end), (t0, t1)


def time_e2e(case: NativeCase, steps: int, warmup: int, world: int, stream):
    """Same step through the public API with the step's inputs in pinned host
    memory: the step's q/k_new/v_new (every call's) and block table, lengths
    and positions are laid out in one pinned staging buffer and copied to the
    device in one transfer, the decode call(s) run on views of the device copy,
    and the outputs of all calls are read back in one transfer, every step,
    inside the timed region."""
    n_calls = case.calls_per_step
    layered = case.layered  # one call over every layer cache (layer-major inputs)
    n_sets = 1 if (n_calls > 1 or layered) else 2  # packed input sets alternated over steps

    def layout():
        segs, off = [], 0
        for n in range(n_calls):
            for k in ("q", "k_new", "v_new"):
                t = case.stacked[k] if layered else case.caches[0][k]
                segs.append((("in", n, k), off, t.shape, t.dtype))
                off += -(-t.numel() * t.element_size() // 256) * 256
        for name, t in (("bt", case.bt), ("sl", case.sl), ("pos", case.pos)):
            segs.append(((name,), off, t.shape, t.dtype))
            off += -(-t.numel() * t.element_size() // 256) * 256
        return segs, off

    segs, total = layout()

    def views(buf):
        out = {}
        for key, off, shape, dtype in segs:
            nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
            out[key] = buf[off:off + nbytes].view(dtype).view(shape)
        return out

    host_packs = []
    for s in range(n_sets):
        hp = torch.empty(total, dtype=torch.uint8).pin_memory()
        v = views(hp)
        for n in range(n_calls):
            src = case.caches[(s * n_calls + n) % len(case.caches)]
            for k in ("q", "k_new", "v_new"):
                v[("in", n, k)].copy_((case.stacked[k] if layered else src[k]).cpu())
        v[("bt",)].copy_(case.bt.cpu())
        v[("sl",)].copy_(case.sl.cpu())
        v[("pos",)].copy_(case.pos.cpu())
        host_packs.append(hp)
    dev_pack = torch.empty(total, dtype=torch.uint8, device=case.out.device)
    dv = views(dev_pack)
    out_d = torch.empty((n_calls,) + tuple(case.out.shape), dtype=case.out.dtype, device=case.out.device)
    out_h = torch.empty(out_d.shape, dtype=out_d.dtype).pin_memory()
    h2d = sum(int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
              for _, _, shape, dtype in segs)
    d2h = out_h.numel() * out_h.element_size()

    def one_step(s):
        dev_pack.copy_(host_packs[s % n_sets], non_blocking=True)
        if layered:
            c = case.stacked
            case.K.kvattn_decode_layers(dv[("in", 0, "q")], dv[("in", 0, "k_new")],
                                        dv[("in", 0, "v_new")], c["k_pages"], c["v_pages"],
                                        dv[("bt",)], dv[("sl",)], dv[("pos",)], out_d[0],
                                        rope_theta=case.wl.rope_theta, scale=case.wl.scale,
                                        workspace=case.ws, k_scales=c["k_scales"],
                                        v_scales=c["v_scales"], stream=stream)
            out_h.copy_(out_d, non_blocking=True)
            return
        idxs = case.step_groups()[s % len(case.step_groups())]
        for n, i in enumerate(idxs):
            c = case.caches[i]
            case.K.kvattn_decode(dv[("in", n, "q")], dv[("in", n, "k_new")], dv[("in", n, "v_new")],
                                 c["k_pages"], c["v_pages"], dv[("bt",)], dv[("sl",)], dv[("pos",)],
                                 out_d[n], rope_theta=case.wl.rope_theta, scale=case.wl.scale,
                                 workspace=case.ws, k_scales=c["k_scales"], v_scales=c["v_scales"],
                                 stream=stream)
        out_h.copy_(out_d, non_blocking=True)

    with torch.cuda.stream(stream):
        for s in range(warmup):
            one_step(s)
        torch.cuda.synchronize()
        barrier(world)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for s in range(steps):
            one_step(s)
        end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    return start.elapsed_time(end), h2d, d2h


def cpu_baseline(name: str, seed: int, budget_s: float = 10.0):
    """The oracle, as it stands, on host copies of the same workload: whole
    decode steps of one cache repeated until the time budget is used."""
    import oracle
    wl = W.make_workload(name, seed=seed)
    t = W.make_tensors(wl, layer=0, device="cpu")
    bits = lambda x: None if x is None else (
        x.contiguous().view(torch.int16).numpy().view(np.uint16).copy()
        if x.dtype == torch.bfloat16 else x.contiguous().numpy().copy())
    h = {k: bits(v) for k, v in t.items()}
    threads = oracle.max_threads()
    seqs = 0
    t0 = time.time()
    n_steps = 0
    # a sequence subset per step keeps one step well under the budget on big configs
    order = np.arange(wl.n_seq)
    chunk = wl.n_seq
    while True:
        mask = np.zeros(wl.n_seq, np.uint8)
        sel = order[(n_steps * chunk) % wl.n_seq:][:chunk]
        mask[sel] = 1
        ts = time.time()
        oracle.decode(h["q"], h["k_new"], h["v_new"], h["k_pages"], h["v_pages"],
                      wl.block_table, wl.seq_lens, wl.positions, wl.rope_theta, wl.scale,
                      h["k_scales"], h["v_scales"], seq_mask=mask, n_threads=threads)
        dt = time.time() - ts
        seqs += int(mask.sum())
        n_steps += 1
        if dt > budget_s / 4 and chunk > 1:
            chunk = max(1, chunk // 2)
        if time.time() - t0 >= budget_s:
            break
    elapsed = time.time() - t0
    # one new token of a sequence needs one decode per layer cache
    value = seqs / elapsed / wl.layers
    return {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{n_steps} oracle steps over {seqs} sequences of one {wl.name} layer cache"
                      f" ({elapsed:.1f} s, fp64, OpenMP over (sequence, KV head)); a step of "
                      f"{wl.layers} layer(s) costs {wl.layers}x one layer"}


def measured_bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def run_prefill_config(kind, steps, warmup, device, stream, seed=0):
    """kvattn_prefill timed from a CUDA graph of one call.

    prefill: SmolLM3-3B-shaped heads (16/4, d 128), 8 prompts of 2048 tokens
             into empty caches (compute-bound: causal attention FLOPs);
    verify:  Qwen3-8B-shaped heads (32/8, d 128) over the Qwen3 workload's 64
             cache lengths, 4 draft tokens each (a speculative step's check;
             bandwidth-bound: the cached K/V are read once per group);
    verify_int8: the same over an int8 cache (codes + per-row fp32 scales).
    """
    from decode_phase_gqa_gb300 import kvattn as K
    if kind == "prefill":
        n_qh, n_kvh, d, theta = 16, 4, 128, 1e6
        ctx = np.zeros(8, np.int64)
        n_new = np.full(8, 2048, np.int64)
    else:
        q3 = W.make_workload("qwen3", seed=seed)
        n_qh, n_kvh, d, theta = q3.n_qh, q3.n_kvh, q3.head_dim, q3.rope_theta
        ctx = q3.seq_lens.astype(np.int64)
        n_new = np.full(len(ctx), 4, np.int64)
    wl = W.make_workload("custom", seed=seed, n_seq=len(ctx), n_qh=n_qh, n_kvh=n_kvh,
                         head_dim=d, page_size=16, rope_theta=theta,
                         kv_dtype="int8" if kind == "verify_int8" else "bf16",
                         lengths=[int(x) for x in ctx + n_new - 1], spare=0.05)
    t = W.make_tensors(wl, device=device)
    g = torch.Generator(device=device).manual_seed(seed + 77)
    T = int(n_new.sum())
    q = torch.randn((T, n_qh, d), generator=g, device=device).to(torch.bfloat16)
    kn = torch.randn((T, n_kvh, d), generator=g, device=device).to(torch.bfloat16)
    vn = torch.randn((T, n_kvh, d), generator=g, device=device).to(torch.bfloat16)
    out = torch.empty_like(q)
    bt = torch.from_numpy(wl.block_table).to(device)
    ss = torch.from_numpy(np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)).to(device)
    cl = torch.from_numpy(ctx.astype(np.int32)).to(device)
    st = torch.zeros(1, dtype=torch.int32, device=device)
    ws = torch.empty(K.kvattn_prefill_workspace_size(T, n_qh, d), dtype=torch.uint8, device=device)

    def call():
        K.kvattn_prefill(q, kn, vn, t["k_pages"], t["v_pages"], bt, ss, cl, out,
                         rope_theta=theta, scale=1.0 / math.sqrt(d), max_new_tokens=int(n_new.max()),
                         k_scales=t.get("k_scales"), v_scales=t.get("v_scales"),
                         dev_status=st, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        call()   # per-device set-up outside the capture
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=stream):
            call()
        for _ in range(warmup):
            gr.replay()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(steps):
            gr.replay()
        t1.record(stream)
        torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise RuntimeError(f"prefill device status {int(st.item()):#x}")
    ms = t0.elapsed_time(t1) / steps

    # End to end through the public API: the call's inputs (new-token rows,
    # block table, row starts, cached lengths) copied every step from pinned
    # host memory, the output read back, all inside the timed region.
    host_in = [(x, x.cpu().pin_memory()) for x in (q, kn, vn, bt, ss, cl)]
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(h.numel() * h.element_size() for _, h in host_in)
    d2h = out_h.numel() * out_h.element_size()

    def e2e_step():
        for dv, hv in host_in:
            dv.copy_(hv, non_blocking=True)
        call()
        out_h.copy_(out, non_blocking=True)

    e2e_steps = max(10, min(steps, 100))
    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise RuntimeError(f"prefill device status {int(st.item()):#x}")
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    keys = float(np.sum(n_new * ctx + n_new * (n_new + 1) // 2))  # sum over new tokens of keys seen
    flops = 4.0 * d * n_qh * keys
    row_bytes = 2 * d + 8 if kind == "verify_int8" else 2 * d * 2  # a K and a V row (+ scales)
    kv_bytes = float(np.sum(ctx + n_new)) * n_kvh * row_bytes
    peak_tf, peak_kind = measured_bf16_peak()
    peak_gb, peak_gb_kind = measured_peak()
    res = {"config": kind, "entry": "kvattn_prefill",
           "workload": ("SmolLM3-3B-shaped heads 16/4, d128: 8 prompts x 2048 new tokens, empty caches"
                        if kind == "prefill" else
                        "Qwen3-8B-shaped heads 32/8, d128: 64 sequences, L log-uniform [128,8192], "
                        "4 draft tokens each" + (", int8 cache" if kind == "verify_int8" else "")),
           "steps": steps, "ms_per_step": ms, "new_tokens_per_s": T / (ms / 1e3),
           "attn_tflops": flops / (ms / 1e3) / 1e12, "bf16_peak_tflops": peak_tf,
           "frac_of_bf16_peak": flops / (ms / 1e3) / 1e12 / peak_tf, "peak_kind": peak_kind,
           "kv_read_gbs": kv_bytes / (ms / 1e3) / 1e9,
           "kv_read_frac_of_peak": kv_bytes / (ms / 1e3) / 1e9 / peak_gb}
    kernels = ("prefill_append_kernel, then the attention kernel (tcgen05 for these prompts) "
               "and its split merge, timed together per library call" if kind == "prefill" else
               "prefill_append_kernel, prefill_short_kernel (4 new tokens x 4 heads a tile) and "
               "the split merge, timed together per library call")
    if kind == "prefill":
        achieved = flops / (ms / 1e3) / 1e12
        res["roofline"] = {"bound": "tensor", "achieved": achieved, "peak": peak_tf,
                           "unit": "TFLOP/s", "frac": achieved / peak_tf, "peak_kind": peak_kind,
                           "algorithmic_flops_per_launch": flops, "launch_us": ms * 1e3,
                           "traffic": None, "kernel": kernels}
    else:
        achieved = kv_bytes / (ms / 1e3) / 1e9
        res["roofline"] = {"bound": "hbm", "achieved": achieved, "peak": peak_gb, "unit": "GB/s",
                           "frac": achieved / peak_gb, "peak_kind": peak_gb_kind,
                           "algorithmic_bytes_per_launch": kv_bytes, "launch_us": ms * 1e3,
                           "traffic": None, "kernel": kernels}
    res["e2e"] = {"value": T / (e2e_ms / 1e3), "unit": "new tokens/s", "ms_per_step": e2e_ms,
                  "steps": e2e_steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    del t, q, kn, vn, out, ws
    torch.cuda.empty_cache()
    return res


ENTRY_LAYERS = "kvattn_decode_layers (one call over the layer caches)"
ENTRY_CALL = "kvattn_decode"


def run_config(name, steps, warmup, rank, world, device, stream, with_e2e=True, layers=None,
               layered=False):
    case = NativeCase(name, seed=1000 * rank, device=device, layers=layers, layered=layered)
    case.capture(stream)
    st = case.check_status()
    if st:
        raise RuntimeError(f"device status {st:#x} on {name}")
    ms, window = time_steps(case, steps, warmup, world, stream)
    ms = max_over_ranks(ms, world, device)
    wl = case.wl
    ms_step = ms / steps
    kv_bytes_step = wl.kv_bytes * wl.layers
    res = {
        "name": name, "ms_per_step": ms_step,
        "tokens_per_s": wl.n_seq * world * steps / (ms / 1e3),
        "kv_gbs": kv_bytes_step * world / (ms_step / 1e3) / 1e9,
        "kv_bytes_per_step": kv_bytes_step,
        "calls_per_step": case.calls_per_step, "copies": case.copies,
        "window": window, "case": case,
    }
    if with_e2e:
        e2e_ms, h2d, d2h = time_e2e(case, steps, warmup, world, stream)
        e2e_ms = max_over_ranks(e2e_ms, world, device)
        res["e2e"] = {"value": wl.n_seq * world * steps / (e2e_ms / 1e3), "unit": "tokens/s",
                      "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}
    return res


def roofline_of(r, world, peak, peak_kind):
    """Roofline of the dominant kernel of one library call: algorithmic K+V
    bytes of the call / the call's event-timed duration (its decode kernel and
    the small merge kernel that follows it, timed together)."""
    case = r["case"]
    per_call_ms = r["ms_per_step"] / r["calls_per_step"]
    call_bytes = r["kv_bytes_per_step"] / r["calls_per_step"]
    achieved = call_bytes / (per_call_ms / 1e3) / 1e9
    return {
        "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
        "frac": achieved / peak, "peak_kind": peak_kind,
        "algorithmic_bytes_per_launch": call_bytes,
        "launch_us": per_call_ms * 1e3,
        "traffic": recorded_traffic(r["name"] + ("_layers" if case.layered else "")),
        "kernel": "decode_mma_kernel (RoPE, append, split-KV attention) with its merge "
                  "kernel, timed together per library call",
    }


def config_entry(r, world, peak, peak_kind):
    """per_config entry of a timed decode configuration."""
    case = r["case"]
    wl = case.wl
    e = {"config": r["name"], "workload": workload_desc(wl),
         "entry": ENTRY_LAYERS if case.layered else ENTRY_CALL,
         "steps": r["steps"], "ms_per_step": r["ms_per_step"],
         "l2_resident": case.l2_resident,
         "tokens_per_s": r["tokens_per_s"], "kv_read_gbs": r["kv_gbs"],
         "kv_read_frac_of_peak": r["kv_gbs"] / world / peak,
         "calls_per_step": r["calls_per_step"],
         "roofline": roofline_of(r, world, peak, peak_kind)}
    if "e2e" in r:
        e["e2e"] = r["e2e"]
    return e


def steps_for(name, layered, peak, budget_ms=300.0):
    """Timed steps of an extra configuration: about budget_ms of device time."""
    wl = W.make_workload(name)
    step_ms = max(wl.kv_bytes * wl.layers / (0.7 * peak * 1e9) * 1e3, 0.01)
    return max(10, min(2000, int(budget_ms / step_ms)))


def native(args, rank, world, local):
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from decode_phase_gqa_gb300 import build as B
    B.build()
    stream = torch.cuda.Stream(device)
    peak, peak_kind = measured_peak()
    layered_main = not args.per_call
    with ClockSampler(local) as clocks:
        main = run_config(args.config, args.steps, args.warmup, rank, world, device, stream,
                          layers=args.layers, layered=layered_main)
    main["steps"] = args.steps
    clk = clocks.summary(*main["window"])
    wl = main["case"].wl
    line = {
        "metric": METRIC,
        "value": main["tokens_per_s"],
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": main["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if wl.kv_dtype == "bf16" else "int8",
        "data": "synthetic (seeded N(0,1) q/k/v and KV pages, no weights)",
        "config": {
            "workload": workload_desc(wl), "n_seq": wl.n_seq, "n_qh": wl.n_qh,
            "n_kvh": wl.n_kvh, "head_dim": wl.head_dim, "page_size": wl.page_size,
            "kv_dtype": wl.kv_dtype, "layer_caches_per_step": wl.layers,
            "entry": ENTRY_LAYERS if main["case"].layered else ENTRY_CALL,
            "kv_bytes_per_step": main["kv_bytes_per_step"],
            "kv_read_gbs": main["kv_gbs"],
            "kv_read_frac_of_peak": main["kv_gbs"] / world / peak,
            "l2": (f"inputs larger than L2: each step reads "
                   f"{main['kv_bytes_per_step'] / 2**20:.0f} MiB of KV"
                   + (f" ({main['copies']} independent caches rotated)"
                      if wl.layers == 1 else f" over {wl.layers} layer caches")),
            "timing": "CUDA events on the launching stream around K steps replayed from "
                      "CUDA graphs of many consecutive steps (no host launch gap inside)",
            "parallelism": f"{world} independent replica(s), one batch per GPU",
        },
        "roofline": roofline_of(main, world, peak, peak_kind),
        "e2e": main["e2e"],
        # decode (with the append) and combine kernels per call
        "gpu_launches": 2 * main["calls_per_step"] * args.steps,
        "clocks": {k: clk[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "impl": "native",
    }
    main_layered = main["case"].layered
    del main["case"]
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.config, seed=0)
    if not args.no_extra_configs:
        extra = []
        for name in W.CONFIG_ORDER + W.EXTRA_CONFIGS:
            wl2 = W.make_workload(name)
            # a multi-layer step is timed both ways: one kvattn_decode_layers
            # call over all layer caches, and one kvattn_decode call per cache
            for layered in ([True, False] if wl2.layers > 1 else [False]):
                if name == args.config and layered == main_layered:
                    continue
                k = steps_for(name, layered, peak)
                r = run_config(name, k, max(3, k // 10), rank, world, device, stream,
                               layered=layered)
                r["steps"] = k
                extra.append(config_entry(r, world, peak, peak_kind))
                del r
                torch.cuda.empty_cache()
        for kind, k in (("prefill", 20), ("verify", 200), ("verify_int8", 200)):
            extra.append(run_prefill_config(kind, k, 3, device, stream))
        line["per_config"] = extra
    return line


# ---------------------------------------------------------- reference ---

def reference(args, rank, world):
    """The oracle as the reference arm: CPU fp64, host cores, bounded samples."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    wl = W.make_workload(args.config, seed=0)
    t = W.make_tensors(wl, layer=0, device="cpu")
    bits = lambda x: None if x is None else (
        x.contiguous().view(torch.int16).numpy().view(np.uint16).copy()
        if x.dtype == torch.bfloat16 else x.contiguous().numpy().copy())
    h = {k: bits(v) for k, v in t.items()}
    threads = oracle.max_threads()

    def step(mask):
        oracle.decode(h["q"], h["k_new"], h["v_new"], h["k_pages"], h["v_pages"],
                      wl.block_table, wl.seq_lens, wl.positions, wl.rope_theta, wl.scale,
                      h["k_scales"], h["v_scales"], seq_mask=mask, n_threads=threads)

    # calibrate a whole-batch step, then size the per-step sample (whole sequences)
    full = np.ones(wl.n_seq, np.uint8)
    ts = time.time()
    step(full)
    full_s = time.time() - ts
    budget = 120.0 / max(1, args.steps + args.warmup)
    per_seq = full_s / wl.n_seq
    n_sample = int(max(1, min(wl.n_seq, budget / max(per_seq, 1e-9))))
    order = np.random.default_rng(0).permutation(wl.n_seq)

    def mask_for(s):
        m = np.zeros(wl.n_seq, np.uint8)
        m[np.take(order, np.arange(s * n_sample, (s + 1) * n_sample), mode="wrap")] = 1
        return m

    for s in range(args.warmup):
        step(mask_for(s))
    seqs = 0
    t0 = time.time()
    for s in range(args.steps):
        m = mask_for(args.warmup + s)
        step(m)
        seqs += int(m.sum())
    elapsed = time.time() - t0
    value = seqs / elapsed / wl.layers
    sample = (f"{n_sample} of {wl.n_seq} sequences per step of one {wl.name} layer cache "
              f"(fp64, OpenMP over (sequence, KV head)); steps of {wl.layers} layer(s) "
              f"scaled as {wl.layers}x one layer")
    return {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed / args.steps * 1e3 * wl.n_seq / n_sample * wl.layers,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), same recipe as the native arm)",
        "config": {"workload": workload_desc(wl), "n_seq": wl.n_seq, "n_qh": wl.n_qh,
                   "n_kvh": wl.n_kvh, "head_dim": wl.head_dim, "page_size": wl.page_size,
                   "kv_dtype": wl.kv_dtype},
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--config", choices=W.CONFIG_ORDER + W.EXTRA_CONFIGS, default=PRIMARY)
    ap.add_argument("--no-extra-configs", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--per-call", action="store_true",
                    help="time a multi-layer config's step as one kvattn_decode call per "
                         "layer cache (default: one kvattn_decode_layers call)")
    ap.add_argument("--layers", type=int, default=None,
                    help="decode at most this many layer caches per step (a smaller case "
                         "for profiling; the default is the workload's own count)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local = dist_setup(use_gpu=args.impl == "native")
    if args.impl == "reference":
        line = reference(args, rank, world)
    else:
        line = native(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
