#!/usr/bin/env python
"""Benchmark of the k-quant batch-1 decode GEMV path on GB300.

A step is one pass of the whole hot path over one synthetic decode token:
the q8 producer(s) followed by the GEMV(s) of the workload, with the weights
resident in HBM.  The default workload is the full Qwen2.5-14B-shaped decode
weight sweep: 48 layers x {q, k, v, o, gate, up, down} plus the 152064 x 5120
output head, 9.011 GB of k-quant weights per step, fed by the fused
rms_norm / SwiGLU / quantize -> q8 producers (every layer's matrices are
distinct device buffers, so one step's inputs exceed L2 many times over).
Workloads smaller than 4x L2 rotate through enough device copies of their
weights.  The sweep's line also reports the four other benchmark
configurations (the 512 x 2048 GEMV, the 7B ffn_down, the 14B attn_v +
ffn_down layer and the head), measured in the same process.

Timing: R >= 5 timed regions of exactly K steps each (CUDA graphs of at most
64 consecutive steps; one graph when K <= 64), CUDA events on the launching
stream with a barrier and synchronize on both sides; the median region is
reported, with the spread.

    python bench.py [--gpus N --steps K --warmup W] [--impl mq|reference]
                    [--workload NAME] [--tokens NT]

Prints ONE JSON line (rank 0).  value = weight content bytes per step /
device time per step (GB/s).  With --tokens NT > 1 every step decodes NT
tokens through the small-batch producers and GEMV: the weights are still
read once per step.  --impl reference times the oracle (plain C,
one host core) on a bounded row sample of the same workload.
Under torchrun (N > 1) every rank runs the same workload on its own GPU
(independent problems, weak scaling, no collective on the data path); the
step time is the max over ranks and value sums the ranks' bytes.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import shutil
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "content GB/s per k-quant GEMV (bytes/kernel time) and % of GB300 HBM peak"
DESCR = {
    "q6k_512x2048": "q6_K 512x2048 GEMV, x -> standalone q8 quantize, batch 1",
    "ffn_down_7b": "Qwen2.5-7B ffn_down: q6_K 3584x18944 (74 super-blocks/row, split-K), "
                   "SwiGLU(g,u)->q8 producer, batch 1",
    "layer_14b": "Qwen2.5-14B attn_v q6_K 1024x5120 + ffn_down q6_K 5120x13824, each fed by "
                 "rms_norm->q8, batch 1",
    "lm_head_14b": "Qwen2.5-14B output head q6_K 152064x5120, rms_norm->q8, batch 1",
    "attn_v_14b": "Qwen2.5-14B attn_v q6_K 1024x5120, rms_norm->q8, batch 1",
    "q6k_2048x4864": "q6_K 2048x4864 GEMV, x -> standalone q8 quantize, batch 1",
    "ffn_down_14b_q5k": "q5_K 5120x13824 (the 14B ffn_down shape), rms_norm->q8, batch 1",
    "ffn_14b": "Qwen2.5-14B FFN: rms_norm->q8 -> gate, up q4_K 13824x5120 -> SwiGLU->q8 -> "
               "down q6_K 5120x13824, batch 1",
    "attn_q_14b": "Qwen2.5-14B attn_q q4_K 5120x5120 (the attn_output shape too), rms_norm->q8, "
                  "batch 1",
    "ffn_gate_14b": "Qwen2.5-14B ffn_gate q4_K 13824x5120 (the ffn_up shape too) as a plain GEMV, "
                    "rms_norm->q8, batch 1",
    "attn_qkv_14b": "Qwen2.5-14B attn q 5120x5120 q4_K, k 1024x5120 q4_K, v 1024x5120 q6_K in one "
                    "grouped launch over one rms_norm->q8 plane, batch 1",
    "sweep_14b": "Qwen2.5-14B decode weight sweep: 48 layers x {q,k,o,gate,up q4_K; v,down q6_K} "
                 "+ q6_K head, fused rms/swiglu/quantize producers, batch 1",
}


# ---------------------------------------------------------------- distributed
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws: int, backend: str):
    import torch.distributed as dist
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if ws > 1 else None


def reduce_max(value: float, dist) -> float:
    """Max of a float over ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(bytes_per_rank_step: float, steps: int, max_ms: float, world: int) -> float:
    """Whole-job GB/s: the bytes every rank processed over the slowest rank's time."""
    return world * bytes_per_rank_step * steps / (max_ms * 1e-3) / 1e9


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle sampling while the GPU runs the workload."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.idx = gpu_index
        self.lines = []
        exe = shutil.which("nvidia-smi")
        if exe:
            self.proc = subprocess.Popen([exe, f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(gpu_index), "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict | None:
        rows = []
        for t, line in self.lines:
            if t0 <= t <= t1:
                f = [s.strip() for s in line.split(",")]
                if len(f) >= 9:
                    rows.append(f)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- measured peaks / profiles
def measured_peak_gbs():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def gemv_source_hash(act: str = "q8", gateup: bool = False, batch: bool = False) -> str:
    """First 16 hex digits of the SHA-256 of the GEMV kernel sources (with
    the gate||up kernel when the workload launches it; the small-batch
    kernel's for nt > 1 tokens)."""
    h = hashlib.sha256()
    main = "gemv_f32.cu" if act == "f32" else "gemv_batch.cu" if batch else "gemv.cu"
    files = [main, "gemv_common.cuh", "layout.h"]
    if gateup:
        files.append("gemv_gateup.cu")
    for f in files:
        with open(os.path.join(ROOT, "quant_quantized_gemv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, act: str = "q8", gateup: bool = False, tokens: int = 1):
    """DRAM bytes (read + write) of the GEMV launches of one step, from the
    committed ncu summary of this workload, if it was taken on the current
    kernel source (else None).  A one-GEMV workload's summary gives them per
    launch (= per step); the small-batch summary per launch and token count
    (traffic_bytes_per_launch_nt<N>)."""
    prefix = "f32_" if act == "f32" else "batch_" if tokens > 1 else ""
    p = os.path.join(ROOT, "profiles", f"gemv_{prefix}{workload}.md")
    if not os.path.exists(p):
        return None
    txt = open(p).read()
    key = f"traffic_bytes_per_launch_nt{tokens}" if tokens > 1 else r"traffic_bytes_per_(?:launch|step)"
    m = re.search(key + r":\s*([0-9.eE+]+)", txt)
    h = re.search(r"source_sha256_16:\s*([0-9a-f]+)", txt)
    if not m or not h or h.group(1) != gemv_source_hash(act, gateup, tokens > 1):
        return None
    return float(m.group(1))


# ---------------------------------------------------------------- workload on the device
class DeviceWorkload:
    """Ops of one decode step: producers writing q8 planes, GEMVs reading them.
    With acts == "f32" every GEMV is the q6_K x f32 GEMV reading its
    producer's f32 output (or its raw input: no quantize op runs)."""

    def __init__(self, name: str, device, l2_bytes: int, group: bool = True, nt: int = 1,
                 fuse: bool = True, acts: str = "q8"):
        import torch
        import quant_quantized_gemv_gb300 as mq
        self.mq = mq
        self.name = name
        self.nt = nt                 # tokens per step (> 1: the small-batch kernels)
        group = group and nt == 1    # the small-batch GEMV takes one matrix per launch
        self.wl = synth.WORKLOADS[name]
        self.f32 = acts == "f32"
        if self.f32:
            if nt != 1 or any(fmt != "q6k" for _, fmt, _, _, _ in self.wl.gemvs):
                raise SystemExit("--act f32: the f32-activation GEMV is q6_K at one token")
            group = fuse = False
        self.dev = device
        self.weight_bytes = self.wl.weight_bytes()
        self.n_copies = max(1, math.ceil(4 * l2_bytes / self.weight_bytes))
        g = synth.rng("bench", name)
        # one host matrix per distinct (fmt, rows, cols): the sweep's 48 layers
        # share content but get distinct device buffers, so nothing is cached
        base = {}
        for _, fmt, rows, cols, _ in self.wl.gemvs:
            if (fmt, rows, cols) not in base:
                W = synth.blocks(fmt, g, rows, cols)
                base[(fmt, rows, cols)] = (W, torch.from_numpy(mq.mq_repack(fmt, W, rows, cols)).to(device))
        self.host_w = {k: v[0] for k, v in base.items()}
        self.ops = []
        self.inputs = []          # (device tensor, host pinned) pairs copied in by e2e
        prev_kind, prev_cols, plane, prev_outputs = None, None, None, []
        def act(n):                              # nt token rows of n values
            return np.stack([synth.normal(g, n) for _ in range(nt)]) if nt > 1 else synth.normal(g, n)

        for gname, fmt, rows, cols, producer in self.wl.gemvs:
            if not (producer == "rms" and prev_kind == "rms" and prev_cols == cols):
                plane = torch.empty(nt * mq.mq_q8_bytes(cols), dtype=torch.uint8, device=device)
                yp = torch.empty((nt, cols) if nt > 1 else cols, dtype=torch.float32, device=device)
                if producer == "rms":
                    x = self._input(act(cols))
                    gain = torch.from_numpy(synth.normal(g, cols, 1.0, 0.1)).to(device)
                    self.ops.append(("rms", x, gain, yp, plane, cols))
                    xsrc = yp
                elif producer == "swiglu":
                    if len(prev_outputs) >= 2 and prev_outputs[-1].numel() == nt * cols and \
                            prev_outputs[-2].numel() == nt * cols:
                        gv, uv = prev_outputs[-2], prev_outputs[-1]     # gate, up outputs
                    else:
                        gv = self._input(act(cols))
                        uv = self._input(act(cols))
                    self.ops.append(("swiglu", gv, uv, yp, plane, cols))
                    xsrc = yp
                else:
                    x = self._input(act(cols))
                    xsrc = x
                    if not self.f32:
                        self.ops.append(("quant", x, plane, cols))
            prev_kind, prev_cols = producer, cols
            W0 = base[(fmt, rows, cols)][1]
            copies = [W0.clone() for _ in range(self.n_copies)]
            y = torch.empty((nt, rows) if nt > 1 else rows, dtype=torch.float32, device=device)
            part = (fmt, copies, rows, y, gname)
            last = self.ops[-1] if self.ops else None
            if self.f32:
                self.ops.append(["gemv32", xsrc, cols, [part], None])
            elif group and last is not None and last[0] == "gemv" and last[1] is plane and \
                    len(last[3]) < mq.MQ_MAX_GROUP:
                last[3].append(part)             # same q8 plane: one launch for the group
            else:
                self.ops.append(["gemv", plane, cols, [part], None])
            prev_outputs.append(y)
        self._pack_inputs()
        if fuse and group and nt == 1:
            self._fuse_gateup()
        for o in self.ops:                       # workspace per GEMV launch (default plan)
            if o[0] == "gemv" and nt == 1:
                o[4] = mq.mq_gemv_group_workspace(self._spec(o), o[2], device=device)
        if self.ops[-1][0] not in ("gemv", "gemv32"):
            raise SystemExit(f"{name}: a step must end with a GEMV (its output is the step's result)")
        self.output = self.ops[-1][3][-1][3]
        gemv_ops = [o for o in self.ops if o[0] in ("gemv", "gateup", "gemv32")]
        self.n_gemv = sum(len(o[3]) for o in gemv_ops)
        self.n_gemv_launches = len(gemv_ops)
        self.n_kernels = len(self.ops)
        self.gemv_bytes = [self._part_alg_bytes(p[0], p[2], o[2], nt, self.f32) for o in gemv_ops
                           for p in o[3]]

    def _fuse_gateup(self):
        """A two-matrix GEMV launch (gate, up) whose outputs feed the next
        op's SwiGLU becomes one gate||up launch with the SwiGLU -> q8 epilogue."""
        out = []
        i = 0
        while i < len(self.ops):
            o = self.ops[i]
            nxt = self.ops[i + 1] if i + 1 < len(self.ops) else None
            if o[0] == "gemv" and len(o[3]) == 2 and nxt is not None and nxt[0] == "swiglu":
                (f0, c0, r0, y0, _), (f1, c1, r1, y1, _) = o[3]
                if f0 == f1 and r0 == r1 and r0 % 32 == 0 and nxt[1] is y0 and nxt[2] is y1:
                    # ("gateup", plane_in, cols, parts, act, plane_out)
                    out.append(["gateup", o[1], o[2], o[3], nxt[3], nxt[4]])
                    i += 2
                    continue
            out.append(o)
            i += 1
        self.ops = out

    def _input(self, arr: np.ndarray):
        import torch
        t = torch.from_numpy(arr).to(self.dev)
        self.inputs.append((t, torch.from_numpy(arr)))
        return t

    def _pack_inputs(self):
        """Place every per-step input in one device buffer (each at a 16-byte
        aligned offset) mirrored by one pinned host buffer, so that a step's
        host-to-device transfer is a single copy."""
        import torch
        offs, total = [], 0
        for t, _ in self.inputs:
            offs.append(total)
            total += -(-t.numel() // 4) * 4
        self.in_dev = torch.zeros(max(total, 4), dtype=torch.float32, device=self.dev)
        self.in_host = torch.zeros(max(total, 4), dtype=torch.float32).pin_memory()
        for (t, h), off in zip(self.inputs, offs):
            self.in_host[off:off + t.numel()] = h.reshape(-1)
            t.set_(self.in_dev.untyped_storage(), off, t.shape)   # ops keep this tensor object
        self.in_dev.copy_(self.in_host)
        self.h2d_bytes = total * 4 if self.inputs else 0
        self.in_off = {id(t): off for (t, _), off in zip(self.inputs, offs)}
        # e2e: inputs read once per element (by quantize or SwiGLU) are read
        # by those producers from pinned host memory in place; rms_norm reads
        # its row once per CTA and the f32 GEMV once per CTA, so inputs that
        # reach either are copied in first (mq_copy)
        once = {id(t) for o in self.ops if o[0] == "quant" for t in (o[1],)} | \
               {id(t) for o in self.ops if o[0] == "swiglu" for t in (o[1], o[2])}
        self.inputs_in_place = bool(self.inputs) and all(id(t) in once for t, _ in self.inputs)

    def host_inputs(self, n: int):
        """n pinned copies of the step input buffer (same layout as in_dev),
        so that consecutive e2e steps read different host lines."""
        return [self.in_host.clone().pin_memory() for _ in range(n)]

    def _in(self, t, host_in):
        """t, or its view in the pinned host buffer host_in when t is a step input."""
        if host_in is None or id(t) not in self.in_off:
            return t
        off = self.in_off[id(t)]
        return host_in[off:off + t.numel()].view(t.shape)

    @staticmethod
    def _part_weight_bytes(fmt, rows, cols) -> int:
        return rows * (cols // 256) * {"q6k": 210, "q4k": 144, "q5k": 176}[fmt]

    @staticmethod
    def _part_alg_bytes(fmt, rows, cols, nt=1, f32=False) -> int:
        wb = rows * (cols // 256) * {"q6k": 210, "q4k": 144, "q5k": 176}[fmt]
        act = (cols // 32) * (34 if fmt == "q6k" else 38)      # codes + fp16 d (+ int32 sum)
        if f32:
            act = 4 * cols                                      # the f32 row
        return wb + nt * (act + 4 * rows)

    @staticmethod
    def _spec(o, c=0):
        return [(fmt, copies[c], rows) for fmt, copies, rows, _, _ in o[3]]

    def _launch(self, o, c, y_last=None):
        """y_last: write the launch's last output there instead (e2e: pinned host)."""
        _, plane, cols, parts, ws = o
        mq = self.mq
        ys = [p[3] for p in parts]
        if y_last is not None:
            ys[-1] = y_last
        if self.nt > 1:
            fmt, copies, rows, _, _ = parts[0]
            fn = getattr(mq, f"mq_gemv_{fmt}_q8_batch")
            fn(copies[c], plane, self.nt, rows, cols, y=ys[0])
        elif len(parts) == 1:
            fmt, copies, rows, _, _ = parts[0]
            fn = getattr(mq, f"mq_gemv_{fmt}_q8")
            fn(copies[c], plane, rows, cols, y=ys[0], ws=ws)
        else:
            mq.mq_gemv_group_q8(self._spec(o, c), plane, cols, ys=ys, ws=ws)

    def _launch32(self, o, c, y_last=None):
        _, xsrc, cols, parts, _ = o
        _, copies, rows, y, _ = parts[0]
        self.mq.mq_gemv_q6k_f32(copies[c], xsrc, rows, cols, y=y if y_last is None else y_last)

    def _launch_gateup(self, o, c):
        _, plane, cols, parts, act, plane_out = o
        (fmt, cg, rows, _, _), (_, cu, _, _, _) = parts
        self.mq.mq_gemv_gateup_swiglu_q8(fmt, cg[c], cu[c], plane, rows, cols, act=act, q8_out=plane_out)

    def launch_op(self, o, k: int):
        """Enqueue one GEMV-type op of step k (weights copy k % n_copies)."""
        c = k % self.n_copies
        if o[0] == "gemv":
            self._launch(o, c)
        elif o[0] == "gemv32":
            self._launch32(o, c)
        elif o[0] == "gateup":
            self._launch_gateup(o, c)

    def run_gemvs(self, k: int, kinds=None):
        """Enqueue only the GEMV launches of step k (for kernel timing), or
        only those of the given op kinds."""
        for o in self.ops:
            if o[0] in ("gemv", "gemv32", "gateup") and (kinds is None or o[0] in kinds):
                self.launch_op(o, k)

    def run(self, k: int, producers_only: bool = False, host_in=None, out=None):
        """Enqueue step k (weights copy k % n_copies) on the current stream;
        with producers_only, just its producer launches (for their timing).
        host_in: a pinned host input buffer whose views the producers read
        in place of the device inputs; out: pinned host tensor the last GEMV
        writes its output into."""
        mq = self.mq
        c = k % self.n_copies
        last = self.ops[-1]
        for o in self.ops:
            kind = o[0]
            if producers_only and kind in ("gemv", "gemv32", "gateup"):
                continue
            b = self.nt > 1
            if kind == "rms":
                (mq.mq_rmsnorm_quant_q8_batch if b else mq.mq_rmsnorm_quant_q8)(
                    self._in(o[1], host_in), o[2], 1e-6, y=o[3], q8=o[4])
            elif kind == "swiglu":
                (mq.mq_swiglu_quant_q8_batch if b else mq.mq_swiglu_quant_q8)(
                    self._in(o[1], host_in), self._in(o[2], host_in), y=o[3], q8=o[4])
            elif kind == "quant":
                (mq.mq_quantize_q8_batch if b else mq.mq_quantize_q8)(self._in(o[1], host_in), q8=o[2])
            elif kind == "gateup":
                self._launch_gateup(o, c)
            elif kind == "gemv32":
                self._launch32(o, c, out if o is last else None)
            else:
                self._launch(o, c, out if o is last else None)


def make_event(timing=True, external=False):
    import torch
    if external:
        return torch.cuda.Event(enable_timing=timing, external=True)
    return torch.cuda.Event(enable_timing=timing)


def capture(fn, stream):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


class StepGraphs:
    """CUDA graphs of consecutive steps of one step function, at most m steps
    each, cached by (first weight copy, length): steps i and i + n_copies use
    the same buffers, so one graph serves every segment with that phase."""

    def __init__(self, fn, n_copies: int, m: int, stream):
        self.fn, self.n_copies, self.m, self.stream = fn, n_copies, max(1, m), stream
        self.cache = {}

    def _segments(self, start: int, k: int):
        s = start
        while s < start + k:
            n = min(self.m, start + k - s)
            yield s, n
            s += n

    def _graph(self, s: int, n: int):
        key = (s % self.n_copies, n)
        if key not in self.cache:
            self.cache[key] = capture(lambda: [self.fn(s + j) for j in range(n)], self.stream)
        return self.cache[key]

    def prepare(self, start: int, k: int):
        """Capture (outside any timed region) every graph enqueue() will use."""
        for s, n in self._segments(start, k):
            self._graph(s, n)

    def enqueue(self, start: int, k: int):
        """Enqueue exactly k steps, start .. start + k - 1."""
        for s, n in self._segments(start, k):
            self._graph(s, n).replay()


def replay_ms(graph, stream, reps: int = 5) -> list:
    """Device time of `reps` replays of a graph, CUDA events on the stream."""
    import torch
    with torch.cuda.stream(stream):
        graph.replay()                                   # warm
    torch.cuda.synchronize()
    out = []
    for _ in range(reps):
        e0, e1 = make_event(), make_event()
        with torch.cuda.stream(stream):
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        e1.synchronize()
        out.append(e0.elapsed_time(e1))
    return out


def spread(vals, scale: float = 1.0, nd: int = 3) -> dict:
    v = sorted(x * scale for x in vals)
    return {"median": round(float(np.median(v)), nd), "min": round(v[0], nd), "max": round(v[-1], nd),
            "n": len(v)}


def kernel_graphs(wl, stream, n_kt: int, kinds=None):
    """One graph of the GEMV launches (of the given op kinds) of n_kt
    consecutive steps back to back, PDL off, rotating weight copies."""
    return capture(lambda: [wl.run_gemvs(i, kinds) for i in range(n_kt)], stream)


def config_report(name: str, dev, l2: int, stream, peak: float, pdl: bool) -> dict:
    """GEMV-alone and chained-step timing of one more workload, measured in
    this process: per GEMV op µs, content GB/s and fraction of the peak."""
    import torch
    import quant_quantized_gemv_gb300 as mq
    wl = DeviceWorkload(name, dev, l2)
    with torch.cuda.stream(stream):
        wl.run(0)
    torch.cuda.synchronize()
    mq.mq_set_pdl(False)
    n_kt = max(wl.n_copies, 16)
    ops = [o for o in wl.ops if o[0] in ("gemv", "gateup")]
    gemvs = []
    for idx, o in enumerate(ops):
        g = capture(lambda o=o: [wl.launch_op(o, i) for i in range(n_kt)], stream)
        t = replay_ms(g, stream)
        us = float(np.median(t)) / n_kt * 1e3
        wbytes = sum(DeviceWorkload._part_weight_bytes(p[0], p[2], o[2]) for p in o[3])
        alg = sum(DeviceWorkload._part_alg_bytes(p[0], p[2], o[2]) for p in o[3])
        gemvs.append({"gemv": "+".join(f"{p[4]} {p[0]} {p[2]}x{o[2]}" for p in o[3]),
                      "us": round(us, 3), "us_spread": spread(t, 1e3 / n_kt),
                      "content_gbs": round(wbytes / (us * 1e-6) / 1e9, 1),
                      "frac": round(alg / (us * 1e-6) / 1e9 / peak, 4)})
        del g
    floor_us = None
    if wl.n_gemv == 1:
        wcopies = ops[0][3][0][1]
        fg = capture(lambda: [mq.mq_read_floor(wcopies[i % wl.n_copies]) for i in range(n_kt)], stream)
        floor_us = round(float(np.median(replay_ms(fg, stream))) / n_kt * 1e3, 3)
        del fg
    mq.mq_set_pdl(pdl)
    m = 16
    sg = StepGraphs(wl.run, wl.n_copies, m, stream)
    nsteps = max(m, wl.n_copies)
    sg.prepare(0, nsteps)
    with torch.cuda.stream(stream):
        sg.enqueue(0, nsteps)
    torch.cuda.synchronize()
    st = []
    for _ in range(5):
        e0, e1 = make_event(), make_event()
        with torch.cuda.stream(stream):
            e0.record(stream)
            sg.enqueue(0, nsteps)
            e1.record(stream)
        e1.synchronize()
        st.append(e0.elapsed_time(e1) / nsteps)
    mq.mq_set_pdl(False)
    step_us = float(np.median(st)) * 1e3
    gemv_us = sum(x["us"] for x in gemvs)
    alg = float(sum(wl.gemv_bytes))
    rep = {"workload": f"{name}: {DESCR[name]}",
           "weight_content_bytes": wl.weight_bytes,
           "gemv_us": round(gemv_us, 3),
           "content_gbs": round(wl.weight_bytes / (gemv_us * 1e-6) / 1e9, 1),
           "frac": round(alg / (gemv_us * 1e-6) / 1e9 / peak, 4),
           "gemvs": gemvs,
           "step_us": round(step_us, 3), "step_spread_us": spread(st, 1e3),
           "step_content_gbs": round(wl.weight_bytes / (step_us * 1e-6) / 1e9, 1),
           "l2": f"{wl.n_copies} rotated weight copies"}
    if floor_us is not None:
        rep["read_floor_us"] = floor_us
        rep["frac_of_read_floor"] = round(floor_us / gemv_us, 4)
    del sg, wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rep


# the benchmark configurations reported beside the headline one (the
# smallest GEMV, the 7B ffn_down, the 14B attn_v + ffn_down layer, the head)
CONFIG_WORKLOADS = ["q6k_512x2048", "ffn_down_7b", "layer_14b", "lm_head_14b"]


def bench_mq(args, ws_, rank, local) -> dict | None:
    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(ws_, "nccl")
    from quant_quantized_gemv_gb300 import build as _b
    if rank == 0 or ws_ == 1:
        _b.build()
    if dist is not None:
        dist.barrier()
    import quant_quantized_gemv_gb300 as mq
    if args.gemv_ring is not None:
        sp = [int(v) for v in str(args.gemv_ring).split(",")]
        mq.mq_set_gemv_ring(sp[0], sp[1] if len(sp) > 1 else -1)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    wl = DeviceWorkload(args.workload, dev, l2, group=args.group, nt=args.tokens, fuse=args.fuse,
                        acts=args.act)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        wl.run(0)                                   # first launches outside capture
    torch.cuda.synchronize()
    K, W, R = args.steps, args.warmup, max(5, args.repeats)

    # ---- step graphs: segments of at most m consecutive steps (PDL edges
    # between all kernels of a segment when enabled); a timed region of K
    # <= m steps is one graph of exactly K steps
    mq.mq_set_pdl(args.pdl)
    m = max(1, min(args.steps_per_graph, K))
    steps = StepGraphs(wl.run, wl.n_copies, m, stream)
    steps.prepare(0, W)
    for r in range(R):                              # repeat r times steps [r*K, (r+1)*K)
        steps.prepare(r * K, K)
    # ---- kernel-timing graphs: the GEMVs of n_kt consecutive steps back to
    # back (no producers, PDL off so no two GEMVs overlap), rotating copies
    mq.mq_set_pdl(False)
    n_kt = max(wl.n_copies, 16) if wl.n_gemv < 8 else 2
    kt_graph = kernel_graphs(wl, stream, n_kt)
    kinds = sorted({o[0] for o in wl.ops if o[0] in ("gemv", "gateup", "gemv32")})
    kind_graphs = {k: kernel_graphs(wl, stream, n_kt, [k]) for k in kinds} if len(kinds) > 1 else {}
    n_prod = sum(1 for o in wl.ops if o[0] in ("rms", "swiglu", "quant"))
    pt_graph = (capture(lambda: [wl.run(i, producers_only=True) for i in range(n_kt)], stream)
                if n_prod else None)
    # the same GEMV launches chained with PDL, as a decode step runs them (each
    # still waits for its predecessor before it reads its plane or writes)
    mq.mq_set_pdl(True)
    kc_graph = kernel_graphs(wl, stream, n_kt) if args.pdl else None
    mq.mq_set_pdl(False)
    # ---- the single-launch read floor of the same weight bytes (one-GEMV
    # workloads): a plain read of each step's weight copy, back to back
    floor_graph = None
    if wl.n_gemv == 1 and args.tokens == 1:
        wcopies = wl.ops[-1][3][0][1]
        floor_graph = capture(lambda: [mq.mq_read_floor(wcopies[i % wl.n_copies]) for i in range(n_kt)],
                              stream)
    mq.mq_set_pdl(args.pdl)
    torch.cuda.synchronize()

    # ---- warm-up, then a clock-sampled window: soak / R timed regions of
    # exactly K steps / soak
    with torch.cuda.stream(stream):
        steps.enqueue(0, W)
    torch.cuda.synchronize()
    sampler = ClockSampler(local) if rank == 0 or ws_ == 1 else None
    t_win0 = time.perf_counter()

    def soak(seconds):
        t_end = time.perf_counter() + seconds
        with torch.cuda.stream(stream):
            while time.perf_counter() < t_end:
                for r in range(R):
                    steps.enqueue(r * K, K)
                torch.cuda.synchronize()

    soak(args.soak)
    region_ms = []
    for r in range(R):
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        start, stop = make_event(), make_event()
        with torch.cuda.stream(stream):
            start.record(stream)
            steps.enqueue(r * K, K)
            stop.record(stream)
        stop.synchronize()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        region_ms.append(reduce_max(start.elapsed_time(stop), dist))
    t_timed1 = time.perf_counter()
    soak(args.soak)
    t_win1 = time.perf_counter()
    if sampler is not None:
        sampler.stop()
    max_ms = float(np.median(region_ms))
    ms_per_step = max_ms / K

    # ---- kernel timing: replay the GEMV-only graph, events around each replay
    kt = replay_ms(kt_graph, stream)
    gemv_step_ms = float(np.median(kt)) / n_kt
    kind_ms = {k: float(np.median(replay_ms(g, stream))) / n_kt for k, g in kind_graphs.items()}
    prod_step_ms = float(np.median(replay_ms(pt_graph, stream))) / n_kt if pt_graph is not None else 0.0
    kc = replay_ms(kc_graph, stream) if kc_graph is not None else None
    floor_ms = float(np.median(replay_ms(floor_graph, stream))) / n_kt if floor_graph is not None else None

    # ---- e2e: the public API, pinned host inputs in, result out, every step
    out_host = torch.empty(wl.output.shape, dtype=torch.float32).pin_memory()
    h2d = wl.h2d_bytes
    d2h = out_host.numel() * 4
    torch.cuda.synchronize()

    # every step reads its own pinned input buffer (rotated like the weight
    # copies, so no step finds the previous one's input lines in L2)
    hosts = wl.host_inputs(wl.n_copies) if wl.inputs else []

    def e2e_step(i):
        hin = hosts[i % len(hosts)] if hosts else None
        if hin is not None and not wl.inputs_in_place:
            mq.mq_copy(wl.in_dev, hin)                   # pinned host -> device, a kernel
        # the producers read in-place inputs over the host link, and the
        # last GEMV writes its rows straight into pinned host memory
        wl.run(i, host_in=hin if wl.inputs_in_place else None, out=out_host)

    n_eager = max(3, min(K, args.e2e_steps))
    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(i)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(n_eager):
            e2e_step(i)
    torch.cuda.synchronize()
    e2e_eager_ms = reduce_max((time.perf_counter() - t0) * 1e3, dist) / n_eager
    # the same steps captured the way a decode loop runs them: K steps per
    # region (graphs of at most m steps), every step with its host input
    # and host result; >= 5 regions, each timed by the wall clock
    e2e = StepGraphs(e2e_step, wl.n_copies, m, stream)
    for r in range(R):
        e2e.prepare(r * K, K)
    with torch.cuda.stream(stream):
        e2e.enqueue(0, K)
    torch.cuda.synchronize()
    e2e_region = []
    for r in range(R):
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            e2e.enqueue(r * K, K)
        torch.cuda.synchronize()
        e2e_region.append(reduce_max((time.perf_counter() - t0) * 1e3, dist))
    e2e_ms = float(np.median(e2e_region)) / K
    mq.mq_set_pdl(False)

    peak, peak_kind = measured_peak_gbs()
    configs = None
    if args.configs and args.workload == "sweep_14b" and args.tokens == 1 and not wl.f32:
        configs = {}
        for i, name in enumerate(CONFIG_WORKLOADS):
            configs[f"config{i}"] = config_report(name, dev, l2, stream, peak, args.pdl)

    if rank != 0:
        return None
    value = weak_scaling_value(wl.weight_bytes, K, max_ms, ws_)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ws_,
        "steps": K, "warmup": W, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if wl.f32 else "i8", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {DESCR[args.workload]}",
                   "activations": ("f32 row (q6_K x f32 GEMV, no quantize producer)" if wl.f32
                                   else "q8 plane"),
                   "tokens_per_step": args.tokens,
                   "weight_content_bytes_per_step": wl.weight_bytes,
                   "gemvs_per_step": wl.n_gemv, "gemv_launches_per_step": wl.n_gemv_launches,
                   "fused_gateup_launches_per_step": sum(1 for o in wl.ops if o[0] == "gateup"),
                   "kernels_per_step": wl.n_kernels,
                   "l2": (f"inputs larger than L2: {wl.weight_bytes / 1e6:.0f} MB of weights per step "
                          f"(L2 {l2 / 1e6:.0f} MB)" if wl.n_copies == 1 else
                          f"{wl.n_copies} rotated weight copies "
                          f"({wl.n_copies * wl.weight_bytes / 1e6:.0f} MB >= 4 x L2 {l2 / 1e6:.0f} MB)"),
                   "timing": f"{R} timed regions of exactly {K} steps, each CUDA graphs of at most {m} "
                             f"consecutive steps ({'one graph of ' + str(K) + ' steps' if K <= m else 'segments'}"
                             f"), CUDA events on the launching stream, barrier + synchronize on both "
                             f"sides; value and ms_per_step from the median region; "
                             f"PDL {'on' if args.pdl else 'off'}",
                   "parallelism": f"replicas{ws_}" if ws_ > 1 else "single GPU",
                   "gemv_ring": args.gemv_ring or "library default"},
        "compute": ("6-bit codes x f32 FMA chains per sub-block, f32 scale combine" if wl.f32 else
                    "int8 x (6-bit|4-bit) dp4a dots, int32 sub-block sums, f32 scale combine"),
        "pct_of_hbm_peak": round(100 * value / ws_ / peak, 2),
        "tokens_per_s": round(ws_ * args.tokens * K / (max_ms * 1e-3), 1),
        "step_ms_spread": spread([x / K for x in region_ms], 1.0, 6),
    }
    alg = float(sum(wl.gemv_bytes))
    achieved = alg / (gemv_step_ms * 1e-3) / 1e9
    traffic = profiled_traffic(args.workload, args.act, "gateup" in kinds, args.tokens)
    line["roofline"] = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                        "unit": "GB/s", "frac": round(achieved / peak, 4),
                        "traffic": traffic, "peak_source": f"{peak_kind} hbm_gbs (copy, burst)",
                        "algorithmic_bytes_per_step": int(alg),
                        "kernel": ("gemv_q6k_f32_kernel (q6_K x f32 row)" if wl.f32 else
                                   "gemv_kernel (q6_K/q4_K/q5_K x q8)" +
                                   (" and gemv_gateup_kernel (gate||up + SwiGLU -> q8)" if "gateup" in kinds else "")
                                   if args.tokens == 1 else
                                   f"gemv_batch_kernel<{args.tokens}> (q6_K/q4_K/q5_K x {args.tokens} q8 rows)"),
                        "gemv_us_per_step": round(gemv_step_ms * 1e3, 3),
                        "gemv_us_spread": spread(kt, 1e3 / n_kt),
                        "how": f"every GEMV launch of {n_kt} steps back to back in one CUDA graph "
                               f"(PDL off), CUDA events around 5 replays, median; achieved = "
                               f"algorithmic bytes per step / GEMV time per step; traffic = ncu DRAM "
                               f"bytes per step from the committed profile when its source hash matches"}
    if kind_ms:
        names = {"gemv": "gemv_kernel", "gateup": "gemv_gateup_kernel", "gemv32": "gemv_q6k_f32_kernel"}
        per = {}
        for k, ms in kind_ms.items():
            ab = float(sum(wl._part_alg_bytes(p[0], p[2], o[2], args.tokens, wl.f32)
                           for o in wl.ops if o[0] == k for p in o[3]))
            nl = sum(1 for o in wl.ops if o[0] == k)
            per[names[k]] = {"launches_per_step": nl, "us_per_step": round(ms * 1e3, 3),
                             "algorithmic_bytes_per_step": int(ab),
                             "achieved": round(ab / (ms * 1e-3) / 1e9, 1),
                             "frac": round(ab / (ms * 1e-3) / 1e9 / peak, 4)}
        line["roofline"]["per_kernel"] = per
    if floor_ms is not None:
        # a plain one-launch read of the same weight copies (mq_read_floor),
        # timed the same way: what any single launch of these bytes costs here
        line["roofline"]["read_floor_us"] = round(floor_ms * 1e3, 3)
        line["roofline"]["read_floor_gbs"] = round(wl.weight_bytes / (floor_ms * 1e-3) / 1e9, 1)
        line["roofline"]["frac_of_read_floor"] = round(floor_ms / gemv_step_ms, 4)
    line["kernel_us"] = {"gemv_per_step_isolated": round(gemv_step_ms * 1e3, 3),
                         "gemv_spread": spread(kt, 1e3 / n_kt),
                         "producers_per_step_isolated": round(prod_step_ms * 1e3, 3),
                         **({"gemv_per_step_pdl_chain": round(float(np.median(kc)) / n_kt * 1e3, 3),
                             "gemv_pdl_chain_achieved_gbs": round(
                                 alg / (float(np.median(kc)) / n_kt * 1e-3) / 1e9, 1),
                             "gemv_pdl_chain_frac": round(
                                 alg / (float(np.median(kc)) / n_kt * 1e-3) / 1e9 / peak, 4)}
                            if kc is not None else {}),
                         "producer_launches_per_step": n_prod,
                         "step": round(ms_per_step * 1e3, 3),
                         "step_spread": spread([x / K for x in region_ms], 1e3),
                         "how": "GEMV launches alone and producer launches alone, each as a graph of "
                                f"{n_kt} steps back to back with PDL off; gemv_per_step_pdl_chain: the "
                                "same GEMV launches with PDL on (each overlaps its ramp with the "
                                "previous launch's tail and still waits for it before touching its "
                                "plane or outputs), context beside roofline.frac, which uses the "
                                "PDL-off time; step: the PDL chain of GEMVs and producers"}
    line["e2e"] = {"value": round(wl.weight_bytes / (e2e_ms * 1e-3) / 1e9 * ws_, 2), "unit": "GB/s",
                   "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d),
                   "d2h_bytes_per_step": int(d2h),
                   "ms_per_step_spread": spread([x / K for x in e2e_region], 1.0, 4),
                   "how": f"public API calls captured as {R} regions of {K} steps (graphs of at most "
                          f"{m} steps); every step takes its inputs from its own pinned host buffer "
                          f"({len(hosts)} rotated) "
                          + ("read in place by the quantize/SwiGLU producers over NVLink-C2C"
                             if wl.inputs_in_place else "copied in by mq_copy (a kernel in the PDL chain)")
                          + "; the last GEMV writes its output rows into pinned host memory; each region "
                            "timed by the wall clock with a synchronize at both ends, median region",
                   "inputs": "in place" if wl.inputs_in_place else "mq_copy",
                   "eager": {"value": round(wl.weight_bytes / (e2e_eager_ms * 1e-3) / 1e9 * ws_, 2),
                             "ms_per_step": round(e2e_eager_ms, 4),
                             "how": f"the same steps as eager Python API calls ({n_eager} steps)"}}
    line["gpu_launches"] = wl.n_kernels * K
    clocks = sampler.summary(t_win0, t_win1) if sampler else None
    line["clocks"] = clocks or {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
    line["clocks_window"] = (f"{args.soak:.1f}s soak + timed regions + {args.soak:.1f}s soak of the same "
                             f"graphs ({(t_timed1 - t_win0):.2f}s to end of timed regions)")
    if configs is not None:
        line["configs"] = configs
    if ws_ == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds, args.tokens, args.act)
    return line


# ---------------------------------------------------------------- oracle (CPU) legs
def oracle_sample(workload: str, rows_cap: int, nt: int = 1):
    """Host inputs for the oracle: each GEMV of the workload truncated to its
    first rows_cap rows, with its producer's f32 inputs for nt tokens."""
    wl = synth.WORKLOADS[workload]
    g = synth.rng("bench", workload)
    items, seen = [], {}
    for gname, fmt, rows, cols, producer in wl.gemvs:
        key = (fmt, rows, cols)
        if key in seen:
            continue
        r = min(rows, rows_cap)
        W = synth.blocks(fmt, g, r, cols)         # the sample's rows only, same distribution
        inps = []
        for _ in range(nt):
            if producer == "rms":
                inps.append((synth.normal(g, cols), synth.normal(g, cols, 1.0, 0.1)))
            elif producer == "swiglu":
                inps.append((synth.normal(g, cols), synth.normal(g, cols)))
            else:
                inps.append((synth.normal(g, cols),))
        seen[key] = True
        items.append((fmt, r, cols, producer, W, inps))
    return items


def oracle_step(items, acts: str = "q8"):
    """One step: every token's producer and GEMV; returns the weight bytes
    (read once per step, as on the GPU)."""
    import oracle
    nbytes = 0
    for fmt, r, cols, producer, W, inps in items:
        for inp in inps:
            if producer == "rms":
                x = oracle.rmsnorm(inp[0], inp[1], 1e-6).astype(np.float32)
            elif producer == "swiglu":
                x = oracle.swiglu(inp[0], inp[1]).astype(np.float32)
            else:
                x = inp[0]
            if acts == "f32":
                oracle.gemv_q6k_f32(W, x, r, cols)
            else:
                d, q, _ = oracle.quantize_q8(x)
                oracle.gemv(fmt, W, d, q, r, cols)
        nbytes += W.nbytes
    return nbytes


def cpu_baseline(workload: str, seconds: float, nt: int = 1, acts: str = "q8") -> dict:
    items = oracle_sample(workload, 512, nt)
    oracle_step(items, acts)                             # warm (page-in, build)
    done, t0 = 0, time.perf_counter()
    n = 0
    while True:
        done += oracle_step(items, acts)
        n += 1
        if time.perf_counter() - t0 >= seconds or n >= 10000:
            break
    dt = time.perf_counter() - t0
    rows = ", ".join(f"{fmt} {r}x{cols}" for fmt, r, cols, _, _, _ in items)
    return {"value": round(done / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} passes over the first <=512 rows of each distinct GEMV ({rows}) with "
                      f"its producer, {nt} token(s) per pass, {acts} activations, single-threaded C "
                      f"oracle, {dt:.1f} s"}


def bench_reference(args, ws_, rank) -> dict | None:
    if rank != 0:
        return None
    items = oracle_sample(args.workload, 512, args.tokens)
    for _ in range(args.warmup):
        oracle_step(items, args.act)
    t0 = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        nbytes += oracle_step(items, args.act)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    rows = ", ".join(f"{fmt} {r}x{cols}" for fmt, r, cols, _, _, _ in items)
    sample = (f"each step: the first <=512 rows of each distinct GEMV ({rows}) with its producer, "
              f"{args.tokens} token(s), {args.act} activations")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": ws_, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32" if args.act == "f32" else "i8",
            "data": "synthetic",
            "config": {"workload": f"{args.workload}: {DESCR[args.workload]}",
                       "tokens_per_step": args.tokens, "sample": sample},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--repeats", type=int, default=5,
                    help="timed regions of exactly --steps steps (at least 5); the median is reported")
    ap.add_argument("--impl", default="mq", choices=["mq", "reference"])
    ap.add_argument("--workload", default="sweep_14b", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--soak", type=float, default=0.6, help="seconds of identical load around the timed steps")
    ap.add_argument("--e2e-steps", type=int, default=20, help="steps of the eager e2e figure")
    ap.add_argument("--steps-per-graph", type=int, default=64,
                    help="most consecutive steps in one CUDA graph")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="with the 14B sweep, skip the per-configuration report of the other four "
                         "benchmark configurations")
    ap.add_argument("--gemv-ring", default=None, metavar="S[,P]",
                    help="weight-ring depth S of the single-token GEMV (0 = none) and the stages P "
                         "requested before the grid-dependency wait (default: the library's)")
    ap.add_argument("--no-pdl", dest="pdl", action="store_false",
                    help="launch without programmatic dependent launch")
    ap.add_argument("--no-group", dest="group", action="store_false",
                    help="one launch per GEMV even when several read the same q8 plane")
    ap.add_argument("--no-fuse", dest="fuse", action="store_false",
                    help="gate and up as a grouped GEMV plus a separate SwiGLU producer instead of "
                         "one gate||up launch with the SwiGLU -> q8 epilogue")
    ap.add_argument("--tokens", type=int, default=1, choices=range(1, 9), metavar="NT",
                    help="tokens per step (1..8); > 1 uses the small-batch producers and GEMV")
    ap.add_argument("--act", default="q8", choices=["q8", "f32"],
                    help="activation form the GEMVs read: the q8 plane (default) or, for q6_K "
                         "workloads at one token, the f32 row through the q6_K x f32 GEMV")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    ws_, rank, local = dist_env()
    if args.impl == "reference":
        line = bench_reference(args, ws_, rank)
    else:
        line = bench_mq(args, ws_, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
