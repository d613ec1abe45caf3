#!/usr/bin/env python
"""Benchmark of the grammar-constrained logit path on GB300.

Headline metric: bitmask-apply HBM throughput (GB/s, and its fraction of the
measured HBM copy bandwidth) on the apply workload -- B=64 bf16 rows padded to
128512 columns, vocab 128256, a 1%-dense grammar-like mask, 32 indexed rows --
and the fused mask + sample rate (rows/s) on the sampling workload -- B=256,
V=131072 bf16, 10% mask, per-row temperature, top_k 50, top_p 0.9, min_p 0.05.

One step = one in-place apply over a batch of the first workload plus one fused
mask + sample over a batch of the second.  Inputs are resident in HBM and rotate
through rings of copies larger than four L2 caches, so no step reads a batch
from L2.  Steps are captured in CUDA graphs (launch gaps are those of a graph
replay; at most 100 steps per graph and at most K/4, so a run times at least
four replays) and
timed with CUDA events on the launching stream; CUDA events between the apply
and sample graph replays split the time per kernel.

The default run then times every configuration of the benchmark list the same
way, one after another (``configs`` in the output line): the tiny apply +
greedy case, the apply workload, the fused workload with its apply alone, the
Zipf top-p sweep (0.5, 0.9, 0.99 and greedy) and the speculative-verify batch
with its apply alone.  Each figure carries its dense algorithmic bytes and the
sector-minimal bytes counted from the actual mask.

    python bench.py [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload default|apply_only|fused_sample|zipf_top_p|
                                speculative_verify|tiny_greedy] [--top-p P]

Prints one JSON line.  ``cpu_baseline`` times the CPU oracle on bounded samples
of the same workloads, on one thread and row-parallel on every host core.
``--impl reference`` times the oracle, row-parallel on every host core, as the
reference arm.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from grammar_constrained_logit_gb300 import synthetic as syn  # noqa: E402

METRIC = "apply_token_bitmask HBM GB/s (% of GB300 peak); fused mask+sample rows/s"
EB = {"f32": 4, "f16": 2, "bf16": 2}


# ------------------------------------------------------------ bytes per unit

def apply_rows(w: syn.Workload) -> int:
    if w.indices is None:
        return w.B
    return int(np.unique(w.indices[(w.indices >= 0) & (w.indices < min(w.B, w.bitmask.shape[0]))]).size)


def apply_bytes(w: syn.Workload) -> int:
    """In place: read + write of every applied logit, plus the mask words."""
    rows = apply_rows(w)
    return 2 * rows * w.vocab_size * EB[w.dtype] + rows * w.bitmask.shape[1] * 4


def sample_bytes(w: syn.Workload, masked: bool = True) -> int:
    """Fused mask + sample: each logit read once, the mask words of masked rows,
    8 bytes of id per row."""
    b = w.B * w.vocab_size * EB[w.dtype] + 8 * w.B
    if masked and w.bitmask is not None:
        b += apply_rows(w) * w.bitmask.shape[1] * 4
    return b


def _applied_rows(w: syn.Workload) -> np.ndarray:
    if w.indices is None:
        return np.arange(w.B)
    lim = min(w.B, w.bitmask.shape[0])
    return np.unique(w.indices[(w.indices >= 0) & (w.indices < lim)])


def _sector_flags(w: syn.Workload, b: int):
    """(any kept, any masked) per 32-byte sector of row b's first vocab_size
    tokens, from the row's mask bits (sectors aligned in memory)."""
    eb = EB[w.dtype]
    words = w.bitmask[b].view(np.uint32)
    bits = np.unpackbits(words.view(np.uint8), bitorder="little")[:w.vocab_size].astype(bool)
    phase = (b * w.stride * eb) % 32 // eb       # tokens before the row in its first sector
    per = 32 // eb
    n = phase + w.vocab_size
    pad_kept = np.zeros(-(-n // per) * per, dtype=bool)
    pad_mask = np.zeros_like(pad_kept)
    pad_kept[phase:n] = bits
    pad_mask[phase:n] = ~bits
    return pad_kept.reshape(-1, per).any(1), pad_mask.reshape(-1, per).any(1)


def sector_minimal_bytes(w: syn.Workload, kind: str) -> int:
    """The bytes a mask-aware kernel must move, counted from the actual mask in
    32-byte DRAM sectors.  In-place apply: every mask word of the applied rows,
    a sector write wherever a token is masked, and a sector read to merge where
    a sector mixes kept and masked tokens (all-kept sectors are not touched).
    Fused mask + sample: the mask words of masked rows, the sectors of masked
    rows that hold a kept token, every sector of unmasked rows, and the ids."""
    eb = EB[w.dtype]
    sec_row = -(-w.vocab_size * eb // 32)
    if kind == "apply":
        rows = _applied_rows(w)
        total = rows.size * w.bitmask.shape[1] * 4
        for b in rows:
            kept, masked = _sector_flags(w, int(b))
            total += 32 * int(masked.sum()) + 32 * int((kept & masked).sum())
        return total
    total = 8 * w.B
    masked_rows = set() if w.bitmask is None else set(int(b) for b in _applied_rows(w))
    for b in range(w.B):
        if b in masked_rows:
            kept, _ = _sector_flags(w, b)
            total += w.bitmask.shape[1] * 4 + 32 * int(kept.sum())
        else:
            total += 32 * sec_row
    return total


def describe(w: syn.Workload) -> str:
    s = f"{w.name}: B={w.B}, V={w.vocab_size} {w.dtype}"
    if w.cols != w.vocab_size or w.stride != w.cols:
        s += f" (row stride {w.stride})"
    if w.bitmask is not None:
        s += f", mask [{w.bitmask.shape[0]}x{w.bitmask.shape[1]}]"
    if w.indices is not None:
        s += f", {apply_rows(w)} indexed rows"
    return s


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str | None):
        self.proc = None
        self.path = None
        self.device_id = device_id

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "20"]
        if self.device_id:
            cmd += ["-i", self.device_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=open(self.path, "w"),
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        seen = set()
        for _, _, flags in rows:
            for n, f in zip(names, flags[1:5]):
                if f.lower().startswith("active"):
                    seen.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": rows[0][1],
                "reasons": sorted(seen), "samples": len(rows)}


# --------------------------------------------------------------- helpers

def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


# the sources each kernel is compiled from (with include/lp.h)
KERNEL_SOURCES = {
    "apply_kernel": ("apply.cu", "common.cuh"),
    "sample_stream_kernel": ("sample.cu", "common.cuh"),
    "sample_finish_kernel": ("sample.cu", "common.cuh"),
}


def kernel_source_hash(kernel: str, read=None) -> str:
    """Hash of the sources `kernel` is built from; `read(path)` gives a file's bytes
    (default: the working tree)."""
    read = read or (lambda rel: open(os.path.join(ROOT, rel), "rb").read())
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        h.update(read(os.path.join("grammar_constrained_logit_gb300", "csrc", f)))
    h.update(read(os.path.join("include", "lp.h")))
    return h.hexdigest()[:16]


def ncu_traffic(kernels, workload: str):
    """DRAM bytes per launch of the given kernels (summed: one hot-path call), from
    the committed ncu captures, if each was taken on its kernel's current
    sources; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    total = 0
    for k in ([kernels] if isinstance(kernels, str) else kernels):
        e = d.get("kernels", {}).get(f"{k}:{workload}")
        if e is None or e.get("source_hash") != kernel_source_hash(k):
            return None
        total += int(e["dram_bytes_per_launch"])
    return total


def make_workload(name: str) -> syn.Workload:
    return syn.WORKLOADS[name]()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value: float, device=None) -> float:
    """Max of a float over all ranks (a timing reduction, not a data-path collective)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Units processed by all ranks per second of the slowest rank (each rank runs
    the same per-rank workload: weak scaling)."""
    return units_per_rank * world / seconds


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------- GPU arm

class Op:
    """One hot-path call on one workload, with a ring of device input copies."""

    def __init__(self, kind: str, w: syn.Workload, ring_bytes_min: int, torch, ops,
                 min_copies: int = 2, row_flags: bool = False):
        self.kind, self.w, self.torch, self.ops = kind, w, torch, ops
        dev = torch.device("cuda")
        st = w.logits
        if w.dtype == "bf16":
            host = torch.from_numpy(st.view(np.int16)).view(torch.bfloat16)
        else:
            host = torch.from_numpy(st)
        touched = apply_bytes(w) if kind == "apply" else sample_bytes(w)
        per_copy = st.nbytes + (0 if w.bitmask is None else w.bitmask.nbytes)
        free = torch.cuda.mem_get_info()[0]
        self.R = int(max(2, min(64, -(-ring_bytes_min // max(touched, 1)))))
        # an apply reads only the bitmask (a few hundred KB a launch), so its copies
        # must not repeat within a graph, or a repeat reads its mask from L2
        self.R = max(self.R, min_copies)
        self.R = max(2, min(self.R, int(0.25 * free // max(per_copy, 1))))
        first = host.to(dev)
        self.logits = [first] + [first.clone() for _ in range(self.R - 1)]
        self.bitmask = None
        if w.bitmask is not None:
            b0 = torch.from_numpy(w.bitmask).to(dev)
            self.bitmask = [b0] + [b0.clone() for _ in range(self.R - 1)]
        self.indices = None if w.indices is None else torch.from_numpy(w.indices).to(dev)
        # the per-row flag selector with its keeps-a-token report, in place of indices
        self.flags = None
        if row_flags and kind == "apply":
            f = np.zeros(w.B, dtype=np.uint8)
            f[np.arange(w.B) if w.indices is None else w.indices] = 1
            self.flags = torch.from_numpy(f).to(dev)
        self.params = {k: torch.from_numpy(w.per_row(k)).to(dev)
                       for k in ("temperature", "top_k", "top_p", "min_p")}
        self.out = torch.empty(w.B, dtype=torch.int64, device=dev)
        # one zero-filled sampler workspace for every replay (the kernels leave it zeroed)
        self.ws = None
        if kind == "sample":
            tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[w.dtype]
            self.ws = torch.zeros(max(1, ops.sample_workspace_bytes(tdt, w.B, w.cols)),
                                  dtype=torch.uint8, device=dev)
        self.bytes = touched
        self.sector_minimal = sector_minimal_bytes(w, kind) if (
            w.bitmask is not None or kind == "sample") else None
        self.units = w.B
        # kernels one call launches: the apply kernel; or the sampler's stream and
        # finish kernels per launch of at most 16384 rows
        self.kernels = 1 if kind == "apply" else 2 * -(-w.B // 16384)

    def launch(self, slot: int, step: int):
        w, ops = self.w, self.ops
        lg = self.logits[slot % self.R][:, :w.cols]
        bm = None if self.bitmask is None else self.bitmask[slot % self.R]
        if self.kind == "apply" and self.flags is not None:
            ops.apply_token_bitmask_rows(lg, bm, self.flags, vocab_size=w.vocab_size, report=True)
        elif self.kind == "apply":
            ops.apply_token_bitmask_inplace(lg, bm, vocab_size=w.vocab_size, indices=self.indices)
        else:
            p = self.params
            ops.mask_and_sample(lg, bm, p["temperature"], p["top_k"], p["top_p"], p["min_p"],
                                seed=w.seed, offset=w.offsets[step % len(w.offsets)],
                                indices=self.indices,
                                vocab_size=w.vocab_size if bm is not None else None,
                                out=self.out, workspace=self.ws)

    def capture(self, nsteps: int, first_step: int):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.launch(0, 0)  # sets kernel attributes before capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for j in range(nsteps):
                self.launch(first_step + j, first_step + j)
        return g


class E2EPipeline:
    """Steps through the public API with host inputs and a host result, the way a
    serving loop overlaps them: step i's upload (pinned host to device, on its own
    stream) runs while step i - 1 is applied and read back; two sets of device
    buffers alternate.  Every step still copies all of its inputs in and its
    result out inside the timed region."""

    def __init__(self, torch, make_set):
        self.torch = torch
        self.sets = [make_set(), make_set()]
        self.up, self.work = torch.cuda.Stream(), torch.cuda.Stream()
        self.ready = [torch.cuda.Event(), torch.cuda.Event()]
        self.free = [torch.cuda.Event(), torch.cuda.Event()]

    def step(self, i, upload, run):
        k = i % 2
        b = self.sets[k]
        with self.torch.cuda.stream(self.up):
            self.up.wait_event(self.free[k])  # the set's previous result is read back
            upload(b)
            self.ready[k].record(self.up)
        with self.torch.cuda.stream(self.work):
            self.work.wait_event(self.ready[k])
            run(b, i)
            self.free[k].record(self.work)

    def time(self, steps, upload, run) -> float:
        torch = self.torch
        for i in range(3):
            self.step(i, upload, run)
        torch.cuda.synchronize()
        cur = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        self.up.wait_stream(cur)
        self.work.wait_stream(cur)
        for i in range(steps):
            self.step(i, upload, run)
        cur.wait_stream(self.up)
        cur.wait_stream(self.work)
        e1.record(cur)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / steps


def _pinned_logits(w: syn.Workload, torch):
    if w.dtype == "bf16":
        return torch.from_numpy(w.logits.view(np.int16)).view(torch.bfloat16).pin_memory()
    return torch.from_numpy(w.logits).pin_memory()


def e2e_apply(w: syn.Workload, steps: int, torch, ops) -> dict:
    """apply_token_bitmask_inplace through the public API: per step the logits,
    bitmask and indices copied in from pinned host memory, the masked logits
    copied back (consecutive steps overlap, E2EPipeline)."""
    dev = torch.device("cuda")
    host = _pinned_logits(w, torch)
    bm_h = torch.from_numpy(w.bitmask).pin_memory()
    idx_h = None if w.indices is None else torch.from_numpy(w.indices).pin_memory()
    out_h = torch.empty_like(host).pin_memory()

    def make_set():
        return {"lg": torch.empty_like(host, device=dev), "bm": torch.empty_like(bm_h, device=dev),
                "idx": None if idx_h is None else torch.empty_like(idx_h, device=dev)}

    def upload(b):
        b["lg"].copy_(host, non_blocking=True)
        b["bm"].copy_(bm_h, non_blocking=True)
        if idx_h is not None:
            b["idx"].copy_(idx_h, non_blocking=True)

    def run(b, i):
        ops.apply_token_bitmask_inplace(b["lg"][:, :w.cols], b["bm"], vocab_size=w.vocab_size,
                                        indices=b["idx"])
        out_h.copy_(b["lg"], non_blocking=True)

    sec = E2EPipeline(torch, make_set).time(steps, upload, run)
    h2d = host.numel() * host.element_size() + bm_h.numel() * 4 + (0 if idx_h is None else idx_h.numel() * 4)
    return {"value": round(apply_bytes(w) / sec / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(out_h.numel() * out_h.element_size()),
            "ms_per_step": round(sec * 1e3, 4),
            "copies": "every step's inputs in and result out; step i's upload overlaps step i-1's apply and read-back"}


def e2e_sample(w: syn.Workload, steps: int, torch, ops) -> dict:
    """mask_and_sample through the public API: per step the logits, bitmask,
    indices and parameters copied in from pinned host memory, the ids copied
    back (consecutive steps overlap, E2EPipeline)."""
    dev = torch.device("cuda")
    host = _pinned_logits(w, torch)
    bm_h = None if w.bitmask is None else torch.from_numpy(w.bitmask).pin_memory()
    idx_h = None if w.indices is None else torch.from_numpy(w.indices).pin_memory()
    par_h = {k: torch.from_numpy(w.per_row(k)).pin_memory()
             for k in ("temperature", "top_k", "top_p", "min_p")}
    ids_h = torch.empty(w.B, dtype=torch.int64).pin_memory()

    def make_set():
        return {"lg": torch.empty_like(host, device=dev),
                "bm": None if bm_h is None else torch.empty_like(bm_h, device=dev),
                "idx": None if idx_h is None else torch.empty_like(idx_h, device=dev),
                "par": {k: torch.empty_like(v, device=dev) for k, v in par_h.items()},
                "ids": torch.empty(w.B, dtype=torch.int64, device=dev)}

    def upload(b):
        b["lg"].copy_(host, non_blocking=True)
        if bm_h is not None:
            b["bm"].copy_(bm_h, non_blocking=True)
        if idx_h is not None:
            b["idx"].copy_(idx_h, non_blocking=True)
        for k in par_h:
            b["par"][k].copy_(par_h[k], non_blocking=True)

    def run(b, i):
        p = b["par"]
        ops.mask_and_sample(b["lg"][:, :w.cols], b["bm"], p["temperature"], p["top_k"], p["top_p"],
                            p["min_p"], seed=w.seed, offset=w.offsets[i % len(w.offsets)],
                            indices=b["idx"], vocab_size=w.vocab_size if bm_h is not None else None,
                            out=b["ids"])
        ids_h.copy_(b["ids"], non_blocking=True)

    sec = E2EPipeline(torch, make_set).time(steps, upload, run)
    h2d = host.numel() * host.element_size() + (0 if bm_h is None else bm_h.numel() * 4) + \
        (0 if idx_h is None else idx_h.numel() * 4) + sum(v.numel() * 4 for v in par_h.values())
    return {"value": round(w.B / sec, 1), "unit": "rows/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(8 * w.B), "ms_per_step": round(sec * 1e3, 4),
            "copies": "every step's inputs in and ids out; step i's upload overlaps step i-1's sampling"}


def roofline(bytes_per_launch: int, sec_per_launch: float, peak: dict, traffic,
             sector_minimal: int | None = None) -> dict:
    achieved = bytes_per_launch / sec_per_launch / 1e9
    r = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak["hbm_gbs"],
         "unit": "GB/s", "frac": round(achieved / peak["hbm_gbs"], 4),
         "peak_source": peak["source"], "traffic": traffic,
         "algorithmic_bytes_per_launch": int(bytes_per_launch),
         "us_per_launch": round(sec_per_launch * 1e6, 3)}
    if sector_minimal is not None:
        r["sector_minimal_bytes_per_launch"] = int(sector_minimal)
        r["frac_sector_minimal"] = round(sector_minimal / sec_per_launch / 1e9 / peak["hbm_gbs"], 4)
    return r


class Timer:
    """Times a plan of ops: K steps in CUDA graphs of G steps, each replay
    bracketed by CUDA events on the launching stream, an untimed write of twice
    the L2 before every replay, W warm-up steps first."""

    def __init__(self, torch, l2: int):
        self.torch, self.l2 = torch, l2
        self.flush = torch.empty(2 * l2, dtype=torch.uint8, device="cuda")
        self.clean = torch.zeros(2 * l2 // 4, dtype=torch.int32, device="cuda")

    def empty_l2(self, r: int):
        """Untimed: a write of twice the L2 evicts every input, then a read of
        another twice the L2 writes those dirty lines back, so that the timed
        kernels neither find their inputs in L2 nor pay for the flush's own
        write-back.  Then the device spins for about 0.25 ms (no memory traffic),
        so that the host has queued the replay before its start event is
        recorded: otherwise a run of one or two replays also times the host's
        submission of its first replay (about 1 us a step on the apply at 20 steps)."""
        self.flush.fill_(r & 0xFF)
        self.sink = self.clean.sum()
        spin = getattr(self.torch.cuda, "_sleep", None)  # a PyTorch test helper
        if spin is not None:
            spin(500_000)

    def run(self, plan, K: int, W: int, G: int, sampler=None):
        torch = self.torch
        graphs = [op.capture(G, 0) for op in plan]
        rem = K % G
        rem_graphs = [op.capture(rem, (K // G) * G) for op in plan] if rem else None
        for _ in range(max(1, -(-W // G))):
            for g in graphs:
                g.replay()
        torch.cuda.synchronize()
        if sampler is not None:
            sampler.start()
        barrier()
        torch.cuda.synchronize()
        reps = K // G
        nrep = reps + (1 if rem else 0)
        ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
        marks = [[(ev(), ev()) for _ in plan] for _ in range(nrep)]
        for r in range(nrep):
            for i, g in enumerate(graphs if r < reps else rem_graphs):
                self.empty_l2(r)
                marks[r][i][0].record()
                g.replay()
                marks[r][i][1].record()
        torch.cuda.synchronize()
        barrier()
        clocks = sampler.stop() if sampler is not None else None
        per_op = [0.0] * len(plan)
        for row in marks:
            for i, (b, e) in enumerate(row):
                per_op[i] += b.elapsed_time(e) / 1e3
        dev = torch.device("cuda")
        total = reduce_max(sum(per_op), dev)
        per_op = [reduce_max(t, dev) for t in per_op]
        del graphs, rem_graphs
        return per_op, total, clocks, nrep


def graph_len(args) -> int:
    """Steps per graph: at most --graph-steps, and at most K/4 so that even a short
    run times at least four replays.  Each replay starts after the L2 has been
    emptied, with the kernels' code and parameters cold as well, which costs
    5-7 us once per replay: a 20-step run (graphs of 5) carries about 1 us of it
    per step, a 2000-step run (graphs of 100) almost none."""
    return max(1, min(args.graph_steps, args.steps // 4 if args.steps >= 4 else 1))


def op_line(op, sec: float, ws: int, peak: dict) -> dict:
    """One op's figures: time per launch, throughput and its roofline (dense and
    sector-minimal bytes)."""
    wl = op.w.name + ("_rows" if op.kind == "apply" and op.flags is not None else "")
    knames = (["apply_kernel"] if op.kind == "apply" else
              ["sample_stream_kernel", "sample_finish_kernel"])
    rf = roofline(op.bytes, sec, peak, ncu_traffic(knames, wl), op.sector_minimal)
    line = {"workload": describe(op.w), "us_per_launch": round(sec * 1e6, 3), "roofline": rf}
    if op.kind == "apply":
        line.update(value=round(whole_job_rate(op.bytes, ws, sec) / 1e9, 2), unit="GB/s")
    else:
        line.update(value=round(whole_job_rate(op.units, ws, sec), 1), unit="rows/s",
                    GBps_algorithmic=rf["achieved"])
    return line


# The per-configuration block of the default run: every configuration of the
# benchmark list, each sampler sub-run and the apply legs, timed one after another.
CONFIGS = [
    ("C1 tiny_greedy (launch-bound; latency reported)", "tiny_greedy", None, ("apply", "sample")),
    ("C2 apply_only", "apply_only", None, ("apply",)),
    ("C3 fused_sample", "fused_sample", None, ("sample", "apply")),
    ("C4 zipf_top_p top_p 0.5", "zipf_top_p", 0.5, ("sample",)),
    ("C4 zipf_top_p top_p 0.9", "zipf_top_p", 0.9, ("sample",)),
    ("C4 zipf_top_p top_p 0.99", "zipf_top_p", 0.99, ("sample",)),
    ("C4 zipf_top_p greedy", "zipf_top_p", "greedy", ("sample",)),
    ("C5 speculative_verify", "speculative_verify", None, ("sample", "apply")),
]


def config_workload(name: str, top_p, base: syn.Workload | None = None):
    w = make_workload(name) if base is None else base
    if name == "zipf_top_p":
        w.temperature, w.top_p = 0.7, 0.9
        if top_p == "greedy":
            w.temperature = 0.0
        elif top_p is not None:
            w.top_p = float(top_p)
    return w


def run_configs(args, timer, torch, ops, ring_min: int, peak: dict, ws: int,
                dev_id) -> dict:
    K, W, G = args.steps, args.warmup, graph_len(args)
    out = {}
    base = None
    for label, name, tp, kinds in CONFIGS:
        if base is None or base.name != name:
            base = None
            torch.cuda.empty_cache()
        base = config_workload(name, tp, base)
        w = base
        plan = [Op(k, w, ring_min, torch, ops, G if k == "apply" else 2) for k in kinds]
        per_op, _, clocks, nrep = timer.run(plan, K, W, G, ClockSampler(dev_id))
        entry = {}
        for op, t in zip(plan, per_op):
            entry["fused_mask_sample" if op.kind == "sample" and w.bitmask is not None
                  else ("sample" if op.kind == "sample" else "apply")] = op_line(op, t / K, ws, peak)
        entry["gpu_launches"] = K * sum(op.kernels for op in plan)
        entry["replays"] = nrep
        entry["clocks"] = clocks
        out[label] = entry
        del plan
    return out


def run_gpu(args) -> dict | None:
    import torch

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from grammar_constrained_logit_gb300 import ops
    from grammar_constrained_logit_gb300 import _lib

    _lib.load()
    dev_props = torch.cuda.get_device_properties(torch.cuda.current_device())
    l2 = int(getattr(dev_props, "L2_cache_size", 128 << 20))
    ring_min = 4 * l2
    K, W = args.steps, args.warmup
    G = graph_len(args)

    plan = []
    if args.workload == "default":
        wa, wf = make_workload("apply_only"), make_workload("fused_sample")
        plan = [Op("apply", wa, ring_min, torch, ops, G), Op("sample", wf, ring_min, torch, ops)]
    elif args.workload == "apply_only":
        plan = [Op("apply", make_workload("apply_only"), ring_min, torch, ops, G,
                   row_flags=args.row_flags)]
    elif args.workload == "tiny_greedy":
        w = make_workload("tiny_greedy")
        plan = [Op("apply", w, ring_min, torch, ops), Op("sample", w, ring_min, torch, ops)]
    else:
        w = config_workload(args.workload, args.top_p if args.workload == "zipf_top_p" else None)
        plan = [Op("sample", w, ring_min, torch, ops)]
        if args.apply_leg and w.bitmask is not None:
            plan.append(Op("apply", w, ring_min, torch, ops, G))

    dev_id = None
    try:
        dev_id = str(dev_props.uuid)
        if not dev_id.startswith("GPU-"):
            dev_id = "GPU-" + dev_id
    except Exception:  # noqa: BLE001
        dev_id = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0] or None
    timer = Timer(torch, l2)
    per_op, total_s, clocks, nrep = timer.run(plan, K, W, G, ClockSampler(dev_id))
    if rank != 0 and args.workload != "default":
        return None

    peak = measured_peaks()
    res = {"metric": METRIC, "n_gpus": ws, "steps": K, "warmup": W,
           "ms_per_step": round(total_s / K * 1e3, 5), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": plan[0].w.dtype,
           "data": "synthetic (seeded generators shaped like the pages' workloads)",
           "gpu_launches": K * sum(op.kernels for op in plan) * ws}
    cfg = {"workload": " + ".join(describe(op.w) + f" [{op.kind}]" for op in plan),
           "l2": f"an untimed write of 2x the {l2 >> 20} MB L2, then a read of another 2x, "
                 "before every graph replay, and inputs in device rings (>= 4x the L2; an "
                 "apply's copies do not repeat within a graph), so no step reads its batch "
                 "from L2",
           "timing": f"CUDA graphs of {G} steps, {nrep} replays; CUDA events on the launch "
                     "stream",
           "parallelism": f"replicas x{ws} (rows shard with no collective)"}
    for op in plan:
        cfg[f"ring_{op.kind}"] = op.R
        if op.flags is not None:
            cfg["selector"] = "per-row flags with the keeps-a-token report (lp_apply_token_bitmask_rows)"
    res["config"] = cfg
    lines = {}
    for op, t in zip(plan, per_op):
        lines.setdefault(op.kind, op_line(op, t / K, ws, peak))
    if "apply" in lines and args.workload in ("default", "apply_only", "tiny_greedy"):
        res["value"], res["unit"] = lines["apply"]["value"], "GB/s"
    else:
        res["value"], res["unit"] = lines["sample"]["value"], "rows/s"
    dominant = max(zip(plan, per_op), key=lambda x: x[1])[0]
    res["roofline"] = dict(lines[dominant.kind]["roofline"])
    res["roofline"]["kernel"] = (
        "apply_kernel" if dominant.kind == "apply" else
        "lp_mask_and_sample call: sample_stream_kernel + sample_finish_kernel, timed together")
    if "apply" in lines:
        res["apply"] = lines["apply"]
    if "sample" in lines:
        res["fused_mask_sample"] = lines["sample"]
    res["clocks"] = clocks

    if not args.no_e2e:
        e2e = {}
        for op in plan:
            if op.kind == "apply" and "apply" not in e2e:
                e2e["apply"] = e2e_apply(op.w, args.e2e_steps, torch, ops)
            elif op.kind == "sample" and "sample" not in e2e:
                e2e["sample"] = e2e_sample(op.w, args.e2e_steps, torch, ops)
        head = e2e.get("apply") if res["unit"] == "GB/s" else e2e.get("sample")
        res["e2e"] = {"value": head["value"], "unit": head["unit"],
                      "h2d_bytes_per_step": sum(v["h2d_bytes_per_step"] for v in e2e.values()),
                      "d2h_bytes_per_step": sum(v["d2h_bytes_per_step"] for v in e2e.values()),
                      "parts": e2e}
    del plan
    torch.cuda.empty_cache()
    if args.workload == "default" and not args.no_configs:
        res["configs"] = run_configs(args, timer, torch, ops, ring_min, peak, ws, dev_id)
    if rank != 0:
        return None
    if not args.no_cpu_baseline and ws == 1:
        res["cpu_baseline"] = cpu_baseline(args)
    return res


# -------------------------------------------------------------- CPU oracle

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _time_for(fn, seconds: float):
    fn()
    n, t0 = 0, time.perf_counter()
    while True:
        fn()
        n += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            return dt / n, n


class OracleJob:
    """One bounded sample of a workload run by the CPU oracle, as it stands, on
    ``threads`` host threads: the rows are split into one contiguous share per
    thread, and each thread runs the oracle's C code on its share (the binding
    releases the interpreter lock during the call)."""

    def __init__(self, kind: str, w: syn.Workload, threads: int, rows_per_thread: int = 0):
        import oracle

        self.kind, self.w, self.threads = kind, w, max(1, threads)
        dt = {"f32": 0, "f16": 1, "bf16": 2}[w.dtype]
        if kind == "apply":
            rows = _applied_rows(w).astype(np.int32)
            self.rows = rows
            self.out = w.logits.copy()
            shares = [c for c in np.array_split(rows, self.threads) if c.size]
            self.calls = [
                (lambda c=c: oracle.apply(w.logits, w.bitmask, dtype=dt, vocab_size=w.vocab_size,
                                          indices=c, cols=w.cols, out=self.out))
                for c in shares]
            self.units = apply_bytes(w) * rows.size / max(apply_rows(w), 1)
            self.desc = f"all {rows.size} applied rows"
        else:
            nr = min(w.B, max(1, rows_per_thread) * self.threads)
            rows = np.sort(np.random.default_rng(0).choice(w.B, size=nr, replace=False))
            self.rows = rows
            shares = [c for c in np.array_split(rows, self.threads) if c.size]
            self.calls = [_oracle_sample_rows(w, c) for c in shares]
            self.units = float(nr)
            self.desc = f"{nr} seeded rows"
        self.pool = None
        if len(self.calls) > 1:
            from concurrent.futures import ThreadPoolExecutor

            self.pool = ThreadPoolExecutor(len(self.calls))

    def __call__(self):
        if self.pool is None:
            self.calls[0]()
        else:
            list(self.pool.map(lambda f: f(), self.calls))

    def close(self):
        if self.pool is not None:
            self.pool.shutdown()

    def rate(self, sec: float):
        if self.kind == "apply":
            return round(self.units / sec / 1e9, 4), "GB/s"
        return round(self.units / sec, 3), "rows/s"


def _oracle_sample_rows(w: syn.Workload, rows: np.ndarray, offset: int = 0):
    import oracle

    pr = {k: w.per_row(k)[rows] for k in ("temperature", "top_k", "top_p", "min_p")}
    dt = {"f32": 0, "f16": 1, "bf16": 2}[w.dtype]
    lg = np.ascontiguousarray(w.logits[rows])
    return lambda: oracle.mask_and_sample(
        lg, dtype=dt, bitmask=w.bitmask, vocab_size=w.vocab_size if w.bitmask is not None else None,
        indices=w.indices, cols=w.cols, temperature=pr["temperature"], top_k=pr["top_k"],
        top_p=pr["top_p"], min_p=pr["min_p"], seed=w.seed, offset=offset, row_ids=rows)


def bench_workloads(workload: str, top_p="0.9"):
    """(kind, workload) pairs of a bench run: the headline apply and fused
    workloads by default, else the selected one."""
    if workload == "default":
        return [("apply", make_workload("apply_only")), ("sample", make_workload("fused_sample"))]
    if workload == "apply_only":
        return [("apply", make_workload("apply_only"))]
    if workload == "tiny_greedy":
        w = make_workload("tiny_greedy")
        return [("apply", w), ("sample", w)]
    return [("sample", config_workload(workload, top_p if workload == "zipf_top_p" else None))]


def cpu_baseline(args) -> dict:
    """The oracle, as it stands, on bounded samples of the bench's workloads: on
    one thread, and row-parallel on every core of this process's affinity set."""
    cores = host_cores()
    parts = {}
    jobs = bench_workloads(args.workload, args.top_p)
    per = args.cpu_seconds / max(2 * len(jobs), 1)
    for kind, w in jobs:
        for threads in (1, cores):
            job = OracleJob(kind, w, threads, rows_per_thread=16 if threads == 1 else 4)
            sec, n = _time_for(job, per)
            job.close()
            v, u = job.rate(sec)
            parts[f"{kind}_{threads}_threads"] = {
                "value": v, "unit": u, "cores": threads,
                "sample": f"{describe(w)}: {job.desc}, {n} repeats"}
    lead = parts[f"{jobs[0][0]}_{cores}_threads"]
    return {"value": lead["value"], "unit": lead["unit"], "cores": cores, "kind": "oracle",
            "sample": lead["sample"] + f"; row-parallel over {cores} host threads, the "
                                       "single-thread figures beside it in parts",
            "parts": parts}


def run_reference(args) -> dict | None:
    """The oracle timed as the reference arm, row-parallel on every host core:
    each step one bounded sample of the workload (the applied rows, or seeded
    sampled rows, sized so the run stays in minutes)."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle

    oracle.build()
    cores = host_cores()
    jobs_in = bench_workloads(args.workload, args.top_p)
    K, W = args.steps, args.warmup
    budget = args.reference_seconds / max(K + W, 1) / len(jobs_in)   # seconds per call
    jobs = []
    for kind, w in jobs_in:
        if kind == "apply":
            jobs.append(OracleJob(kind, w, cores))
        else:
            probe = OracleJob(kind, w, 1, rows_per_thread=1)
            t1, _ = _time_for(probe, 0.2)
            per_thread = int(max(1, min(-(-w.B // cores), budget / max(t1, 1e-9))))
            jobs.append(OracleJob(kind, w, cores, rows_per_thread=per_thread))
    times = [0.0] * len(jobs)
    for _ in range(W):
        for job in jobs:
            job()
    for _ in range(K):
        for i, job in enumerate(jobs):
            t0 = time.perf_counter()
            job()
            times[i] += time.perf_counter() - t0
    for job in jobs:
        job.close()
    res = {"impl": "reference", "metric": METRIC, "n_gpus": 1, "steps": K, "warmup": W,
           "ms_per_step": round(sum(times) / max(K, 1) * 1e3, 4), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": jobs_in[0][1].dtype,
           "data": "synthetic (seeded generators shaped like the pages' workloads)",
           "gpu_launches": 0}
    parts = {}
    for job, t in zip(jobs, times):
        v, u = job.rate(t / max(K, 1))
        parts[job.kind] = {"value": v, "unit": u,
                           "sample": f"{describe(job.w)}: {job.desc} per step, row-parallel "
                                     f"over {cores} host threads"}
    head = parts.get("apply") or parts.get("sample")
    res["value"], res["unit"] = head["value"], head["unit"]
    res["config"] = {"workload": " + ".join(describe(w) for _, w in jobs_in),
                     "parallelism": f"CPU oracle, row-parallel over {cores} host threads"}
    res["cpu_baseline"] = {"value": head["value"], "unit": head["unit"], "cores": cores,
                           "kind": "oracle", "sample": head["sample"], "parts": parts}
    res["e2e"] = {"value": head["value"], "unit": head["unit"], "h2d_bytes_per_step": 0,
                  "d2h_bytes_per_step": 0}
    if "sample" in parts and "apply" in parts:
        res["fused_mask_sample"] = parts["sample"]
    return res


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="default",
                    choices=["default", *syn.WORKLOADS.keys()])
    ap.add_argument("--top-p", default="0.9", help="zipf_top_p: 0.5, 0.9, 0.99 or greedy")
    ap.add_argument("--graph-steps", type=int, default=100)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=90.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--row-flags", action="store_true",
                    help="apply_only: select the rows by per-row flags and report which keep a "
                         "token (lp_apply_token_bitmask_rows) instead of indices")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="default run: skip the per-configuration block")
    ap.add_argument("--apply-leg", action="store_true",
                    help="a sampler workload with a mask: also time the in-place apply alone")
    args = ap.parse_args(argv)
    res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
