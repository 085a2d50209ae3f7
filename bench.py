"""Benchmark of the paged-KV decode hot path on GB300.

One step = the whole hot path over one batch: the append of each sequence's
new token and the decode over its paged context, as one fused call (pa_verify
with one query per sequence; --unfused times pa_cache_write then pa_decode),
with the inputs resident in HBM. The headline workload is the 32k-context decode (8 sequences x 32768
tokens, 12 query / 2 KV heads, head_dim 128, bf16, 16384-block pool). The
64-sequence decode, the Qwen2-1.5B-shaped decode and the fused speculative
verify are measured too and reported under "per_config".

Metric: achieved KV-read bandwidth (algorithmic K+V bytes of every valid token
per step / step time, GB/s) and microseconds per call. Timing uses CUDA events
on the launching stream, with L2 flushed (a 256 MiB write, then a 256 MiB read
that retires the write-backs) before every timed step, each step timed on its
own. Every workload is also timed as a layer loop ("layer_loop"): many calls
back to back between one event pair, rotating over per-layer copies of the
pool so that no call finds its K/V in L2, as a decode step calls attention
once per layer. rank 0 prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload c4] [--no-extra]

--impl reference times the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload, on the host cores. --prefill
times the paged prefill workloads alone; --record-traffic stores an ncu
capture's DRAM bytes.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from paged_kv_decode_pa_gb300 import accounting, inputs  # noqa: E402

METRIC = "paged-decode attention: achieved KV-read HBM GB/s (% of peak), µs per call"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="c4", choices=["c2", "c3", "c4", "c5"])
    ap.add_argument("--kv", default="bf16", choices=["bf16", "int8"],
                    help="KV pool format (int8: bytes + scales, dequantised inside the kernel)")
    ap.add_argument("--no-extra", action="store_true", help="skip the per_config measurements")
    ap.add_argument("--kernel", default="auto", choices=["auto", "mma", "simt"])
    ap.add_argument("--split-tokens", type=int, default=0)
    ap.add_argument("--buckets", action="store_true",
                    help="also time the Qwen2-shaped decode step per batch bucket (1..64), direct and as "
                         "CUDA-graph replays")
    ap.add_argument("--graph", action="store_true",
                    help="time each step as a replay of a captured CUDA graph of the step")
    ap.add_argument("--unfused", action="store_true",
                    help="time a decode step as two calls, pa_cache_write then pa_decode")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU baseline sample budget")
    ap.add_argument("--record-traffic", nargs=2, metavar=("WORKLOAD", "NCU_CSV"),
                    help="store the DRAM bytes of an ncu capture (`ncu -i REPORT --page raw --csv` output) "
                         "for WORKLOAD (c4, c3, c5, c4_int8, ...) in profiles/decode_traffic.json; no GPU")
    ap.add_argument("--prefill", action="store_true",
                    help="time only the paged prefill workloads (both kernels, --steps calls each) and print "
                         "their line")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; timing reduction only)

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        import torch

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# What each workload times: the configs as specified, with the 64-request
# decode (c3) run as its bucket of 64 rows, 57 sequences plus 7 padded rows
# that attend only to the spare block.
TIMED_OVERRIDES = {"c3": {"padded_rows": 7}}


def timed_spec(name: str):
    base = inputs.CONFIGS[name]
    over = TIMED_OVERRIDES.get(name)
    return inputs.Spec(**{**base.__dict__, **over}) if over else base


def timed_workload(name: str, seed=None):
    spec = timed_spec(name)
    return inputs.generate(spec, seed=spec.seed if seed is None else seed)


def rank_workload(name: str, rank: int):
    """This rank's replica of a workload: same shapes, its own seed (weak scaling)."""
    return timed_workload(name, seed=timed_spec(name).seed + 1000 * rank)


def whole_job_gbs(kv_bytes_per_rank: int, world: int, ms_step_max: float) -> float:
    """Whole-job KV-read rate: the bytes every rank read in one step, over the
    slowest rank's step time."""
    return kv_bytes_per_rank * world / (ms_step_max * 1e-3) / 1e9


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# measured peaks, clocks, ncu traffic

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


# Device sources each timed kernel is built from (with include/pa.h): a
# recorded traffic figure stays valid while these files are unchanged.
TRAFFIC_SOURCES = {
    "attn_mma": ("attn_mma.cu", "mma_tile.cuh", "pa_device.cuh"),
    "attn_q8": ("attn_q8.cu", "q8.cuh", "mma_tile.cuh", "pa_device.cuh"),
}


def traffic_kernel(workload: str) -> str:
    return "attn_q8" if workload.endswith("_int8") else "attn_mma"


def header_code(text: str) -> str:
    """include/pa.h without its comments and blank space: what a kernel sees."""
    import re

    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel: str = "attn_mma") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_pa_gb300", "csrc")
    for name in TRAFFIC_SOURCES[kernel]:
        h.update(open(os.path.join(csrc, name), "rb").read())
    h.update(header_code(open(os.path.join(ROOT, "include", "pa.h")).read()).encode())
    return h.hexdigest()[:16]


def record_traffic(workload: str, csv_path: str) -> dict:
    """Store one ncu capture's DRAM bytes for a workload in
    profiles/decode_traffic.json. csv_path: `ncu -i <report> --page raw --csv`
    output holding one launch of the workload's attention kernel."""
    import csv

    rows = list(csv.reader(open(csv_path)))
    hdr = rows[0]
    data = [r for r in rows[2:] if len(r) == len(hdr)]
    if len(data) != 1:
        raise SystemExit(f"{csv_path}: expected one captured launch, found {len(data)}")
    rec = dict(zip(hdr, data[0]))
    units = dict(zip(hdr, rows[1]))
    scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}

    def nbytes(name):
        return int(round(float(rec[name].replace(",", "")) * scale[units[name]]))

    tscale = {"ns": 1e-3, "nsecond": 1e-3, "us": 1.0, "usecond": 1.0, "ms": 1e3, "msecond": 1e3}
    dur_us = float(rec["gpu__time_duration.sum"].replace(",", "")) * tscale[units["gpu__time_duration.sum"]]
    kernel = traffic_kernel(workload)
    if kernel not in rec.get("Kernel Name", ""):
        raise SystemExit(f"{csv_path}: captured {rec.get('Kernel Name')!r}, expected {kernel}")
    rd, wr = nbytes("dram__bytes_read.sum"), nbytes("dram__bytes_write.sum")
    entry = {"kernel": rec.get("Kernel Name"), "kernel_source_hash": kernel_source_hash(kernel),
             "dram_bytes_per_launch": rd + wr, "dram_read_bytes": rd, "dram_write_bytes": wr,
             "ncu_duration_us": round(dur_us, 3)}
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        allrec = json.load(open(path))
    except Exception:
        allrec = {}
    allrec[workload] = entry
    with open(path, "w") as f:
        json.dump(allrec, f, indent=1)
        f.write("\n")
    return entry


def ncu_record(workload: str):
    """The committed ncu record of a workload's attention kernel (DRAM bytes and
    duration of one launch), if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        rec = json.load(open(path))
    except Exception:
        return None
    entry = rec.get(workload)
    if not entry or entry.get("kernel_source_hash") != kernel_source_hash(traffic_kernel(workload)):
        return None
    return entry


def ncu_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current kernels."""
    entry = ncu_record(workload)
    return entry.get("dram_bytes_per_launch") if entry else None


# ---------------------------------------------------------------------------
# GPU arm

class DecodeStep:
    """Device-resident buffers of one workload and the call(s) of one step.

    A decode step appends each sequence's new token and attends. By default it
    is the single fused call (pa_verify with one query per sequence, which is
    pa_cache_write followed by pa_decode in one launch); with fused=False it is
    the two calls. A verify workload's step is pa_verify.
    """

    def __init__(self, w, device, split_tokens=0, kernel="auto", fused=True, kv="bf16"):
        import paged_kv_decode_pa_gb300 as pa

        self.pa = pa
        self.w = w
        self.kv = kv
        self.dev = device
        self.split = split_tokens
        self.kernel = kernel
        self.scales = {}
        if kv == "int8":  # a seeded int8 pool for the same tables and lengths
            pool = inputs.q8_pool(w)
            self.kc = pa.to_torch(pool.k_codes, device)
            self.vc = pa.to_torch(pool.v_codes, device)
            self.scales = {"k_scale": pa.to_torch(pool.k_scale, device),
                           "v_scale": pa.to_torch(pool.v_scale, device)}
        else:
            self.kc = pa.to_torch(w.k_cache, device)
            self.vc = pa.to_torch(w.v_cache, device)
        self.q = pa.to_torch(w.q, device)
        self.k_new = pa.to_torch(w.k_new, device)
        self.v_new = pa.to_torch(w.v_new, device)
        self.slots = pa.to_torch(w.slot_mapping, device)
        self.tables = pa.to_torch(w.block_tables, device)
        self.lens = pa.to_torch(w.context_lens, device)
        self.out = self.q.new_empty(self.q.shape)
        s = w.spec
        self.nq = s.num_queries
        self.fused = fused or self.nq > 1
        self.q4 = self.q if self.q.dim() == 4 else self.q.unsqueeze(1)
        self.out4 = self.out if self.out.dim() == 4 else self.out.unsqueeze(1)
        self.ws = pa.new_workspace(s.batch, self.nq, s.q_heads, s.kv_heads, w.max_context_len, device,
                                   split_tokens)

    def rebind(self, q, k_new, v_new, slots, tables, lens):
        """A copy of this step that reads its per-step inputs from other device
        tensors (same shapes); caches, output and workspace are shared."""
        import copy

        st = copy.copy(self)
        st.q, st.k_new, st.v_new, st.slots, st.tables, st.lens = q, k_new, v_new, slots, tables, lens
        st.q4 = q if q.dim() == 4 else q.unsqueeze(1)
        return st

    def write(self):
        self.pa.pa_cache_write(self.kc, self.vc, self.k_new, self.v_new, self.slots, **self.scales)

    def attend(self):
        w = self.w
        if not self.fused:
            self.pa.pa_decode(self.kc, self.vc, self.q, self.tables, self.lens, w.max_context_len, w.scale,
                              self.ws, out=self.out, split_tokens=self.split, kernel=self.kernel, **self.scales)
        else:
            self.pa.pa_verify(self.kc, self.vc, self.q4, self.k_new, self.v_new, self.slots, self.tables,
                              self.lens, w.max_context_len, w.scale, self.ws, out=self.out4,
                              split_tokens=self.split, kernel=self.kernel, **self.scales)

    def run(self):
        """One whole step."""
        if not self.fused:
            self.write()
        self.attend()

    def capture(self):
        """Record one step in a CUDA graph, as an engine does per batch bucket
        ("From 183 ms to 19 ms per decode step", section "4. CUDA graphs per
        batch bucket"); every buffer the graph reads is owned by this object."""
        import torch

        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.run()  # warm the library's per-device set-up outside the capture
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.run()
        torch.cuda.synchronize()


def make_l2_flush(device):
    """Return a function that leaves L2 holding nothing the timed step reads.

    It writes a buffer larger than L2, then reads a second one: the read
    evicts the dirty lines the write left, so their write-back to HBM happens
    here and not inside the timed region (where it would compete with the
    kernel's reads).
    """
    import torch

    dirty = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    clean = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)

    def flush():
        dirty.fill_(1)
        clean.sum()

    return flush


def gpu_hold(us: float = 150.0):
    """A short device-side delay before a timed region (outside it), so that
    the host has enqueued the step before the GPU reaches the start event."""
    import torch

    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None:
        sleep(int(us * 2000))  # cycles at about 2 GHz


def time_steps(step: DecodeStep, steps: int, warmup: int, flush, graph: bool = False):
    """Per-step CUDA-event times (ms) of the whole step and of its attention call.

    With graph=True each step is one replay of the captured step graph (both
    returned lists are then the replay time).
    """
    import torch

    for _ in range(warmup):
        flush()
        step.run()
    torch.cuda.synchronize()
    if graph:
        step.capture()
        for _ in range(warmup):
            flush()
            step.graph.replay()
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for k in range(steps):
            flush()
            gpu_hold()
            ev[k][0].record()
            step.graph.replay()
            ev[k][1].record()
        torch.cuda.synchronize()
        t = [e[0].elapsed_time(e[1]) for e in ev]
        return t, t
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for k in range(steps):
        flush()
        gpu_hold()
        ev[k][0].record()
        if not step.fused:
            step.write()
        ev[k][1].record()
        step.attend()
        ev[k][2].record()
    torch.cuda.synchronize()
    total = [e[0].elapsed_time(e[2]) for e in ev]
    attend = [e[1].elapsed_time(e[2]) for e in ev]
    return total, attend


def time_e2e(step: DecodeStep, steps: int, warmup: int, flush):
    """The same step through the public API from pinned host memory: every step
    uploads its small inputs (q, new K/V rows, slots, block tables, lengths) with
    one copy from a pinned staging buffer, calls libpa on the device views, and
    copies the output back; both copies are inside the timed region."""
    import torch

    from paged_kv_decode_pa_gb300.staging import StepStaging

    pa = step.pa
    w = step.w
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
    tens = {n: pa.to_torch(getattr(w, n), "cpu") for n in names}
    stage = StepStaging({n: (tuple(t.shape), t.dtype) for n, t in tens.items()}, step.dev)
    for n, t in tens.items():
        stage.host[n].copy_(t)
    d = stage.dev
    view = step.rebind(d["q"], d["k_new"], d["v_new"], d["slot_mapping"], d["block_tables"], d["context_lens"])
    out_host = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    h2d = stage.upload_bytes
    d2h = out_host.numel() * out_host.element_size()

    def one():
        stage.upload()
        view.run()
        out_host.copy_(view.out, non_blocking=True)

    for _ in range(warmup):
        flush()
        one()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for k in range(steps):
        flush()
        ev[k][0].record()
        one()
        ev[k][1].record()
    torch.cuda.synchronize()
    return [e[0].elapsed_time(e[1]) for e in ev], h2d, d2h


def step_bytes(w, fused=True, kv="bf16"):
    s = w.spec
    eb = accounting.elem_bytes(s.dtype)
    fused_write = fused or s.num_queries > 1
    if kv == "int8":
        att = accounting.decode_bytes_q8(w.context_lens, s.q_heads, s.kv_heads, s.head_dim, s.num_queries,
                                         fused_write=fused_write)
        return att, 0
    att = accounting.decode_bytes(w.context_lens, s.q_heads, s.kv_heads, s.head_dim, eb, s.num_queries,
                                  fused_write=fused_write)
    write = 0 if fused_write else accounting.cache_write_bytes(len(w.slot_mapping), s.kv_heads, s.head_dim, eb)
    return att, write


def measure_graph_buckets(device, flush, steps: int = 20) -> dict:
    """The engine pattern of one CUDA graph per batch bucket ("From 183 ms to
    19 ms per decode step", section "4. CUDA graphs per batch bucket"): for
    each bucket a Qwen2-1.5B-shaped decode step (pa_cache_write of one token per
    sequence, then pa_decode) over fixed buffers, timed as direct launches and
    as a replay of its captured graph."""
    out = {}
    for batch in (1, 2, 4, 8, 16, 32, 64):
        w = inputs.make("c2", batch=batch, num_blocks=max(4096, batch * 40))
        st = DecodeStep(w, device, fused=False)
        direct, _ = time_steps(st, steps, 3, flush)
        replay, _ = time_steps(st, steps, 3, flush, graph=True)
        out[str(batch)] = {"direct_us": round(statistics.mean(direct) * 1e3, 2),
                           "graph_replay_us": round(statistics.mean(replay) * 1e3, 2),
                           "kv_mb": round(step_bytes(w, False)[0]["kv"] / 1e6, 2)}
        del st
    return out


def prefill_flops(context_lens, chunks, q_heads: int, head_dim: int = 128) -> int:
    """Tensor-core flops of a causal prefill: each query row's score and value
    products over its visible positions, 2 * head_dim each."""
    f = 0
    for L, n in zip(context_lens, chunks):
        vis = np.arange(int(L) - int(n), int(L)) + 1
        f += int(np.maximum(vis, 0).sum()) * q_heads * 4 * head_dim
    return f


def prefill_bytes(context_lens, chunks, q_heads: int, kv_heads: int, head_dim: int = 128) -> int:
    """Algorithmic HBM bytes of a paged prefill (bf16): every query row read and
    every output row written once, and each sequence's visible K and V read once."""
    rows = int(sum(chunks)) * q_heads * head_dim * 2
    kv = int(sum(context_lens)) * kv_heads * 2 * head_dim * 2
    return 2 * rows + kv


def measure_prefill(device, flush, steps: int = 10) -> dict:
    """Paged prefill (next row 2): the 64-request workload's prompts (64 x 256
    tokens, 16/8 heads, no prefix) and a long chunk (8 sequences, 2048 tokens
    after a 2048-token prefix, 12/2 heads). Each is reported against the roof
    its arithmetic intensity puts it under: the measured bf16 peak when its
    flops per algorithmic byte exceed the ridge point (peak flops over the
    measured HBM bandwidth), else the measured HBM bandwidth."""
    import torch

    import paged_kv_decode_pa_gb300 as pa

    out = {}
    peak = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak = float(json.load(f)["bf16_tflops"])
    except Exception:
        peak = 1900.0
    for name, lens, chunks, hq, hkv, nb in (("prefill_64x256", (256,) * 64, (256,) * 64, 16, 8, 1100),
                                              ("prefill_8x2048_after_2048", (4096,) * 8, (2048,) * 8, 12, 2, 2100)):
        w = inputs.custom(batch=len(lens), q_heads=hq, kv_heads=hkv, context_lens=lens, num_blocks=nb, seed=61,
                          num_queries=max(chunks))
        rw = inputs.ragged(w, list(chunks))
        kc, vc = pa.to_torch(w.k_cache, device), pa.to_torch(w.v_cache, device)
        q, qs = pa.to_torch(rw.q, device), pa.to_torch(rw.query_start, device)
        tb, ln = pa.to_torch(w.block_tables, device), pa.to_torch(w.context_lens, device)
        o = torch.empty_like(q)
        fl = prefill_flops(lens, chunks, hq)
        nbytes = prefill_bytes(lens, chunks, hq, hkv)
        hbm, _ = hbm_peak()
        tensor_bound = fl / nbytes > peak * 1e12 / (hbm * 1e9)
        for kernel, suffix in (("tc", ""), ("mma", "_mma")):
            ts = []
            for k in range(steps + 3):
                flush()
                gpu_hold()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                pa.pa_prefill(kc, vc, q, qs, tb, ln, w.max_context_len, w.scale, rw.max_queries, out=o,
                              kernel=kernel)
                e1.record()
                torch.cuda.synchronize()
                if k >= 3:
                    ts.append(e0.elapsed_time(e1))
            us = statistics.mean(ts) * 1e3
            rec = {"kernel": kernel, "us_per_call": round(us, 2), "gflop": round(fl / 1e9, 2),
                   "tflops": round(fl / (us * 1e-6) / 1e12, 1), "algorithmic_mb": round(nbytes / 1e6, 1),
                   "achieved_gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                   "frac_of_measured_bf16": round(fl / (us * 1e-6) / 1e12 / peak, 3),
                   "frac_of_measured_hbm": round(nbytes / (us * 1e-6) / 1e9 / hbm, 3)}
            rec["bound"] = "tensor" if tensor_bound else "hbm"
            out[name + suffix] = rec
    return out


def launches_per_step(w, step, split: int, kernel: str, kv: str) -> int:
    """libpa kernels one step launches: the append when it is not fused, the
    attention kernel, the log-sum-exp merge when a call has several splits
    (tensor-core paths), and, for an int8 pool whose (sequence, KV head) rows
    span several row groups, the quantised append ahead of a fused verify."""
    from paged_kv_decode_pa_gb300 import _lib

    s = w.spec
    max_ctx = w.max_context_len
    if split:
        size = split
    elif max_ctx > _lib.PA_LONG_CONTEXT_TOKENS:
        size = _lib.PA_DEFAULT_SPLIT_LONG_INT8 if kv == "int8" else _lib.PA_DEFAULT_SPLIT_LONG
    else:
        size = _lib.PA_DEFAULT_SPLIT_TOKENS_INT8 if kv == "int8" else _lib.PA_DEFAULT_SPLIT_TOKENS
    splits = max(1, -(-max_ctx // size))
    n = (0 if step.fused else 1) + 1
    tensor_core = kv == "int8" or (kernel in ("auto", "mma") and s.dtype == "bf16")
    if tensor_core and splits > 1:
        n += 1
    rows = s.num_queries * (s.q_heads // s.kv_heads)
    if kv == "int8" and step.fused and rows > 16:
        n += 1
    return n


def measure_extra(name, device, steps, flush, split, kernel, fused=True, graph=False, kv="bf16"):
    w = timed_workload(name)
    st = DecodeStep(w, device, split, kernel, fused, kv)
    total, attend = time_steps(st, steps, 3, flush, graph)
    att, _ = step_bytes(w, fused, kv)
    us = statistics.mean(attend) * 1e3
    peak, _ = hbm_peak()
    gbs = att["total"] / (us * 1e-6) / 1e9
    rec = {"workload": w.spec.description, "us_per_call": round(us, 2),
           "us_per_call_p10_p90": [round(np.percentile(attend, 10) * 1e3, 2),
                                   round(np.percentile(attend, 90) * 1e3, 2)],
           "kv_bytes": att["kv"], "algorithmic_bytes": att["total"],
           "kv_gbs": round(att["kv"] / (us * 1e-6) / 1e9, 1), "achieved_gbs": round(gbs, 1),
           "frac_of_measured_hbm": round(gbs / peak, 3), "frac_of_8tbs": round(gbs / 8000.0, 3),
           "us_per_call_median": round(statistics.median(attend) * 1e3, 2),
           "call": ("pa_verify (fused write)" if w.spec.num_queries > 1 else
                    "pa_verify, one query per sequence (fused append + decode)" if fused else "pa_decode"),
           "l2": "flushed (write + read) before each call", "kv": kv}
    # Warm variant: no flush between calls, so whatever of the working set
    # fits in L2 (129 MB) is read from there.
    _, warm = time_steps(st, steps, 3, lambda: None, graph)
    rec["warm_us_per_call"] = round(statistics.mean(warm) * 1e3, 2)
    rec["warm_achieved_gbs"] = round(att["total"] / (statistics.mean(warm) * 1e-3) / 1e9, 1)
    rec["layer_loop"] = time_layer_loop(st, att["total"], flush)
    rec["kernels"] = call_kernels(w, st, split, kv)
    del st
    return rec


def layer_count(kv_bytes: int, l2_bytes: int = 129 * 10**6) -> int:
    """Layers whose pools a layer loop rotates through: enough that between two
    calls on the same pool the others stream more K/V than L2 holds."""
    return min(16, max(2, 1 + -(-l2_bytes // max(1, kv_bytes))))


def time_layer_loop(step: DecodeStep, call_bytes: int, flush, reps: int = 3) -> dict:
    """The contract's way of timing: many calls back to back between one pair of
    CUDA events, as a decode step calls attention once per layer. Each layer has
    its own copy of the pool (same tables, lengths and contents, different
    memory), and the calls rotate through them, so no call finds its K/V in L2
    (the pools read in between exceed it). Per-call inputs (q, new rows, tables)
    are shared, as the layers of one step share them."""
    import copy

    import torch

    nl = layer_count(step_kv_bytes(step))
    layers = [step]
    for _ in range(nl - 1):
        st = copy.copy(step)
        st.kc, st.vc = step.kc.clone(), step.vc.clone()
        st.scales = {k: v.clone() for k, v in step.scales.items()}
        layers.append(st)
    calls = nl * max(2, -(-24 // nl))
    for st in layers:
        st.attend()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        flush()
        gpu_hold()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for i in range(calls):
            layers[i % nl].attend()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3 / calls)
    us = statistics.median(times)
    peak, _ = hbm_peak()
    gbs = call_bytes / (us * 1e-6) / 1e9
    del layers
    return {"layers": nl, "calls": calls, "us_per_call": round(us, 2), "achieved_gbs": round(gbs, 1),
            "frac_of_measured_hbm": round(gbs / peak, 3),
            "timing": "one event pair around all calls, median of 3; calls rotate over per-layer pool copies "
                      "so each call's K/V was last read nl-1 calls earlier (not in L2)"}


def step_kv_bytes(step: DecodeStep) -> int:
    return step_bytes(step.w, step.fused, step.kv)[0]["kv"]


def call_kernels(w, step, split: int, kv: str) -> list:
    """The libpa kernels one call launches, in order (see launches_per_step)."""
    names = []
    s = w.spec
    if not step.fused:
        names.append("cache_write_q8_kernel" if kv == "int8" else "cache_write_kernel")
    rows = s.num_queries * (s.q_heads // s.kv_heads)
    if kv == "int8" and step.fused and rows > 16:
        names.append("cache_write_q8_kernel")
    names.append("attn_q8_kernel" if kv == "int8" else
                 ("attn_simt_kernel" if (step.kernel == "simt" or s.dtype == "f32") else "attn_mma_kernel"))
    if launches_per_step(w, step, split, step.kernel, kv) > len(names):
        names.append("merge_kernel")
    return names


def run_native(args):
    import torch

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import paged_kv_decode_pa_gb300 as pa
    from paged_kv_decode_pa_gb300 import _lib

    _lib.load()  # fails loudly if the library is missing
    w = rank_workload(args.workload, rank)
    step = DecodeStep(w, device, args.split_tokens, args.kernel, fused=not args.unfused, kv=args.kv)
    flush = make_l2_flush(device)

    att, write = step_bytes(w, step.fused, args.kv)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        t0 = time.perf_counter()
        total, attend = time_steps(step, args.steps, args.warmup, flush, args.graph)
        wall = time.perf_counter() - t0
    torch.cuda.synchronize()
    barrier(world)
    ms_step = max_over_ranks(statistics.mean(total), world, device)
    ms_attend = max_over_ranks(statistics.mean(attend), world, device)
    status = pa.pa_workspace_status(step.ws)
    if status:
        raise RuntimeError(f"device status flags {status:#x} during the benchmark")

    e2e_ms, h2d, d2h = time_e2e(step, max(5, args.steps // 2), 3, flush)
    e2e_step = max_over_ranks(statistics.mean(e2e_ms), world, device)

    value = whole_job_gbs(att["kv"], world, ms_step)
    peak, peak_kind = hbm_peak()
    achieved = att["total"] / (ms_attend * 1e-3) / 1e9
    traffic_key = args.workload if args.kv == "bf16" else f"{args.workload}_{args.kv}"
    traffic = ncu_traffic(traffic_key)
    ncu_rec = ncu_record(traffic_key)
    kernels = call_kernels(w, step, args.split_tokens, args.kv)
    loop = time_layer_loop(step, att["total"], flush)

    extra = {}
    if not args.no_extra and rank == 0:
        for name in ("c2", "c3", "c5"):
            if name != args.workload:
                extra[name] = measure_extra(name, device, 20, flush, args.split_tokens, args.kernel,
                                            not args.unfused, args.graph)
        if args.buckets:
            extra["graph_buckets_c2"] = measure_graph_buckets(device, flush)
        extra.update(measure_prefill(device, flush))
        # The int8 pool (the next row of the scope): the same workloads with
        # dequantisation fused into the attention kernel.
        for name in ("c4", "c3", "c5"):
            extra[name + "_int8"] = measure_extra(name, device, 20, flush, args.split_tokens, "auto",
                                                  not args.unfused, args.graph, kv="int8")

    cpu = cpu_baseline(w, args.cpu_seconds, args.kv) if rank == 0 else None

    if rank == 0:
        s = w.spec
        line = {
            "metric": METRIC,
            "value": round(value, 1),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_step, 5),
            "us_per_call": round(ms_attend * 1e3, 2),
            "us_per_call_median": round(statistics.median(attend) * 1e3, 2),
            "us_per_call_p10_p90": [round(float(np.percentile(attend, 10)) * 1e3, 2),
                                    round(float(np.percentile(attend, 90)) * 1e3, 2)],
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": s.dtype if args.kv == "bf16" else "int8 pool, bf16 queries",
            "data": "synthetic (seeded N(0,1) bf16; no dataset or weights involved)",
            "config": {
                "workload": f"{args.workload}: {s.description}",
                "batch": s.batch, "q_heads": s.q_heads, "kv_heads": s.kv_heads, "head_dim": s.head_dim,
                "block_size": s.block_size, "num_blocks": s.num_blocks,
                "context_tokens": int(w.context_lens.sum()),
                "split_tokens": args.split_tokens or (
                    f"default: {_lib.PA_DEFAULT_SPLIT_TOKENS_INT8 if args.kv == 'int8' else _lib.PA_DEFAULT_SPLIT_TOKENS}"
                    f" up to {_lib.PA_LONG_CONTEXT_TOKENS} tokens, "
                    f"{_lib.PA_DEFAULT_SPLIT_LONG_INT8 if args.kv == 'int8' else _lib.PA_DEFAULT_SPLIT_LONG} "
                    f"beyond"),
                "kernel": args.kernel,
                "kv": args.kv,
                "launch": "CUDA graph replay of the step" if args.graph else "direct launches",
                "step": ("pa_cache_write (one new token per sequence) + pa_decode" if not step.fused
                         else "pa_verify with one query per sequence: fused append of the new token "
                              "+ decode, one launch" if s.num_queries == 1
                         else "pa_verify (fused write of the new tokens + causal attention)"),
                "l2": "flushed before every timed step (256 MiB write, then 256 MiB read so that the "
                      "write-backs finish; outside the timed region)",
                "parallelism": f"replicas x{world} (independent sequences per GPU)",
            },
            "roofline": {
                "bound": "hbm",
                "kernel": ("the timed call: " + " + ".join(kernels) + " (" +
                           ("pa_verify with one query per sequence: fused append + decode"
                            if step.fused and s.num_queries == 1 else
                            "pa_verify" if step.fused else "pa_cache_write + pa_decode") + ")"),
                "achieved": round(achieved, 1),
                "peak": peak,
                "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "peak_kind": f"{peak_kind} (bf16 copy, read+write)",
                "frac_of_8tbs_nominal": round(achieved / 8000.0, 4),
                "algorithmic_bytes_per_launch": att["total"],
                "traffic": traffic,
                # The attention kernel alone, from the committed ncu record of
                # this workload (one launch, cold cache, serialised): the call
                # above also pays the event pair, the launch and the merge.
                "attention_kernel_ncu_us": ncu_rec.get("ncu_duration_us") if ncu_rec else None,
                "attention_kernel_frac_ncu": (round(att["total"] / (ncu_rec["ncu_duration_us"] * 1e-6) / 1e9 / peak, 4)
                                              if ncu_rec else None),
            },
            "layer_loop": loop,
            "cpu_baseline": cpu,
            "e2e": {"value": round(whole_job_gbs(att["kv"], world, e2e_step), 1), "unit": "GB/s",
                    "ms_per_step": round(e2e_step, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "path": "one pinned host -> device copy of the step's inputs (StepStaging), the step's libpa call(s), "
                            "device -> host copy of the output"},
            "gpu_launches": launches_per_step(w, step, args.split_tokens, args.kernel, args.kv) * args.steps,
            "clocks": clocks.summary(),
            "wall_s_timed_loop": round(wall, 3),
            "per_config": extra,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# CPU baseline: the fp64 oracle, as it stands, on a bounded sample

def cpu_baseline(w, budget_s: float, kv_format: str = "bf16"):
    import oracle

    cores = os.cpu_count() or 1
    oracle.set_threads(cores)
    s = w.spec
    if kv_format == "int8":
        # The oracle's int8 attention: dequantise the pool (fp32), then the fp64 attention.
        pool = inputs.q8_pool(w)
        kc, vc = oracle.dequant_q8(pool.k_codes, pool.v_codes, pool.k_scale, pool.v_scale)
        q = oracle.bf16_bits_to_f64(w.q).astype(np.float32)
    else:
        kc, vc = w.k_cache, w.v_cache
        q = w.q
    done, elapsed = 0, 0.0
    chunk = max(1, min(s.batch, cores))
    used_threads = min(cores, chunk)
    while done < s.batch and elapsed < budget_s:
        b1 = min(s.batch, done + chunk)
        t0 = time.perf_counter()
        oracle.attend(kc, vc, q, w.block_tables, w.context_lens, w.scale, (done, b1))
        elapsed += time.perf_counter() - t0
        done = b1
    if kv_format == "int8":
        kv = accounting.q8_kv_read_bytes(w.context_lens[:done], s.kv_heads, s.head_dim)
    else:
        kv = accounting.kv_read_bytes(w.context_lens[:done], s.kv_heads, s.head_dim, accounting.elem_bytes(s.dtype))
    return {"value": round(kv / elapsed / 1e9, 3), "unit": "GB/s", "cores": used_threads,
            "kind": "oracle",
            "sample": f"{done} of {s.batch} sequences ({int(w.context_lens[:done].sum())} tokens), "
                      f"fp64 C oracle with OpenMP, {elapsed:.2f} s"}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return
    import oracle

    cores = os.cpu_count() or 1
    oracle.set_threads(cores)
    base = inputs.CONFIGS[args.workload]
    w = inputs.generate(base)
    s = w.spec
    # One step = the oracle on a bounded sample of the sequences (one per core).
    sample = max(1, min(s.batch, cores))
    per_step_budget = 120.0 / max(1, args.steps + args.warmup)
    times = []
    for k in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        n = 0
        while n < s.batch:
            b1 = min(s.batch, n + sample)
            oracle.attend(w.k_cache, w.v_cache, w.q, w.block_tables, w.context_lens, w.scale, (n, b1))
            n = b1
            if time.perf_counter() - t0 > per_step_budget:
                break
        dt = time.perf_counter() - t0
        if k >= args.warmup:
            times.append((dt, n))
    eb = accounting.elem_bytes(s.dtype)
    total_t = sum(t for t, _ in times)
    total_kv = sum(accounting.kv_read_bytes(w.context_lens[:n], s.kv_heads, s.head_dim, eb) for _, n in times)
    value = total_kv / total_t / 1e9
    ms = total_t / len(times) * 1e3
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": f"{args.workload}: {s.description}",
                   "step": "fp64 CPU oracle attention over a bounded sample of the sequences"},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": min(cores, sample),
                         "kind": "oracle", "sample": f"up to {per_step_budget:.1f} s of sequences per step"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_prefill_only(args):
    """One JSON line with the prefill measurements alone (profiling runs)."""
    import torch

    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    res = measure_prefill(device, make_l2_flush(device), steps=max(1, args.steps))
    print(json.dumps({"metric": "paged prefill throughput", "unit": "TFLOP/s", "steps": args.steps,
                      "dtype": "bf16", "data": "synthetic", "per_config": res}), flush=True)


def main():
    args = parse_args()
    if args.record_traffic:
        print(json.dumps(record_traffic(*args.record_traffic)))
    elif args.prefill:
        run_prefill_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
