#!/usr/bin/env python
"""Benchmark of the sparse MLA hot path on one GB300 (or N replicas).

A step is one sparse-MLA decode of the bf16 decode batch: 64 requests x 64 heads, top-k
2048 over contexts of 8K-32K tokens in a page_size-64 cache with shuffled pages (slot
resolution, gather, both contractions, online softmax, epilogue and the split merge, all in
the library's kernels). The headline is decode queries/s with its HBM roofline; every other
workload is a line item of the same JSON line, timed the same way:
  decode_fp8    128 requests x 64 heads, e4m3 cache, contexts 4K-46K
  decode_mixed  128 requests x 16 heads, bf16, contexts 16K-46K
  prefill       8192 new tokens, 64 heads, groups of 2 (union build + attention)
  prefill_mixed 8192 new tokens on 24576 cached, 16 heads, groups of 8
  prefill_fp8   the 8192-token prefill over an e4m3 cache
  gather_probe  the bf16 batch's 131072 rows read with no arithmetic (the gather ceiling)
  topk          top-k selection of 64 indexer rows of 8K-32K scores
  tensor_probe  one half-tile's MMA group, 400 times on every SM (the contractions' ceiling)
Decode items report HBM GB/s on algorithmic and on gathered bytes against the measured copy
peak; prefill items report executed, union and useful TFLOP/s against the bf16 peak and
their executed rate against the tensor probe's.

Timing: W untimed warm-up steps, then K steps each bracketed by CUDA events on the
launching stream, with a 256 MB buffer written before every step (outside the events) so
that L2 starts cold; barrier + synchronize on both sides; max over ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl svt|reference] [--phase-trace]
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-MLA decode queries/s + gather HBM GB/s; grouped prefill TFLOP/s"
UNIT = "queries/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# dram__bytes_read.sum and dram__bytes_write.sum of one decode call of the bf16 batch (every
# kernel of the call), keyed by the hash of the sources it was measured on (stale -> null),
# with the flush the capture ran after.
TRAFFIC_BY_SOURCE = {
    # earlier sources, flushed by a 256 MB write alone: the writes were the flush buffer's
    # dirty lines evicted by the gather (the decode itself writes 4.2 MB of output)
    "ac42cc583c934f36": (158.648832e6, 60.999424e6, "256 MB write"),
    "6a36a901a86fcc23": (159.517184e6, 58.950400e6, "256 MB write"),
    # TMA Q^T, bulk-copy cluster merge, column-group softmax barriers
    "d700b230a6228da8": (159.347712e6, 60.956416e6, "256 MB write"),
    # the same with the resolvers' first-round length read and the softmax's per-segment bounds
    "4ff596103d408444": (159.387392e6, 60.962304e6, "256 MB write"),
    # the cluster merge storing its channels straight from registers (and the tensor probe's
    # entry point in the API source)
    "4293d95688b1c4ae": (159.183360e6, 60.931840e6, "256 MB write"),
    # one kernel per cache type and mode, waits out of line in the e4m3 and prefill kernels
    "895581153be257dc": (157.544448e6, 61.046272e6, "256 MB write"),
    # the prefill kernels' mode fixed at compile time (the decode kernels' code unchanged)
    "3b8854cb7d11f6cb": (157.325568e6, 61.010432e6, "256 MB write"),
    # the API source with the union-tile prefill's entry point (the decode kernels unchanged)
    "89f3154b7fd2c791": (157.413888e6, 60.970496e6, "256 MB write"),
    # the trace build's mid-launch prefill window and row-set switch stamps (the decode kernels'
    # code unchanged)
    "66995d98d7f56091": (157.3632e6, 59.189248e6, "256 MB write"),
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["svt", "reference"], default="svt")
    ap.add_argument("--no-prefill", action="store_true", help="skip the grouped-prefill line item")
    ap.add_argument("--no-topk", action="store_true", help="skip the top-k selection line item")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-items", action="store_true", help="only the headline decode (with e2e and CPU legs)")
    ap.add_argument("--decode-T", type=int, default=64, help="decode batch size (64 = the benchmark workload)")
    ap.add_argument("--prefill-T", type=int, default=8192)
    ap.add_argument("--phase-trace", action="store_true",
                    help="build the phase-trace library and print per-phase times of the attention kernel")
    ap.add_argument("--item", choices=["decode_fp8", "decode_mixed", "prefill", "prefill_mixed", "prefill_fp8",
                                       "prefill_union_tile", "prefill_mixed_union_tile", "tensor_probe"],
                    help="run that one line item alone and print it (for profiling one workload)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


class ClockSampler:
    """SM clock and clock-event (throttle) reasons, sampled every 0.2 ms while running.

    Reads through NVML (the driver's libnvidia-ml, read-only queries) so that even a timed
    region of a few milliseconds gets samples; falls back to nvidia-smi at 200 ms when NVML
    cannot be loaded."""

    # nvmlClocksEventReason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, cuda_index: int):
        self.cuda_index = cuda_index
        self.samples = []  # (sm_mhz, reasons bitmask)
        self.max_mhz = None
        self._stop = threading.Event()
        self.thread = None
        self.proc = None
        self.lines = []
        self.nvml = None
        self.handle = None

    def _nvml_open(self) -> bool:
        import ctypes
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return False
            h = ctypes.c_void_p()
            ok = False
            try:
                import torch
                bus = getattr(torch.cuda.get_device_properties(self.cuda_index), "pci_bus_id", None)
                if isinstance(bus, int):
                    bus = None
                if bus:
                    ok = nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
            except Exception:
                ok = False
            if not ok:
                vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
                idx = int(vis.split(",")[self.cuda_index]) if vis and vis.split(",")[0].isdigit() else self.cuda_index
                ok = nv.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(h)) == 0
            if not ok:
                return False
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.nvml, self.handle = nv, h
            return True
        except OSError:
            return False

    def _nvml_loop(self):
        import ctypes
        nv, h = self.nvml, self.handle
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and get_reasons(h, ctypes.byref(rs)) == 0:
                self.samples.append((float(clk.value), int(rs.value)))
            time.sleep(0.0002)

    def start(self):
        # the timed loop holds the GIL between its CUDA calls: a short switch interval lets the
        # sampling thread run every ~0.1 ms instead of once per 5 ms (longer than the region)
        self._switch = sys.getswitchinterval()
        sys.setswitchinterval(1e-4)
        if self._nvml_open():
            self.thread = threading.Thread(target=self._nvml_loop, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.cuda_index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read_smi, daemon=True)
        self.thread.start()

    def _read_smi(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        sys.setswitchinterval(getattr(self, "_switch", 0.005))
        if self.nvml is not None:
            self._stop.set()
            self.thread.join(timeout=2)
            if not self.samples:
                return None
            reasons = set()
            for _, r in self.samples:
                for bit, name in self.REASONS.items():
                    if r & bit:
                        reasons.add(name)
            return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                    "reasons": sorted(reasons), "samples": len(self.samples), "source": "nvml, 0.2 ms"}
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi, 200 ms"}


def dist_setup(args):
    """Rank layout from torchrun's environment; NCCL on GPUs, gloo where there is no CUDA."""
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if torch.cuda.is_available():
        torch.cuda.set_device(local if world > 1 else 0)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank: int, ms_max: float, world: int) -> float:
    """Whole-job units per second: every rank processes its own copy of the workload (weak
    scaling), and the job takes as long as its slowest rank."""
    return units_per_rank * world / (ms_max / 1000.0)


def source_hash() -> str:
    """Hash of the sources of the decode kernels the roofline line times and of their launch plan."""
    h = hashlib.sha256()
    for name in ("attention.cu", "merge.cu", "api.cu"):
        with open(os.path.join(ROOT, "sparse_mla_attention_top_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def decode_bytes(w) -> dict:
    live = int(np.count_nonzero(w.topk >= 0))
    gathered = live * w.row_bytes
    other = (w.T * w.H * 576 * 2 + w.T * w.H * 512 * 2 + w.T * w.H * 4   # q, out, lse
             + w.T * w.K * 4 + live * 4)                                   # top-k list, page-table reads
    flops = 2 * w.H * live * (576 + 512)
    return {"gathered": gathered, "algorithmic": gathered + other, "flops": flops, "live": live}


L2_NOTE = "256 MB buffer written before each step, outside the events"


def headline_config(w, world: int) -> dict:
    """The headline workload's config: the same dict in both arms."""
    return {"workload": w.name, "T": w.T, "H": w.H, "top_k": w.K, "page_size": w.page_size,
            "kv_dtype": "bf16" if w.kv_dtype == 0 else "e4m3", "contexts": "uniform 8192..32768",
            "l2": L2_NOTE, "parallelism": f"replicas x{world}"}


def cpu_baseline(w, budget_s: float = 15.0):
    """The oracle as it stands, on the host cores, over a bounded sample of the queries."""
    import oracle

    oracle.build()
    t0 = time.perf_counter()
    oracle.decode(w.q_bits, w.kv, w.kv_dtype, w.num_pages, w.page_size, w.topk, w.scale,
                  block_table=w.block_table, seq_lens=w.seq_lens, query_ids=[0])
    one = max(time.perf_counter() - t0, 1e-3)
    cores = oracle.num_threads()
    n = int(max(1, min(w.T, budget_s / one * cores)))
    ids = np.arange(n) % w.T
    t0 = time.perf_counter()
    oracle.decode(w.q_bits, w.kv, w.kv_dtype, w.num_pages, w.page_size, w.topk, w.scale,
                  block_table=w.block_table, seq_lens=w.seq_lens, query_ids=ids)
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} of the {w.T} queries of the bf16 decode batch, all {w.H} heads, fp64, OpenMP over queries",
            "seconds": round(dt, 3)}


def run_reference(args):
    from sparse_mla_attention_top_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return
    w = W.decode_bf16_batch(args.decode_T)
    for _ in range(args.warmup):
        cpu_baseline(w, budget_s=2.0)
    vals = [cpu_baseline(w, budget_s=8.0) for _ in range(args.steps)]
    value = statistics.median(v["value"] for v in vals)
    cb = dict(vals[0])
    cb["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * w.T / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": headline_config(w, args.gpus),
            "cpu_baseline": cb, "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def rowset_kept_counts(enc: np.ndarray, lens: np.ndarray, H: int) -> np.ndarray:
    """Per 64-row half of each group, the union entries live for one of its members (the
    attention kernel walks only those)."""
    w = enc.view(np.uint32)
    valid = (np.arange(w.shape[1])[None, :] < lens[:, None]) & (w != 0xFFFFFFFF)
    m = w >> 24
    out = []
    for h in range(2):
        lo, hi = h * 64 // H, (h * 64 + 63) // H
        bits = ((2 << hi) - 1) & ~((1 << lo) - 1)
        out.append(np.count_nonzero(valid & ((m & bits) != 0), axis=1))
    return np.stack(out, axis=1).astype(np.int64).ravel()


class Flusher:
    """Leaves L2 cold between timed steps by writing a 256 MB buffer (twice the L2), as the
    pages' benchmark does (vLLM PR #63104, bench_shardq_rank.py). The buffer's dirty lines
    are written back while the next step runs: that step's DRAM write counter includes them."""

    def __init__(self, dev):
        import torch

        self.wr = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.wr.zero_()


def time_steps(step, steps, flush, stream):
    import torch

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s, e in evs:
        flush()
        s.record(stream)
        step()
        e.record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in evs]


def dev_inputs(S, w, dev):
    import torch

    return dict(kv=S.KVCache(torch.from_numpy(w.kv).to(dev), w.num_pages, w.page_size, w.kv_dtype),
                q=torch.from_numpy(w.q_bits.view(np.int16)).to(dev).view(torch.bfloat16),
                topk=torch.from_numpy(w.topk).to(dev), bt=torch.from_numpy(w.block_table).to(dev),
                seq=torch.from_numpy(w.seq_lens).to(dev), req=torch.from_numpy(w.req_of_token).to(dev))


def bench_decode(S, w, dev, stream, flush, steps, warmup, hbm_peak, ws=None):
    """One decode workload resident in HBM: per-call time and its HBM roofline."""
    import torch

    d = dev_inputs(S, w, dev)
    out = torch.empty((w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)
    ws = S.Workspace(dev) if ws is None else ws

    def step():
        S.sparse_mla_decode(d["q"], d["kv"], d["topk"], w.scale, block_table=d["bt"], seq_lens=d["seq"], out=out,
                            lse=lse, ws=ws)

    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize()
    assert ws.read_status() == 0, f"device status flagged an error during warm-up ({w.name})"
    times = time_steps(step, steps, flush, stream)
    assert ws.read_status() == 0, f"device status flagged an error ({w.name})"
    nb = decode_bytes(w)
    ms = statistics.mean(times)
    ws_need = S.svt.lib().svt_sparse_mla_decode_workspace_size(w.T, w.H, w.K, 0)
    return {"workload": w.name, "ms": ms, "ms_median": statistics.median(times), "queries_per_s": w.T / (ms / 1e3),
            "algorithmic_bytes": nb["algorithmic"], "gathered_bytes": nb["gathered"],
            "gbs_algorithmic": nb["algorithmic"] / (ms / 1e3) / 1e9, "gbs_gathered": nb["gathered"] / (ms / 1e3) / 1e9,
            "frac_of_hbm_peak": nb["algorithmic"] / (ms / 1e3) / 1e9 / hbm_peak,
            "frac_of_hbm_peak_gathered": nb["gathered"] / (ms / 1e3) / 1e9 / hbm_peak,
            "tflops": nb["flops"] / (ms / 1e3) / 1e12,
            "launches_per_call": 2 if ws_need > 256 else 1, "_times": times, "_d": d, "_out": out, "_lse": lse}


def bench_prefill(S, pw, dev, stream, flush, steps, warmup, bf16_peak, union_tile=False):
    """One grouped-prefill workload: slot resolution + union build, then attention, timed apart
    (union_tile: the two-CTA union-tile kernel instead of the row-set kernel)."""
    import torch

    d = dev_inputs(S, pw, dev)
    ws = S.Workspace(dev)
    slots = torch.empty_like(d["topk"])
    groups = (pw.T + pw.G - 1) // pw.G
    enc = torch.empty((groups, pw.G * pw.K), dtype=torch.int32, device=dev)
    lens = torch.empty((groups,), dtype=torch.int32, device=dev)
    pout = torch.empty((pw.T, pw.H, 512), dtype=torch.bfloat16, device=dev)
    plse = torch.empty((pw.T, pw.H), dtype=torch.float32, device=dev)

    def union_step():
        S.resolve_topk_slots(d["topk"], block_table=d["bt"], seq_lens=d["seq"], req_of_token=d["req"],
                             page_size=pw.page_size, num_pages=pw.num_pages, out=slots, ws=ws)
        S.build_group_union(slots, pw.G, pw.num_slots, enc=enc, lens=lens, ws=ws)

    def attn_step():
        S.sparse_mla_prefill_grouped(d["q"], pw.G, d["kv"], enc, lens, pw.K, pw.scale, out=pout, lse=plse, ws=ws,
                                     union_tile=union_tile)

    for _ in range(max(3, warmup)):
        union_step()
        attn_step()
    torch.cuda.synchronize()
    assert ws.read_status() == 0, f"device status flagged an error ({pw.name})"
    ut = time_steps(union_step, steps, flush, stream)
    at = time_steps(attn_step, steps, flush, stream)
    assert ws.read_status() == 0, f"device status flagged an error ({pw.name})"
    lens_h = lens.cpu().numpy().astype(np.int64)
    live = np.count_nonzero(pw.topk >= 0, axis=1)
    # Executed MMA flops: each 64-row half of a group walks the union entries live for one of
    # its members, in 64-entry half-tiles (64 KV rows x 64 query rows x (576 + 512) MACs
    # each, the last one padded). A 128-row tile over the whole union would execute `union`
    # flops instead; useful flops count each query's own live entries.
    kept = rowset_kept_counts(enc.cpu().numpy(), lens_h, pw.H)
    if union_tile:
        # every group's 128 rows over its whole union, in 64-entry tiles (the last one padded)
        executed = float(2 * 128 * 64 * ((lens_h + 63) // 64).sum() * (576 + 512))
    else:
        executed = float(2 * 64 * 64 * ((kept + 63) // 64).sum() * (576 + 512))
    union = float(2 * 128 * lens_h.sum() * (576 + 512))
    useful = float(2 * pw.H * live.sum() * (576 + 512))
    a_ms, u_ms = statistics.mean(at), statistics.mean(ut)
    return {"workload": pw.name, "kv_dtype": "bf16" if pw.kv_dtype == 0 else "e4m3",
            "kernel": "union tile (pair_prefill_kernel)" if union_tile else "row-sets (tile_attention_kernel)",
            "union_ms": round(u_ms, 4), "attention_ms": round(a_ms, 4), "step_ms": round(u_ms + a_ms, 4),
            "tflops_executed": executed / (a_ms / 1e3) / 1e12,
            "tflops_union": union / (a_ms / 1e3) / 1e12,
            "tflops_useful": useful / (a_ms / 1e3) / 1e12,
            "tflops_step_useful": useful / ((a_ms + u_ms) / 1e3) / 1e12,
            "union_lists": float(lens_h.mean() / live.mean()),
            "frac_of_bf16_peak": executed / (a_ms / 1e3) / 1e12 / bf16_peak,
            "frac_of_bf16_peak_useful": useful / (a_ms / 1e3) / 1e12 / bf16_peak,
            "peak_tflops": bf16_peak}


def bench_probe(S, w, d, dev, stream, flush, steps, hbm_peak):
    """The decode batch's rows read with no arithmetic, three ways, in the list's order and
    sorted by slot: the gather's own ceiling next to the decode."""
    import torch

    ws = S.Workspace(dev)
    slots = S.resolve_topk_slots(d["topk"], block_table=d["bt"], seq_lens=d["seq"], page_size=w.page_size,
                                 num_pages=w.num_pages, ws=ws).view(-1)
    slots = slots[slots >= 0].contiguous()
    sorted_slots = torch.sort(slots).values.contiguous()
    n = slots.numel()
    out = torch.empty((n,), dtype=torch.int32, device=dev)
    gathered = n * w.row_bytes
    res = {"rows": n, "row_bytes": w.row_bytes, "gathered_bytes": gathered}
    names = {0: "cp_async_16B", 1: "bulk_row", 2: "ld_16B_regs"}
    for order, sl in (("list_order", slots), ("sorted", sorted_slots)):
        for mode in (0, 1, 2):
            def step(sl=sl, mode=mode):
                S.gather_probe(d["kv"], sl, mode, out=out, ws=ws)

            for _ in range(3):
                step()
            torch.cuda.synchronize()
            t = time_steps(step, steps, flush, stream)
            ms = statistics.median(t)
            res[f"{names[mode]}_{order}"] = {"ms": ms, "gbs": gathered / (ms / 1e3) / 1e9,
                                             "frac_of_hbm_peak": gathered / (ms / 1e3) / 1e9 / hbm_peak}
    assert ws.read_status() == 0
    return res


# one 64-row half-tile's contractions: S^T (64 x 64 x 576) and PV (512 x 64 x 64), 2 flops per MAC
HALF_TILE_FLOP = 2 * 64 * 64 * (576 + 512)


def bench_tensor_probe(S, dev, stream, flush, steps, bf16_peak, reps=400):
    """One half-tile's MMA group of the attention kernels, `reps` times on one CTA per SM,
    with nothing else running: the contractions' own cost, the ceiling the grouped prefill's
    half-tiles run against."""
    import torch

    rng = np.random.default_rng(12)
    mk = lambda shape: torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16).to(dev)  # noqa: E731
    k_rows, q = mk((64, 576)), mk((64, 576))
    pt = torch.from_numpy(rng.random((64, 64)).astype(np.float32)).to(torch.bfloat16).to(dev)
    grid = torch.cuda.get_device_properties(dev).multi_processor_count
    ws = S.Workspace(dev)
    box = {}

    def step():
        box["r"] = S.tensor_probe(k_rows, q, pt, reps=reps, grid=grid, ws=ws)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    t = time_steps(step, steps, flush, stream)
    assert ws.read_status() == 0
    ms = statistics.median(t)
    cycles = box["r"][2].cpu().numpy()
    us_half = ms * 1e3 / reps
    tflops = grid * HALF_TILE_FLOP * reps / (ms / 1e3) / 1e12
    return {"grid": grid, "reps": reps, "ms": ms, "us_per_half_tile": us_half,
            "cycles_per_half_tile_median": float(np.median(cycles)) / reps,
            "mflop_per_half_tile": HALF_TILE_FLOP / 1e6, "tflops": tflops, "frac_of_bf16_peak": tflops / bf16_peak}


def bench_topk(S, W, dev, stream, flush, steps, warmup, hbm_peak, T):
    import torch

    tw = W.topk_batch(T)
    t_scores = torch.from_numpy(tw.scores).to(dev)
    t_lens = torch.from_numpy(tw.lens).to(dev)
    t_out = torch.empty((tw.T, tw.K), dtype=torch.int32, device=dev)

    def topk_step():
        S.topk_select(t_scores, tw.K, lens=t_lens, out=t_out)

    for _ in range(max(3, warmup)):
        topk_step()
    torch.cuda.synchronize()
    tt = time_steps(topk_step, steps, flush, stream)
    t_ms = statistics.mean(tt)
    t_bytes = float(tw.lens.astype(np.int64).sum() * 4 + tw.T * tw.K * 4)  # scores read once, lists written
    return {"workload": tw.name, "ms": round(t_ms, 4), "queries_per_s": tw.T / (t_ms / 1e3),
            "algorithmic_bytes": t_bytes, "gbs": t_bytes / (t_ms / 1e3) / 1e9,
            "frac_of_hbm_peak": t_bytes / (t_ms / 1e3) / 1e9 / hbm_peak}


def public(item: dict) -> dict:
    return {k: v for k, v in item.items() if not k.startswith("_")}


# ------------------------------------------------------------------------------ phase trace

TRACE_HEAD, TRACE_G, TRACE_EV = 48, 48, 16
TRACE_PREFILL_FROM = 1000  # grouped-prefill launches stamp half-tiles 1000 .. 1047 (attention.cu)


def analyse_trace(tr: np.ndarray, window: bool = False) -> dict:
    """Per-phase times (µs) from the stamps of one traced launch ([CTAs, slots] uint64): see
    the slot map in attention.cu. Medians over CTAs (and over half-tiles where per half-tile).
    window: the stamps are of half-tiles from the middle of the launch (grouped prefill), so
    the first half-tile's times are not reported."""
    tr = tr.astype(np.int64)
    ctas = tr[tr[:, 0] != 0]
    if len(ctas) == 0:
        return {"ctas": 0}
    gt0, c0, gt1, c9 = ctas[:, 0], ctas[:, 1], ctas[:, 15], ctas[:, 9]
    ghz = float(np.median((c9 - c0) / np.maximum(gt1 - gt0, 1)))
    us = lambda cyc: float(cyc) / ghz / 1e3  # noqa: E731
    n_half = ctas[:, 14]
    ev = ctas[:, TRACE_HEAD:].reshape(len(ctas), TRACE_G, TRACE_EV)
    out = {"ctas": int(len(ctas)), "sm_ghz": ghz, "half_tiles_per_cta_median": float(np.median(n_half)),
           "launch_span_us": float(gt1.max() - gt0.min()) / 1e3,
           "cta_start_spread_us": float(gt0.max() - gt0.min()) / 1e3,
           "cta_span_us_median": float(np.median(gt1 - gt0)) / 1e3}
    rel = lambda col: [us(x) for x in (col - c0)]  # noqa: E731
    out["setup_us"] = float(np.median(rel(ctas[:, 2])))
    out["first_q_issued_us"] = float(np.median(rel(ctas[:, 3])))
    first_slots = ctas[:, 4]
    ok = first_slots != 0
    if np.any(ok):
        out["first_slots_resolved_us"] = float(np.median([us(x) for x in (first_slots - c0)[ok]]))
    has0 = ev[:, 0, 1] != 0
    if np.any(has0) and not window:
        out["first_rows_landed_us"] = float(np.median([us(x) for x in (ev[has0, 0, 1] - c0[has0])]))
        out["first_s_issued_us"] = float(np.median([us(x) for x in (ev[has0, 0, 2] - c0[has0])]))
        out["first_p_written_us"] = float(np.median([us(x) for x in (ev[has0, 0, 4] - c0[has0])]))
    periods, fill_lat, s_lat, sm_lat, pv_gap, wait_rows, wait_buf = [], [], [], [], [], [], []
    sm_ld, sm_bar, sm_exp, sm_arrive = [], [], [], []
    for i in range(len(ctas)):
        n = int(np.count_nonzero(ev[i, :, 2])) if window else int(min(n_half[i], TRACE_G))
        if n < 4:
            continue
        e = ev[i, :n]
        periods.extend(np.diff(e[2:n - 1, 2]).tolist())
        for g in range(2, n - 1):
            fill_lat.append(e[g, 1] - e[g, 7])         # fill issued -> rows landed
            s_lat.append(e[g, 3] - e[g, 2])            # S^T issued -> softmax sees it done
            sm_lat.append(e[g, 4] - e[g, 3])           # softmax: S^T done -> P^T written
            pv_gap.append(e[g, 5] - e[g, 4])           # P^T written -> PV issued
            prev = max(e[g, 0], e[g - 1, 2])           # S issuer ready for g (buffer free, previous issued)
            wait_rows.append(max(0, e[g, 1] - prev))   # ... then waited for the rows
            wait_buf.append(max(0, e[g, 0] - e[g - 1, 2]))  # waited for the softmax to free the buffer
            sm_ld.append(e[g, 8] - e[g, 3])            # softmax: S^T read from TMEM
            sm_bar.append(e[g, 9] - e[g, 8])           # ... scaled, masked, maxima agreed (named barrier)
            sm_exp.append(e[g, 10] - e[g, 9])          # ... exponentials, P^T stored
            sm_arrive.append(e[g, 4] - e[g, 10])       # ... proxy fence and arrival
    med = lambda v: float(np.median([us(x) for x in v])) if v else None  # noqa: E731
    out.update({"half_tile_period_us": med(periods), "fill_issue_to_landed_us": med(fill_lat),
                "s_issue_to_done_us": med(s_lat), "softmax_us": med(sm_lat), "p_to_pv_issue_us": med(pv_gap),
                "s_issuer_wait_rows_us": med(wait_rows), "s_issuer_wait_buffer_us": med(wait_buf),
                "softmax_tmem_load_us": med(sm_ld), "softmax_scale_max_us": med(sm_bar),
                "softmax_exp_store_us": med(sm_exp), "softmax_fence_arrive_us": med(sm_arrive)})
    last_p = []
    for i in range(len(ctas) if not window else 0):
        n = int(min(n_half[i], TRACE_G))
        if n > 0 and n_half[i] <= TRACE_G:
            last_p.append(ctas[i, 7] - ev[i, n - 1, 4])
    out["last_p_to_roles_done_us"] = med(last_p)
    out["epilogue_us"] = med((ctas[:, 6] - ctas[:, 5])[ctas[:, 6] != 0].tolist())
    merged = ctas[:, 8] != 0
    out["cluster_merge_us"] = med((ctas[merged, 8] - ctas[merged, 7]).tolist()) if np.any(merged) else None
    if np.any(merged):
        # the merge's steps (slots 24-27, 16, 17, 21, 22, 18 in order): headers written, O^T in
        # registers, messages packed, past the cluster barrier, copies issued, messages landed,
        # weights, past their barrier, own channels combined and stored
        m = ctas[merged]
        steps = [("lse_headers", 7, 24), ("o_from_tmem", 24, 25), ("pack", 25, 26), ("cluster_barrier", 26, 27),
                 ("issue_copies", 27, 16), ("copies_land", 16, 17), ("weights", 17, 21), ("weights_barrier", 21, 22),
                 ("combine_and_store", 22, 18), ("final_barrier", 18, 8)]
        if all(np.all(m[:, b] != 0) for _, _, b in steps):
            out["cluster_merge_steps_us"] = {name: med((m[:, b] - m[:, a]).tolist()) for name, a, b in steps}
    out["roles_done_us"] = float(np.median(rel(ctas[:, 7])))
    out["end_us"] = float(np.median(rel(ctas[:, 9])))
    return out


def analyse_boundaries(tr: np.ndarray) -> dict:
    """What a row-set switch costs in the middle of a grouped-prefill launch: for each traced
    half-tile that opens a segment (stamp 12 = 1) with three more after it, the S^T issue
    times around it against the launch's steady half-tile period, and the steps the switch
    waits for (µs, medians over the switches of all CTAs)."""
    tr = tr.astype(np.int64)
    ctas = tr[tr[:, 0] != 0]
    if len(ctas) == 0:
        return {"switches": 0}
    gt0, c0, gt1, c9 = ctas[:, 0], ctas[:, 1], ctas[:, 15], ctas[:, 9]
    ghz = float(np.median((c9 - c0) / np.maximum(gt1 - gt0, 1)))
    us = lambda cyc: float(cyc) / ghz / 1e3  # noqa: E731
    ev = ctas[:, TRACE_HEAD:].reshape(len(ctas), TRACE_G, TRACE_EV)
    inner, cols = [], {k: [] for k in ("period_into", "period_1", "period_2", "period_3", "extra_over_4",
                                      "epilogue", "first_p_to_pv", "first_s_done_to_epilogue_done",
                                      "first_softmax", "s_issue_after_prev", "first_rows_wait",
                                      "prev_s_issued_to_q_issued", "q_issued_to_q_seen", "q_seen_to_s_issued",
                                      "prev_s_done_to_q_issued", "q_seen_to_buffer_free", "rows_to_fenced",
                                      "fenced_to_s_accepted", "prev_pv_issued_to_s_accepted",
                                      "prev_p_to_prev_pv_issued", "steady_fenced_to_s_accepted")}
    seg_len = []
    for i in range(len(ctas)):
        e = ev[i]
        n = int(np.count_nonzero(e[:, 2]))
        idx = e[:n, 12]
        for k in range(1, n):
            if idx[k] > 1 and idx[k - 1] >= 1:
                inner.append(e[k, 2] - e[k - 1, 2])
        for k in range(1, n - 3):
            if idx[k] != 1 or idx[k - 1] < 1 or not np.all(idx[k + 1:k + 4] > 1):
                continue
            seg_len.append(int(idx[k - 1]))
            cols["period_into"].append(e[k, 2] - e[k - 1, 2])
            cols["period_1"].append(e[k + 1, 2] - e[k, 2])
            cols["period_2"].append(e[k + 2, 2] - e[k + 1, 2])
            cols["period_3"].append(e[k + 3, 2] - e[k + 2, 2])
            cols["extra_over_4"].append(e[k + 3, 2] - e[k - 1, 2])
            cols["epilogue"].append(e[k, 13] - e[k - 1, 4])
            cols["first_p_to_pv"].append(e[k, 5] - e[k, 4])
            cols["first_s_done_to_epilogue_done"].append(e[k, 13] - e[k, 3])
            cols["first_softmax"].append(e[k, 4] - e[k, 13])
            cols["s_issue_after_prev"].append(e[k, 2] - e[k - 1, 2])
            cols["first_rows_wait"].append(max(0, e[k, 1] - e[k, 0]))
            cols["prev_s_issued_to_q_issued"].append(e[k, 14] - e[k - 1, 2])
            cols["q_issued_to_q_seen"].append(e[k, 15] - e[k, 14])
            cols["q_seen_to_s_issued"].append(e[k, 2] - e[k, 15])
            cols["prev_s_done_to_q_issued"].append(e[k, 14] - e[k - 1, 3])
            cols["q_seen_to_buffer_free"].append(e[k, 0] - e[k, 15])
            cols["rows_to_fenced"].append(e[k, 11] - e[k, 1])
            cols["fenced_to_s_accepted"].append(e[k, 2] - e[k, 11])
            cols["prev_pv_issued_to_s_accepted"].append(e[k, 2] - e[k - 1, 5])
            cols["prev_p_to_prev_pv_issued"].append(e[k - 1, 5] - e[k - 1, 4])
            cols["steady_fenced_to_s_accepted"].append(e[k + 2, 2] - e[k + 2, 11])
    if not inner or not cols["period_into"]:
        return {"switches": 0}
    steady = float(np.median(inner))
    out = {"switches": len(cols["period_into"]), "steady_period_us": us(steady),
           "half_tiles_per_cta_median": float(np.median(ctas[:, 14])),
           "segments_per_cta_median": float(np.median(ctas[:, 23])),
           "roles_done_per_half_tile_us": float(np.median([us(x) for x in (ctas[:, 7] - c0) / np.maximum(ctas[:, 14], 1)])),
           "previous_segment_half_tiles_median": float(np.median(seg_len))}
    for k, v in cols.items():
        if k == "extra_over_4":
            out["switch_extra_us"] = float(np.median([us(x - 4 * steady) for x in v]))
        else:
            out[k + "_us"] = float(np.median([us(x) for x in v]))
    return out


PAIR_TRACE_FROM = 1000  # the union-tile kernel stamps tiles 1000 .. 1047 of each CTA (pair_prefill.cu)


def analyse_pair_trace(tr: np.ndarray) -> dict:
    """Per-step times (µs) of the union-tile prefill kernel from one traced launch: tiles
    PAIR_TRACE_FROM .. + 47 of each CTA, the middle of a long launch (see the slot map in
    pair_prefill.cu). Medians over CTAs and tiles."""
    tr = tr.astype(np.int64)
    ctas = tr[tr[:, 1] != 0]
    if len(ctas) == 0:
        return {"ctas": 0}
    gt0, c0, gt1, c9 = ctas[:, 0], ctas[:, 1], ctas[:, 15], ctas[:, 9]
    ghz = float(np.median((c9 - c0) / np.maximum(gt1 - gt0, 1)))
    ev = ctas[:, TRACE_HEAD:].reshape(len(ctas), TRACE_G, TRACE_EV).astype(np.float64)

    def step(ea, eb, off=0):
        vals = []
        for k in range(2, TRACE_G - 4):
            a, b = ev[:, k, ea], ev[:, k + off, eb]
            ok = (a > 1) & (b > 1)
            vals.extend(((b - a)[ok] / ghz / 1e3).tolist())
        return float(np.median(vals)) if vals else None

    moved = ev[:, 2:TRACE_G - 4, 0]
    return {"ctas": int(len(ctas)), "sm_ghz": ghz, "tiles": f"{PAIR_TRACE_FROM}..{PAIR_TRACE_FROM + TRACE_G - 1}",
            "launch_span_us": float(gt1.max() - gt0.min()) / 1e3,
            "tile_period_us": step(2, 2, 1),
            "s_issuer_rows_landed_to_s_issued_us": step(1, 2),
            "s_issued_to_next_rows_landed_us": step(2, 1, 1),
            "softmax_sees_s_to_peer_partial_us": step(3, 4),
            "softmax_partial_to_masks_us": step(4, 5),
            "softmax_masks_to_maxima_agreed_us": step(5, 10),
            "softmax_agreed_to_p_buffer_free_us": step(10, 11),
            "softmax_p_rows_stored_us": step(11, 6),
            "softmax_loop_us": step(3, 3, 1),
            "pv_own_p_to_peer_p_us": step(7, 8),
            "pv_peer_p_to_issued_us": step(8, 9),
            "pv_issued_to_rows_landed_4_tiles_on_us": step(9, 1, 4),
            "tiles_moving_maxima": float((moved == 1).mean())}


def run_phase_trace(args):
    """Builds the phase-trace library, runs the bf16 decode batch, the e4m3 batch and the
    grouped prefill once each (after warm-up and an L2 flush) and prints per-phase times."""
    import torch

    from sparse_mla_attention_top_gb300 import build as B
    from sparse_mla_attention_top_gb300 import svt
    from sparse_mla_attention_top_gb300 import workloads as W

    svt.use_library(B.build(trace=True))
    import sparse_mla_attention_top_gb300 as S

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    flush = Flusher(dev)
    L = S.svt.lib()
    L.svt_trace_attach.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    slots_per_cta = L.svt_trace_slots()
    assert slots_per_cta == TRACE_HEAD + TRACE_G * TRACE_EV
    buf = torch.zeros((1024, slots_per_cta), dtype=torch.int64, device=dev)
    res = {"trace": "phase stamps of one launch (clock64 per SM; medians over CTAs)"}

    def traced(step, label, window=False):
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        buf.zero_()
        L.svt_trace_attach(ctypes.c_void_p(buf.data_ptr()), buf.numel() * 8)
        flush()
        step()
        torch.cuda.synchronize()
        L.svt_trace_attach(None, 0)
        res[label] = analyse_trace(buf.cpu().numpy(), window=window)
        if window:
            res[label + "_row_set_switch"] = analyse_boundaries(buf.cpu().numpy())

    for name, w in (("decode_bf16", W.decode_bf16_batch(args.decode_T)), ("decode_fp8", W.decode_fp8_batch())):
        d = dev_inputs(S, w, dev)
        ws = S.Workspace(dev)
        traced(lambda: S.sparse_mla_decode(d["q"], d["kv"], d["topk"], w.scale, block_table=d["bt"],
                                           seq_lens=d["seq"], ws=ws), name)
        del d
    pw = W.grouped_prefill(args.prefill_T)
    d = dev_inputs(S, pw, dev)
    ws = S.Workspace(dev)
    slots = S.resolve_topk_slots(d["topk"], block_table=d["bt"], seq_lens=d["seq"], req_of_token=d["req"],
                                 page_size=pw.page_size, num_pages=pw.num_pages, ws=ws)
    enc, lens = S.build_group_union(slots, pw.G, pw.num_slots, ws=ws)
    traced(lambda: S.sparse_mla_prefill_grouped(d["q"], pw.G, d["kv"], enc, lens, pw.K, pw.scale, ws=ws),
           "prefill_bf16", window=True)
    # the union-tile kernel: its own slot map, mid-launch tiles
    for _ in range(3):
        S.sparse_mla_prefill_grouped(d["q"], pw.G, d["kv"], enc, lens, pw.K, pw.scale, ws=ws, union_tile=True)
    torch.cuda.synchronize()
    buf.zero_()
    L.svt_trace_attach(ctypes.c_void_p(buf.data_ptr()), buf.numel() * 8)
    flush()
    S.sparse_mla_prefill_grouped(d["q"], pw.G, d["kv"], enc, lens, pw.K, pw.scale, ws=ws, union_tile=True)
    torch.cuda.synchronize()
    L.svt_trace_attach(None, 0)
    res["prefill_bf16_union_tile"] = analyse_pair_trace(buf.cpu().numpy())
    print(json.dumps(res), flush=True)


def run_item(args):
    """One line item alone (same timing as in the full run), printed as {item: {...}}."""
    import torch

    import sparse_mla_attention_top_gb300 as S
    from sparse_mla_attention_top_gb300 import build as B
    from sparse_mla_attention_top_gb300 import workloads as W

    B.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    hbm_peak, bf16_peak, _, _ = peaks()
    flush = Flusher(dev)
    if args.item.startswith("decode"):
        w = W.decode_fp8_batch() if args.item == "decode_fp8" else W.mixed_decode()
        item = public(bench_decode(S, w, dev, stream, flush, args.steps, args.warmup, hbm_peak))
    elif args.item == "tensor_probe":
        item = bench_tensor_probe(S, dev, stream, flush, args.steps, bf16_peak)
    else:
        pw = {"prefill": W.grouped_prefill, "prefill_mixed": W.mixed_prefill, "prefill_fp8": W.grouped_prefill_fp8,
              "prefill_union_tile": W.grouped_prefill, "prefill_mixed_union_tile": W.mixed_prefill}[args.item](
                  args.prefill_T)
        item = bench_prefill(S, pw, dev, stream, flush, args.steps, args.warmup, bf16_peak,
                             union_tile=args.item.endswith("union_tile"))
    print(json.dumps({args.item: item}), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    if args.phase_trace:
        run_phase_trace(args)
        return
    if args.item:
        run_item(args)
        return
    import torch

    import sparse_mla_attention_top_gb300 as S
    from sparse_mla_attention_top_gb300 import build as B
    from sparse_mla_attention_top_gb300 import workloads as W

    world, rank, local = dist_setup(args)
    if rank == 0:
        B.build()
    barrier(world)
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    hbm_peak, bf16_peak, bf16_sust, peak_src = peaks()
    flush = Flusher(dev)

    # ---- headline: the bf16 decode batch, resident in HBM
    w = W.decode_bf16_batch(args.decode_T)
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    head = bench_decode(S, w, dev, stream, flush, args.steps, args.warmup, hbm_peak)
    barrier(world)
    times = head["_times"]
    ms = max_over_ranks(statistics.mean(times), world)
    ms_med = max_over_ranks(statistics.median(times), world)
    nb = decode_bytes(w)
    value = replica_throughput(w.T, ms, world)
    achieved = nb["algorithmic"] / (ms / 1000.0) / 1e9
    th = source_hash()
    d = head["_d"]

    # ---- end to end: host buffers in, results out, through the public API. The step's inputs
    # (q and the top-k lists) sit back to back in one pinned host buffer and go over in one
    # copy; the results (out and lse) sit back to back in one device buffer and come back in
    # one copy.
    e2e = None
    if not args.no_e2e:
        ws = S.Workspace(dev)
        q_bytes, tk_bytes = w.T * w.H * 576 * 2, w.T * w.K * 4
        out_bytes, lse_bytes = w.T * w.H * 512 * 2, w.T * w.H * 4
        in_h = torch.empty(q_bytes + tk_bytes, dtype=torch.uint8).pin_memory()
        in_h[:q_bytes].copy_(torch.from_numpy(w.q_bits.view(np.uint8).reshape(-1)))
        in_h[q_bytes:].copy_(torch.from_numpy(w.topk.view(np.uint8).reshape(-1)))
        in_d = torch.empty_like(in_h, device=dev)
        res_d = torch.empty(out_bytes + lse_bytes, dtype=torch.uint8, device=dev)
        res_h = torch.empty_like(res_d, device="cpu").pin_memory()
        q_d = in_d[:q_bytes].view(torch.bfloat16).view(w.T, w.H, 576)
        topk_d = in_d[q_bytes:].view(torch.int32).view(w.T, w.K)
        out = res_d[:out_bytes].view(torch.bfloat16).view(w.T, w.H, 512)
        lse = res_d[out_bytes:].view(torch.float32).view(w.T, w.H)

        def e2e_step():
            in_d.copy_(in_h, non_blocking=True)
            S.sparse_mla_decode(q_d, d["kv"], topk_d, w.scale, block_table=d["bt"], seq_lens=d["seq"], out=out,
                                lse=lse, ws=ws)
            res_h.copy_(res_d, non_blocking=True)

        for _ in range(max(3, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        ref_out, ref_lse = head["_out"], head["_lse"]
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), "end-to-end results differ"
        barrier(world)
        et = time_steps(e2e_step, args.steps, flush, stream)
        barrier(world)
        ems = max_over_ranks(statistics.mean(et), world)
        e2e = {"value": replica_throughput(w.T, ems, world), "unit": UNIT, "ms_per_step": ems,
               "h2d_bytes_per_step": q_bytes + tk_bytes, "d2h_bytes_per_step": out_bytes + lse_bytes}

    # ---- the other workloads, each a line item timed the same way
    items = {}
    psteps = max(3, args.steps // 2)
    if not args.no_items:
        items["gather_probe"] = bench_probe(S, w, d, dev, stream, flush, psteps, hbm_peak)
    del d, head["_d"]
    if not args.no_items:
        for key, fn in (("decode_fp8", W.decode_fp8_batch), ("decode_mixed", W.mixed_decode)):
            it = bench_decode(S, fn(), dev, stream, flush, args.steps, args.warmup, hbm_peak)
            items[key] = public(it)
            del it
    if not args.no_topk:
        items["topk"] = bench_topk(S, W, dev, stream, flush, psteps, args.warmup, hbm_peak, args.decode_T)
    if not args.no_prefill:
        tp = bench_tensor_probe(S, dev, stream, flush, psteps, bf16_peak)
        items["tensor_probe"] = tp
        items["prefill"] = bench_prefill(S, W.grouped_prefill(args.prefill_T), dev, stream, flush, psteps,
                                         args.warmup, bf16_peak)
        if not args.no_items:
            items["prefill_union_tile"] = bench_prefill(S, W.grouped_prefill(args.prefill_T), dev, stream, flush,
                                                        psteps, args.warmup, bf16_peak, union_tile=True)
            items["prefill_mixed"] = bench_prefill(S, W.mixed_prefill(args.prefill_T), dev, stream, flush, psteps,
                                                   args.warmup, bf16_peak)
            items["prefill_fp8"] = bench_prefill(S, W.grouped_prefill_fp8(args.prefill_T), dev, stream, flush,
                                                 psteps, args.warmup, bf16_peak)
        # the prefill's executed rate against the same half-tiles' MMAs with nothing else running
        for key in ("prefill", "prefill_mixed", "prefill_fp8"):  # the row-set kernel's half-tiles
            if key in items:
                items[key]["frac_of_tensor_probe"] = items[key]["tflops_executed"] / tp["tflops"]

    # one clock record over every timed region above and the short warm-ups between them: a
    # single region is too short for more than one NVML sample
    clk = clocks.stop()
    if clk is not None:
        clk["window"] = "every timed region of this run and the warm-ups between them"

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(w)

    if rank == 0:
        tr = TRAFFIC_BY_SOURCE.get(th)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_median": ms_med, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": headline_config(w, world),
            "gather_gbs": nb["gathered"] / (ms / 1000.0) / 1e9,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak,
                         "frac_gathered": nb["gathered"] / (ms / 1000.0) / 1e9 / hbm_peak,
                         "traffic": (tr[0] + tr[1]) if tr else None,
                         "traffic_read": tr[0] if tr else None, "traffic_write": tr[1] if tr else None,
                         "traffic_flush": tr[2] if tr else None,
                         "kernel": ("tile_attention_kernel + streamk_merge_kernel (one decode call, timed together)"
                                    if head["launches_per_call"] == 2 else "tile_attention_kernel (one decode call)"),
                         "algorithmic_bytes": nb["algorithmic"], "gathered_bytes": nb["gathered"],
                         "peak_source": peak_src, "source_hash": th},
            "clocks": clk, "gpu_launches": head["launches_per_call"] * args.steps, "e2e": e2e, "cpu_baseline": cpu,
        }
        line.update(items)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
