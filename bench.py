#!/usr/bin/env python
"""Benchmark of the sparse MLA hot path on one GB300 (or N replicas).

A step is one sparse-MLA decode of the bf16 decode batch: 64 requests x 64 heads, top-k
2048 over contexts of 8K-32K tokens in a page_size-64 cache with shuffled pages (slot
resolution, gather, both contractions, online softmax, epilogue and the split merge, all in
the library's kernels). The headline is decode queries/s; gather GB/s and the roofline are
reported beside it, and the grouped prefill (8192 new tokens, 64 heads, groups of 2) is
measured after it as a second line item (union build + attention, TFLOP/s).

Timing: W untimed warm-up steps, then K steps each bracketed by CUDA events on the
launching stream, with a 256 MB buffer written before every step (outside the events) so
that L2 starts cold; barrier + synchronize on both sides; max over ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl svt|reference]
"""

from __future__ import annotations

import argparse
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

# dram__bytes_read.sum + dram__bytes_write.sum of one decode call (attention_kernel and
# streamk_merge_kernel), keyed by the hash of their sources it was measured on (stale -> null).
TRAFFIC_BY_SOURCE = {
    # full-size capture (profiles/decode_bf16_attention_ncu.md, ncu --cache-control none after
    # bench.py's own L2 flush): the cluster-merged attention kernel (no merge kernel on this plan)
    "ac42cc583c934f36": (158.648832 + 60.999424) * 1e6,
    # the same kernel after the prefill row-set compaction (decode path unchanged in effect)
    "6a36a901a86fcc23": (159.517184 + 58.950400) * 1e6,
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
    ap.add_argument("--decode-T", type=int, default=64, help="decode batch size (64 = the benchmark workload)")
    ap.add_argument("--prefill-T", type=int, default=8192)
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
            "config": {"workload": w.name, "T": w.T, "H": w.H, "top_k": w.K, "page_size": w.page_size},
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


def time_steps(step, steps, flush, stream):
    import torch

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s, e in evs:
        flush.zero_()
        s.record(stream)
        step()
        e.record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in evs]


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
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

    # ---- decode batch, resident in HBM
    w = W.decode_bf16_batch(args.decode_T)
    kv = S.KVCache(torch.from_numpy(w.kv).to(dev), w.num_pages, w.page_size, w.kv_dtype)
    q = torch.from_numpy(w.q_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    topk = torch.from_numpy(w.topk).to(dev)
    bt = torch.from_numpy(w.block_table).to(dev)
    seq = torch.from_numpy(w.seq_lens).to(dev)
    out = torch.empty((w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.T, w.H), dtype=torch.float32, device=dev)
    ws = S.Workspace(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    # one attention kernel per decode call, plus the split merge when any query's list is split
    # between CTAs (the workspace then holds partial results beyond the status header)
    ws_need = S.svt.lib().svt_sparse_mla_decode_workspace_size(w.T, w.H, w.K, 0)
    launches_per_step = 2 if ws_need > 256 else 1

    def step():
        S.sparse_mla_decode(q, kv, topk, w.scale, block_table=bt, seq_lens=seq, out=out, lse=lse, ws=ws)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert ws.read_status() == 0, "device status flagged an error during warm-up"
    barrier(world)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    times = time_steps(step, args.steps, flush, stream)
    barrier(world)
    ms = max_over_ranks(statistics.mean(times), world)
    ms_med = max_over_ranks(statistics.median(times), world)
    nb = decode_bytes(w)
    value = replica_throughput(w.T, ms, world)
    achieved = nb["algorithmic"] / (ms / 1000.0) / 1e9
    th = source_hash()

    # ---- end to end: host buffers in, results out, through the public API
    e2e = None
    if not args.no_e2e:
        q_h = torch.from_numpy(w.q_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
        topk_h = torch.from_numpy(w.topk).pin_memory()
        out_h = torch.empty((w.T, w.H, 512), dtype=torch.bfloat16).pin_memory()
        lse_h = torch.empty((w.T, w.H), dtype=torch.float32).pin_memory()
        q_d, topk_d = torch.empty_like(q), torch.empty_like(topk)

        def e2e_step():
            q_d.copy_(q_h, non_blocking=True)
            topk_d.copy_(topk_h, non_blocking=True)
            o, l = S.sparse_mla_decode(q_d, kv, topk_d, w.scale, block_table=bt, seq_lens=seq, out=out, lse=lse,
                                       ws=ws)
            out_h.copy_(o, non_blocking=True)
            lse_h.copy_(l, non_blocking=True)

        for _ in range(max(3, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        et = time_steps(e2e_step, args.steps, flush, stream)
        barrier(world)
        ems = max_over_ranks(statistics.mean(et), world)
        e2e = {"value": replica_throughput(w.T, ems, world), "unit": UNIT, "ms_per_step": ems,
               "h2d_bytes_per_step": q_h.numel() * 2 + topk_h.numel() * 4,
               "d2h_bytes_per_step": out_h.numel() * 2 + lse_h.numel() * 4}

    # ---- top-k selection line item (the indexer's last step, on the decode batch's contexts)
    topk_item = None
    if not args.no_topk:
        tw = W.topk_batch(args.decode_T)
        t_scores = torch.from_numpy(tw.scores).to(dev)
        t_lens = torch.from_numpy(tw.lens).to(dev)
        t_out = torch.empty((tw.T, tw.K), dtype=torch.int32, device=dev)

        def topk_step():
            S.topk_select(t_scores, tw.K, lens=t_lens, out=t_out)

        for _ in range(max(3, args.warmup)):
            topk_step()
        torch.cuda.synchronize()
        tt = time_steps(topk_step, max(3, args.steps // 2), flush, stream)
        t_ms = statistics.mean(tt)
        t_bytes = float(tw.lens.astype(np.int64).sum() * 4 + tw.T * tw.K * 4)  # scores read once, lists written
        topk_item = {"workload": tw.name, "ms": round(t_ms, 4), "queries_per_s": tw.T / (t_ms / 1e3),
                     "algorithmic_bytes": t_bytes, "gbs": t_bytes / (t_ms / 1e3) / 1e9,
                     "frac_of_hbm_peak": t_bytes / (t_ms / 1e3) / 1e9 / hbm_peak}

    # ---- grouped prefill line item (union + attention)
    prefill = None
    if not args.no_prefill:
        pw = W.grouped_prefill(args.prefill_T)
        pkv = S.KVCache(torch.from_numpy(pw.kv).to(dev), pw.num_pages, pw.page_size, pw.kv_dtype)
        pq = torch.from_numpy(pw.q_bits.view(np.int16)).to(dev).view(torch.bfloat16)
        ptopk = torch.from_numpy(pw.topk).to(dev)
        pbt = torch.from_numpy(pw.block_table).to(dev)
        pseq = torch.from_numpy(pw.seq_lens).to(dev)
        preq = torch.from_numpy(pw.req_of_token).to(dev)
        slots = torch.empty_like(ptopk)
        groups = (pw.T + pw.G - 1) // pw.G
        enc = torch.empty((groups, pw.G * pw.K), dtype=torch.int32, device=dev)
        lens = torch.empty((groups,), dtype=torch.int32, device=dev)
        pout = torch.empty((pw.T, pw.H, 512), dtype=torch.bfloat16, device=dev)
        plse = torch.empty((pw.T, pw.H), dtype=torch.float32, device=dev)

        def union_step():
            S.resolve_topk_slots(ptopk, block_table=pbt, seq_lens=pseq, req_of_token=preq, page_size=pw.page_size,
                                 num_pages=pw.num_pages, out=slots, ws=ws)
            S.build_group_union(slots, pw.G, pw.num_slots, enc=enc, lens=lens, ws=ws)

        def attn_step():
            S.sparse_mla_prefill_grouped(pq, pw.G, pkv, enc, lens, pw.K, pw.scale, out=pout, lse=plse, ws=ws)

        for _ in range(max(3, args.warmup)):
            union_step()
            attn_step()
        torch.cuda.synchronize()
        assert ws.read_status() == 0
        psteps = max(3, args.steps // 2)
        ut = time_steps(union_step, psteps, flush, stream)
        at = time_steps(attn_step, psteps, flush, stream)
        lens_h = lens.cpu().numpy().astype(np.int64)
        live = np.count_nonzero(pw.topk >= 0, axis=1)
        # Executed MMA flops: each 64-row half of a group walks the union entries live for one
        # of its members, in 64-entry half-tiles (64 KV rows x 64 query rows x (576 + 512) MACs
        # each, the last one padded). A 128-row tile over the whole union would execute
        # `union` flops instead; useful flops count each query's own live entries.
        kept = rowset_kept_counts(enc.cpu().numpy(), lens_h, pw.H)
        executed = float(2 * 64 * 64 * ((kept + 63) // 64).sum() * (576 + 512))
        union = float(2 * 128 * lens_h.sum() * (576 + 512))
        useful = float(2 * pw.H * live.sum() * (576 + 512))
        a_ms, u_ms = statistics.mean(at), statistics.mean(ut)
        prefill = {"workload": pw.name, "union_ms": round(u_ms, 4), "attention_ms": round(a_ms, 4),
                   "step_ms": round(u_ms + a_ms, 4),
                   "tflops_executed": executed / (a_ms / 1e3) / 1e12,
                   "tflops_union": union / (a_ms / 1e3) / 1e12,
                   "tflops_useful": useful / (a_ms / 1e3) / 1e12,
                   "tflops_step_useful": useful / ((a_ms + u_ms) / 1e3) / 1e12,
                   "union_lists": float(lens_h.mean() / live.mean()),
                   "frac_of_bf16_peak": executed / (a_ms / 1e3) / 1e12 / bf16_peak,
                   "peak_tflops": bf16_peak, "peak_source": peak_src}

    # one clock record over every timed region above (decode, end to end, top-k, prefill) and
    # the short warm-ups between them: a single region is too short for more than one NVML sample
    clk = clocks.stop()
    if clk is not None:
        clk["window"] = "decode, e2e, top-k and prefill timed regions and the warm-ups between them"

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(w)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_median": ms_med, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "T": w.T, "H": w.H, "top_k": w.K, "page_size": w.page_size,
                       "kv_dtype": "bf16", "contexts": "uniform 8192..32768", "l2": "256 MB flush before each step",
                       "parallelism": f"replicas x{world}"},
            "gather_gbs": nb["gathered"] / (ms / 1000.0) / 1e9,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": TRAFFIC_BY_SOURCE.get(th),
                         "kernel": ("tile_attention_kernel + streamk_merge_kernel (one decode call, timed together)"
                                    if launches_per_step == 2 else "tile_attention_kernel (one decode call)"),
                         "algorithmic_bytes": nb["algorithmic"], "peak_source": peak_src, "source_hash": th},
            "clocks": clk, "gpu_launches": launches_per_step * args.steps, "e2e": e2e, "cpu_baseline": cpu,
            "prefill": prefill,
            "topk": topk_item,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
