#!/usr/bin/env python
"""Benchmark of the GB300 Invariant Bit Packing codec.

Headline: decompress-gather throughput in GB/s of uncompressed output rows on the
dense GNN-feature workload (2,000,000 x 128 FP32, column c ~ N(mu_c, sigma_c),
rows L2-normalised; T = 0.9, B = 32), one step = one gather of 100,000
Zipf(1.0) row indices from slots held in page-locked host memory and read
zero-copy by the kernel. The same run also reports, each with its roofline:
  * the HBM-resident gather of the same store (slots in device memory);
  * metadata build and compression throughput (the preprocessing stages);
  * space saving of the store (bitmask + row sizes from ibp_query);
  * the end-to-end figure through the C ABI with host buffers (index upload,
    gather, download of the gathered rows inside the timed region);
  * the oracle (plain single-threaded C++) timed on the host cores on a bounded
    sample, as a CPU baseline.

python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload W]
Under torchrun (N > 1) every rank runs an independent replica of the workload
(no collective on the data path); rank 0 prints one JSON line with the
whole-job throughput over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import ibp_inputs as gen  # noqa: E402
import lossless_bit_level_gb300 as ibp  # noqa: E402

METRIC = "IBP decompress-gather GB/s (uncompressed out) & space saving %, vs roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20

WORKLOADS = {
    # name: rows factory, dtype code, T, B, batch size, index sampler, residency, description
    "gnn_dense": dict(
        rows=lambda: gen.gnn_dense(), dtype=ibp.FP32, T=0.9, B=32, batch=100_000,
        index=lambda n, k, part: gen.zipf_indices(n, k, 1.0, part=part, workload=gen.GNN_DENSE),
        residency="host",
        desc="dense GNN features 2,000,000 x 128 FP32 (col N(mu_c,sigma_c), rows L2-normalised), "
             "T=0.9, B=32; gather 100,000 Zipf(1.0) indices per step from pinned host slots "
             "(zero-copy)"),
    "gnn_sparse": dict(
        rows=lambda: gen.gnn_sparse(), dtype=ibp.FP32, T=0.9, B=32, batch=100_000,
        index=lambda n, k, part: gen.uniform_indices(n, k, part=part, workload=gen.GNN_SPARSE),
        residency="host",
        desc="sparse GNN features 500,000 x 512 FP32 (1.0 w.p. 0.01), T=0.9, B=32; gather "
             "100,000 uniform indices per step from pinned host slots (zero-copy)"),
    "tiny": dict(
        rows=lambda: gen.tiny_fp32(), dtype=ibp.FP32, T=0.9, B=32, batch=1024,
        index=lambda n, k, part: gen.uniform_indices(n, k, part=part, workload=gen.TINY),
        residency="device",
        desc="tiny FP32 4096 x 128 N(0,0.05), T=0.9, B=32; gather 1024 uniform indices, HBM"),
    "dlrm_table": dict(
        rows=lambda: gen.dlrm_table(0), dtype=ibp.FP32, T=0.95, B=32, batch=65_536,
        index=lambda n, k, part: gen.zipf_indices(n, k, 1.05, part=part, workload=gen.DLRM),
        residency="host",
        desc="one DLRM embedding table 1,000,000 x 128 FP32 U(-1e-3,1e-3), T=0.95, B=32; "
             "gather 65,536 Zipf(1.05) lookups per step from pinned host slots (zero-copy)"),
    "llm_kv": dict(
        rows=lambda: gen.llm_kv(0, 0), dtype=ibp.BF16, T=0.9, B=64, batch=32_768,
        index=lambda n, k, part: np.arange(k, dtype=np.int64) % n,
        residency="host",
        desc="LLM K cache of one layer, 8 x 4096 tokens x (32 heads x 128) BF16 N(0,1) with 41 "
             "channels x10, T=0.9, B=64; every row streamed in order per step from pinned "
             "host slots (zero-copy)"),
    "llm_down": dict(
        rows=lambda: gen.llm_weight(0, "down"), dtype=ibp.BF16, T=0.9, B=64, batch=4096,
        index=lambda n, k, part: np.arange(k, dtype=np.int64) % n,
        residency="host",
        desc="LLM FFN down-projection weight 4096 x 11008 BF16 N(0,0.02), T=0.9, B=64; every "
             "row streamed in order per step from pinned host slots (zero-copy)"),
}


# the legs that follow the timed gather, in the order they run
LEGS = ("hbm", "e2e", "stages", "dedup", "select", "packed", "positions", "offload", "dlrm26",
        "configs")


# ----------------------------------------------------------------------------- utilities

def env_rank():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def measured_peaks():
    try:
        with open(PEAKS_FILE) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="ibp_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        smax = max(r[1] for r in rows)
        loaded = [r for r in rows if r[2] > 200.0] or rows
        reasons = set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for r in rows:
            for name, val in zip(names[1:], r[3][1:]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": smax,
                "samples": len(rows), "reasons": sorted(reasons)}


def clocks_rejected(clk) -> bool:
    if not clk:
        return False
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    if bad & set(clk["reasons"]):
        return True
    return clk["sm_mhz"] < 0.5 * clk["sm_max_mhz"] and "sw_power_cap" not in clk["reasons"]


def event_pair(stream):
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    return a, b


def recorded_traffic(key):
    """DRAM / host-link bytes per gather launch from the committed ncu summary
    (profiles/gather_traffic.json), or None when the gather kernel source changed
    since those counters were taken."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "gather_traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    h = hashlib.sha256()
    for p in ("ibp_gather.cu", "ibp_device.cuh"):
        with open(os.path.join(ROOT, "lossless_bit_level_gb300", "csrc", p), "rb") as f:
            h.update(f.read())
    if rec.get("kernel_source_sha256") != h.hexdigest():
        return None
    return rec.get("captures", {}).get(key)


def measure_link(dev, nbytes=1 << 30, reps=10):
    """Pinned host -> device copy bandwidth (cudaMemcpyAsync through torch), device ->
    pinned host, and the zero-copy read probe kernel over the same pinned buffer."""
    host = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    host.fill_(1)
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream()
    best_h2d = best_d2h = best_probe = 0.0
    sink = torch.zeros(2, dtype=torch.int32, device=dev)
    for _ in range(reps):
        a, b = event_pair(s)
        a.record(s)
        d.copy_(host, non_blocking=True)
        b.record(s)
        b.synchronize()
        best_h2d = max(best_h2d, nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
        a.record(s)
        host.copy_(d, non_blocking=True)
        b.record(s)
        b.synchronize()
        best_d2h = max(best_d2h, nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
        a.record(s)
        ibp.probe_read(host, sink)
        b.record(s)
        b.synchronize()
        best_probe = max(best_probe, nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    # both directions at once (two streams, half the buffer each way): the
    # denominator of the end-to-end leg, whose steps move rows both ways
    half = nbytes // 2
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    best_bidir = 0.0
    for _ in range(reps):
        a, b = event_pair(s)
        a.record(s)
        s1.wait_event(a)
        s2.wait_event(a)
        with torch.cuda.stream(s1):
            d[:half].copy_(host[:half], non_blocking=True)
        with torch.cuda.stream(s2):
            host[half:].copy_(d[half:], non_blocking=True)
        s.wait_stream(s1)
        s.wait_stream(s2)
        b.record(s)
        b.synchronize()
        best_bidir = max(best_bidir, nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    del host, d
    return {"h2d_memcpy_gbs": best_h2d, "d2h_memcpy_gbs": best_d2h,
            "bidirectional_memcpy_gbs": best_bidir,
            "zero_copy_read_gbs": best_probe, "bytes": nbytes, "reps": reps}


def host_placement(dev):
    """Where the page-locked buffers can live relative to the GPU, read from sysfs and
    the process status (read-only): the GPU's NUMA node, the nodes online, and the
    CPUs and memory nodes this process may use. With a single node every pinned
    buffer is local to the GPU."""
    out = {}
    bus = None
    try:
        q = subprocess.run(["nvidia-smi", f"--id={dev.index or 0}", "--query-gpu=pci.bus_id",
                            "--format=csv,noheader"], capture_output=True, text=True, timeout=20)
        bus = q.stdout.strip() or bus
    except (OSError, subprocess.SubprocessError):
        pass
    if bus:
        dom, rest = bus.split(":", 1)
        sysfs = f"/sys/bus/pci/devices/{dom[-4:].lower()}:{rest.lower()}/numa_node"
        try:
            out["gpu_numa_node"] = int(open(sysfs).read().strip())
        except (OSError, ValueError):
            out["gpu_numa_node"] = None
        out["gpu_pci"] = bus
    try:
        out["nodes_online"] = open("/sys/devices/system/node/online").read().strip()
    except OSError:
        out["nodes_online"] = None
    try:
        for line in open("/proc/self/status"):
            if line.startswith(("Cpus_allowed_list", "Mems_allowed_list")):
                k, v = line.split(":", 1)
                out[k.strip().lower()] = v.strip()
    except OSError:
        pass
    return out


def measure_hbm_copy(dev, nbytes=1 << 30, reps=10):
    a_t = torch.empty(nbytes // 2, dtype=torch.bfloat16, device=dev).fill_(1)
    b_t = torch.empty_like(a_t)
    s = torch.cuda.current_stream()
    best = 0.0
    for _ in range(reps):
        a, b = event_pair(s)
        a.record(s)
        b_t.copy_(a_t)
        b.record(s)
        b.synchronize()
        best = max(best, 2 * nbytes / (a.elapsed_time(b) * 1e-3) / 1e9)
    return best


def measure_launch_floor(dev, flush, reps=20):
    """CUDA-event time of a one-element kernel right after the L2 flush, the way a
    gather step is timed: the floor that any single-launch step pays (launch,
    dispatch and the two event records), in seconds (mean after 3 warm-ups)."""
    tiny = torch.zeros(1, dtype=torch.int32, device=dev)
    s = torch.cuda.current_stream()
    ts = []
    for k in range(reps + 3):
        flush()
        a, b = event_pair(s)
        a.record(s)
        tiny.add_(1)
        b.record(s)
        b.synchronize()
        if k >= 3:
            ts.append(a.elapsed_time(b) * 1e-3)
    return float(np.mean(ts))


def job_throughput(t_local: float, bytes_per_step_local: float, dist=None, device=None):
    """Whole-job throughput of independent replicas: every rank processed
    bytes_per_step_local per step; the job's step time is the slowest rank's, so the
    value is the sum of all ranks' bytes over that time. Returns (t_step, GB/s)."""
    world = 1
    total = bytes_per_step_local
    t = t_local
    if dist is not None and dist.is_initialized():
        world = dist.get_world_size()
        tt = torch.tensor([t_local, bytes_per_step_local], dtype=torch.float64, device=device)
        tmax = tt[:1].clone()
        dist.all_reduce(tmax, op=dist.ReduceOp.MAX)
        tsum = tt[1:].clone()
        dist.all_reduce(tsum, op=dist.ReduceOp.SUM)
        t, total = float(tmax.item()), float(tsum.item())
    return t, total / t / 1e9


# ----------------------------------------------------------------------------- the codec

class Store:
    def __init__(self, words_np, dtype, T, B, residency, dev):
        self.n, self.L = words_np.shape
        self.dtype, self.T, self.B, self.residency, self.dev = dtype, T, B, residency, dev
        self.raw_bytes = self.L * words_np.dtype.itemsize
        self.slot_bytes = ibp.slot_bytes(self.L, dtype)
        tdt = torch.int32 if words_np.dtype.itemsize == 4 else torch.int16
        npv = np.int32 if words_np.dtype.itemsize == 4 else np.int16
        src = torch.from_numpy(words_np.view(npv))
        if residency == "host":
            self.rows = torch.empty(src.shape, dtype=tdt, pin_memory=True)
            self.rows.copy_(src)
            self.slots = torch.empty((self.n, self.slot_bytes), dtype=torch.uint8,
                                     pin_memory=True)
        else:
            self.rows = src.to(dev)
            self.slots = torch.empty((self.n, self.slot_bytes), dtype=torch.uint8, device=dev)
        self.word_dtype = tdt
        self.meta = torch.zeros(4, dtype=torch.int32, device=dev)
        self.scratch = torch.empty(ibp.meta_scratch_bytes() // 4, dtype=torch.int32, device=dev)
        self.bitmask = torch.zeros(((self.n + 31) // 32,), dtype=torch.int32, device=dev)
        self.row_bits = torch.zeros((self.n,), dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.stats_t = torch.zeros(10, dtype=torch.int32, device=dev)
        # under several ranks the metadata is that of every rank's rows together:
        # local bit counts, one all-reduce of 33 int64 values, then the threshold
        self.sharded = False
        self.counters = torch.zeros(32, dtype=torch.int64, device=dev)

    def build_meta(self):
        if self.sharded:
            from lossless_bit_level_gb300.sharded import sharded_meta
            sharded_meta(self.rows, self.T, self.B, self.meta, self.counters, dtype=self.dtype)
        else:
            ibp.build_meta(self.rows, self.T, self.B, self.meta, self.scratch, dtype=self.dtype)

    def compress(self):
        ibp.compress(self.rows, self.B, self.meta, self.slots, self.bitmask, self.row_bits,
                     self.status, dtype=self.dtype)

    def gather(self, idx, out, status=None):
        ibp.decompress_gather(self.slots, self.n, self.L, self.dtype, self.B, self.bitmask,
                              self.meta, idx, out, status)

    def stats(self):
        return ibp.query(self.bitmask, self.row_bits, self.n, self.L, self.dtype)

    def stored_per_row(self):
        bits = self.row_bits.cpu().numpy().view(np.uint32).astype(np.int64)
        bm = self.bitmask.cpu().numpy().view(np.uint32)
        r = np.arange(self.n)
        flags = (bm[r // 32] >> (r % 32).astype(np.uint32)) & 1
        return np.where(flags == 1, 4 * ((bits + 31) // 32), self.raw_bytes)


class MaskSelect:
    """The saving-aware mask selection of a store's rows (meta + candidate table)."""

    def __init__(self, store):
        self.store = store
        dev = store.meta.device
        self.meta = torch.zeros(4, dtype=torch.int32, device=dev)
        self.scratch = torch.empty(ibp.meta_select_scratch_bytes() // 4, dtype=torch.int32,
                                   device=dev)
        self.cand = torch.zeros((ibp.MAX_MASK_CANDIDATES, 4), dtype=torch.int32, device=dev)

    def run(self):
        st = self.store
        ibp.build_meta_select(st.rows, st.T, st.B, self.meta, self.scratch, self.cand,
                              dtype=st.dtype)


def mask_select_leg(store, wl, batches, out, steps, warmup, flush, barrier, reps, table_raw,
                    out_bytes, residency, link, hbm_peak):
    """The saving-aware mask variant: time the selection over the table, recompress
    the store with the chosen mask (into the same slot buffer; the legs of the
    threshold mask are done by then) and time the same gather on it."""
    sel = MaskSelect(store)
    sel_t, _ = time_stage(sel.run, reps, flush)
    torch.cuda.synchronize()
    cands = ibp.read_candidates(sel.cand)
    sstore = Store.__new__(Store)
    sstore.__dict__.update(store.__dict__)
    sstore.meta = sel.meta
    sstore.bitmask = torch.zeros_like(store.bitmask)
    sstore.row_bits = torch.zeros_like(store.row_bits)
    sstore.status = torch.zeros_like(store.status)
    sstore.compress()
    torch.cuda.synchronize()
    assert int(sstore.status.item()) == 0
    st = sstore.stats()
    stored = sstore.stored_per_row()
    per_step, clk = timed_gather(sstore, batches, out, max(50, steps // 4), warmup, flush,
                                 barrier)
    ts = float(np.mean(per_step))
    gathered = float(np.mean([stored[b.cpu().numpy()].sum() for b in batches]))

    class Sized:  # the same store read through the sized gather (row sizes from row_bits)
        def gather(self, idx, o, st=None):
            ibp.decompress_gather_sized(sstore.slots, sstore.n, sstore.L, sstore.dtype, sstore.B,
                                        sstore.bitmask, sstore.row_bits, sstore.meta, idx, o, st)

    per_sized, clk_sized = timed_gather(Sized(), batches, out, max(50, steps // 4), warmup,
                                        flush, barrier)
    t_sized = float(np.mean(per_sized))
    peak = link["h2d_memcpy_gbs"] if residency == "host" else hbm_peak
    sel_frac = 2 * table_raw / sel_t / 1e9 / peak
    mask = int(sel.meta[0].item()) & 0xFFFFFFFF
    g = {"value": out_bytes / ts / 1e9, "unit": "GB/s", "ms_per_step": ts * 1e3,
         "stored_bytes_per_launch": gathered, "clocks": clk,
         "sized": {"value": out_bytes / t_sized / 1e9, "unit": "GB/s",
                   "ms_per_step": t_sized * 1e3, "clocks": clk_sized,
                   "note": "ibp_decompress_gather_sized: each row's stored bytes only"}}
    if residency == "host":
        g["link_frac_algorithmic"] = gathered / ts / 1e9 / peak
    else:
        alg = wl["batch"] * 8 + gathered + out_bytes
        g["hbm_frac"] = alg / ts / 1e9 / hbm_peak
    return sstore, {
        "mask": f"{mask:#010x}", "bitval": f"{int(sel.meta[1].item()) & 0xFFFFFFFF:#010x}",
        "candidates": [{"mask": f"{m:#010x}", "stored_bytes": b} for m, _, b in cands],
        "space_saving_pct": 100.0 * (1.0 - st.stored_bytes / st.raw_bytes),
        "space_saving_gathered_pct": 100.0 * (1.0 - gathered / out_bytes),
        "select": {"ms": sel_t * 1e3, "gbs_raw_in": table_raw / sel_t / 1e9,
                   "frac": sel_frac, "bound": "host_link" if residency == "host" else "hbm",
                   "reads_rows": 2},
        "gather": g}


class PackedStore:
    """A packed store (rows end to end) of every row of a slotted store."""

    def __init__(self, store, where, dev):
        self.n, self.L, self.dtype, self.B, self.meta = (store.n, store.L, store.dtype, store.B,
                                                         store.meta)
        self.offsets = torch.zeros(self.n + 1, dtype=torch.int64, device=dev)
        scratch = torch.empty(ibp.pack_scratch_bytes(self.n) // 8, dtype=torch.int64,
                              device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        ibp.pack_offsets(store.bitmask, store.row_bits, self.n, self.L, self.dtype, self.offsets,
                         scratch, status=self.status)
        self.total = int(self.offsets[-1].item())
        if where == "host":
            self.packed = torch.empty(self.total, dtype=torch.uint8, pin_memory=True)
        else:
            self.packed = torch.empty(self.total, dtype=torch.uint8, device=dev)
        self.bitmask = torch.zeros_like(store.bitmask)
        self.row_bits = torch.zeros_like(store.row_bits)
        self.pack_fn = lambda: ibp.pack(store.slots, self.n, self.L, self.dtype, store.bitmask,
                                        store.row_bits, self.offsets, self.packed, self.bitmask,
                                        self.row_bits, status=self.status)
        self.pack_fn()
        torch.cuda.synchronize()
        assert int(self.status.item()) == 0

    def gather(self, idx, out, status=None):
        ibp.decompress_gather_packed(self.packed, self.offsets, self.n, self.L, self.dtype,
                                     self.B, self.bitmask, self.meta, idx, out, status)


def packed_leg(sstore, wl, batches, out, steps, warmup, flush, barrier, table_raw, out_bytes,
               link, hbm_peak, dev):
    """The packed store ("cache-compression mode") of the table compressed with the
    saving-aware mask, in pinned host memory and in HBM: the same gathers, reading
    exactly each row's stored bytes (16-byte rounded)."""
    res = {"store": "rows compressed with the saving-aware mask, packed end to end"}
    for where in ("host", "device"):
        ps = PackedStore(sstore, where, dev)
        pt, _ = time_stage(ps.pack_fn, 3, flush)
        per_step, clk = timed_gather(ps, batches, out, max(50, steps // 4), warmup, flush,
                                     barrier)
        ts = float(np.mean(per_step))
        off = ps.offsets.cpu().numpy()
        entry = np.diff(off)
        gathered = float(np.mean([entry[b.cpu().numpy()].sum() for b in batches]))
        r = {"value": out_bytes / ts / 1e9, "unit": "GB/s", "ms_per_step": ts * 1e3,
             "packed_bytes": ps.total, "capacity_gain": table_raw / ps.total,
             "entry_bytes_per_launch": gathered, "pack_ms": pt * 1e3, "clocks": clk}
        if where == "host":
            r["link_frac_algorithmic"] = gathered / ts / 1e9 / link["h2d_memcpy_gbs"]
        else:
            alg = wl["batch"] * 24 + gathered + out_bytes  # index, two offsets, entry, row
            r["hbm_frac"] = alg / ts / 1e9 / hbm_peak
        res[where] = r
        del ps
        torch.cuda.empty_cache()
    return res


def positions_leg(store, wl, batches, out, steps, warmup, flush, barrier, reps, table_raw,
                  out_bytes, link, hbm_peak, dev, thresholds=(None, 0.99)):
    """Per-position metadata (one mask/bitval per element position of a row): the
    metadata build, the compression and the same gathers, at the workload's T and at
    T = 0.99; then block-position metadata (one pair per position within a block) at
    the workload's T. Compresses into the store's slot buffer (the other legs are
    done)."""
    n, L, dt, B = store.n, store.L, store.dtype, store.B
    pm = torch.zeros(L, dtype=torch.int32, device=dev)
    pb = torch.zeros(L, dtype=torch.int32, device=dev)
    scratch = torch.empty(ibp.meta_positions_scratch_bytes(L, dt) // 8, dtype=torch.int64,
                          device=dev)
    bitmask = torch.zeros_like(store.bitmask)
    row_bits = torch.zeros_like(store.row_bits)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    res = {"metadata_bytes": 8 * L, "block_positions_metadata_bytes": 8 * B}
    modes = [(f"T={wl['T'] if T is None else T}", wl["T"] if T is None else T, False)
             for T in thresholds]
    modes.append((f"block_positions T={wl['T']}", wl["T"], True))
    for key, T, per_block in modes:
        build = ibp.build_meta_block_positions if per_block else ibp.build_meta_positions

        def meta():
            build(store.rows, T, B, pm, pb, scratch, dtype=dt)

        def comp():
            ibp.compress_positions(store.rows, B, pm, pb, store.slots, bitmask, row_bits, dtype=dt)

        mt, _ = time_stage(meta, reps, flush)
        ct, _ = time_stage(comp, reps, flush)
        torch.cuda.synchronize()
        bits = row_bits.cpu().numpy().view(np.uint32).astype(np.int64)
        bm = bitmask.cpu().numpy().view(np.uint32)
        r = np.arange(n)
        comp_flag = (bm[r // 32] >> (r % 32).astype(np.uint32)) & 1
        stored = np.where(comp_flag == 1, 4 * ((bits + 31) // 32), store.raw_bytes)

        class G:
            def gather(self, idx, o, st=None):
                ibp.decompress_gather_positions(store.slots, n, L, dt, B, bitmask, pm, pb, idx, o,
                                                status)

        per_step, clk = timed_gather(G(), batches, out, max(50, steps // 4), warmup, flush,
                                     barrier)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ts = float(np.mean(per_step))
        peak = link["h2d_memcpy_gbs"] if store.residency == "host" else hbm_peak
        res[key] = {
            "space_saving_pct": 100.0 * (1.0 - stored.sum() / table_raw),
            "build_meta_ms": mt * 1e3, "build_meta_frac": table_raw / mt / 1e9 / peak,
            "compress_ms": ct * 1e3,
            "gather": {"value": out_bytes / ts / 1e9, "unit": "GB/s", "ms_per_step": ts * 1e3,
                       "clocks": clk, "frac_of_" + ("link" if store.residency == "host" else "hbm"):
                       out_bytes / ts / 1e9 / peak if store.residency == "host" else
                       (wl["batch"] * 8 + out_bytes + out_bytes) / ts / 1e9 / peak}}
    return res


def dedup_launches(store):
    """Kernel launches of one de-duplicated gather: clear, claiming gather and copy for
    rows of at most 32 blocks and 4 KiB (one gather unit each); a separate hash pass
    before the gather for longer rows."""
    block_bytes = store.B * ibp.WIDTH[store.dtype] // 8
    nb = -(-store.L // store.B)
    seg_blocks = max(1, min(nb, 32, 4096 // block_bytes))
    return 3 if nb <= seg_blocks else 4


def dedup_leg(store, wl, batches, out, steps, warmup, flush, barrier, out_bytes, link, hbm_peak,
              dev):
    """The same gathers through ibp_decompress_gather_dedup: each distinct row of a batch
    read and decoded once, then copied to every position that names it. The link
    bytes it needs are the stored bytes of the distinct rows."""
    scratch = torch.empty(ibp.gather_dedup_scratch_bytes(wl["batch"], store.L, store.dtype,
                                                         store.B),
                          dtype=torch.uint8, device=dev)

    class Dedup:
        def gather(self, idx, o, st=None):
            ibp.decompress_gather_dedup(store.slots, store.n, store.L, store.dtype, store.B,
                                        store.bitmask, store.meta, idx, o, scratch, st)

    per_step, clk = timed_gather(Dedup(), batches, out, max(50, steps // 4), warmup, flush,
                                 barrier)
    ts = float(np.mean(per_step))
    stored = store.stored_per_row()
    host_idx = [b.cpu().numpy() for b in batches]
    distinct = float(np.mean([np.unique(b).size / b.size for b in host_idx]))
    distinct_bytes = float(np.mean([stored[np.unique(b)].sum() for b in host_idx]))
    # the output matches the plain gather's
    check = torch.empty_like(out)
    store.gather(batches[0], check)
    Dedup().gather(batches[0], out)
    torch.cuda.synchronize()
    assert torch.equal(check, out)
    del scratch, check
    torch.cuda.empty_cache()
    r = {"value": out_bytes / ts / 1e9, "unit": "GB/s", "ms_per_step": ts * 1e3, "clocks": clk,
         "distinct_fraction": distinct, "distinct_stored_bytes_per_launch": distinct_bytes,
         "launches_per_call": dedup_launches(store)}
    if store.residency == "host":
        r["link_frac_distinct_bytes"] = distinct_bytes / ts / 1e9 / link["h2d_memcpy_gbs"]
    else:
        r["hbm_frac"] = (wl["batch"] * 8 + distinct_bytes + 2 * out_bytes) / ts / 1e9 / hbm_peak
    return r


def dlrm_batched_leg(dev, flush, barrier, steps, warmup, hbm_peak, n_tables=26,
                     lookups=65_536, n_rows=1_000_000):
    """All 26 DLRM tables (1,000,000 x 128 FP32 each, per-table metadata T = 0.95,
    B = 32, slots in HBM) and one Zipf(1.05) lookup batch of 65,536 rows per table:
    26 separate gathers per step against one batched gather of all 26 jobs."""
    L, T, B = 128, 0.95, 32
    stores, jobs, outs = [], [], []
    stored_total = 0
    for t in range(n_tables):
        words = gen.dlrm_table(t, n_rows).view(np.uint32)
        n = words.shape[0]
        rows = torch.from_numpy(words.view(np.int32)).to(dev)
        meta = torch.zeros(4, dtype=torch.int32, device=dev)
        scr = torch.empty(ibp.meta_scratch_bytes() // 4, dtype=torch.int32, device=dev)
        ibp.build_meta(rows, T, B, meta, scr, dtype=ibp.FP32)
        slots = torch.empty((n, ibp.slot_bytes(L, ibp.FP32)), dtype=torch.uint8, device=dev)
        bm = torch.zeros(((n + 31) // 32,), dtype=torch.int32, device=dev)
        rb = torch.zeros((n,), dtype=torch.int32, device=dev)
        ibp.compress(rows, B, meta, slots, bm, rb, None, dtype=ibp.FP32)
        ix = gen.zipf_indices(n, lookups, 1.05, part=t, workload=gen.DLRM)
        bits = rb.cpu().numpy().view(np.uint32).astype(np.int64)
        comp = (bm.cpu().numpy().view(np.uint32)[np.arange(n) // 32] >>
                (np.arange(n) % 32).astype(np.uint32)) & 1
        stored = np.where(comp == 1, 4 * ((bits + 31) // 32), 4 * L)
        stored_total += int(stored[ix].sum())
        out = torch.empty((lookups, L), dtype=torch.int32, device=dev)
        stores.append((slots, n, bm, meta))
        jobs.append((slots, n, bm, meta, torch.from_numpy(ix).to(dev), out))
        outs.append(out)
        del rows, words
    torch.cuda.synchronize()
    out_bytes = n_tables * lookups * 4 * L
    alg = n_tables * lookups * 8 + stored_total + out_bytes
    s = torch.cuda.current_stream()

    def separate():
        for slots, n, bm, meta, ix, out in jobs:
            ibp.decompress_gather(slots, n, L, ibp.FP32, B, bm, meta, ix, out)

    def batched():
        ibp.decompress_gather_batched(jobs, L, ibp.FP32, B)

    res = {"workload": f"{n_tables} DLRM tables {n_rows:,} x 128 FP32 in HBM, {lookups} "
                       "Zipf(1.05) lookups per table per step", "output_bytes_per_step": out_bytes,
           "algorithmic_bytes_per_step": alg}
    for name, fn in (("separate_calls", separate), ("batched_call", batched)):
        class G:
            def gather(self, idx, o, st=None):
                fn()
        per_step, clk = timed_gather(G(), [None], None, max(20, steps // 10), warmup, flush,
                                     barrier)
        t = float(np.mean(per_step))
        res[name] = {"value": out_bytes / t / 1e9, "unit": "GB/s", "ms_per_step": t * 1e3,
                     "hbm_frac": alg / t / 1e9 / hbm_peak, "clocks": clk}
    # every table's rows come back exactly
    for (slots, n, bm, meta, ix, out), t in zip(jobs, range(n_tables)):
        if t % 9 == 0:
            words = gen.dlrm_table(t, n_rows).view(np.uint32)
            assert np.array_equal(out.cpu().numpy().view(np.uint32), words[ix.cpu().numpy()])
    del stores, jobs, outs
    torch.cuda.empty_cache()
    return res


def offload_leg(dev, n_steps=8, token_counts=(256, 4096)):
    """Overlapped offload pipeline on one LLaMA-7B-shaped decoder layer (q, k, v, o
    4096 x 4096; gate, up 11008 x 4096; down 4096 x 11008; BF16 N(0, 0.02)) kept
    compressed in page-locked host memory (threshold mask per tensor, T = 0.9,
    B = 64) and streamed n_steps times through two device buffer sets while a
    consumer runs one bf16 matmul per weight (tokens x in) @ (in x out). Per-layer
    time for the compressed and the raw (cudaMemcpyAsync) loaders, overlapped with
    the consumer and serialised with it."""
    from lossless_bit_level_gb300.offload import CompressedTensor, OffloadPipeline, raw_loader

    layer, raw = [], {}
    for name in gen.LLM_MATRICES:
        w = gen.llm_weight(0, name)
        t = CompressedTensor.from_words(w, ibp.BF16, 0.9, 64, dev)
        h = torch.empty(w.shape, dtype=torch.int16, pin_memory=True)
        h.copy_(torch.from_numpy(w.view(np.int16)))
        raw[id(t)] = h
        layer.append(t)
        del w
    layers = [layer]
    raw_bytes = sum(t.raw_bytes for t in layer)
    stored = sum(t.stored_bytes() for t in layer)
    res = {"workload": "one LLaMA-7B-shaped decoder layer, 7 BF16 weights N(0, 0.02), "
                       f"streamed {n_steps} times; consumer: one bf16 matmul per weight",
           "raw_bytes_per_layer": raw_bytes, "stored_bytes_per_layer": stored,
           "saving_pct": 100.0 * (1.0 - stored / raw_bytes), "tokens": {}}
    for tokens in token_counts:
        xh = torch.randn(tokens, gen.LLM_HIDDEN, dtype=torch.bfloat16, device=dev)
        xf = torch.randn(tokens, gen.LLM_FFN, dtype=torch.bfloat16, device=dev)

        def consume(l, bufs):
            for t, b in zip(layers[l], bufs):
                x = xf if t.row_elems == gen.LLM_FFN else xh
                torch.matmul(x, b.view(torch.bfloat16).t())

        r = {}
        warm = [t.empty_like(dev) for t in layer]
        for _ in range(3):  # library start-up of the consumer's matmul shapes
            consume(0, warm)
        torch.cuda.synchronize()
        del warm
        for mode, load, overlap in (("ibp_overlap", None, True), ("raw_overlap", raw_loader(raw), True),
                                    ("ibp_serial", None, False), ("raw_serial", raw_loader(raw), False)):
            pipe = OffloadPipeline(layers, dev, load=load, overlap=overlap)
            pipe.run(3, consume)
            pipe.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(pipe.loader)
            pipe.compute.wait_event(a)
            pipe.run(n_steps, consume)
            b.record(pipe.compute)
            b.synchronize()
            r[mode + "_ms_per_layer"] = a.elapsed_time(b) / n_steps
            del pipe
        s = torch.cuda.current_stream()
        bufs = [t.empty_like(dev) for t in layer]
        consume(0, bufs)
        a, b = event_pair(s)
        a.record(s)
        for _ in range(n_steps):
            consume(0, bufs)
        b.record(s)
        b.synchronize()
        r["compute_only_ms_per_layer"] = a.elapsed_time(b) / n_steps
        r["speedup_vs_raw_overlap"] = r["raw_overlap_ms_per_layer"] / r["ibp_overlap_ms_per_layer"]
        r["ibp_decode_link_gbs"] = stored / (r["ibp_serial_ms_per_layer"] -
                                            r["compute_only_ms_per_layer"]) / 1e6
        res["tokens"][str(tokens)] = r
        del bufs, xh, xf
    for t in layer:
        assert int(t.status.item()) == 0
    del layers, layer, raw
    torch.cuda.empty_cache()
    return res


def time_stage(fn, reps, flush=None):
    s = torch.cuda.current_stream()
    ts = []
    for _ in range(reps):
        if flush is not None:
            flush()
        a, b = event_pair(s)
        a.record(s)
        fn()
        b.record(s)
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e-3)
    return min(ts), statistics.median(ts)


def timed_gather(store, batches, out, steps, warmup, flush, barrier):
    """W warm-up steps, then K timed steps; per-step CUDA events on the launch stream
    (the L2 flush between steps sits outside the events). The clock sampler starts
    before the warm-up, so that the warm-up steps, not the first timed one, absorb
    whatever the pause of its start-up leaves behind. Returns seconds per step list
    and the clock summary."""
    s = torch.cuda.current_stream()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with ClockSampler(torch.cuda.current_device()) as clk:
        for k in range(warmup):
            flush()
            store.gather(batches[k % len(batches)], out)
        barrier()
        torch.cuda.synchronize()
        for k in range(steps):
            flush()
            starts[k].record(s)
            store.gather(batches[k % len(batches)], out)
            ends[k].record(s)
        torch.cuda.synchronize()
        barrier()
    per_step = [a.elapsed_time(b) * 1e-3 for a, b in zip(starts, ends)]
    return per_step, clk.summary()


def run_e2e(store, host_batches, steps, warmup, dev):
    """Through the public API with host buffers: pinned index batch -> device, gather,
    gathered rows -> pinned host, all inside the timed region of each step. Steps
    rotate over four streams with their own buffers, so that the read-back of one
    step (device -> host) overlaps the gathers of the next ones (host -> device); every
    step still makes both copies. (Measured: 1, 2, 3, 4 streams give 103, 138, 156,
    160 GB/s on the dense GNN workload; the host link carries ~340 GB/s in both
    directions at once.)"""
    n_idx = host_batches[0].numel()
    ns = 4
    streams = [torch.cuda.Stream(device=dev) for _ in range(ns)]
    idx_d = [torch.empty(n_idx, dtype=torch.int64, device=dev) for _ in range(ns)]
    out_d = [torch.empty((n_idx, store.L), dtype=store.word_dtype, device=dev) for _ in range(ns)]
    out_h = [torch.empty((n_idx, store.L), dtype=store.word_dtype, pin_memory=True)
             for _ in range(ns)]
    main = torch.cuda.current_stream()

    def step(k):
        j = k % ns
        with torch.cuda.stream(streams[j]):
            idx_d[j].copy_(host_batches[k % len(host_batches)], non_blocking=True)
            store.gather(idx_d[j], out_d[j])
            out_h[j].copy_(out_d[j], non_blocking=True)

    for k in range(warmup):
        step(k)
    torch.cuda.synchronize()
    a, b = event_pair(main)
    a.record(main)
    for st in streams:
        st.wait_event(a)
    for k in range(steps):
        step(k)
    for st in streams:
        main.wait_stream(st)
    b.record(main)
    b.synchronize()
    t = a.elapsed_time(b) * 1e-3 / steps
    return {"value": n_idx * store.raw_bytes / t / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": n_idx * 8, "d2h_bytes_per_step": n_idx * store.raw_bytes,
            "ms_per_step": t * 1e3, "streams": ns}


# ----------------------------------------------------------------------------- five configs

def _sig(x, nd=3):
    """x rounded to nd significant digits (the per-config summary is kept short)."""
    if x is None or x == 0 or not np.isfinite(x):
        return x
    return float(f"{x:.{nd}g}")


def time_steps(fn, steps, warmup, flush):
    """warmup untimed calls, then steps calls, each after an L2 flush and timed with
    CUDA events on the launch stream; mean seconds per call. fn(k) runs step k."""
    s = torch.cuda.current_stream()
    for k in range(warmup):
        flush()
        fn(k)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for k in range(steps):
        flush()
        starts[k].record(s)
        fn(k)
        ends[k].record(s)
    torch.cuda.synchronize()
    return float(np.mean([a.elapsed_time(b) for a, b in zip(starts, ends)])) * 1e-3


class TableBench:
    """One table of a workload, measured the way every config is: rows and slots in
    HBM, metadata and compression timed (raw input per second; compression's roofline
    counts the rows read, the stored bytes and the bitmask/row-size words written),
    then gathers of index batches (or in-order streams of whole tables, idx None)
    from the slots in HBM and from a copy of them in page-locked host memory."""

    def __init__(self, words, dtype, T, B, dev, flush, hbm_peak):
        self.st = Store(words, dtype, T, B, "device", dev)
        self.dev, self.flush, self.hbm_peak = dev, flush, hbm_peak
        st = self.st
        self.t_meta, _ = time_stage(st.build_meta, 3, flush)
        self.t_comp, _ = time_stage(st.compress, 3, flush)
        torch.cuda.synchronize()
        assert int(st.status.item()) == 0
        self.stats = st.stats()
        self.stored = st.stored_per_row()
        self.raw = st.n * st.raw_bytes
        self.comp_alg = self.raw + float(self.stored.sum()) + 4 * ((st.n + 31) // 32) + 4 * st.n
        self.host_slots = None

    def slots(self, where):
        if where == "device":
            return self.st.slots
        if self.host_slots is None:
            self.host_slots = torch.empty(self.st.slots.shape, dtype=torch.uint8, pin_memory=True)
            self.host_slots.copy_(self.st.slots)
        return self.host_slots

    def gather(self, where, batches_np, steps=10, warmup=3):
        """Mean seconds per gather of batches_np[k % len] (None: every row in order
        through ibp_decompress_range), and the output checked on the device against
        the rows of the last batch."""
        st = self.st
        slots = self.slots(where)
        if batches_np is None:
            out = torch.empty_like(st.rows)

            def fn(k):
                ibp.decompress_range(slots, st.n, st.L, st.dtype, st.B, st.bitmask, st.meta, 0,
                                     st.n, out, st.status)
        else:
            batches = [torch.from_numpy(b).to(self.dev) for b in batches_np]
            out = torch.empty((batches_np[0].size, st.L), dtype=st.word_dtype, device=self.dev)

            def fn(k):
                ibp.decompress_gather(slots, st.n, st.L, st.dtype, st.B, st.bitmask, st.meta,
                                      batches[k % len(batches)], out, st.status)
        t = time_steps(fn, steps, warmup, self.flush)
        torch.cuda.synchronize()
        assert int(st.status.item()) == 0
        want = st.rows if batches_np is None else st.rows[batches[(steps - 1) % len(batches)]]
        assert torch.equal(out, want), "gathered rows differ from the originals"
        del out
        return t

    def summary(self):
        st = self.st
        return {"rows": st.n, "save_pct": _sig(100.0 * (1.0 - self.stats.stored_bytes / self.raw)),
                "meta_GBs": _sig(self.raw / self.t_meta / 1e9),
                "comp_GBs": _sig(self.raw / self.t_comp / 1e9),
                "comp_frac": _sig(self.comp_alg / self.t_comp / 1e9 / self.hbm_peak)}


def gather_entry(t, n_idx, row_bytes, stored_gathered, distinct_stored, where, h2d, hbm_peak,
                 index_bytes=8):
    """One gather result: GB/s of output rows and the roofline fraction. HBM: (index +
    stored + output bytes) / t over the device copy. Host slots: stored bytes of the
    gathered rows (duplicates counted) / t over the pinned H2D copy, and the same for
    the distinct rows only (each distinct row crosses the link at least once, so the
    true link fraction lies at or above it)."""
    out_bytes = n_idx * row_bytes
    e = {"ms": _sig(t * 1e3), "GBs": _sig(out_bytes / t / 1e9)}
    if where == "device":
        alg = n_idx * index_bytes + stored_gathered + out_bytes
        e["frac"] = _sig(alg / t / 1e9 / hbm_peak)
        e["alg_MB"] = _sig(alg / 1e6)
    else:
        e["link_frac"] = _sig(stored_gathered / t / 1e9 / h2d)
        e["link_frac_distinct"] = _sig(distinct_stored / t / 1e9 / h2d)
        e["link_MB"] = _sig(stored_gathered / 1e6)
    return e


def configs_leg(dev, flush, hbm_peak, link, main):
    """Every configuration of the workload set, measured in one pass (inputs generated
    from the seeded recipe, the big ones in parallel host threads):
      tiny FP32 4096 x 128, 1024 uniform indices, HBM;
      dense GNN 2,000,000 x 128 (the headline store, from the main measurement) plus
        1,000,000-index gathers from HBM whose output (512 MB) exceeds L2, Zipf(1.0)
        and uniform;
      sparse GNN 500,000 x 512, 100,000 uniform indices, host and HBM;
      DLRM: table 0 (65,536 Zipf(1.05) lookups, host and HBM) and all 26 tables in
        HBM, one lookup batch per table per step, 26 separate calls vs one batched call;
      LLM BF16: layer 0's seven weights and its K and V caches (8 x 4096 tokens), each
        tensor streamed in order through ibp_decompress_range from host and from HBM
        (the weights also with one launch per row geometry: a batched call for the six
        with 4096-element rows, a range call for the down-projection); summed over the
        layer (the other 31 layers have the same shapes and
        distributions, so a layer's time scales by 32 for the model).
    Every gather's output is checked against the original rows on the device."""
    import concurrent.futures as cf

    h2d = link["h2d_memcpy_gbs"]
    res = {}
    pool = cf.ThreadPoolExecutor(max_workers=max(2, min(16, os.cpu_count() or 2)))
    # the big inputs are generated in the background while the small configs run
    dlrm_f = [pool.submit(gen.dlrm_table, t) for t in range(26)]
    llm_f = {name: pool.submit(gen.llm_weight, 0, name) for name in gen.LLM_MATRICES}
    llm_f["K"] = pool.submit(gen.llm_kv, 0, 0)
    llm_f["V"] = pool.submit(gen.llm_kv, 0, 1)
    sparse_f = pool.submit(gen.gnn_sparse)

    def table_config(words, dtype, T, B, batches_np, wheres, steps=10):
        tb = TableBench(words, dtype, T, B, dev, flush, hbm_peak)
        r = tb.summary()
        for where in wheres:
            t = tb.gather(where, batches_np, steps=steps)
            if batches_np is None:
                n_idx, g_st, d_st, ib = tb.st.n, float(tb.stored.sum()), float(tb.stored.sum()), 0
            else:
                n_idx = batches_np[0].size
                g_st = float(np.mean([tb.stored[b].sum() for b in batches_np]))
                d_st = float(np.mean([tb.stored[np.unique(b)].sum() for b in batches_np]))
                ib = 8
            r["hbm" if where == "device" else "host"] = gather_entry(
                t, n_idx, tb.st.raw_bytes, g_st, d_st, where, h2d, hbm_peak, ib)
        return tb, r

    # tiny: a correctness config (0.5 MB of output per launch is launch-bound)
    words = gen.tiny_fp32().view(np.uint32)
    b = [gen.uniform_indices(words.shape[0], 1024, part=k, workload=gen.TINY) for k in range(4)]
    tb, res["tiny"] = table_config(words, ibp.FP32, 0.9, 32, b, ("device",), steps=20)
    del tb

    # dense GNN: the headline store's figures, and a large HBM batch
    res["gnn_dense"] = main
    words = gen.gnn_dense().view(np.uint32)
    big = [gen.zipf_indices(words.shape[0], 1_000_000, 1.0, part=100 + k,
                            workload=gen.GNN_DENSE) for k in range(2)]
    tb = TableBench(words, ibp.FP32, 0.9, 32, dev, flush, hbm_peak)
    t = tb.gather("device", big, steps=6)
    g_st = float(np.mean([tb.stored[x].sum() for x in big]))
    res["gnn_dense"]["hbm_1M_idx"] = gather_entry(t, big[0].size, tb.st.raw_bytes, g_st, g_st,
                                                  "device", h2d, hbm_peak)
    # the same size with uniform indices: few duplicates, so nearly every byte counted
    # is a DRAM byte (Zipf's hot rows are served from L2)
    uni = [gen.uniform_indices(words.shape[0], 1_000_000, part=200 + k, workload=gen.GNN_DENSE)
           for k in range(2)]
    t = tb.gather("device", uni, steps=6)
    g_st = float(np.mean([tb.stored[x].sum() for x in uni]))
    res["gnn_dense"]["hbm_1M_uniform"] = gather_entry(t, uni[0].size, tb.st.raw_bytes, g_st,
                                                      g_st, "device", h2d, hbm_peak)
    del tb, words, big, uni
    torch.cuda.empty_cache()

    # sparse GNN
    words = sparse_f.result().view(np.uint32)
    b = [gen.uniform_indices(words.shape[0], 100_000, part=k, workload=gen.GNN_SPARSE)
         for k in range(4)]
    tb, res["gnn_sparse"] = table_config(words, ibp.FP32, 0.9, 32, b, ("host", "device"))
    del tb, words
    torch.cuda.empty_cache()

    # DLRM: table 0 alone, then the 26 tables in HBM
    L, T, B, lookups = 128, 0.95, 32, 65_536
    tables, jobs, stored_g = [], [], 0
    for t_id in range(26):
        words = dlrm_f[t_id].result().view(np.uint32)
        dlrm_f[t_id] = None
        ix = gen.zipf_indices(words.shape[0], lookups, 1.05, part=t_id, workload=gen.DLRM)
        if t_id == 0:
            tb, r = table_config(words, ibp.FP32, T, B, [ix], ("host", "device"))
            res["dlrm"] = {"table0": r}
            tb.host_slots = None
        else:
            tb = TableBench(words, ibp.FP32, T, B, dev, flush, hbm_peak)
        st = tb.st
        stored_g += int(tb.stored[ix].sum())
        out = torch.empty((lookups, L), dtype=torch.int32, device=dev)
        jobs.append((st.slots, st.n, st.bitmask, st.meta, torch.from_numpy(ix).to(dev), out))
        st.rows = None  # rows are not needed past compression; keep HBM use down
        tables.append(tb)
        del words
    out_bytes = 26 * lookups * 4 * L
    alg = 26 * lookups * 8 + stored_g + out_bytes

    def separate(k):
        for slots, n, bm, meta, ix, out in jobs:
            ibp.decompress_gather(slots, n, L, ibp.FP32, B, bm, meta, ix, out)

    def batched(k):
        ibp.decompress_gather_batched(jobs, L, ibp.FP32, B)

    d = {"save_pct": _sig(100.0 * (1.0 - sum(x.stats.stored_bytes for x in tables) /
                                   sum(x.raw for x in tables))),
         "comp_GBs": _sig(sum(x.raw for x in tables) / sum(x.t_comp for x in tables) / 1e9),
         "comp_frac": _sig(sum(x.comp_alg for x in tables) / sum(x.t_comp for x in tables) /
                           1e9 / hbm_peak)}
    for name, fn in (("separate_hbm", separate), ("batched_hbm", batched)):
        t = time_steps(fn, 8, 3, flush)
        d[name] = {"ms": _sig(t * 1e3), "GBs": _sig(out_bytes / t / 1e9),
                   "frac": _sig(alg / t / 1e9 / hbm_peak)}
    torch.cuda.synchronize()
    for j in (0, 13, 25):  # rows back exactly (the tables' rows are regenerated)
        ref = torch.from_numpy(gen.dlrm_table(j).view(np.int32)).to(dev)
        assert torch.equal(jobs[j][5], ref[jobs[j][4]])
        del ref
    res["dlrm"]["tables26"] = d
    del tables, jobs
    torch.cuda.empty_cache()

    # LLM: one decoder layer, every row of each tensor streamed in order
    parts = {"weights": [*gen.LLM_MATRICES], "kv": ["K", "V"]}
    acc = {}
    kept = []  # the weights' HBM stores, for the one-launch-per-row-geometry decode
    for part, names in parts.items():
        a = dict(raw=0, stored=0, t_comp=0.0, comp_alg=0.0, host=0.0, device=0.0)
        for name in names:
            words = llm_f[name].result()
            llm_f[name] = None
            tb = TableBench(words, ibp.BF16, 0.9, 64, dev, flush, hbm_peak)
            a["raw"] += tb.raw
            a["stored"] += int(tb.stats.stored_bytes)
            a["t_comp"] += tb.t_comp
            a["comp_alg"] += tb.comp_alg
            for where in ("host", "device"):
                a[where] += tb.gather(where, None, steps=6)
            if part == "weights":
                tb.host_slots = None
                kept.append(tb)
            del tb, words
            torch.cuda.empty_cache()
        acc[part] = a
    pool.shutdown()

    # the same weights decoded with one launch per row geometry: the tensors with
    # 4096-element rows in one batched call (their rows in order as index lists), the
    # down-projection (11008-element rows) in one range call
    geo = {}
    for tb in kept:
        geo.setdefault(tb.st.L, []).append(tb)
    calls, alg_b = [], 0.0
    for L_g, tbs in geo.items():
        if len(tbs) == 1:
            st = tbs[0].st
            out = torch.empty_like(st.rows)
            calls.append(lambda k, st=st, out=out, L_g=L_g: ibp.decompress_range(
                st.slots, st.n, L_g, ibp.BF16, 64, st.bitmask, st.meta, 0, st.n, out))
            alg_b += float(tbs[0].stored.sum()) + tbs[0].raw
            checks = [(out, st.rows)]
        else:
            jobs_w = []
            for tb in tbs:
                st = tb.st
                out = torch.empty_like(st.rows)
                jobs_w.append((st.slots, st.n, st.bitmask, st.meta,
                               torch.arange(st.n, dtype=torch.int64, device=dev), out))
                alg_b += float(tb.stored.sum()) + tb.raw + 8 * st.n
            calls.append(lambda k, jobs_w=jobs_w, L_g=L_g: ibp.decompress_gather_batched(
                jobs_w, L_g, ibp.BF16, 64))
            checks = [(j[5], tb.st.rows) for j, tb in zip(jobs_w, tbs)]
        geo[L_g] = checks

    def per_geometry(k):
        for c in calls:
            c(k)

    t_b = time_steps(per_geometry, 6, 3, flush)
    torch.cuda.synchronize()
    for checks in geo.values():
        for out, rows in checks:
            assert torch.equal(out, rows), "decoded weights differ from the originals"
    weights_batched = {"ms": _sig(t_b * 1e3), "GBs": _sig(acc["weights"]["raw"] / t_b / 1e9),
                       "frac": _sig(alg_b / t_b / 1e9 / hbm_peak), "launches": len(calls)}
    del kept, geo, calls
    torch.cuda.empty_cache()

    def llm_entry(a):
        e = {"save_pct": _sig(100.0 * (1.0 - a["stored"] / a["raw"])),
             "comp_GBs": _sig(a["raw"] / a["t_comp"] / 1e9),
             "comp_frac": _sig(a["comp_alg"] / a["t_comp"] / 1e9 / hbm_peak)}
        e["host"] = gather_entry(a["host"], 1, a["raw"], a["stored"], a["stored"], "host", h2d,
                                 hbm_peak)
        e["hbm"] = gather_entry(a["device"], 1, a["raw"], a["stored"], a["stored"], "device",
                                h2d, hbm_peak, index_bytes=0)
        return e

    layer = {k: acc["weights"][k] + acc["kv"][k] for k in acc["weights"]}
    res["llm_layer0"] = {"all": llm_entry(layer), "weights": llm_entry(acc["weights"]),
                         "kv": llm_entry(acc["kv"]),
                         "note": "ms per layer; 32 layers of the same shapes: x32"}
    res["llm_layer0"]["weights"]["hbm_per_geometry"] = weights_batched
    return res


# ----------------------------------------------------------------------------- oracle arm

def oracle_sample(wl, seconds_budget=10.0, sample_rows=200_000, all_cores_budget=4.0):
    """The oracle (as written) on a bounded sample of the workload: a prefix table of
    sample_rows rows is built once (meta + compress by the oracle), then batches of
    the workload's batch size, drawn with the workload's index distribution over the
    prefix, are gathered until the time budget is spent. Returns the single-thread
    figure and the figure of the same oracle run on every host core, each batch split
    into one index range per thread (the library releases the interpreter lock while
    it runs, and its calls share no state)."""
    import concurrent.futures as cf

    import oracle

    rows = wl["rows_prefix"](sample_rows)
    words = rows.view(np.uint32) if rows.dtype == np.float32 else rows
    n, L = words.shape
    mask, bitval = oracle.build_meta(words, wl["T"])
    slots, bitmask, _ = oracle.compress(words, wl["B"], mask, bitval)
    out = np.empty((wl["batch"], L), dtype=words.dtype)
    row_bytes = L * words.dtype.itemsize

    def run(budget, gather):
        total_bytes, total_t, k = 0, 0.0, 0
        while total_t < budget and k < 64:
            idx = wl["index"](n, wl["batch"], 1000 + k)
            t0 = time.perf_counter()
            gather(idx)
            total_t += time.perf_counter() - t0
            total_bytes += idx.size * row_bytes
            k += 1
        return total_bytes / total_t / 1e9, total_t, k

    def one(idx, o):
        _, rc = oracle.decompress_gather(slots, n, L, words.dtype, wl["B"], bitmask, mask,
                                         bitval, idx, out=o)
        assert rc == 0

    gbs, secs, k = run(seconds_budget, lambda idx: one(idx, out))
    single = {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
              "sample": f"{k} gathers of {wl['batch']} indices ({wl['index_desc']}) over a "
                        f"{n}-row prefix table compressed by the oracle; single thread",
              "seconds": secs, "batches": k}
    cores = os.cpu_count() or 1
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        def split(idx):
            cuts = np.linspace(0, idx.size, cores + 1).astype(np.int64)
            futs = [ex.submit(one, idx[a:b], out[a:b]) for a, b in zip(cuts[:-1], cuts[1:])
                    if b > a]
            for f in futs:
                f.result()
        gbs_all, secs_all, k_all = run(all_cores_budget, split)
    every = {"value": gbs_all, "unit": "GB/s", "cores": cores, "kind": "oracle",
             "sample": f"{k_all} gathers of {wl['batch']} indices over the same table, each "
                       f"split into {cores} index ranges, one thread each",
             "seconds": secs_all, "batches": k_all}
    return single, every


# ----------------------------------------------------------------------------- main

def workload_table(name):
    wl = dict(WORKLOADS[name])
    wl["name"] = name
    if name == "gnn_dense":
        wl["rows_prefix"] = lambda n: gen.gnn_dense(n)
        wl["index_desc"] = "Zipf(1.0)"
    elif name == "gnn_sparse":
        wl["rows_prefix"] = lambda n: gen.gnn_sparse(min(n, 500_000))
        wl["index_desc"] = "uniform"
    elif name == "tiny":
        wl["rows_prefix"] = lambda n: gen.tiny_fp32(min(n, 4096))
        wl["index_desc"] = "uniform"
    elif name == "llm_kv":
        wl["rows_prefix"] = lambda n: gen.llm_kv(0, 0, n_rows=min(n, 32_768))
        wl["index_desc"] = "in-order"
    elif name == "llm_down":
        wl["rows_prefix"] = lambda n: gen.llm_weight(0, "down", n_rows=min(n, 4096))
        wl["index_desc"] = "in-order"
    else:
        wl["rows_prefix"] = lambda n: gen.dlrm_table(0, min(n, 1_000_000))
        wl["index_desc"] = "Zipf(1.05)"
    return wl


def run_reference(args, wl):
    """The oracle arm: the plain C++ oracle, as written, on the host cores. Each step
    gathers a bounded sample of one batch (a prefix of the batch's indices, sized so
    that the whole run stays within a few minutes) from a prefix table that the
    oracle itself built; the value is GB/s of rebuilt rows, as for the GPU arm."""
    rank, _, world = env_rank()
    if rank != 0:
        return 0
    import oracle

    steps, warmup = max(1, args.steps), max(0, args.warmup)
    prefix_rows = 200_000
    rows = wl["rows_prefix"](prefix_rows)
    words = rows.view(np.uint32) if rows.dtype == np.float32 else rows
    n, L = words.shape
    mask, bitval = oracle.build_meta(words, wl["T"])
    slots, bitmask, _ = oracle.compress(words, wl["B"], mask, bitval)
    out = np.empty((wl["batch"], L), dtype=words.dtype)
    # calibrate: seconds per index of the oracle gather on this host
    probe = wl["index"](n, min(wl["batch"], 20_000), 999)
    t0 = time.perf_counter()
    oracle.decompress_gather(slots, n, L, words.dtype, wl["B"], bitmask, mask, bitval, probe,
                             out=out)
    per_index = (time.perf_counter() - t0) / probe.size
    budget = 120.0 / (steps + warmup)
    per_step = int(max(256, min(wl["batch"], budget / max(per_index, 1e-9))))
    batches = [wl["index"](n, wl["batch"], 2000 + (k % 20))[:per_step] for k in range(20)]
    for k in range(warmup):
        oracle.decompress_gather(slots, n, L, words.dtype, wl["B"], bitmask, mask, bitval,
                                 batches[k % 20], out=out)
    t0 = time.perf_counter()
    for k in range(steps):
        oracle.decompress_gather(slots, n, L, words.dtype, wl["B"], bitmask, mask, bitval,
                                 batches[k % 20], out=out)
    t = (time.perf_counter() - t0) / steps
    value = per_step * L * words.dtype.itemsize / t / 1e9
    sample = (f"each step gathers the first {per_step} of a {wl['batch']}-index "
              f"{wl['index_desc']} batch over a {n}-row prefix table built by the oracle; "
              "single thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": f"u{8 * words.dtype.itemsize}",
        "data": "synthetic",
        "config": {"workload": wl["desc"]},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ibp", "reference"], default="ibp")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="gnn_dense")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quick", action="store_true", help="skip the HBM-resident and e2e legs")
    ap.add_argument("--legs", default=None,
                    help="run only these of the legs after the timed gather (comma-separated: "
                         f"{','.join(LEGS)}); default: all of them unless --quick")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the pass over every configuration (default workload only)")
    ap.add_argument("--residency", choices=["host", "device"], default=None,
                    help="override where slots and rows live (default: the workload's)")
    ap.add_argument("--indices", choices=["zipf", "uniform"], default=None,
                    help="override the workload's index distribution")
    ap.add_argument("--tables", type=int, default=26,
                    help="DLRM workload: tables in the batched-gather leg")
    ap.add_argument("--rows", type=int, default=None,
                    help="use only the first ROWS rows of the table (smaller profiling cases)")
    args = ap.parse_args()
    steps = args.steps if args.steps is not None else 2000
    warmup = args.warmup if args.warmup is not None else 20
    args.steps, args.warmup = steps, warmup
    if warmup < 3 and args.impl == "ibp":
        raise SystemExit("at least 3 warm-up steps are required")
    legs = None if args.legs is None else set(args.legs.split(","))
    if legs is not None and not legs <= set(LEGS):
        raise SystemExit(f"unknown legs: {sorted(legs - set(LEGS))}")
    wl = workload_table(args.workload)
    if args.residency:
        wl["residency"] = args.residency
    if args.indices == "uniform":
        wl["index"] = lambda n, k, part: gen.uniform_indices(n, k, part=part, workload=0)
        wl["index_desc"] = "uniform"
        wl["desc"] += " [indices overridden: uniform]"
    if args.rows:
        k = args.rows
        wl["rows"] = lambda: wl["rows_prefix"](k)
    if args.impl == "reference":
        return run_reference(args, wl)

    rank, local_rank, world = env_rank()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", torch.cuda.current_device())

    def barrier():
        if dist is not None:
            dist.barrier()

    from lossless_bit_level_gb300 import build_lib
    build_lib.build()
    ibp.load()

    peaks = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    hbm_peak_src = "measured" if "hbm_gbs" in peaks else "fallback"

    # inputs: generated on the host (seeded), resident where the workload says
    rows_np = wl["rows"]()
    words = rows_np.view(np.uint32) if rows_np.dtype == np.float32 else rows_np
    del rows_np
    store = Store(words, wl["dtype"], wl["T"], wl["B"], wl["residency"], dev)
    store.sharded = world > 1
    n, L = store.n, store.L
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def flush():
        # write a buffer larger than L2, then read it back so that the lines left in
        # L2 are clean (no write-back of the flush data charged to the next step)
        flush_buf.fill_(1)
        flush_buf.sum()

    link = measure_link(dev)
    hbm_copy_now = measure_hbm_copy(dev)
    launch_floor = measure_launch_floor(dev, flush)
    torch.cuda.empty_cache()

    # preprocessing stages (timed with CUDA events; raw input bytes per second)
    reps = 5
    meta_t, _ = time_stage(store.build_meta, reps, flush)
    comp_t, _ = time_stage(store.compress, reps, flush)
    torch.cuda.synchronize()
    assert int(store.status.item()) == 0
    st = store.stats()
    stored = store.stored_per_row()
    table_raw = n * store.raw_bytes

    # index batches (distinct per step, cycled)
    nb = 20
    host_batches = [torch.from_numpy(wl["index"](n, wl["batch"], k)).pin_memory()
                    for k in range(nb)]
    batches = [b.to(dev) for b in host_batches]
    out = torch.empty((wl["batch"], L), dtype=store.word_dtype, device=dev)
    gathered_stored = np.array([stored[b.numpy()].sum() for b in host_batches], dtype=np.int64)

    attempt = 0
    while True:
        per_step, clk = timed_gather(store, batches, out, steps, warmup, flush, barrier)
        attempt += 1
        if not clocks_rejected(clk) or attempt >= 2:
            break
    out_bytes = wl["batch"] * store.raw_bytes
    t_step, value = job_throughput(float(np.mean(per_step)), out_bytes, dist, dev)
    stored_per_step = float(np.mean([gathered_stored[k % nb] for k in range(steps)]))
    link_bytes = stored_per_step  # compressed bytes crossing the link per launch
    residency = wl["residency"]
    idx_key = "/uniform" if args.indices == "uniform" else ""
    rec = recorded_traffic(f"{args.workload}/{residency}{idx_key}") if not args.rows else None
    if residency == "host":
        achieved = link_bytes / t_step / 1e9
        peak = link["h2d_memcpy_gbs"]
        traffic = rec["sysmem_read_bytes"] if rec else None
        roofline = {"bound": "host_link", "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "traffic": traffic,
                    "traffic_kind": "ncu sysmem read bytes per launch (bytes that crossed the link; "
                                    "duplicate rows served from L1/L2 do not)",
                    "traffic_frac": (traffic / t_step / 1e9 / peak) if traffic else None,
                    "peak_source": "pinned host->device cudaMemcpyAsync, 1 GiB, best of 10, "
                                   "measured in this run",
                    "algorithmic_bytes_per_launch": link_bytes}
    else:
        alg = wl["batch"] * 8 + stored_per_step + out_bytes
        achieved = alg / t_step / 1e9
        traffic = (rec["dram_read_bytes"] + rec["dram_write_bytes"]) if rec else None
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved / hbm_peak, "traffic": traffic,
                    "peak_source": f"{hbm_peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                    "algorithmic_bytes_per_launch": alg}

    def want(leg):
        return (not args.quick) if legs is None else leg in legs

    extra = {}
    # HBM-resident gather of the same store
    if residency == "host" and want("hbm"):
        dstore = Store.__new__(Store)
        dstore.__dict__.update(store.__dict__)
        dstore.slots = store.slots.to(dev)
        dstore.residency = "device"
        per_step_h, clk_h = timed_gather(dstore, batches, out, max(50, steps // 4), warmup,
                                         flush, barrier)
        th = float(np.mean(per_step_h))
        alg = wl["batch"] * 8 + stored_per_step + out_bytes
        rec_d = recorded_traffic(f"{args.workload}/device{idx_key}") if not args.rows else None
        extra["hbm_resident"] = {
            "value": out_bytes / th / 1e9, "unit": "GB/s", "ms_per_step": th * 1e3,
            "roofline": {"bound": "hbm", "achieved": alg / th / 1e9, "peak": hbm_peak,
                         "unit": "GB/s", "frac": alg / th / 1e9 / hbm_peak,
                         "traffic": (rec_d["dram_read_bytes"] + rec_d["dram_write_bytes"])
                         if rec_d else None,
                         "peak_source": f"{hbm_peak_src} hbm_gbs",
                         "algorithmic_bytes_per_launch": alg},
            "clocks": clk_h}
        del dstore
    if want("e2e"):
        extra["e2e"] = run_e2e(store, host_batches, max(20, steps // 10), warmup, dev)
    if residency == "host" and want("e2e"):
        # bytes over the link per step: the rows the gather reads (the ncu-measured
        # link bytes when recorded, else the stored bytes), the index batch up,
        # the rows back down
        up = (rec["sysmem_read_bytes"] if rec else stored_per_step) + wl["batch"] * 8
        both = up + out_bytes
        t_e = extra["e2e"]["ms_per_step"] * 1e-3
        extra["e2e"]["roofline"] = {
            "bound": "host_link_both_directions", "achieved": both / t_e / 1e9,
            "peak": link["bidirectional_memcpy_gbs"], "unit": "GB/s",
            "frac": both / t_e / 1e9 / link["bidirectional_memcpy_gbs"],
            "link_bytes_per_step": both}
    # preprocessing stages with rows and slots in HBM
    if residency == "host" and want("stages"):
        dstore = Store.__new__(Store)
        dstore.__dict__.update(store.__dict__)
        dstore.rows = store.rows.to(dev)
        dstore.slots = torch.empty((n, store.slot_bytes), dtype=torch.uint8, device=dev)
        dstore.bitmask = torch.zeros_like(store.bitmask)
        dstore.row_bits = torch.zeros_like(store.row_bits)
        dstore.status = torch.zeros_like(store.status)
        mt, _ = time_stage(dstore.build_meta, reps, flush)
        ct, _ = time_stage(dstore.compress, reps, flush)
        sel_d = MaskSelect(dstore)
        sdt, _ = time_stage(sel_d.run, reps, flush)
        torch.cuda.synchronize()
        same = bool(torch.equal(dstore.bitmask, store.bitmask))
        comp_bytes = table_raw + float(stored.sum())
        extra["stages_hbm"] = {
            "build_meta": {"gbs_raw_in": table_raw / mt / 1e9, "ms": mt * 1e3,
                           "frac_of_hbm": table_raw / mt / 1e9 / hbm_peak},
            "compress": {"gbs_raw_in": table_raw / ct / 1e9, "ms": ct * 1e3,
                         "frac_of_hbm": comp_bytes / ct / 1e9 / hbm_peak,
                         "same_bitmask_as_host_run": same},
            "build_meta_select": {"gbs_raw_in": table_raw / sdt / 1e9, "ms": sdt * 1e3,
                                  "frac_of_hbm": 2 * table_raw / sdt / 1e9 / hbm_peak,
                                  "reads_rows": 2}}
        del dstore, sel_d
        torch.cuda.empty_cache()
    # before the mask-selection leg, which recompresses into the store's slots
    if want("dedup"):
        extra["dedup"] = dedup_leg(store, wl, batches, out, steps, warmup, flush, barrier,
                                   out_bytes, link, hbm_peak, dev)
    if want("select") or want("packed"):  # the packed store is made of the selected mask
        sstore, mask_select = mask_select_leg(store, wl, batches, out, steps, warmup, flush,
                                              barrier, reps, table_raw, out_bytes, residency,
                                              link, hbm_peak)
        if want("select"):
            extra["mask_select"] = mask_select
        if want("packed"):
            extra["packed"] = packed_leg(sstore, wl, batches, out, steps, warmup, flush,
                                         barrier, table_raw, out_bytes, link, hbm_peak, dev)
        del sstore
    # per-position tables are built for rows up to 16 KiB
    if store.raw_bytes <= 16384 and want("positions"):
        extra["positions"] = positions_leg(store, wl, batches, out, steps, warmup, flush,
                                           barrier, reps, table_raw, out_bytes, link,
                                           hbm_peak, dev)
    if args.workload == "gnn_dense" and want("offload"):
        extra["offload"] = offload_leg(dev)
    if args.workload == "dlrm_table" and want("dlrm26"):
        extra["dlrm_26_tables"] = dlrm_batched_leg(dev, flush, barrier, steps, warmup,
                                                   hbm_peak, n_tables=args.tables,
                                                   n_rows=args.rows or 1_000_000)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": f"u{8 * words.dtype.itemsize}",
        "data": "synthetic",
        "config": {"workload": wl["desc"], "rows": n, "row_elems": L, "T": wl["T"],
                   "block_elems": wl["B"], "batch": wl["batch"], "residency": residency,
                   "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write, then read)",
                   "parallelism": f"{world} independent replica(s)",
                   "meta_exchange": ("all-reduce of 32 bit counters + element count"
                                     if world > 1 else None)},
        "space_saving_pct": 100.0 * (1.0 - st.stored_bytes / st.raw_bytes),
        "space_saving_gathered_pct": 100.0 * (1.0 - stored_per_step / out_bytes),
        "bit_saving_pct": 100.0 * (1.0 - st.total_bits / (8.0 * st.raw_bytes)),
        "rows_compressed_pct": 100.0 * st.n_compressed / st.n_rows,
        "metadata_bytes": 16, "bitmask_bytes": 4 * ((n + 31) // 32),
        "meta": {"mask": f"{int(store.meta[0].item()) & 0xFFFFFFFF:#010x}",
                 "bitval": f"{int(store.meta[1].item()) & 0xFFFFFFFF:#010x}"},
        "roofline": roofline,
        "clocks": clk,
        "gpu_launches": steps,
        "stages": {
            "build_meta": {"gbs_raw_in": table_raw / meta_t / 1e9, "ms": meta_t * 1e3,
                           "residency": residency},
            "compress": {"gbs_raw_in": table_raw / comp_t / 1e9, "ms": comp_t * 1e3,
                         "residency": residency},
        },
        "link": link, "host_placement": host_placement(dev),
        "hbm_copy_gbs_this_run": hbm_copy_now,
        "launch_floor_us": {"value": launch_floor * 1e6,
                            "what": "CUDA-event time of a one-element kernel after the L2 "
                                    "flush, timed like a gather step"},
        "e2e": extra.pop("e2e", None),
    }
    line.update(extra)
    if residency == "host":
        line["stages"]["build_meta"]["frac_of_link"] = table_raw / meta_t / 1e9 / link[
            "h2d_memcpy_gbs"]
        line["stages"]["compress"]["link_bytes_gbs"] = (table_raw + float(stored.sum())) / \
            comp_t / 1e9
    else:
        line["stages"]["build_meta"]["frac_of_hbm"] = table_raw / meta_t / 1e9 / hbm_peak
        line["stages"]["compress"]["frac_of_hbm"] = (table_raw + float(stored.sum())) / \
            comp_t / 1e9 / hbm_peak
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"], line["cpu_baseline_all_cores"] = oracle_sample(wl)
    if (args.workload == "gnn_dense" and want("configs") and not args.no_configs and
            not args.rows and residency == "host"):
        # every configuration, summarised in one short object at the end of the line
        distinct = float(np.mean([stored[np.unique(hb.numpy())].sum()
                                  for hb in host_batches]))
        main_cfg = {
            "rows": n, "save_pct": _sig(line["space_saving_pct"]),
            "meta_GBs": _sig(table_raw / meta_t / 1e9),
            "comp_host_GBs": _sig(table_raw / comp_t / 1e9),
            "host": gather_entry(t_step, wl["batch"], store.raw_bytes, stored_per_step, distinct,
                                 "host", link["h2d_memcpy_gbs"], hbm_peak)}
        if roofline.get("traffic_frac"):
            main_cfg["host"]["link_frac_ncu"] = _sig(roofline["traffic_frac"])
        if "stages_hbm" in line:
            main_cfg["comp_GBs"] = _sig(line["stages_hbm"]["compress"]["gbs_raw_in"])
            main_cfg["comp_frac"] = _sig(line["stages_hbm"]["compress"]["frac_of_hbm"])
        if "hbm_resident" in line:
            h = line["hbm_resident"]
            main_cfg["hbm"] = {"ms": _sig(h["ms_per_step"]), "GBs": _sig(h["value"]),
                               "frac": _sig(h["roofline"]["frac"]),
                               "alg_MB": _sig(h["roofline"]["algorithmic_bytes_per_launch"] / 1e6)}
        del store
        torch.cuda.empty_cache()
        with ClockSampler(torch.cuda.current_device()) as clk_c:
            cfgs = configs_leg(dev, flush, hbm_peak, link, main_cfg)
        cfgs["clocks"] = clk_c.summary()
        line["configs"] = cfgs
    if rank == 0:
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
