"""Benchmark of the paged-KV input-preparation path on one GB300.

One step = one pass of the whole hot path over one batch: the fused
prepare_batch (sort, query_start_loc, positions, input_ids, seq_lens, per-group
slot_mapping and block-table gather) followed by the KV store of every layer of
every group.  The headline workload is the large step (4096 requests, 16384
scheduled tokens, block size 32, W 4096, fp8 KV lines of 1 KiB, 80 layers each
with its own 28,610-block cache), the largest single-GPU configuration.

  value     scheduled tokens/s with every input already in HBM (device-side
            schedule, K/V in device memory), CUDA events on the launching
            stream;
  e2e       the same metric through the host-buffer API: the schedule from host
            arrays (pkv_prepare_batch, which stages and copies it), the K/V
            lines of every layer copied from pinned host memory, and the
            prepared query_start_loc/seq_lens read back, all inside the timed
            region (wall clock);
  roofline  the dominant kernel (the multi-layer KV store) against the measured
            HBM copy bandwidth;
  cpu_baseline  the CPU oracle on a bounded sample of the same workload.

``--impl reference`` times the CPU oracle alone on the same workload and
prints its own line.  Multi-process runs (torchrun, N > 1) are independent
replicas: the path has no cross-GPU exchange.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "scheduled tokens/s through prepare_batch+kv_cache_write; KV-write HBM GB/s vs peak"
UNIT = "tokens/s"
L2_BYTES = 129 << 20


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------
def prepare_bytes(wl) -> int:
    """What the fused prepare must move: per request the row id, count and
    completed_tokens read and index_mapping, query_start_loc, seq_lens written
    (24 B); per token the token id read and position + input_id written (12 B);
    per group per token the block-table entry read and the int64 slot written
    (12 B), and per group per request the W-entry table row read and written
    (8 W B)."""
    n, T = wl.num_scheduled_requests, wl.total_tokens
    b = 24 * n + 12 * T
    for g in wl.groups:
        b += 12 * T + 8 * n * g.max_blocks_per_req
    return b


def prepare_bytes_live(wl) -> int:
    """The same with only the live block-table entries gathered (per group per
    request ceil(seq_len / bs) entries read and written)."""
    reqs = wl.requests()
    n, T = wl.num_scheduled_requests, wl.total_tokens
    b = 24 * n + 12 * T
    for g in wl.groups:
        live = 0
        for h, c in wl.schedule:
            seq = reqs[h].num_computed + c
            live += min(-(-seq // g.block_size), g.max_blocks_per_req)
        b += 12 * T + 8 * live
    return b


def paged_entries(wl, group) -> int:
    """Live block-table entries of the step in one group: sum ceil(seq_len / bs)."""
    reqs = wl.requests()
    g = wl.groups[group]
    return sum(min(-(-(reqs[h].num_computed + c) // g.block_size), g.max_blocks_per_req)
               for h, c in wl.schedule)


def paged_bytes(wl, group) -> int:
    """What the paged (CSR) table build must move for one group: per request
    index_mapping and seq_lens read, seq_lens read again for last_page_len,
    kv_indptr and last_page_len written (20 B); per live entry the table entry
    read and written (8 B)."""
    return 20 * wl.num_scheduled_requests + 4 + 8 * paged_entries(wl, group)


def kv_bytes_per_layer_group(wl) -> int:
    """K and V line read and written per token, plus the int64 slot."""
    T = wl.total_tokens
    return 4 * wl.line_bytes * T + 8 * T


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class NvmlSampler:
    """SM clock, clock-event reasons and power read from the driver's NVML
    library every 2 ms on a thread of this process (read-only queries), so
    that even a timed region of a few tens of milliseconds holds samples;
    nvidia-smi (below) samples every 50 ms at best."""

    # reason bits of NVML's clock-event reason mask (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch, device: int):
        import ctypes
        self.C = ctypes
        self.rows = []
        self.stop_flag = threading.Event()
        self.thread = None
        self.lib = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(device)
            rc = -1
            if hasattr(props, "pci_bus_id"):
                bus = (f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:"
                       f"{props.pci_device_id:02X}.0").encode()
                rc = lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus),
                                                          ctypes.byref(self.handle))
            if rc != 0:
                rc = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(device),
                                                       ctypes.byref(self.handle))
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
            mx = ctypes.c_uint(0)   # clock type 1 below and in _run: the SM clock
            if (rc != 0 or self.reasons_fn is None
                    or lib.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) != 0):
                lib.nvmlShutdown()
                return
            self.max_mhz = mx.value
            self.lib = lib
        except (OSError, AttributeError):
            self.lib = None

    def start(self):
        if self.lib is None:
            return
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def _run(self):
        C, lib, h = self.C, self.lib, self.handle
        mhz, reasons, mw = C.c_uint(0), C.c_ulonglong(0), C.c_uint(0)
        while not self.stop_flag.is_set():
            t = time.time()
            if (lib.nvmlDeviceGetClockInfo(h, 1, C.byref(mhz)) == 0
                    and self.reasons_fn(h, C.byref(reasons)) == 0):
                if lib.nvmlDeviceGetPowerUsage(h, C.byref(mw)) != 0:
                    mw.value = 0
                self.rows.append((t, mhz.value, reasons.value, mw.value / 1e3))
            time.sleep(0.002)

    def stop(self):
        if self.thread is not None:
            self.stop_flag.set()
            self.thread.join(timeout=5)
        if self.lib is not None:
            self.lib.nvmlShutdown()
            self.lib = None

    def summary(self, t0, t1):
        rows = [r for r in self.rows if t0 <= r[0] <= t1]
        if not rows:
            return None
        reasons = set()
        for _, _, bits, _ in rows:
            reasons.update(name for bit, name in self.REASONS.items() if bits & bit)
        return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(r[1] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": round(max(r[3] for r in rows), 1)}


class ClockSampler:
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(1.0)   # let nvidia-smi start sampling before the timed region

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    @staticmethod
    def sample_time(field, fallback):
        """nvidia-smi's own timestamp (local time, ms), else when the line was
        read (a pipe may deliver lines late, in batches)."""
        try:
            day, ms = field.rsplit(".", 1)
            return time.mktime(time.strptime(day, "%Y/%m/%d %H:%M:%S")) + int(ms) / 1e3
        except (ValueError, OverflowError):
            return fallback

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            ts = self.sample_time(parts[0], ts)
            if not (t0 <= ts <= t1 + 0.05):
                continue
            try:
                rows.append(dict(sm=float(parts[2]), max=float(parts[3]),
                                 power=float(parts[4]) if parts[4] not in ("[N/A]", "") else 0.0,
                                 hw=parts[6], hwt=parts[7], swt=parts[8], pcap=parts[9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                    "samples": 0}
        reasons = set()
        for r in rows:
            if r["hw"].lower() == "active":
                reasons.add("hw_slowdown")
            if r["hwt"].lower() == "active":
                reasons.add("hw_thermal_slowdown")
            if r["swt"].lower() == "active":
                reasons.add("sw_thermal_slowdown")
            if r["pcap"].lower() == "active":
                reasons.add("sw_power_cap")
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


# ---------------------------------------------------------------------------
# traffic figure committed from an ncu capture
# ---------------------------------------------------------------------------
def kernel_source_digest() -> str:
    h = hashlib.sha256()
    for name in ("pkv_kvwrite.cu", "pkv_common.cuh", "pkv_async.cuh"):
        with open(os.path.join(ROOT, "paged_kv_prep_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(units_per_launch: float):
    """dram bytes per launch of the KV-store kernel from the committed ncu
    summary, scaled to this launch's tokens x layers, or None if the summary is
    missing or was taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", "kv_write_large_step.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_src = re.search(r"kernel source digest:\s*`?([0-9a-f]+)", text)
    m_b = re.search(r"dram bytes per unit:\s*([0-9.eE+]+)", text)
    if not m_src or not m_b or m_src.group(1) != kernel_source_digest():
        return None
    return float(m_b.group(1)) * units_per_launch


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------
class DeviceStep:
    """All inputs resident in HBM: the schedule as device arrays, one K/V source
    and one K/V cache pair per layer per group."""

    def __init__(self, wl, torch, pkv, workloads, multi_layer=True):
        self.wl = wl
        self.torch = torch
        self.pkv = pkv
        self.multi_layer = multi_layer
        groups = workloads.group_tuples(wl)
        t = time.time()
        self.st = pkv.State(wl.max_reqs, wl.max_model_len, groups)
        self.rows_map = workloads.apply_ops(self.st, wl)
        self.rows, self.ns = workloads.schedule_arrays(wl, self.rows_map)
        self.T = int(self.ns.sum())
        self.n = len(self.ns)
        dev = "cuda"
        self.d_rows = torch.tensor(self.rows, dtype=torch.int32, device=dev)
        self.d_ns = torch.tensor(self.ns, dtype=torch.int32, device=dev)
        self.batch = self.st.alloc_batch(self.n, self.T)
        line = wl.line_bytes
        self.ks, self.vs, self.kcs, self.vcs = [], [], [], []
        for g, spec in enumerate(wl.groups):
            num_slots = spec.num_blocks * spec.block_size
            ks, vs, kcs, vcs = [], [], [], []
            for layer in range(wl.num_layers):
                k, v = workloads.kv_sources(wl, layer, g, device=dev)
                ks.append(k)
                vs.append(v)
                kcs.append(torch.empty(num_slots, line, dtype=torch.uint8, device=dev))
                vcs.append(torch.empty(num_slots, line, dtype=torch.uint8, device=dev))
            self.ks.append(ks)
            self.vs.append(vs)
            self.kcs.append(kcs)
            self.vcs.append(vcs)
        # the per-step calls, marshalled once (the same buffers every step)
        # the schedule arrays are written once, here, never by a step's kernels
        self.prep_call = pkv.PrepareDeviceCall(self.st, self.d_rows, self.d_ns, self.T, self.batch,
                                               flags=pkv.SCHEDULE_SETTLED)
        self.prep_call_full = self.prep_call
        self.prep_call_live = pkv.PrepareDeviceCall(
            self.st, self.d_rows, self.d_ns, self.T, self.batch,
            flags=pkv.LIVE_TABLES | pkv.SCHEDULE_SETTLED)
        # every (layer, group) item of the step in one launch
        items = [(self.ks[g][layer], self.vs[g][layer], self.kcs[g][layer], self.vcs[g][layer],
                  self.batch.slot_mapping[g])
                 for g in range(len(wl.groups)) for layer in range(wl.num_layers)]
        self.step_call = pkv.KvStepCall(items)
        # optional paged (CSR) table of group 0 between prepare and store
        self.paged_out = None
        self.paged = False
        torch.cuda.synchronize()
        log(f"[bench] {wl.name}: n={self.n} T={self.T} setup {time.time() - t:.1f}s, "
            f"{torch.cuda.memory_allocated() / 2**30:.1f} GiB on device")

    def launches_per_step(self):
        items = self.wl.num_layers * len(self.wl.groups)
        return 1 + (-(-items // 128) if self.multi_layer else items)

    def prepare(self, stream):
        self.prep_call(stream.cuda_stream)

    def store(self, stream):
        pkv = self.pkv
        if self.multi_layer:
            self.step_call(stream.cuda_stream)
            return
        for g in range(len(self.wl.groups)):
            for layer in range(self.wl.num_layers):
                pkv.kv_cache_write(self.ks[g][layer], self.vs[g][layer], self.kcs[g][layer],
                                   self.vcs[g][layer], self.batch.slot_mapping[g],
                                   stream=stream)

    def paged_tables(self, stream):
        if self.paged_out is None:
            cap = self.n * self.wl.groups[0].max_blocks_per_req
            self.paged_out = self.st.kv_indices(0, self.batch.index_mapping,
                                                self.batch.seq_lens, capacity=cap)
        self.st.kv_indices(0, self.batch.index_mapping, self.batch.seq_lens,
                           capacity=self.paged_out[1].numel(), out=self.paged_out,
                           stream=stream)

    def step(self, stream):
        self.prepare(stream)
        if self.paged:
            self.paged_tables(stream)
        self.store(stream)


def time_device(ds, steps, warmup, torch, barrier):
    """Whole-step time plus per-kernel durations (events on the launching
    stream around each launch)."""
    s = torch.cuda.current_stream()
    for _ in range(warmup):
        ds.step(s)
    torch.cuda.synchronize()
    barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    ev_p = [torch.cuda.Event(enable_timing=True) for _ in range(steps)] if ds.paged else None
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    start.record(s)
    for k in range(steps):
        a, b, c = ev[k]
        a.record(s)
        ds.prepare(s)
        b.record(s)
        if ds.paged:
            ds.paged_tables(s)
            ev_p[k].record(s)
        ds.store(s)
        c.record(s)
    end.record(s)
    end.synchronize()
    t1 = time.time()
    torch.cuda.synchronize()
    barrier()
    total_ms = start.elapsed_time(end)
    prep = [a.elapsed_time(b) for a, b, _ in ev]
    if ds.paged:
        ds.paged_ms = [ev[k][1].elapsed_time(ev_p[k]) for k in range(steps)]
        store = [ev_p[k].elapsed_time(ev[k][2]) for k in range(steps)]
    else:
        store = [b.elapsed_time(c) for _, b, c in ev]
    return total_ms, prep, store, (t0, t1)


def time_steps(ds, steps, warmup, torch, barrier):
    """Steps back to back with no event between the kernels (PDL lets each
    launch overlap the kernel before it): total milliseconds."""
    s = torch.cuda.current_stream()
    for _ in range(warmup):
        ds.step(s)
    torch.cuda.synchronize()
    barrier()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(s)
    for _ in range(steps):
        ds.step(s)
    end.record(s)
    end.synchronize()
    barrier()
    return start.elapsed_time(end)


def time_e2e(wl, ds, steps, warmup, torch):
    """Through the host-buffer API: host schedule -> pkv_prepare_batch (staged
    and copied by the library), every layer's K/V lines copied from pinned
    host memory, then the prepared query_start_loc and seq_lens read back."""
    pkv = ds.pkv
    s = torch.cuda.current_stream()
    host_k = [[t.cpu().pin_memory() for t in ks] for ks in ds.ks]
    host_v = [[t.cpu().pin_memory() for t in vs] for vs in ds.vs]
    out_qsl = torch.empty(ds.n + 1, dtype=torch.int32).pin_memory()
    out_sl = torch.empty(ds.n, dtype=torch.int32).pin_memory()
    h2d = 8 * ds.n + sum(t.numel() for ks in host_k for t in ks) + \
        sum(t.numel() for vs in host_v for t in vs)
    d2h = 4 * (ds.n + 1) + 4 * ds.n

    # the KV store reading each layer's K/V straight from pinned host memory
    # (mapped into the device's address space; the bytes cross NVLink-C2C
    # inside the kernel instead of through separate copies)
    items = [(host_k[g][layer], host_v[g][layer], ds.kcs[g][layer], ds.vcs[g][layer],
              ds.batch.slot_mapping[g])
             for g in range(len(wl.groups)) for layer in range(wl.num_layers)]
    direct_call = ds.pkv.KvStepCall(items)

    def staged():
        ds.st.prepare_batch(ds.rows, ds.ns, out=ds.batch, stream=s)
        for g in range(len(wl.groups)):
            for layer in range(wl.num_layers):
                ds.ks[g][layer].copy_(host_k[g][layer], non_blocking=True)
                ds.vs[g][layer].copy_(host_v[g][layer], non_blocking=True)
        ds.step_call(s.cuda_stream)
        out_qsl.copy_(ds.batch.query_start_loc, non_blocking=True)
        out_sl.copy_(ds.batch.seq_lens, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    def direct():
        ds.st.prepare_batch(ds.rows, ds.ns, out=ds.batch, stream=s)
        direct_call(s.cuda_stream)
        out_qsl.copy_(ds.batch.query_start_loc, non_blocking=True)
        out_sl.copy_(ds.batch.seq_lens, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    # for comparison only (not an end-to-end figure: the K/V lines are not
    # copied): the host schedule and the read-back, K/V already on the device
    host_call = pkv.PrepareHostCall(ds.st, ds.batch)

    def kv_on_device():
        host_call(ds.rows, ds.ns, stream=s.cuda_stream)
        ds.step_call(s.cuda_stream)
        out_qsl.copy_(ds.batch.query_start_loc, non_blocking=True)
        out_sl.copy_(ds.batch.seq_lens, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    def wall(one):
        for _ in range(warmup):
            one()
        torch.cuda.synchronize()
        t = time.perf_counter()
        for _ in range(steps):
            one()
        dt = time.perf_counter() - t
        if int(out_qsl[-1]) != ds.T:
            raise RuntimeError("e2e: query_start_loc[n] != T")
        return dt

    res = {name: wall(one)
           for name, one in (("staged_copies", staged), ("kernel_reads_pinned_host", direct))}
    return res, h2d, d2h, wall(kv_on_device)


def other_configs(torch, pkv, workloads, steps=300, warmup=10):
    """The medium configurations (one layer per step): tokens/s from steps
    back to back, and each kernel's fraction of the measured peak from CUDA
    events around its launches (a separate run of the same steps: the events
    between kernels add their own cost and stop PDL's launch overlap)."""
    peak, _ = measured_peaks()
    res = {}
    for name in ("mixed_prefill", "two_groups"):
        wl = workloads.build(name, seed=0)
        ds = DeviceStep(wl, torch, pkv, workloads)
        total_ms, prep, store, _ = time_device(ds, steps, warmup, torch, lambda: None)
        plain_ms = time_steps(ds, steps, warmup, torch, lambda: None)
        kv_b = kv_bytes_per_layer_group(wl) * wl.num_layers * len(wl.groups)
        p_us, s_us = statistics.mean(prep) * 1e3, statistics.mean(store) * 1e3
        res[name] = {"n": ds.n, "T": ds.T, "groups": len(wl.groups),
                     "tokens_per_s": ds.T * steps / (plain_ms / 1e3),
                     "us_per_step": round(plain_ms * 1e3 / steps, 2),
                     "us_per_step_with_kernel_events": round(total_ms * 1e3 / steps, 2),
                     "prepare_us": round(p_us, 2),
                     "prepare_frac": round(prepare_bytes(wl) / (p_us * 1e-6) / 1e9 / peak, 4),
                     "kv_store_us": round(s_us, 2),
                     "kv_store_frac": round(kv_b / (s_us * 1e-6) / 1e9 / peak, 4)}
        ds.st.close()
        del ds
        torch.cuda.empty_cache()
    return res


def apply_latency(torch, pkv, workloads, steps=100):
    """Host wall time of applying one decode step's scheduler output to the
    state (256 running requests append a sampled token, and a block when they
    cross a block boundary; 4 finish and 4 arrive): one call per request
    against one pkv_apply_step (from Python lists, and from the same output
    already packed as int32 CSR arrays, as an engine would hold it),
    synchronised after every step."""
    import numpy as np

    res = {}
    def packed(fin, new, cached, G):
        def csr(lists):
            off = np.zeros(len(lists) + 1, np.int32)
            off[1:] = np.cumsum([len(x) for x in lists])
            flat = (np.concatenate([np.asarray(x, np.int32) for x in lists])
                    if off[-1] else np.zeros(0, np.int32))
            return off, flat
        nt = csr([x[0] for x in new])
        ct = csr([x[1] for x in cached])
        nb = [csr([x[2][g] for x in new]) for g in range(G)]
        cb = [csr([x[3][g] for x in cached]) for g in range(G)]
        return (np.asarray(fin, np.int32), nt[0], nt[1], np.array([x[1] for x in new], np.int32),
                [b[0] for b in nb], [b[1] for b in nb], np.array([x[0] for x in cached], np.int32),
                ct[0], ct[1], np.array([x[2] for x in cached], np.int32),
                [b[0] for b in cb], [b[1] for b in cb])

    for mode in ("per_request_calls", "apply_step", "apply_step_arrays"):
        wl = workloads.decode_heavy(seed=3, max_ctx=4096)
        wl.max_model_len = 8192
        for g in wl.groups:
            g.max_blocks_per_req = 512
        st = pkv.State(wl.max_reqs + 8, wl.max_model_len, workloads.group_tuples(wl))
        rows = list(workloads.apply_ops(st, wl).values())
        rng = np.random.default_rng(0)
        ntok = {r: st.row_info(r)["n_tokens"] for r in rows}
        nxt = 0
        s = torch.cuda.current_stream()
        times = []
        for step in range(steps):
            fin = rows[:4]
            rows = rows[4:]
            new = [(rng.integers(0, 128000, 64), 0, [np.arange(4, dtype=np.int32) + nxt])
                   for _ in range(4)]
            nxt = (nxt + 16) % 100000
            cached = []
            for r in rows:
                blocks = [np.array([(nxt + r) % 100000], np.int32)] if ntok[r] % 16 == 0 else \
                    [np.zeros(0, np.int32)]
                cached.append((r, [int(rng.integers(0, 128000))], ntok[r], blocks))
            args = packed(fin, new, cached, len(wl.groups)) if mode == "apply_step_arrays" else None
            t = time.perf_counter()
            if mode == "apply_step_arrays":
                got = st.apply_step_arrays(*args, stream=s).tolist()
            elif mode == "apply_step":
                got = st.apply_step(fin, new, cached, stream=s)
            else:
                for r in fin:
                    st.remove_request(r, stream=s)
                got = [st.add_request(tk, nc, b, stream=s) for tk, nc, b in new]
                for r, tk, nc, b in cached:
                    st.update_request(r, b, tk, nc, stream=s)
            s.synchronize()
            times.append((time.perf_counter() - t) * 1e6)
            for r, tk, nc, b in cached:
                ntok[r] += 1
            for r in got:
                ntok[r] = 64
            rows = rows + got
        st.close()
        res[mode] = round(statistics.median(times[5:]), 1)
    res["requests_per_step"] = 256
    return res


def prefix_cache_bench(torch, pkv, workloads, reps=20):
    """Prefix-cache keys of every full block of the large step's requests
    (block size 32, all known tokens) and a match of all of them against an
    index holding the first half of the requests' blocks."""
    peak, _ = measured_peaks()
    wl = workloads.large_step(seed=0, num_layers=1, pool=28610)
    groups = workloads.group_tuples(wl)
    st = pkv.State(wl.max_reqs, wl.max_model_len, groups)
    rows = list(workloads.apply_ops(st, wl).values())
    bs = wl.groups[0].block_size
    s = torch.cuda.current_stream()
    off, keys = st.block_keys(rows, bs)
    tokens = sum(st.row_info(r)["n_tokens"] for r in rows)
    hashed = int(off[-1]) * bs
    rows_np = np.array(rows, np.int32)
    off_np = np.zeros(len(rows) + 1, np.int32)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize()
    ev[0].record(s)
    for _ in range(reps):
        st.block_keys_into(rows_np, bs, off_np, keys, stream=s.cuda_stream)
    ev[1].record(s)
    ev[1].synchronize()
    keys_us = ev[0].elapsed_time(ev[1]) * 1e3 / reps
    half = int(off[len(rows) // 2])
    pc = pkv.PrefixCache(1 << 22)
    pc.insert(keys[:half].contiguous(),
              torch.arange(half, dtype=torch.int32, device="cuda"))
    d_off = torch.tensor(off, dtype=torch.int32, device="cuda")
    caps = torch.tensor([(st.row_info(r)["n_tokens"] - 1) // bs for r in rows],
                        dtype=torch.int32, device="cuda")
    hits_t = torch.empty(len(rows), dtype=torch.int32, device="cuda")
    ids_t = torch.empty(int(off[-1]), dtype=torch.int32, device="cuda")
    pc.match_into(keys, d_off, caps, hits_t, ids_t)
    torch.cuda.synchronize()
    ev[0].record(s)
    for _ in range(reps):
        pc.match_into(keys, d_off, caps, hits_t, ids_t, stream=s.cuda_stream)
    ev[1].record(s)
    ev[1].synchronize()
    match_us = ev[0].elapsed_time(ev[1]) * 1e3 / reps
    hits, _ = pc.match(keys, d_off, caps)
    res = {"requests": len(rows), "blocks": int(off[-1]), "block_size": bs,
           "keys_us": round(keys_us, 1),
           "keys_tokens_per_s": hashed / (keys_us * 1e-6),
           "keys_hbm_frac": round(hashed * 4 / (keys_us * 1e-6) / 1e9 / peak, 4),
           "match_us": round(match_us, 1),
           "matched_blocks": int(hits.sum().item()), "tokens_known": tokens}
    pc.close()
    st.close()
    torch.cuda.empty_cache()
    return res


def allocate_bench(torch, pkv, workloads, reps=50):
    """allocate_slots for the large step's 4096 requests, each holding the
    blocks of its history only: the first call hands out every block the
    step writes; later calls find nothing missing.  Every call runs the
    admission and the id moves on the GPU and waits for the result; `gpu_us`
    is the stream's time from before the staging copy to after the result
    copy (CUDA events on the call's stream), `wall_us` the host time."""
    import numpy as np

    wl = workloads.large_step(seed=0, num_layers=1)
    spec = wl.groups[0]
    reqs = wl.requests()
    st = pkv.State(wl.max_reqs, wl.max_model_len, workloads.group_tuples(wl))
    rows, ns, used = [], [], set()
    for h, c in wl.schedule:
        r = reqs[h]
        held = r.blocks[0][: -(-r.num_computed // spec.block_size)]
        used.update(int(b) for b in held)
        rows.append(st.add_request(r.token_ids, r.num_computed, [held]))
        ns.append(c)
    free = np.array([b for b in range(spec.num_blocks) if b not in used], np.int32)
    st.pool_reset(0, free)
    rows_np, ns_np = np.array(rows, np.int32), np.array(ns, np.int32)
    s = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def one():
        torch.cuda.synchronize()
        a.record(s)
        t = time.perf_counter()
        res = st.allocate_slots(rows_np, ns_np, stream=s)
        wall = (time.perf_counter() - t) * 1e6
        b.record(s)
        b.synchronize()
        return res, a.elapsed_time(b) * 1e3, wall

    (adm, nb), first_gpu, first_wall = one()
    gpu, wall = [], []
    for _ in range(reps):
        _, g_us, w_us = one()
        gpu.append(g_us)
        wall.append(w_us)
    st.close()
    return {"requests": len(rows), "admitted": int(adm), "new_blocks": int(nb.sum()),
            "first_call": {"gpu_us": round(first_gpu, 1), "wall_us": round(first_wall, 1)},
            "no_blocks_missing": {"gpu_us_median": round(statistics.median(gpu), 1),
                                  "wall_us_median": round(statistics.median(wall), 1)},
            "where": "admission and id moves on the GPU (plan, pop and push kernels); "
                     "the host validates, stages and copies the result back"}


def latency_small(torch, pkv, workloads, iters=200):
    """Step latency of the launch-bound small batches (prepare + one layer's
    KV store): GPU time, host wall time through the host-buffer API, and the
    device path replayed from a CUDA graph."""
    res = {}
    for name in ("tiny", "decode_heavy"):
        wl = workloads.build(name, seed=0)
        ds = DeviceStep(wl, torch, pkv, workloads)
        s = torch.cuda.current_stream()
        for _ in range(10):
            ds.step(s)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(s)
        for _ in range(iters):
            ds.step(s)
        b.record(s)
        b.synchronize()
        gpu_us = a.elapsed_time(b) * 1000 / iters
        # host-buffer API, synchronised every step: the output buffers
        # marshalled once (PrepareHostCall), the host schedule passed each step
        host_call = pkv.PrepareHostCall(ds.st, ds.batch)
        sh = s.cuda_stream
        wall = []
        for _ in range(iters):
            t = time.perf_counter()
            host_call(ds.rows, ds.ns, stream=sh)
            ds.store(s)
            s.synchronize()
            wall.append((time.perf_counter() - t) * 1e6)
        # CUDA graph of the device-schedule path
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream()
        cs.wait_stream(s)
        with torch.cuda.stream(cs):
            ds.step(cs)
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=cs):
                ds.step(torch.cuda.current_stream())
        torch.cuda.synchronize()
        gw = []
        for _ in range(iters):
            t = time.perf_counter()
            g.replay()
            torch.cuda.current_stream().synchronize()
            gw.append((time.perf_counter() - t) * 1e6)
        res[name] = {"n": ds.n, "T": ds.T, "gpu_us_per_step": round(gpu_us, 2),
                     "host_api_wall_us_median": round(statistics.median(wall), 1),
                     "graph_replay_wall_us_median": round(statistics.median(gw), 1)}
        ds.st.close()
        del ds, g
        torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# CPU oracle timing
# ---------------------------------------------------------------------------
class OracleStep:
    """The oracle's prepare on the full batch plus its KV store for `layers`
    layers of every group (all of them by default), observed, not scaled.
    Host memory holds two layers' caches and sources per group; the layers of
    a step cycle over them, so each layer's store moves the same bytes into a
    cache of the full per-layer size."""

    def __init__(self, wl, layers=None):
        import oracle
        import pkv_workloads as workloads

        self.oracle = oracle
        self.wl = wl
        self.orc = oracle.OracleState(wl.max_reqs, wl.max_model_len,
                                      workloads.group_tuples(wl))
        self.rows_map = workloads.apply_ops(self.orc, wl)
        self.rows, self.ns = workloads.schedule_arrays(wl, self.rows_map)
        self.layers = wl.num_layers if layers is None else max(1, min(layers, wl.num_layers))
        self.held = min(2, self.layers)
        ref = self.orc.prepare_batch(self.rows, self.ns)
        self.slots = ref["slot_mapping"]
        rng = np.random.default_rng(0)
        T, line = wl.total_tokens, wl.line_bytes
        self.src = [(rng.integers(0, 256, (T, line), dtype=np.uint8),
                     rng.integers(0, 256, (T, line), dtype=np.uint8))
                    for _ in range(self.held)]
        self.caches = []
        for g, spec in enumerate(wl.groups):
            ns = spec.num_blocks * spec.block_size
            self.caches.append([(np.zeros((ns, line), np.uint8), np.zeros((ns, line), np.uint8))
                                for _ in range(self.held)])
        for per_group in self.caches:          # touch every page before timing
            for kc, vc in per_group:
                kc.fill(1)
                vc.fill(1)

    def run(self):
        """One step: returns (prepare seconds, store seconds for its layers)."""
        t = time.perf_counter()
        self.orc.prepare_batch(self.rows, self.ns)
        tp = time.perf_counter() - t
        t = time.perf_counter()
        for layer in range(self.layers):
            k, v = self.src[layer % self.held]
            for g in range(len(self.wl.groups)):
                kc, vc = self.caches[g][layer % self.held]
                self.oracle.kv_write(k, v, kc, vc, self.slots[g])
        ts = time.perf_counter() - t
        return tp, ts

    def step_seconds(self, tp, ts):
        """The whole step's time: observed when every layer ran, else the
        sampled layers' store time scaled to all of them."""
        return tp + ts * self.wl.num_layers / self.layers

    def sample_text(self):
        what = (f"the full {self.wl.name} batch (n={len(self.ns)}, T={int(self.ns.sum())})")
        if self.layers == self.wl.num_layers:
            store = (f"its KV store of all {self.wl.num_layers} layers per group (two host "
                     f"cache pairs of the full per-layer size, used in turn), every step observed")
        else:
            store = (f"its KV store of {self.layers} of {self.wl.num_layers} layers per group, "
                     f"the store time scaled to all layers")
        return f"oracle prepare_batch on {what} plus {store}; single thread"


def cpu_baseline(wl, budget_s=12.0):
    os_ = OracleStep(wl)
    steps = []
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s or len(steps) < 3:
        steps.append(os_.step_seconds(*os_.run()))
    step = statistics.median(steps)
    return {"value": wl.total_tokens / step, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": os_.sample_text() + f"; median of {len(steps)} steps",
            "ms_per_step": step * 1e3, "host": host_info()}


def host_info():
    """Core count and CPU model: /proc/cpuinfo's model name (x86) or CPU part
    number (Arm), and lscpu's model name where lscpu is installed (it names
    the Arm part, e.g. Neoverse-V2 for part 0xd4f)."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part", "hardware")):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    name = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                name = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    info = {"nproc": os.cpu_count(), "machine": platform.machine(), "cpu": model}
    if name and name != model:
        info["cpu_model"] = name
    return info


# ---------------------------------------------------------------------------
def workload_config(wl, world):
    """The `config` object of both arms' lines (the same workload)."""
    kv = kv_bytes_per_layer_group(wl) * wl.num_layers * len(wl.groups)
    return {"workload": wl.name, "requests": len(wl.schedule),
            "scheduled_tokens": wl.total_tokens,
            "block_size": wl.groups[0].block_size,
            "max_blocks_per_req": wl.groups[0].max_blocks_per_req,
            "layers": wl.num_layers, "kv_groups": len(wl.groups),
            "kv_dtype": wl.kv_dtype, "line_bytes": wl.line_bytes,
            "pool_blocks_per_layer": wl.groups[0].num_blocks,
            "l2": (f"inputs larger than L2: each step streams {kv / 2**30:.1f} GiB of K/V "
                   f"through the {L2_BYTES >> 20} MiB L2") if kv > L2_BYTES else
                  (f"inputs smaller than L2 ({kv / 2**20:.0f} MiB of K/V per step): no flush, "
                   "a parity and latency case, not the headline"),
            "parallelism": "replicas" if world > 1 else "single GPU"}


def max_over_ranks(ms: float, dist) -> float:
    """The slowest rank's time (every rank gets it); ms itself on one rank."""
    if not dist:
        return ms
    import torch

    t = torch.tensor([ms], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0])


def whole_job_value(world: int, tokens_per_step: int, steps: int, ms: float) -> float:
    """Scheduled tokens per second over all replicas: every rank runs the
    same step on its own GPU (weak scaling), timed by the slowest rank."""
    return world * tokens_per_step * steps / (ms / 1e3)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        return world, rank, local, dist
    return 1, 0, 0, None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="large_step")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--layers", type=int, default=None,
                    help="override the workload's layer count (small profiling cases)")
    ap.add_argument("--pool-blocks", type=int, default=None,
                    help="override the large step's per-layer pool (small profiling cases)")
    ap.add_argument("--line-bytes", type=int, default=None,
                    help="override the K/V line size (one head; a multiple of 16): small "
                         "profiling cases of the batch build, whose work does not depend on it")
    ap.add_argument("--per-layer-calls", action="store_true",
                    help="time one kv_cache_write call per layer instead of one launch")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-latency", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world, rank, local, dist = dist_setup()
    import pkv_workloads as workloads

    kw = {}
    if args.pool_blocks is not None:
        if args.workload != "large_step":
            ap.error("--pool-blocks applies to the large step only")
        kw["pool"] = args.pool_blocks
    wl = workloads.build(args.workload, seed=args.seed, **kw)
    if args.layers is not None:
        wl.num_layers = args.layers
    if args.line_bytes is not None:
        if args.line_bytes < 16 or args.line_bytes % 16 or args.line_bytes % wl.elem_size:
            ap.error("--line-bytes must be a positive multiple of 16")
        wl.num_heads, wl.head_dim = 1, args.line_bytes // wl.elem_size

    if args.impl == "reference":
        if rank != 0:
            return
        # every layer each step when warm-up plus K steps fit in about three
        # minutes, else a stated sample of the layers (time scaled)
        budget = 180.0 / (args.steps + args.warmup)
        probe = OracleStep(wl, layers=1)
        probe.run()
        tp, ts = probe.run()
        del probe
        layers = wl.num_layers
        if tp + ts * wl.num_layers > budget:
            layers = max(1, int((budget - tp) / max(ts, 1e-9)))
        os_ = OracleStep(wl, layers=layers)
        for _ in range(args.warmup):
            os_.run()
        t = time.perf_counter()
        steps_s = []
        for _ in range(args.steps):
            steps_s.append(os_.step_seconds(*os_.run()))
        wall = time.perf_counter() - t
        per = sum(steps_s) / len(steps_s)
        value = wl.total_tokens / per
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "int32/u8", "data": "synthetic", "impl": "reference",
                "config": workload_config(wl, world),
                "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                                 "sample": os_.sample_text(), "host": host_info()},
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0},
                "wall_s": wall}
        print(json.dumps(line), flush=True)
        return

    import torch

    import paged_kv_prep_gb300 as pkv
    from paged_kv_prep_gb300 import build as pbuild

    pbuild.build()
    torch.cuda.set_device(local)
    barrier = (lambda: dist.barrier()) if dist else (lambda: None)

    ds = DeviceStep(wl, torch, pkv, workloads, multi_layer=not args.per_layer_calls)
    clocks = ClockSampler(local)
    clocks.start()
    nvml = NvmlSampler(torch, local)
    nvml.start()
    total_ms, prep, store, (t0, t1) = time_device(ds, args.steps, args.warmup, torch, barrier)
    nvml.stop()
    total_ms = max_over_ranks(total_ms, dist)
    ms_per_step = total_ms / args.steps
    value = whole_job_value(world, ds.T, args.steps, total_ms)
    err = ds.st.get_error()
    if err:
        raise RuntimeError(f"device error word set during the run: {err}")

    peak, peak_kind = measured_peaks()
    kv_launch_bytes = kv_bytes_per_layer_group(wl) * wl.num_layers * len(wl.groups)
    store_ms = statistics.mean(store)
    prep_ms = statistics.mean(prep)
    kv_gbs = kv_launch_bytes / (store_ms / 1e3) / 1e9
    prep_gbs = prepare_bytes(wl) / (prep_ms / 1e3) / 1e9
    units = wl.num_layers * len(wl.groups) * ds.T
    # the committed figure is for the one-launch store; per-layer calls have none
    traffic = committed_traffic(units) if not args.per_layer_calls else None
    roofline = {"bound": "hbm", "achieved": round(kv_gbs, 1), "peak": peak, "unit": "GB/s",
                "frac": round(kv_gbs / peak, 4), "traffic": traffic,
                "kernel": "kv_write_kernel (every layer and group of a step in one launch)"
                if not args.per_layer_calls else "kv_write_kernel (one launch per layer)",
                "algorithmic_bytes_per_step": kv_launch_bytes,
                "launches_per_step": ds.launches_per_step() - 1,
                "peak_source": f"{peak_kind} hbm_gbs (copy, burst)"}
    prep_roof = {"bound": "hbm", "achieved": round(prep_gbs, 1), "peak": peak, "unit": "GB/s",
                 "frac": round(prep_gbs / peak, 4), "avg_us": round(prep_ms * 1e3, 2),
                 "algorithmic_bytes_per_launch": prepare_bytes(wl)}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int32/u8", "data": "synthetic",
            "config": workload_config(wl, world),
            "roofline": roofline,
            "kernels": {"prepare_batch": prep_roof,
                        "kv_store_avg_us": round(store_ms * 1e3, 2)},
            "gpu_launches": ds.launches_per_step() * args.steps,
            "clocks": None}

    # the same step without events between its kernels (the timed region
    # above records three per step, which also stop PDL's launch overlap)
    k_p = max(10, min(300, args.steps))
    p_ms = max_over_ranks(time_steps(ds, k_p, args.warmup, torch, barrier), dist)
    step_plain = {"value": whole_job_value(world, ds.T, k_p, p_ms), "ms_per_step": p_ms / k_p,
                  "steps": k_p}

    # variant: only the live block-table entries gathered (PKV_LIVE_TABLES)
    ds.prep_call = ds.prep_call_live
    k_v = max(10, min(300, args.steps))
    v_ms, v_prep, v_store, _ = time_device(ds, k_v, args.warmup, torch, barrier)
    v_ms = max_over_ranks(v_ms, dist)
    ds.prep_call = ds.prep_call_full
    v_prep_us = statistics.mean(v_prep) * 1e3
    line["variants"] = {"no_kernel_events": step_plain, "live_tables": {
        "value": whole_job_value(world, ds.T, k_v, v_ms), "ms_per_step": v_ms / k_v, "steps": k_v,
        "prepare_us": round(v_prep_us, 2),
        "prepare_algorithmic_bytes": prepare_bytes_live(wl),
        "prepare_frac": round(prepare_bytes_live(wl) / (v_prep_us * 1e-6) / 1e9 / peak, 4)}}

    # variant: live tables plus the paged (CSR) table of group 0 (pkv_kv_indices)
    ds.prep_call = ds.prep_call_live
    ds.paged = True
    v_ms, _, _, _ = time_device(ds, k_v, args.warmup, torch, barrier)
    v_ms = max_over_ranks(v_ms, dist)
    ds.paged = False
    ds.prep_call = ds.prep_call_full
    p_us = statistics.mean(ds.paged_ms) * 1e3
    pb = paged_bytes(wl, 0)
    line["variants"]["paged_tables"] = {
        "value": whole_job_value(world, ds.T, k_v, v_ms), "ms_per_step": v_ms / k_v, "steps": k_v,
        "kv_indices_us": round(p_us, 2), "entries": paged_entries(wl, 0),
        "algorithmic_bytes": pb, "frac": round(pb / (p_us * 1e-6) / 1e9 / peak, 4)}
    err = ds.st.get_error()
    if err:
        raise RuntimeError(f"device error word set during the paged-table variant: {err}")

    # clocks: nvidia-smi samples every 50 ms, and K steps of the large step
    # last well under that, so the sampled window is the timed steps plus the
    # device-resident measurements of the same workload right after them
    t_dev_end = time.time()
    clocks.stop()
    smi = clocks.summary(t0, t_dev_end)
    smi["window"] = (f"{t_dev_end - t0:.2f} s from the start of the timed steps "
                     "through the no-event, live-table and paged-table runs")
    inside = nvml.summary(t0, t1)
    if inside is not None:
        # the timed steps themselves, every 2 ms; a reason seen by either
        # sampler is reported
        inside["window"] = f"the {t1 - t0:.3f} s of the timed steps (NVML, every 2 ms)"
        inside["reasons"] = sorted(set(inside["reasons"]) | set(
            r for r in smi["reasons"] if r != "no samples"))
        inside["nvidia_smi"] = smi
        line["clocks"] = inside
    else:
        line["clocks"] = smi
    if not args.no_e2e:
        k_e2e = max(3, min(20, args.steps))
        res, h2d, d2h, dev_s = time_e2e(wl, ds, k_e2e, 3, torch)
        dev_ms = max_over_ranks(dev_s * 1e3, dist)
        res = {k: max_over_ranks(v * 1e3, dist) / 1e3 for k, v in sorted(res.items())}
        best = min(res, key=res.get)
        el = res[best]
        line["e2e"] = {"value": whole_job_value(world, ds.T, k_e2e, el * 1e3), "unit": UNIT,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": el / k_e2e * 1e3, "steps": k_e2e, "path": best,
                       "ms_per_step_by_path": {k: round(v / k_e2e * 1e3, 3)
                                               for k, v in res.items()},
                       "kv_on_device": {
                           "value": whole_job_value(world, ds.T, k_e2e, dev_ms), "unit": UNIT,
                           "ms_per_step": dev_ms / k_e2e,
                           "h2d_bytes_per_step": 8 * ds.n, "d2h_bytes_per_step": d2h,
                           "what": "host schedule and read-back through the API, K/V already "
                                   "in device memory (not end to end: no K/V copies)"}}
    ds.st.close()
    del ds
    torch.cuda.empty_cache()

    if not args.no_latency and rank == 0:
        line["small_batch_latency"] = latency_small(torch, pkv, workloads)
        line["medium_configs"] = other_configs(torch, pkv, workloads)
        line["scheduler_apply_wall_us"] = apply_latency(torch, pkv, workloads)
        line["prefix_cache"] = prefix_cache_bench(torch, pkv, workloads)
        line["allocate_slots"] = allocate_bench(torch, pkv, workloads)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
