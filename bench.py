#!/usr/bin/env python3
"""Benchmark of the GB300 KV-cache write path.

One step = one call of the write path over one batch of the workload (the
batch's K rows and V rows scattered into the caches at its slot indices).
Default workload (the headline): the strided copy, the largest single-GPU
configuration -- fp16 K and V as column views of a fused QKV tensor
[65536, 6144] (token stride 12,288 B), int32 slots into a 2,097,152-slot
cache, 537 MB moved per call.  Other workloads with ``--workload``.

Protocol (``--impl ours``):
  * inputs already in HBM; every step uses the next batch of a pool of
    distinct batches (K/V rows and slot sets) whose total size exceeds 4x the
    L2 cache, or one batch larger than twice the L2, so consecutive steps
    never hit L2 for their inputs;
  * the steps run back to back from CUDA graphs of recorded calls;
  * W warm-up steps and one untimed replay that uploads the timed graphs,
    then exactly K timed steps bracketed by barrier + synchronise; a short
    device-side delay before the opening CUDA event keeps the host's
    submission out of the bracket; events on the launching stream; max over
    ranks;
  * clocks sampled with nvidia-smi during the timed region;
  * ``per_config``: every configuration (and, with ``--suite all``, the
    further rows) timed the same way, with the command's K and W, plus the
    same calls over a region of at least ``--long-ms``;
  * ``e2e``: the same steps with each step's inputs coming from pinned host
    memory and the step's status read back into host memory, inside the
    timed region;
  * ``cpu_baseline``: the CPU oracle on a bounded sample of the same
    workload, on one thread and on all host threads (rank 0, N=1 only).

``--impl reference`` times the CPU oracle as the reference arm on the same
metric and configuration and prints its own JSON line.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KV write tokens/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
L2_BYTES = 129 * 1000 * 1000
FALLBACK_HBM_GBS = 6800.0

DESCRIPTIONS = {
    "tiny": "tiny copy: T=16, H_kv=2, D=64 bf16, cache 256 slots, int32 indices",
    "decode": "decode copy: T=256, H_kv=8, D=128 bf16 (2048 B rows), cache 1,048,576 slots, "
              "int64 distinct random slots",
    "prefill": "prefill copy: T=32768, H_kv=8, D=128 bf16, page_size 64, 512 whole pages in "
               "random order, cache 4,194,304 slots, int32",
    "fp8": "fused FP8 write: T=8192, H_kv=8, D=128 bf16 4*N(0,1) with 0.1% outliers, "
           "inv_scale=448/amax (use_scale=1), e4m3fn cache 1,048,576 slots, page_size 32, int64",
    "fp8_noscale": "fused FP8 write as fp8 with use_scale=0",
    "fp8_dynamic": "dynamic FP8 write: the fp8 batch with per-(token, head) scales computed in "
                   "the kernel (amax/448 per head, stored per slot as fp32), e4m3fn cache "
                   "1,048,576 slots, page_size 32, int64",
    "fp8_dynamic_token": "dynamic FP8 write as fp8_dynamic with one scale per token row "
                         "(amax over the 1024 elements of the K or V row)",
    "fp8_e5m2": "FP8 write into an e5m2 cache: the fp8 batch, per-tensor inv_scale=57344/amax, "
                "kv_store_fp8_ex",
    "fp8_page": "FP8 write with per-page scales: the fp8 batch, one fp32 inverse scale per "
                "32-slot page (32,768 pages, inv_k * 2^-3..2^0), kv_store_fp8_ex",
    "paged": "paged copy: the prefill batch into 4-D pages [65536, 64, 8, 128] padded by one "
             "slot per page (page stride 133,120 B), int32",
    "strided": "strided copy: fp16 K/V views into QKV [65536, 6144] (token stride 12,288 B), "
               "cache 2,097,152 slots, int32",
    "odd": "odd-size copy: fp16 H_kv=1, D=576 (1152 B rows), 1280 B slot stride, "
           "cache 2,097,152 slots, int32",
    "gather_prefill": "gather (inverse of prefill): T=32768 rows (512 whole pages) of H_kv=8, "
                      "D=128 bf16 from a 4,194,304-slot cache, int32",
    "gather_decode": "gather (inverse of decode): T=256 rows of H_kv=8, D=128 bf16 from a "
                     "1,048,576-slot cache, int64",
    "gather_fp8": "dequantising gather (inverse of fp8): T=8192 e4m3fn rows x (1/inv) -> bf16, "
                  "1,048,576-slot cache, page_size 32, int64",
    "absmax": "per-tensor scale pass: max |x| of the fp8 batch's K and V (8192 x 8 x 128 bf16 "
              "each) and inv = 448/amax on the device",
    "fp8_tensor_dynamic": "fused dynamic per-tensor FP8 write: the fp8 batch, amax of K and of V "
                          "over the batch, inv = 448/amax and the e4m3fn write in one call "
                          "(kv_store_fp8_dynamic_tensor, two launches)",
}

DEFAULT_STEPS = {"tiny": 200000, "decode": 200000, "prefill": 10000, "fp8": 50000,
                 "fp8_noscale": 50000, "strided": 5000, "odd": 10000, "gather_decode": 200000,
                 "gather_fp8": 50000, "absmax": 50000, "fp8_dynamic": 50000, "paged": 10000,
                 "fp8_dynamic_token": 50000, "fp8_e5m2": 50000, "fp8_page": 50000,
                 "gather_prefill": 10000, "fp8_tensor_dynamic": 50000}


# ---------------------------------------------------------------------------
# Distributed plumbing (one process per GPU; weak scaling, no data exchange)
# ---------------------------------------------------------------------------

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend):
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float, device=None) -> float:
        if self.pg is None:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# Peaks, clocks
# ---------------------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs: STREAM-style copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (no measured peak file)"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str, period_ms: int = 50):
        self.cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-i", str(gpu_index), "-lms", str(period_ms)]
        self.proc = None
        self.lines = []
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def mark(self):
        self.marks.append(time.monotonic())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        return self.summary()

    def summary(self):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(t=ts, sm=float(parts[1]), smax=float(parts[2]),
                                 reasons=parts[4], hw=parts[5], hwt=parts[6], swt=parts[7],
                                 pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        t0, t1 = (self.marks[0], self.marks[-1]) if len(self.marks) >= 2 else (0, 1e30)
        inside = [r for r in rows if t0 - 0.06 <= r["t"] <= t1 + 0.06] or rows
        reasons = set()
        for r in inside:
            if r["hw"] == "Active":
                reasons.add("hw_slowdown")
            if r["hwt"] == "Active":
                reasons.add("hw_thermal_slowdown")
            if r["swt"] == "Active":
                reasons.add("sw_thermal_slowdown")
            if r["pcap"] == "Active":
                reasons.add("sw_power_cap")
        return {"sm_mhz": statistics.median(r["sm"] for r in inside),
                "sm_max_mhz": max(r["smax"] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


# ---------------------------------------------------------------------------
# Workload pools on the device
# ---------------------------------------------------------------------------

class Pool:
    """Device-resident batches of one workload plus the caches they write.

    Batch 0 is the workload's own seeded data; further batches (used to keep
    consecutive steps out of L2) hold N(0,1) rows drawn on the device and
    fresh slot sets with the same structure (distinct random slots, or whole
    random pages for the prefill workload).
    """

    def __init__(self, name: str, device, pool_bytes: int, seed: int = 1234, n_slots=None):
        import torch
        self.name = name
        w = load_workload(name, n_slots)
        self.w = w
        self.dev = device
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        T, H, D = w.T, w.H, w.D
        src_dtype = torch.bfloat16 if w.src_dtype == "bf16" else torch.float16
        self.src_dtype = src_dtype
        idx_dtype = torch.int64 if w.indices.dtype == np.int64 else torch.int32
        self.in_bytes_per_batch = 2 * w.row_bytes * T + w.indices.itemsize * T
        shared = bool(w.notes.get("shared_source"))
        src_batch_bytes = w.k.nbytes if shared else 2 * w.k.nbytes
        nb = max(1, min(256, -(-pool_bytes // max(1, src_batch_bytes))))
        if src_batch_bytes >= 2 * L2_BYTES:
            nb = 1
        self.num_batches = nb
        self.k, self.v, self.idx = [], [], []
        host_k = torch.from_numpy(w.k.view(np.int16)).to(device).view(src_dtype)
        host_v = host_k if shared else torch.from_numpy(w.v.view(np.int16)).to(device).view(src_dtype)
        for b in range(nb):
            if b == 0:
                kb, vb = host_k, host_v
                ib = torch.from_numpy(w.indices).to(device)
            else:
                kb = torch.randn(host_k.shape, generator=g, device=device).to(src_dtype)
                vb = kb if shared else torch.randn(host_v.shape, generator=g, device=device).to(src_dtype)
                ib = self._slots(g, idx_dtype)
            self.k.append(kb)
            self.v.append(vb)
            self.idx.append(ib)
        # caches (for the gather workloads: seeded random content to read back)
        if w.kind == "gather":
            words = w.cache_bytes // 2
            self.kc = torch.randint(-32768, 32767, (words,), generator=g, dtype=torch.int16,
                                    device=device)
            self.vc = torch.randint(-32768, 32767, (words,), generator=g, dtype=torch.int16,
                                    device=device)
        elif w.kind == "gather_fp8":
            nbytes = w.cache_bytes
            self.kc = torch.randint(0, 256, (nbytes,), generator=g, dtype=torch.uint8, device=device)
            self.vc = torch.randint(0, 256, (nbytes,), generator=g, dtype=torch.uint8, device=device)
        elif w.kind == "absmax":
            self.kc = torch.zeros(1, dtype=torch.uint8, device=device)
            self.vc = torch.zeros(1, dtype=torch.uint8, device=device)
        elif w.kind == "copy":
            words = w.cache_bytes // 2
            self.kc = torch.full((words,), w.sentinel, dtype=torch.int16, device=device)
            self.vc = torch.full((words,), w.sentinel, dtype=torch.int16, device=device)
        else:
            nbytes = w.cache_bytes
            self.kc = torch.full((nbytes,), w.sentinel, dtype=torch.uint8, device=device)
            self.vc = torch.full((nbytes,), w.sentinel, dtype=torch.uint8, device=device)
        if w.kind == "fp8_dyn":       # per-slot fp32 scale caches (per head or per row)
            self.groups = w.H if w.notes.get("scale_mode", "token_head") == "token_head" else 1
            self.ks = torch.full((w.n_slots * self.groups,), -1.0, dtype=torch.float32,
                                 device=device)
            self.vs = torch.full_like(self.ks, -1.0)
        if w.notes.get("scale_mode") == "page":     # one inverse scale per cache page
            self.page_inv = [torch.from_numpy(w.notes["page_inv_k"]).to(device),
                             torch.from_numpy(w.notes["page_inv_v"]).to(device)]
        self.inv = torch.tensor([w.inv_k, w.inv_v], dtype=torch.float32, device=device)
        self.scale = torch.ones(2, dtype=torch.float32, device=device) / self.inv
        self.amax_inv = torch.zeros(4, dtype=torch.float32, device=device)
        self.absmax_work = torch.zeros(4, dtype=torch.int32, device=device)
        self.dyn_work = torch.zeros(3, dtype=torch.int64, device=device)   # fused dynamic write
        self.dyn_scale = torch.zeros(2, dtype=torch.float32, device=device)
        self.err = torch.zeros(2, dtype=torch.int64, device=device)
        self.i64 = idx_dtype == torch.int64
        # kernels one call launches: kv_absmax_inv with a workspace reduces and
        # finishes; the fused dynamic write reduces and writes
        dyn = w.notes.get("scale_mode") == "tensor_dynamic"
        self.launches_per_call = 2 if w.kind == "absmax" or dyn else 1

    def _slots(self, g, idx_dtype):
        import torch
        w = self.w
        if w.notes.get("whole_pages"):
            ps = w.page_size
            pages = torch.randperm(w.n_slots // ps, generator=g, device=self.dev)[: w.T // ps]
            s = (pages[:, None] * ps + torch.arange(ps, device=self.dev)[None, :]).reshape(-1)
        else:
            s = torch.randperm(w.n_slots, generator=g, device=self.dev)[: w.T]
        return s.to(idx_dtype)

    def algorithmic_bytes(self) -> int:
        return self.w.algorithmic_bytes()

    def views(self, b):
        """Device addresses and byte strides of batch b (source views inside QKV)."""
        w = self.w
        e = 2
        kbase = self.k[b].data_ptr() + w.k_view[0]
        vbase = self.v[b].data_ptr() + w.v_view[0]
        strides = (w.k_view[1], w.k_view[2], w.k_view[3], w.v_view[1], w.v_view[2], w.v_view[3],
                   w.slot_stride, w.cache_head_stride, w.cache_elem,
                   w.slot_stride, w.cache_head_stride, w.cache_elem)
        return kbase, vbase, strides

    def call(self, b, stream_handle, k_ptr=None, v_ptr=None, idx_ptr=None) -> int:
        import fp8_quant_gb300 as kv
        w = self.w
        kbase, vbase, strides = self.views(b)
        k_ptr = kbase if k_ptr is None else k_ptr
        v_ptr = vbase if v_ptr is None else v_ptr
        idx_ptr = self.idx[b].data_ptr() if idx_ptr is None else idx_ptr
        idt = 1 if self.i64 else 0
        if w.kind == "copy" and w.paged:
            return kv.raw.kv_store_paged(k_ptr, v_ptr, self.kc.data_ptr(), self.vc.data_ptr(),
                                         idx_ptr, idt, 1, w.T, w.H, w.D, 2, strides, w.page_size,
                                         w.page_stride, w.page_stride, w.n_slots, w.num_split,
                                         self.err.data_ptr(), stream_handle)
        if w.kind == "copy":
            return kv.raw.kv_store(k_ptr, v_ptr, self.kc.data_ptr(), self.vc.data_ptr(), idx_ptr,
                                   idt, 1, w.T, w.H, w.D, 2, strides, w.n_slots, w.num_split,
                                   self.err.data_ptr(), stream_handle)
        if w.kind == "fp8_dyn":
            return kv.raw.kv_store_fp8_ex(k_ptr, v_ptr, self.kc.data_ptr(), self.vc.data_ptr(),
                                          idx_ptr, idt, 1, w.T, w.H, w.D,
                                          1 if w.src_dtype == "bf16" else 0, strides, w.page_size,
                                          w.page_stride, w.page_stride, w.n_slots, 0,
                                          3 if self.groups > 1 else 2, None, None,
                                          self.ks.data_ptr(), self.vs.data_ptr(), self.groups,
                                          self.err.data_ptr(), stream_handle)
        if w.notes.get("scale_mode") == "tensor_dynamic":
            return kv.raw.kv_store_fp8_dynamic_tensor(
                k_ptr, v_ptr, self.kc.data_ptr(), self.vc.data_ptr(), idx_ptr, idt, 1, w.T, w.H,
                w.D, 1 if w.src_dtype == "bf16" else 0, strides, w.page_size, w.page_stride,
                w.page_stride, w.n_slots, 0, self.dyn_scale.data_ptr(),
                self.dyn_scale.data_ptr() + 4, self.dyn_work.data_ptr(), self.err.data_ptr(),
                stream_handle)
        if w.notes.get("scale_mode") == "page":
            return kv.raw.kv_store_fp8_ex(k_ptr, v_ptr, self.kc.data_ptr(), self.vc.data_ptr(),
                                          idx_ptr, idt, 1, w.T, w.H, w.D,
                                          1 if w.src_dtype == "bf16" else 0, strides, w.page_size,
                                          w.page_stride, w.page_stride, w.n_slots, 0, 4,
                                          self.page_inv[0].data_ptr(), self.page_inv[1].data_ptr(),
                                          None, None, 0, self.err.data_ptr(), stream_handle)
        if w.notes.get("fmt") == "e5m2":
            return kv.raw.kv_store_fp8_ex(k_ptr, v_ptr, self.kc.data_ptr(), self.vc.data_ptr(),
                                          idx_ptr, idt, 1, w.T, w.H, w.D,
                                          1 if w.src_dtype == "bf16" else 0, strides, w.page_size,
                                          w.page_stride, w.page_stride, w.n_slots, 1, 1,
                                          self.inv.data_ptr(), self.inv.data_ptr() + 4, None,
                                          None, 1, self.err.data_ptr(), stream_handle)
        if w.kind == "absmax":
            return kv.raw.kv_absmax_inv(k_ptr, v_ptr, 1 if w.src_dtype == "bf16" else 0, w.T, w.H,
                                        w.D, strides, 448.0, self.amax_inv.data_ptr(),
                                        self.amax_inv.data_ptr() + 8,
                                        self.absmax_work.data_ptr(), stream_handle)
        if w.kind == "gather":
            return kv.raw.kv_gather(self.kc.data_ptr(), self.vc.data_ptr(), k_ptr, v_ptr, idx_ptr,
                                    idt, 1, w.T, w.H, w.D, 2, strides, w.n_slots,
                                    self.err.data_ptr(), stream_handle)
        if w.kind == "gather_fp8":
            return kv.raw.kv_gather_fp8(self.kc.data_ptr(), self.vc.data_ptr(), k_ptr, v_ptr,
                                        idx_ptr, idt, 1, w.T, w.H, w.D,
                                        1 if w.src_dtype == "bf16" else 0, strides, w.page_size,
                                        w.page_stride, w.page_stride, w.n_slots,
                                        self.scale.data_ptr(), self.scale.data_ptr() + 4, 1,
                                        self.err.data_ptr(), stream_handle)
        return kv.raw.kv_store_fp8(k_ptr, v_ptr, self.kc.data_ptr(), self.vc.data_ptr(), idx_ptr,
                                   idt, 1, w.T, w.H, w.D, 1 if w.src_dtype == "bf16" else 0,
                                   strides, w.page_size, w.page_stride, w.page_stride, w.n_slots,
                                   self.inv.data_ptr() if w.use_scale else None,
                                   self.inv.data_ptr() + 4 if w.use_scale else None,
                                   w.use_scale, self.err.data_ptr(), stream_handle)


def capture_graphs(torch, fn_step, steps: int, chunk: int):
    """CUDA graphs that run `steps` steps: (graph, steps_in_graph) list."""
    graphs = []
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    done = 0
    sizes = []
    full, rem = divmod(steps, chunk)
    if full:
        sizes.append((chunk, full))
    if rem:
        sizes.append((rem, 1))
    step_ctr = [0]
    for size, reps in sizes:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(size):
                fn_step(step_ctr[0])
                step_ctr[0] += 1
        graphs.append((g, size, reps))
        done += size * reps
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return graphs


def run_graphs(graphs):
    for g, _, reps in graphs:
        for _ in range(reps):
            g.replay()


# Device-side delay enqueued before the opening event of a timed region, in
# GPU clock cycles (about 0.1 ms): the host submits the region's work while
# the GPU is still busy with it, so the events bracket device time only and
# not the host's submission latency.
_HOLD_CYCLES = 200_000


def time_region(torch, dist, fn, device):
    """Device time of fn()'s work on the current stream, in ms (max over ranks)."""
    dist.barrier()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(_HOLD_CYCLES)
    e0.record(st)
    fn()
    e1.record(st)
    torch.cuda.synchronize()
    dist.barrier()
    ms = e0.elapsed_time(e1)
    return dist.max(ms, device=device)


def measure_calls(torch, dist, device, step, steps, warmup, chunk, long_ms=0.0):
    """Per-call device time of `step` (one call of the path) run back to back
    from CUDA graphs: `warmup` untimed calls, one untimed replay that uploads
    the timed graphs, then exactly `steps` timed calls.  With long_ms > 0 the
    same calls are also timed over a region of at least long_ms (graphs of up
    to `chunk` calls replayed), which resolves calls of a microsecond or two
    better than a short region can."""
    graphs = capture_graphs(torch, step, steps, min(steps, chunk))
    warm = capture_graphs(torch, step, warmup, min(warmup, chunk))
    run_graphs(warm)
    run_graphs(graphs)
    torch.cuda.synchronize()
    del warm
    ms = time_region(torch, dist, lambda: run_graphs(graphs), device)
    out = {"us_per_call": ms * 1e3 / steps, "calls": steps}
    del graphs
    if long_ms > 0:
        per_ms = max(ms / steps, 1e-6)
        want = max(steps, int(math.ceil(long_ms / per_ms)))
        size = min(want, chunk)
        reps = -(-want // size)
        lg = capture_graphs(torch, step, size, size)
        run_graphs(lg)
        torch.cuda.synchronize()
        g = lg[0][0]

        def replay():
            for _ in range(reps):
                g.replay()

        ms_l = time_region(torch, dist, replay, device)
        out["us_per_call_long"] = ms_l * 1e3 / (reps * size)
        out["calls_long"] = reps * size
        del lg
    return out


def single_call_cold_us(torch, pool, stream_handle, reps=30):
    """Median device time of one call with L2 flushed before it (informational).

    A short device-side delay after the flush keeps the GPU busy while the
    host submits the call, so the events bracket device time only, not the
    host's submission latency."""
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=pool.dev)
    times = []
    st = torch.cuda.current_stream()
    for r in range(reps):
        flush.fill_(float(r))
        torch.cuda._sleep(_HOLD_CYCLES)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        rc = pool.call(r % pool.num_batches, stream_handle)
        e1.record(st)
        assert rc == 0
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3)
    del flush
    return statistics.median(times)


# ---------------------------------------------------------------------------
# CPU oracle timing
# ---------------------------------------------------------------------------

def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


_ORACLE_CACHE = {}


def oracle_buffers(name, w):
    """Host caches (full size; only written pages are ever touched), the
    source rows and the strides of workload `name` for the CPU oracle."""
    import oracle
    if name not in _ORACLE_CACHE:
        cache_bytes = 1 if w.kind == "absmax" else w.cache_bytes
        if w.kind == "fp8_dyn":
            _ORACLE_CACHE[name + "/scales"] = (np.empty(w.n_slots * w.H, dtype=np.float32),
                                               np.empty(w.n_slots * w.H, dtype=np.float32))
        k = np.ascontiguousarray(w.k).view(np.uint8).reshape(-1).copy()
        v = k if w.notes.get("shared_source") else \
            np.ascontiguousarray(w.v).view(np.uint8).reshape(-1).copy()
        _ORACLE_CACHE[name] = (np.empty(cache_bytes, dtype=np.uint8),
                               np.empty(cache_bytes, dtype=np.uint8), k, v,
                               oracle.Strides(k_token=w.k_view[1], k_head=w.k_view[2],
                                              k_dim=w.k_view[3], v_token=w.v_view[1],
                                              v_head=w.v_view[2], v_dim=w.v_view[3],
                                              kc_slot=w.slot_stride, kc_head=w.cache_head_stride,
                                              kc_dim=w.cache_elem, vc_slot=w.slot_stride,
                                              vc_head=w.cache_head_stride, vc_dim=w.cache_elem))
    return _ORACLE_CACHE[name]


def oracle_job(name, w):
    """The oracle's write loop for workload `name` as a job that runs on POSIX
    threads over token ranges (kinds whose oracle call takes a token range:
    the flat and paged copies and the per-tensor FP8 write), else None."""
    import oracle
    if w.kind not in ("copy", "fp8") or "fmt" in w.notes or "scale_mode" in w.notes:
        return None
    kc, vc, k, v, st = oracle_buffers(name, w)
    if w.kind == "copy":
        return oracle.ThreadedJob("copy_paged" if w.paged else "copy", k, v, kc, vc, w.indices,
                                  st, w.H, w.D, w.n_slots, elem_bytes=2, page_size=w.page_size,
                                  kc_page_stride=w.page_stride, vc_page_stride=w.page_stride,
                                  k_off=w.k_view[0], v_off=w.v_view[0])
    return oracle.ThreadedJob("fp8", k, v, kc, vc, w.indices, st, w.H, w.D, w.n_slots,
                              src_dtype=w.src_dtype, page_size=w.page_size,
                              kc_page_stride=w.page_stride, vc_page_stride=w.page_stride,
                              inv_k=w.inv_k, inv_v=w.inv_v, use_scale=w.use_scale,
                              k_off=w.k_view[0], v_off=w.v_view[0])


def oracle_tokens_per_s(name: str, seconds: float, threads: int = 1):
    """Time the CPU oracle (as it stands) on a bounded sample of the workload:
    its batch, repeated for about `seconds`.  Kinds with a token-range oracle
    call run on `threads` POSIX threads, thread i repeating its own token
    range of the batch (no interpreter lock, no hand-off between threads);
    the others run on one thread.  Returns (tokens/s, sample, threads used)."""
    w = load_workload(name)
    job = oracle_job(name, w)
    if job is not None:
        used = max(1, min(threads, w.T))
        job.run(used)                        # first touch of the written pages
        done, el, _ = job.run(used, seconds, 3)
        sample = (f"{done} tokens: {used} POSIX thread{'s' if used > 1 else ''}, each "
                  f"repeating its own token range of the workload's batch of {w.T} tokens for "
                  f"{el:.1f} s (full-size host caches)")
        return done / el, sample, used
    oracle_step(name, w, w.T)                # loads the oracle and touches the written pages
    n = 0
    t0 = time.perf_counter()
    while True:
        oracle_step(name, w, w.T)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds and n >= 3:
            break
    sample = (f"{n} repetitions of the workload's batch of {w.T} tokens ({el:.1f} s, one "
              f"thread, full-size host caches)")
    return n * w.T / el, sample, 1


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def pool_batches(w, pool_bytes: int) -> int:
    """Distinct input batches a Pool of `pool_bytes` rotates through (one when
    a single batch already exceeds twice the L2)."""
    shared = bool(w.notes.get("shared_source"))
    src_batch_bytes = w.k.nbytes if shared else 2 * w.k.nbytes
    if src_batch_bytes >= 2 * L2_BYTES:
        return 1
    return max(1, min(256, -(-pool_bytes // max(1, src_batch_bytes))))


def line_config(name, w, world, pool_bytes, slots=None):
    """The `config` object of the JSON line: what the workload is, identical
    for both arms."""
    nb = pool_batches(w, pool_bytes)
    in_bytes = 2 * w.row_bytes * w.T + w.indices.itemsize * w.T
    return {
        "workload": DESCRIPTIONS[name] + ("" if slots is None
                                          else f" [cache reduced to {slots} slots]"),
        "tokens_per_step": w.T,
        "bytes_per_step": w.algorithmic_bytes(),
        "parallelism": f"replicas x{world}",
        "l2": (f"inputs rotate over {nb} batches ({nb * in_bytes / 1e6:.0f} MB read per cycle) "
               + ("> L2 (129 MB)" if nb * in_bytes > L2_BYTES else
                  "< L2 (129 MB): L2-resident, parity-only size")
               if nb > 1 else
               f"one batch: {in_bytes / 1e6:.0f} MB read and {(w.algorithmic_bytes() - in_bytes) / 1e6:.0f}"
               f" MB written per step, each larger than L2 (129 MB)"),
    }


# ---------------------------------------------------------------------------
# Arms
# ---------------------------------------------------------------------------

def run_reference(args, dist):
    """The CPU oracle as the reference arm (rank 0 only): each step writes the
    workload's batch (or, if that would not fit the time budget, its first
    tokens) through the oracle on all host threads."""
    if dist.rank != 0:
        return
    name = args.workload
    w = load_workload(name)
    threads = host_threads()
    job = oracle_job(name, w)
    if job is not None:
        used = max(1, min(threads, w.T))
        job.run(used)                                # first touch
        t0 = time.perf_counter()
        job.run(used)
        rate = w.T / (time.perf_counter() - t0)
        run = lambda n: job.run(used, 0.0, 1, num_tokens=n)
    else:
        used = 1
        oracle_step(name, w, w.T)
        t0 = time.perf_counter()
        oracle_step(name, w, w.T)
        rate = w.T / (time.perf_counter() - t0)
        run = lambda n: oracle_step(name, w, n)
    per_step_s = 150.0 / max(1, args.steps + args.warmup)
    tokens = max(1, min(w.T, int(rate * per_step_s)))
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        run(tokens)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = args.steps * tokens / total
    config = line_config(name, w, args.gpus, args.pool_mb << 20)
    if tokens < w.T:
        config["tokens_per_step"] = tokens
        config["bytes_per_step"] = w.algorithmic_bytes() * tokens // w.T
    how = ("one thread" if used == 1 else
           f"{used} POSIX threads, one token range each")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype_of(w), "data": "synthetic",
        "config": config,
        "achieved_gbs": value * w.algorithmic_bytes() / w.T / 1e9,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
                         "sample": f"each step: {'the' if tokens == w.T else 'the first'} "
                                   f"{tokens} of the workload's {w.T} tokens through the CPU "
                                   f"oracle, {how} ({cpu_model()})"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def load_workload(name, n_slots=None):
    import workloads as wl
    kw = {} if n_slots is None else {"n_slots": n_slots}
    if name == "fp8_noscale":
        return wl.fp8(use_scale=0, **kw)
    return wl.WORKLOADS[name](**kw)


def oracle_step(name, w, tokens, t_begin=0):
    """Tokens [t_begin, tokens) of the workload through the CPU oracle, from
    this thread."""
    import oracle
    key = name
    oracle_buffers(name, w)
    kc, vc, k, v, st = _ORACLE_CACHE[key]
    if w.kind == "absmax":
        oracle.absmax_inv(k, v, st, tokens, w.H, w.D, w.src_dtype)
    elif w.kind == "gather":
        oracle.gather_copy(kc, vc, k, v, w.indices, st, w.H, w.D, 2, w.n_slots, t_end=tokens)
    elif w.kind == "gather_fp8":
        oracle.gather_fp8(kc, vc, k, v, w.indices, st, w.H, w.D, w.src_dtype, w.page_size,
                          w.page_stride, w.page_stride, w.n_slots, 1.0 / w.inv_k, 1.0 / w.inv_v,
                          1, t_end=tokens)
    elif w.kind == "copy" and w.paged:
        oracle.store_copy_paged(k, v, kc, vc, w.indices, st, w.H, w.D, 2, w.page_size,
                                w.page_stride, w.page_stride, w.n_slots, k_off=w.k_view[0],
                                v_off=w.v_view[0], t_end=tokens)
    elif w.kind == "copy":
        oracle.store_copy(k, v, kc, vc, w.indices, st, w.H, w.D, 2, w.n_slots,
                          k_off=w.k_view[0], v_off=w.v_view[0], t_begin=t_begin, t_end=tokens)
    elif w.kind == "fp8_dyn":
        ks, vs = _ORACLE_CACHE[key + "/scales"]
        mode = w.notes.get("scale_mode", "token_head")
        oracle.store_fp8_ex(k, v, kc, vc, w.indices, st, w.H, w.D, w.src_dtype, w.page_size,
                            w.page_stride, w.page_stride, w.n_slots, fmt="e4m3fn",
                            scale_mode=mode, k_scales=ks, v_scales=vs,
                            scales_slot_stride=w.H if mode == "token_head" else 1, t_end=tokens)
    elif w.notes.get("scale_mode") == "tensor_dynamic":
        _, inv = oracle.absmax_inv(k, v, st, tokens, w.H, w.D, w.src_dtype, 448.0,
                                   k_off=w.k_view[0], v_off=w.v_view[0])
        oracle.store_fp8_ex(k, v, kc, vc, w.indices, st, w.H, w.D, w.src_dtype, w.page_size,
                            w.page_stride, w.page_stride, w.n_slots, fmt="e4m3fn",
                            scale_mode="tensor", inv_k=float(inv[0]), inv_v=float(inv[1]),
                            t_end=tokens)
    elif w.notes.get("scale_mode") == "page":
        oracle.store_fp8_ex(k, v, kc, vc, w.indices, st, w.H, w.D, w.src_dtype, w.page_size,
                            w.page_stride, w.page_stride, w.n_slots, fmt="e4m3fn",
                            scale_mode="page", k_scales=w.notes["page_inv_k"],
                            v_scales=w.notes["page_inv_v"], t_end=tokens)
    elif w.notes.get("fmt") == "e5m2":
        oracle.store_fp8_ex(k, v, kc, vc, w.indices, st, w.H, w.D, w.src_dtype, w.page_size,
                            w.page_stride, w.page_stride, w.n_slots, fmt="e5m2",
                            scale_mode="tensor", inv_k=w.inv_k, inv_v=w.inv_v, t_end=tokens)
    else:
        oracle.store_fp8(k, v, kc, vc, w.indices, st, w.H, w.D, w.src_dtype, w.page_size,
                         w.page_stride, w.page_stride, w.n_slots, w.inv_k, w.inv_v,
                         w.use_scale, t_begin=t_begin, t_end=tokens)


def dtype_of(w):
    if w.kind == "absmax":
        return f"f32 ({w.src_dtype} in)"
    if w.kind in ("fp8", "fp8_dyn"):
        return f"f32 ({w.src_dtype} in, {w.notes.get('fmt', 'e4m3fn')} out)"
    if w.kind == "gather_fp8":
        return f"f32 (e4m3fn in, {w.src_dtype} out)"
    return w.src_dtype


# The configurations the write path is measured on (decode with its row
# splits, prefill, the fused FP8 write with and without the scale, the
# strided QKV views, the odd row size), then the further rows: paged pages,
# e5m2, dynamic scales, the gathers and the per-tensor scale pass.
SUITE_CONFIGS = ("decode", "prefill", "fp8", "fp8_noscale", "strided", "odd")
SUITE_MORE = ("paged", "fp8_e5m2", "fp8_page", "fp8_dynamic", "fp8_dynamic_token", "gather_decode",
              "gather_prefill", "gather_fp8", "absmax", "fp8_tensor_dynamic")
HEADLINE = "strided"


def pool_step(kv, pool):
    """step(i): one call of the path on batch i (mod the pool's batches)."""
    import torch

    def step(i):
        rc = pool.call(i % pool.num_batches, torch.cuda.current_stream().cuda_stream)
        if rc != 0:
            raise RuntimeError(f"launch failed: {kv.kv_status_str(rc)}")
    return step


def fractions(entry, bytes_per_call, tokens, peak):
    """GB/s, tokens/s and roofline fraction of an entry's per-call times."""
    for key, tag in (("us_per_call", ""), ("us_per_call_long", "_long")):
        if key in entry:
            us = entry[key]
            entry["gbs" + tag] = bytes_per_call / (us * 1e-6) / 1e9
            entry["frac" + tag] = entry["gbs" + tag] / peak
            entry["tokens_per_s" + tag] = tokens / (us * 1e-6)
    return entry


def suite_entry(args, dist, torch, kv, device, name, peak, pool=None):
    """Per-call time of workload `name` in the headline's protocol: the
    command's steps and warm-up (else the workload's defaults), plus a long
    region of at least --long-ms; decode adds its row splits and the
    launch floor."""
    own = pool is None
    if own:
        pool = Pool(name, device, pool_bytes=args.pool_mb << 20, seed=1234 + dist.rank)
    steps = args.steps if args.steps_given else DEFAULT_STEPS[name]
    warm = args.warmup if args.warmup_given else max(3, steps // 20)
    w = pool.w
    e = measure_calls(torch, dist, device, pool_step(kv, pool), steps, warm, args.graph_chunk,
                      args.long_ms)
    e["launches_per_call"] = pool.launches_per_call
    fractions(e, pool.algorithmic_bytes(), w.T, peak)
    if name == "decode":
        e["by_num_split"] = {}
        saved = w.num_split
        try:
            for split in (1, 2, 4):
                if split > 1 and w.row_bytes % (split * 128):
                    continue
                w.num_split = split
                sub = measure_calls(torch, dist, device, pool_step(kv, pool), steps, warm,
                                    args.graph_chunk, args.long_ms)
                e["by_num_split"][str(split)] = fractions(sub, pool.algorithmic_bytes(), w.T,
                                                          peak)
        finally:
            w.num_split = saved
        # an empty kernel with the decode launch's shape and hand-over: the
        # per-launch floor under a decode call
        warps = floor_warps(pool)

        def floor_step(i):
            rc = kv.raw.kv_launch_floor(warps, torch.cuda.current_stream().cuda_stream)
            if rc != 0:
                raise RuntimeError(kv.kv_status_str(rc))

        f = measure_calls(torch, dist, device, floor_step, steps, warm, args.graph_chunk,
                          args.long_ms)
        f["warps"] = warps
        e["launch_floor"] = f
    e["single_call_cold_us"] = single_call_cold_us(torch, pool,
                                                   torch.cuda.current_stream().cuda_stream)
    st, nbad, _ = kv.kv_error_poll(pool.err)
    if st != kv.KVStatus.OK:
        raise RuntimeError(f"{nbad} out-of-range slots in the benchmark data")
    if own:
        del pool
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return e


def floor_warps(pool):
    """Warps of work in one call of the pool's copy workload (its launch shape)."""
    w = pool.w
    parts = w.num_split
    if parts == 0:      # the automatic split of the library for these row sizes
        sms = 152
        try:
            import torch
            sms = torch.cuda.get_device_properties(pool.dev).multi_processor_count
        except Exception:
            pass
        parts = 1
        chunks = w.row_bytes // 32
        units = 2 * w.T
        while (units * parts < sms * 16 and chunks % (2 * parts) == 0
               and chunks // (2 * parts) >= 32 and parts < 8):
            parts *= 2
    return 2 * w.T * parts


def run_ours(args, dist):
    import torch
    import fp8_quant_gb300 as kv
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU path)")
    torch.cuda.set_device(dist.local_rank)
    device = torch.device("cuda", dist.local_rank)
    kv.load_library()
    name = args.workload
    peak, peak_src = hbm_peak()
    pool = Pool(name, device, pool_bytes=args.pool_mb << 20, seed=1234 + dist.rank,
                n_slots=args.slots)
    w = pool.w
    T = w.T
    step = pool_step(kv, pool)

    # --- headline: exactly --steps timed calls ------------------------------
    graphs = capture_graphs(torch, step, args.steps, min(args.steps, args.graph_chunk))
    warm_graphs = capture_graphs(torch, step, args.warmup, min(args.warmup, args.graph_chunk))
    run_graphs(warm_graphs)
    del warm_graphs
    run_graphs(graphs)                      # untimed replay: uploads the timed graphs
    torch.cuda.synchronize()

    visible = [x.strip() for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    clocks = ClockSampler(visible[dist.local_rank] if len(visible) > dist.local_rank
                          else str(dist.local_rank))
    clocks.start()
    time.sleep(0.3)
    clocks.mark()
    ms = time_region(torch, dist, lambda: run_graphs(graphs), device)
    clocks.mark()
    clock_summary = clocks.stop()
    del graphs

    st, nbad, _ = kv.kv_error_poll(pool.err)
    if st != kv.KVStatus.OK:
        raise RuntimeError(f"{nbad} out-of-range slots in the benchmark data")

    bytes_per_step = pool.algorithmic_bytes()
    sec_per_step = ms / 1e3 / args.steps
    value = dist.world * T / sec_per_step
    achieved_gbs = bytes_per_step / sec_per_step / 1e9

    # --- the same calls over a long region, and cold single calls ------------
    head = {"us_per_call": ms * 1e3 / args.steps, "calls": args.steps}
    if args.long_ms > 0:
        longer = measure_calls(torch, dist, device, step, args.steps, args.warmup,
                               args.graph_chunk, args.long_ms)
        head["us_per_call_long"] = longer["us_per_call_long"]
        head["calls_long"] = longer["calls_long"]
    head["launches_per_call"] = pool.launches_per_call
    fractions(head, bytes_per_step, T, peak)
    head["single_call_cold_us"] = single_call_cold_us(torch, pool,
                                                      torch.cuda.current_stream().cuda_stream)

    # --- end to end: pinned host inputs, result back to the host ------------
    e2e = run_e2e(args, dist, torch, kv, pool, device)

    # --- every configuration in the same protocol ----------------------------
    per_config = {}
    if args.suite != "none" and args.slots is None:
        names = SUITE_CONFIGS + (SUITE_MORE if args.suite == "all" else ())
        del pool
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        pool = None
        for other in names:
            if other == name:
                per_config[other] = head
                continue
            try:
                per_config[other] = suite_entry(args, dist, torch, kv, device, other, peak)
            except Exception as exc:     # recorded, not fatal: the headline stands
                per_config[other] = {"error": f"{type(exc).__name__}: {exc}"}
                torch.cuda.synchronize()
                torch.cuda.empty_cache()

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        rate1, sample1, _ = oracle_tokens_per_s(name, args.cpu_seconds / 2)
        rate, sample, used = oracle_tokens_per_s(name, args.cpu_seconds / 2, host_threads())
        cpu = {"value": rate, "unit": "tokens/s", "cores": used, "kind": "oracle",
               "sample": sample + f"; host CPU: {cpu_model()}",
               "one_thread": {"value": rate1, "sample": sample1}}

    traffic = load_traffic(name)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype_of(w), "data": "synthetic",
        "config": line_config(name, w, dist.world, args.pool_mb << 20, args.slots),
        "timing": {
            "protocol": "CUDA graphs of back-to-back calls; a device-side delay before the "
                        "opening CUDA event so that the events bracket device time only; "
                        "events on the launching stream",
            "upload_replays": 1,
            "headline": head,
        },
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peak, "unit": "GB/s",
                     "frac": achieved_gbs / peak, "traffic": traffic,
                     "peak_source": peak_src,
                     "kernel": "kv_copy_rows" if w.kind == "copy" else w.kind},
        "per_config": per_config,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * (pool.launches_per_call if pool is not None
                                      else head["launches_per_call"]),
        "clocks": clock_summary,
    }
    if dist.rank == 0:
        print(json.dumps(line), flush=True)


# The sources each workload's kernels are compiled from: the shared device and
# host headers plus the translation unit that holds the workload's kernel (the
# public header holds declarations and documentation only).
_COMMON_SOURCES = ("fp8_quant_gb300/csrc/kv_abi.h", "fp8_quant_gb300/csrc/kv_device.cuh",
                   "fp8_quant_gb300/csrc/kv_host.h")


def kernel_source_hash(name: str) -> str:
    """sha256 over the sources of workload `name`'s kernels: what the traffic
    counters in profiles/ were taken with."""
    import hashlib
    unit = ("kv_gather.cu" if name.startswith("gather") else
            "kv_scale.cu" if name == "absmax" else
            "kv_fp8_ex.cu" if name.startswith("fp8_dynamic") else "kvstore.cu")
    files = _COMMON_SOURCES + ("fp8_quant_gb300/csrc/" + unit,)
    h = hashlib.sha256()
    for f in files:
        h.update(f.encode())
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def load_traffic(name):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    workload's kernel sources have changed since those counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            entry = json.load(f)["workloads"][name]
        if not kernel_source_hash(name).startswith(entry["sources_sha256_prefix"]):
            return None
        return entry["bytes"]
    except Exception:
        return None


def run_e2e(args, dist, torch, kv, pool, device):
    """Steps whose inputs come from pinned host memory every time.

    Each batch's K rows, V rows and slot ids sit in one pinned host buffer
    (256-byte aligned segments), so a step is one host->device copy into a
    device staging buffer, the kv_store/kv_store_fp8 call on the staged
    inputs, and a device->host read of the error record."""
    w = pool.w
    nb = pool.num_batches
    if w.kind.startswith("gather"):
        return run_e2e_gather(args, dist, torch, kv, pool, device)
    shared = bool(w.notes.get("shared_source"))
    align = lambda n: (n + 255) // 256 * 256
    kbytes = pool.k[0].numel() * pool.k[0].element_size()
    vbytes = 0 if shared else pool.v[0].numel() * pool.v[0].element_size()
    ibytes = pool.idx[0].numel() * pool.idx[0].element_size()
    off_v = align(kbytes)
    off_i = off_v + align(vbytes)
    total = off_i + ibytes
    hosts = []
    for b in range(nb):
        h = torch.empty(total, dtype=torch.uint8).pin_memory()
        h[:kbytes].copy_(pool.k[b].reshape(-1).view(torch.uint8).cpu())
        if not shared:
            h[off_v:off_v + vbytes].copy_(pool.v[b].reshape(-1).view(torch.uint8).cpu())
        h[off_i:off_i + ibytes].copy_(pool.idx[b].view(torch.uint8).cpu())
        hosts.append(h)
    stage = torch.empty(total, dtype=torch.uint8, device=device)
    err_host = torch.zeros(2, dtype=torch.int64).pin_memory()
    d2h = err_host.numel() * err_host.element_size()
    base = stage.data_ptr()

    def step(i):
        b = i % nb
        stage.copy_(hosts[b], non_blocking=True)
        kbase = base + w.k_view[0]
        vbase = (base if shared else base + off_v) + w.v_view[0]
        rc = pool.call(b, torch.cuda.current_stream().cuda_stream, kbase, vbase, base + off_i)
        if rc != 0:
            raise RuntimeError(kv.kv_status_str(rc))
        err_host.copy_(pool.amax_inv.view(torch.int64) if w.kind == "absmax" else pool.err,
                       non_blocking=True)

    def step_zero_copy(i):
        # the kernel reads the batch straight from pinned host memory over
        # NVLink-C2C: the host -> device transfer happens inside the call
        b = i % nb
        hbase = hosts[b].data_ptr()
        kbase = hbase + w.k_view[0]
        vbase = (hbase if shared else hbase + off_v) + w.v_view[0]
        rc = pool.call(b, torch.cuda.current_stream().cuda_stream, kbase, vbase, hbase + off_i)
        if rc != 0:
            raise RuntimeError(kv.kv_status_str(rc))
        if w.kind == "absmax":
            err_host.copy_(pool.amax_inv.view(torch.int64), non_blocking=True)
        else:   # the record lands in pinned host memory by a chained kernel
            rc = kv.raw.kv_error_snapshot(pool.err.data_ptr(), err_host.data_ptr(),
                                          torch.cuda.current_stream().cuda_stream)
            if rc != 0:
                raise RuntimeError(kv.kv_status_str(rc))

    steps = max(3, min(args.steps, args.e2e_steps))
    out = {}
    for name, fn in (("staged", step), ("zero_copy", step_zero_copy)):
        graphs = capture_graphs(torch, fn, steps, min(steps, args.graph_chunk))
        run_graphs(graphs)
        torch.cuda.synchronize()
        ms = time_region(torch, dist, lambda: run_graphs(graphs), device)
        out[name] = dist.world * w.T / (ms / 1e3 / steps)
        del graphs
    best = max(out, key=out.get)
    # zero-copy moves only what the kernel reads over the link: the K and V
    # rows (not the Q columns of a fused QKV batch) and the slot ids
    h2d = {"staged": total,
           "zero_copy": 2 * w.row_bytes * w.T + (0 if w.kind == "absmax" else ibytes)}
    how = {"staged": "every step: one pinned host -> device copy of the batch (K, V, slot ids "
                     "packed) into a device buffer, the call on the staged inputs, and a "
                     "device -> host read of the error record; back-to-back from CUDA graphs",
           "zero_copy": "every step: the call reads the batch (K, V, slot ids) directly from "
                        "pinned host memory over NVLink-C2C, then kv_error_snapshot writes the "
                        "error record into pinned host memory; back-to-back from CUDA graphs"}
    return {"value": out[best], "unit": "tokens/s", "h2d_bytes_per_step": h2d[best],
            "d2h_bytes_per_step": d2h, "steps": steps, "mode": best, "how": how[best],
            "by_mode": out}


def run_e2e_gather(args, dist, torch, kv, pool, device):
    """Gather steps as a KV offload: the slot ids go host -> device, the
    gathered K and V rows and the error record come back device -> host."""
    w = pool.w
    nb = pool.num_batches
    host_i = [pool.idx[b].cpu().pin_memory() for b in range(nb)]
    di = torch.empty_like(pool.idx[0])
    out_k = torch.empty_like(pool.k[0])
    out_v = torch.empty_like(pool.v[0])
    host_k = torch.empty(out_k.shape, dtype=out_k.dtype).pin_memory()
    host_v = torch.empty(out_v.shape, dtype=out_v.dtype).pin_memory()
    err_host = torch.zeros(2, dtype=torch.int64).pin_memory()
    h2d = host_i[0].numel() * host_i[0].element_size()
    d2h = 2 * out_k.numel() * out_k.element_size() + err_host.numel() * 8

    def step(i):
        b = i % nb
        di.copy_(host_i[b], non_blocking=True)
        rc = pool.call(b, torch.cuda.current_stream().cuda_stream, out_k.data_ptr(),
                       out_v.data_ptr(), di.data_ptr())
        if rc != 0:
            raise RuntimeError(kv.kv_status_str(rc))
        host_k.copy_(out_k, non_blocking=True)
        host_v.copy_(out_v, non_blocking=True)
        err_host.copy_(pool.err, non_blocking=True)

    def step_zero_copy(i):
        # slot ids read from pinned host memory and rows written straight into
        # pinned host memory by the kernel; the record follows by a chained kernel
        b = i % nb
        rc = pool.call(b, torch.cuda.current_stream().cuda_stream, host_k.data_ptr(),
                       host_v.data_ptr(), host_i[b].data_ptr())
        if rc != 0:
            raise RuntimeError(kv.kv_status_str(rc))
        rc = kv.raw.kv_error_snapshot(pool.err.data_ptr(), err_host.data_ptr(),
                                      torch.cuda.current_stream().cuda_stream)
        if rc != 0:
            raise RuntimeError(kv.kv_status_str(rc))

    steps = max(3, min(args.steps, args.e2e_steps))
    out = {}
    for name, fn in (("staged", step), ("zero_copy", step_zero_copy)):
        graphs = capture_graphs(torch, fn, steps, min(steps, args.graph_chunk))
        run_graphs(graphs)
        torch.cuda.synchronize()
        ms = time_region(torch, dist, lambda: run_graphs(graphs), device)
        out[name] = dist.world * w.T / (ms / 1e3 / steps)
        del graphs
    best = max(out, key=out.get)
    how = {"staged": "every step: slot ids pinned host -> device, the gather, and the gathered "
                     "K/V rows plus the error record device -> pinned host by copies; from CUDA "
                     "graphs",
           "zero_copy": "every step: the gather reads the slot ids from pinned host memory and "
                        "writes the K/V rows straight into pinned host memory over NVLink-C2C, "
                        "then kv_error_snapshot writes the error record there; from CUDA graphs"}
    return {"value": out[best], "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "mode": best, "how": how[best],
            "by_mode": out}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(DESCRIPTIONS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--suite", default="all", choices=["all", "configs", "none"],
                    help="after the headline, time every configuration (configs) and the "
                         "further rows (all) in the same protocol")
    ap.add_argument("--long-ms", type=float, default=10.0,
                    help="also time each workload's calls over a region of at least this "
                         "many ms (0: off)")
    ap.add_argument("--pool-mb", type=int, default=512)
    ap.add_argument("--graph-chunk", type=int, default=1000)
    ap.add_argument("--e2e-steps", type=int, default=20000)
    ap.add_argument("--cpu-seconds", type=float, default=20.0,
                    help="CPU oracle timing: half on one thread, half on all host threads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--slots", type=int, default=None,
                    help="override the cache size in slots (small profiler captures; "
                         "no suite)")
    a = ap.parse_args(argv)
    a.steps_given = a.steps is not None
    a.warmup_given = a.warmup is not None
    if a.steps is None:
        a.steps = DEFAULT_STEPS[a.workload] if a.impl == "ours" else 20
    if a.warmup is None:
        a.warmup = max(3, a.steps // 20) if a.impl == "ours" else 3
    if a.warmup < 3:
        ap.error("--warmup must be at least 3")
    if a.steps < 1:
        ap.error("--steps must be positive")
    return a


def main(argv=None):
    args = parse_args(argv)
    dist = Dist()
    if args.impl == "reference":
        if dist.rank == 0:
            run_reference(args, dist)
        return
    import torch
    if torch.cuda.is_available():
        torch.cuda.set_device(dist.local_rank)   # before the process group binds a device
    dist.init("nccl")
    try:
        run_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
